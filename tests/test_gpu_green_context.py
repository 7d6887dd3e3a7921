"""The library on a green context (an SM partition of the device): kernels
launched on a stream of a partition run on its SMs only, and the persistent
grids (GEMM, quantizers) are sized for that partition.  Results must equal
those on an ordinary stream bit for bit.  The partition is made through the
CUDA driver's green-context API (cuDevSmResourceSplitByCount,
cuGreenCtxCreate, cuGreenCtxStreamCreate), loaded with ctypes."""
import ctypes

import pytest
import torch

import int8_mixed_precision_row_gb300 as m
from int8_mixed_precision_row_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


class _DevResource(ctypes.Structure):  # CUdevResource, ABI version 1
    _fields_ = [("type", ctypes.c_int), ("pad", ctypes.c_ubyte * 92), ("sm_count", ctypes.c_uint),
                ("min_partition", ctypes.c_uint), ("alignment", ctypes.c_uint),
                ("rest", ctypes.c_ubyte * 36)]


@pytest.fixture(scope="module")
def partition():
    from int8_mixed_precision_row_gb300 import build
    build.build()
    m.load()
    torch.zeros(1, device=DEV)  # the primary context exists
    try:
        cu = ctypes.CDLL("libcuda.so.1")
    except OSError:
        pytest.skip("libcuda not loadable")
    P = ctypes.c_void_p
    dev = ctypes.c_int()
    assert cu.cuDeviceGet(ctypes.byref(dev), 0) == 0
    whole = _DevResource()
    if cu.cuDeviceGetDevResource(dev, ctypes.byref(whole), 1) != 0:
        pytest.skip("green contexts not supported here")
    part = (_DevResource * 1)()
    n = ctypes.c_uint(1)
    rest = _DevResource()
    assert cu.cuDevSmResourceSplitByCount(part, ctypes.byref(n), ctypes.byref(whole),
                                          ctypes.byref(rest), 0, 64) == 0
    desc, gctx, stream = P(), P(), P()
    assert cu.cuDevResourceGenerateDesc(ctypes.byref(desc), part, 1) == 0
    assert cu.cuGreenCtxCreate(ctypes.byref(gctx), desc, dev, 1) == 0
    assert cu.cuGreenCtxStreamCreate(ctypes.byref(stream), gctx, 1, 0) == 0
    yield torch.cuda.ExternalStream(stream.value), part[0].sm_count, whole.sm_count
    torch.cuda.synchronize()
    cu.cuStreamDestroy_v2(stream)
    cu.cuGreenCtxDestroy(gctx)


def test_gemm_and_quantizers_on_a_partition(partition):
    stream, sms, total = partition
    assert 0 < sms < total
    M, N, K = 2048, 2312, 4096   # 80 pair tiles: more than the partition's pairs
    A = synth.bf16_normal((M, K), 51).to(DEV)
    B = synth.bf16_normal((K, N), 52).to(DEV)
    ws = torch.empty(m.int8mp_mm_workspace_size(), dtype=torch.uint8, device=DEV)

    C = synth.bf16_normal((1024, 2048), 56).to(DEV)   # the one-launch kernels of small operands

    def run(s):
        with torch.cuda.stream(s):
            cm = torch.zeros(K, dtype=torch.float32, device=DEV)
            qa, sa = m.int8mp_quantize_rows_colmax(A, cm, codes=m.INT8MP_CODES_F16)
            qb, sb = m.int8mp_quantize_rowwise(B, axis=m.INT8MP_GROUP_COLS, mode=m.INT8MP_SR,
                                               seed=7, codes=m.INT8MP_CODES_F16)
            out = m.int8mp_scaled_mm(qa, sa, qb, sb, layout=m.INT8MP_AxB, workspace=ws)
            acc = m.int8mp_mm_s32(qa, qb, layout=m.INT8MP_AxB, workspace=ws)
            qr, sr = m.int8mp_quantize_rowwise(C, mode=m.INT8MP_SR, seed=8,
                                               codes=m.INT8MP_CODES_F16)
            qc, sc = m.int8mp_quantize_rowwise(C, axis=m.INT8MP_GROUP_COLS, mode=m.INT8MP_SR,
                                               seed=9, codes=m.INT8MP_CODES_F16)
        s.synchronize()
        return qa, sa, qb, sb, out, acc, cm, qr, sr, qc, sc

    ref = run(torch.cuda.current_stream())
    got = run(stream)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_linear_layer_on_a_partition(partition):
    stream, _, _ = partition
    T, N, K = 4096, 2048, 2048
    X = synth.bf16_normal((T, K), 53).to(DEV)
    W = synth.bf16_normal((N, K), 54, std=0.02).to(DEV)
    dY = synth.bf16_normal((T, N), 55, std=1e-3).to(DEV)
    cfg = m.linear_cfg(mode=m.INT8MP_SR, seed=11)

    def run(s):
        with torch.cuda.stream(s):
            absmax = torch.empty(2 * K, dtype=torch.float32, device=DEV)
            Y = m.int8mp_linear_fwd_save(X, W, absmax, cfg)
            dX, dW = m.int8mp_linear_bwd_saved(dY, X, W, absmax, cfg)
        s.synchronize()
        return Y, dX, dW

    ref = run(torch.cuda.current_stream())
    got = run(stream)
    for a, b in zip(got, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
