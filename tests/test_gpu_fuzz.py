"""Seeded random shapes through every entry point of the C ABI, against the
oracle: quantization by rows, by columns in both code layouts, with column
maxima and from them, two matrices' rows in one launch; the matmul in the
three layouts, int32 and scaled, with and without the split-tail workspace;
the linear layer forward and backward.  Shapes are drawn so that most cases
are ragged (rows, columns and K off the tile sizes) and small enough for the
oracle; every result must match bit for bit."""
import numpy as np
import pytest
import torch

import int8_mixed_precision_row_gb300 as m
import oracle
from helpers import bf16_bits
from int8_mixed_precision_row_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CASES = 40


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_mixed_precision_row_gb300 import build
    build.build()
    m.load()


def _rng(case):
    return np.random.default_rng(1000 + case)


def _input(rows, cols, seed):
    return synth.bf16_normal((rows, cols), seed, outlier_frac=0.01, outlier_scale=20.0)


def _codes_np(q):
    q = q.cpu()
    return q.float().to(torch.int8).numpy() if q.dtype == torch.float16 else q.numpy()


def _f32_bits(t):
    return t.cpu().contiguous().view(torch.int32).numpy()


def _col_absmax_bits(x):
    return x.float().abs().amax(dim=0).contiguous().view(torch.int32).numpy()


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_quantization(case):
    g = _rng(case)
    rows = int(g.integers(1, 700))
    cols = 8 * int(g.integers(1, 400))
    pad = 8 * int(g.integers(0, 3))
    mode = int(g.integers(0, 2))
    codes = int(g.integers(0, 2))
    seed, off = int(g.integers(0, 1 << 40)), int(g.integers(0, 1 << 34))
    sid = int(g.integers(0, 6))
    base = _input(rows, cols + pad, 7 * case + 1)
    x = base[:, :cols]
    xd = base.to(DEV)[:, :cols]
    kw = dict(mode=mode, seed=seed, offset=off, stream_id=sid, codes=codes)
    bits = bf16_bits(base)
    # rows
    q, s = m.int8mp_quantize_rowwise(xd, axis=m.INT8MP_GROUP_ROWS, **kw)
    qr, sr = oracle.quantize(bits, axis=0, mode=mode, seed=seed, offset=off, stream_id=sid,
                             cols=cols)
    np.testing.assert_array_equal(_f32_bits(s), sr.view(np.int32))
    np.testing.assert_array_equal(_codes_np(q), qr)
    # columns, codes in the input's layout, and the same from recorded maxima
    qc, sc = m.int8mp_quantize_rowwise(xd, axis=m.INT8MP_GROUP_COLS, **kw)
    qcr, scr = oracle.quantize(bits, axis=1, mode=mode, seed=seed, offset=off, stream_id=sid,
                               cols=cols)
    np.testing.assert_array_equal(_f32_bits(sc), scr.view(np.int32))
    np.testing.assert_array_equal(_codes_np(qc), np.ascontiguousarray(qcr.T))
    cm = torch.zeros(cols, dtype=torch.float32, device=DEV)
    q2, s2 = m.int8mp_quantize_rows_colmax(xd, cm, **kw)
    assert torch.equal(q2.view(torch.uint8), q.view(torch.uint8)) and torch.equal(s2, s)
    np.testing.assert_array_equal(_f32_bits(cm), _col_absmax_bits(x))
    qc2, sc2 = m.int8mp_quantize_cols_absmax(xd, cm, **kw)
    assert torch.equal(qc2.view(torch.uint8), qc.view(torch.uint8)) and torch.equal(sc2, sc)
    # columns written transposed (whole 8-row groups)
    if rows % 8 == 0:
        qt, st = m.int8mp_quantize_rowwise(xd, axis=m.INT8MP_GROUP_COLS_T, **kw)
        np.testing.assert_array_equal(_f32_bits(st), scr.view(np.int32))
        np.testing.assert_array_equal(_codes_np(qt), qcr)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_rows_batch(case):
    g = _rng(50 + case)
    cols = 8 * int(g.integers(1, 800))
    r0, r1 = int(g.integers(1, 3000)), int(g.integers(1, 600))
    mode, codes = int(g.integers(0, 2)), int(g.integers(0, 2))
    seed = int(g.integers(0, 1 << 40))
    offs = [int(g.integers(0, 1 << 34)), int(g.integers(0, 1 << 34))]
    sids = [int(g.integers(0, 6)), int(g.integers(0, 6))]
    with_cm = bool(g.integers(0, 2))
    xs = [_input(r0, cols, 11 * case + 2), _input(r1, cols, 11 * case + 3)]
    cms = [torch.zeros(cols, dtype=torch.float32, device=DEV) for _ in xs] if with_cm else None
    got = m.int8mp_quantize_rows_batch([x.to(DEV) for x in xs], mode=mode, seed=seed,
                                       offsets=offs, stream_ids=sids, codes=codes, colmaxes=cms)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    for i, x in enumerate(xs):
        qr, sr = oracle.quantize(bf16_bits(x), axis=0, mode=mode, seed=seed, offset=offs[i],
                                 stream_id=sids[i])
        np.testing.assert_array_equal(_f32_bits(got[i][1]), sr.view(np.int32))
        np.testing.assert_array_equal(_codes_np(got[i][0]), qr)
        if with_cm:
            np.testing.assert_array_equal(_f32_bits(cms[i]), _col_absmax_bits(x))


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_cols_batch(case):
    # two matrices' column groups in one call: one launch when both have at
    # most 2048 rows (most cases here), each matrix's passes otherwise
    g = _rng(70 + case)
    cols = 8 * int(g.integers(1, 400))
    r0, r1 = int(g.integers(1, 2600)), int(g.integers(1, 2100))
    mode, codes = int(g.integers(0, 2)), int(g.integers(0, 2))
    seed = int(g.integers(0, 1 << 40))
    offs = [int(g.integers(0, 1 << 34)), int(g.integers(0, 1 << 34))]
    sids = [int(g.integers(0, 6)), int(g.integers(0, 6))]
    xs = [_input(r0, cols, 13 * case + 4), _input(r1, cols, 13 * case + 5)]
    got = m.int8mp_quantize_cols_batch([x.to(DEV) for x in xs], mode=mode, seed=seed,
                                       offsets=offs, stream_ids=sids, codes=codes)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    for i, x in enumerate(xs):
        qr, sr = oracle.quantize(bf16_bits(x), axis=1, mode=mode, seed=seed, offset=offs[i],
                                 stream_id=sids[i])
        np.testing.assert_array_equal(_f32_bits(got[i][1]), sr.view(np.int32))
        np.testing.assert_array_equal(_codes_np(got[i][0]), np.ascontiguousarray(qr.T))


def _rand_codes(shape, g):
    return torch.from_numpy(g.integers(-127, 128, size=shape).astype(np.int8))


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz_matmul(case):
    g = _rng(100 + case)
    # up to ~1,100 pair tiles' worth of M x N with small K, or a long K
    M = int(g.integers(1, 2600))
    N = 8 * int(g.integers(1, 330))
    K = 16 * int(g.integers(1, 40 if g.integers(0, 2) else 700))
    layout = int(g.integers(0, 3))
    if layout == m.INT8MP_ATxB:
        M = 8 * max(1, M // 8)
    ws = bool(g.integers(0, 2))
    a = _rand_codes((K, M) if layout == m.INT8MP_ATxB else (M, K), g)
    b = _rand_codes((N, K) if layout == m.INT8MP_AxBT else (K, N), g)
    ad, bd = a.half().to(DEV), b.half().to(DEV)
    acc = m.int8mp_mm_s32(ad, bd, layout=layout, workspace=True if ws else None)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    rows = np.unique(np.r_[0, M - 1, g.integers(0, M, size=24)])
    a_rows = (a.numpy().T if layout == m.INT8MP_ATxB else a.numpy())[rows]
    b_nk = b.numpy() if layout == m.INT8MP_AxBT else np.ascontiguousarray(b.numpy().T)
    ref = oracle.mm_s32(a_rows, b_nk, len(rows), N, K)
    np.testing.assert_array_equal(acc.cpu().numpy()[rows], ref)
    sa = torch.from_numpy(g.random(M).astype(np.float32) + 0.25)
    sb = torch.from_numpy(g.random(N).astype(np.float32) + 0.25)
    out = m.int8mp_scaled_mm(ad, sa.to(DEV), bd, sb.to(DEV), layout=layout,
                             workspace=True if ws else None)
    ref = oracle.scaled_mm(a_rows, sa.numpy()[rows], b_nk, sb.numpy(), len(rows), N, K)
    np.testing.assert_array_equal(out.cpu().view(torch.int16).numpy()[rows].view(np.uint16), ref)


@pytest.mark.parametrize("case", range(CASES // 2))
def test_fuzz_linear(case):
    # random per-pass switches (a pass at 0 runs in BF16) and, for every
    # other case, the forward pass that saves X's and W's column absmax and
    # the backward pass that takes them
    from test_gpu_parity import _bf16_pass_close
    g = _rng(200 + case)
    T = 16 * int(g.integers(1, 80))
    N = 16 * int(g.integers(1, 80))
    K = 16 * int(g.integers(1, 80))
    mode = int(g.integers(0, 2))
    seed, off = int(g.integers(0, 1 << 40)), int(g.integers(0, 1 << 30))
    f, gi, gw = (1, 1, 1) if case % 3 == 0 else tuple(int(v) for v in g.integers(0, 2, size=3))
    saved = case % 2 == 1
    X = _input(T, K, 300 + case)
    W = synth.bf16_normal((N, K), 400 + case, std=0.02)
    dY = synth.bf16_normal((T, N), 500 + case, std=1e-3)
    cfg = m.linear_cfg(mode=mode, seed=seed, offset=off, int8_fwd=f, int8_grad_in=gi,
                       int8_grad_w=gw)
    Xd, Wd, dYd = X.to(DEV), W.to(DEV), dY.to(DEV)
    if saved:
        absmax = torch.empty(2 * K, dtype=torch.float32, device=DEV)
        Y = m.int8mp_linear_fwd_save(Xd, Wd, absmax, cfg)
        dX, dW = m.int8mp_linear_bwd_saved(dYd, Xd, Wd, absmax, cfg)
    else:
        Y = m.int8mp_linear_fwd(Xd, Wd, cfg)
        dX, dW = m.int8mp_linear_bwd(dYd, Xd, Wd, cfg)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    kw = dict(mode=mode, seed=seed, offset=off)
    Yr = oracle.linear_fwd_cfg(bf16_bits(X), bf16_bits(W), int8_fwd=f, **kw)
    dXr, dWr = oracle.linear_bwd_cfg(bf16_bits(dY), bf16_bits(X), bf16_bits(W), int8_grad_in=gi,
                                     int8_grad_w=gw, **kw)
    xf, wf, gf = X.float(), W.float(), dY.float()
    for got, ref, int8, a, b, what in ((Y, Yr, f, xf, wf, "forward"),
                                       (dX, dXr, gi, gf, wf.T.contiguous(), "grad input"),
                                       (dW, dWr, gw, gf.T.contiguous(), xf.T.contiguous(),
                                        "grad weight")):
        if int8:
            np.testing.assert_array_equal(bf16_bits(got.cpu()), ref, err_msg=what)
        else:
            _bf16_pass_close(got, ref, a, b, what)
