"""Parity of the benchmark's timed step itself, at its full size.

The headline number times `bench.LayerStep.run`: per linear, X and W
quantized by rows in one launch that also records their column absmax
(int8mp_quantize_rows_batch), the forward matmul, dY by rows recording its
column absmax (int8mp_quantize_rows_colmax), W, dY and X by columns from
those maxima (int8mp_quantize_cols_absmax), and the grad-input and
grad-weight matmuls (int8mp_scaled_mm_ws in the A @ B and A.T @ B layouts).
These tests run that sequence through the same LayerStep methods, at
T = 16 x 2048 on the Llama2-1B shapes, and compare with the oracle after
every call: the column maxima, every code and every scale in full, and a
sample of output rows of the three matmuls (an output row depends only on
its own row of the first operand, so a sampled row is exact).  Then a whole
`run()` must give those same outputs.  Stochastic rounding ("Quantized model
training" README, the SR rows of the INT8 mixed precision training table)
is covered on q and down.

The layer entry points the end-to-end figure uses (int8mp_linear_fwd_save /
int8mp_linear_bwd_saved) are checked the same way at full size.
"""
import numpy as np
import pytest
import torch

import bench
import int8_mixed_precision_row_gb300 as m
import oracle
from helpers import bf16_bits, bits_to_f32
from int8_mixed_precision_row_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_mixed_precision_row_gb300 import build
    build.build()
    m.load()


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    idx = set(rng.choice(n, size=k - 2, replace=False).tolist()) | {0, n - 1}
    return np.array(sorted(idx))


def _colmax_ref(xb):
    """max |x| over each column of bf16 bits [rows, cols], as fp32."""
    return np.abs(bits_to_f32(xb)).max(axis=0).astype(np.float32)


def _f32_equal(got_t, ref, what):
    got = got_t.detach().cpu().numpy().astype(np.float32)
    if not np.array_equal(got.view(np.int32), ref.astype(np.float32).view(np.int32)):
        bad = np.flatnonzero(got.view(np.int32) != ref.astype(np.float32).view(np.int32))
        pytest.fail(f"{what}: {bad.size} of {ref.size} values differ, first at {bad[0]} "
                    f"({got.ravel()[bad[0]]!r} vs {ref.ravel()[bad[0]]!r})")


def _codes_equal(got_f16, ref_i8, what):
    got = got_f16.to(torch.int8).cpu().numpy()
    if not np.array_equal(got, ref_i8):
        bad = np.argwhere(got != ref_i8)
        pytest.fail(f"{what}: {len(bad)} of {ref_i8.size} codes differ, first at {bad[0]}")


def _rows_equal(got_t, idx, ref, what):
    got = bf16_bits(got_t[torch.from_numpy(idx).to(got_t.device)].cpu())
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        pytest.fail(f"{what}: {len(bad)} of {ref.size} sampled outputs differ, first at {bad[0]}")


STEP_CASES = [
    ("q", oracle.RNE), ("gate", oracle.RNE), ("down", oracle.RNE),
    ("q", oracle.SR), ("down", oracle.SR),
]


@pytest.mark.parametrize("name,mode", STEP_CASES)
def test_timed_step_sequence_full_size(name, mode):
    seed, offset = 5, 3 << 20
    step = bench.LayerStep(synth.LLAMA2_1B, mode, torch.device(DEV), only={name})
    l = step.linears[0]
    X, W, dY = step.host[name]
    T, K = X.shape
    N = W.shape[0]
    assert T == 32768
    xb, wb, gb = bf16_bits(X), bf16_bits(W), bf16_bits(dY)
    kw = dict(mode=mode, seed=seed, offset=offset)
    cm = l["colmax"]
    cx, cw, cg = cm[:K], cm[K:2 * K], cm[2 * K:]
    rows_t = _sample(T, 8, 11)
    rows_n = _sample(N, 4, 12)

    # forward: X and W by rows in one launch, with their column maxima
    step.colmax_all.zero_()
    (qx, sx), (qw, sw) = step._q_rows2(l["X"], l["W"], cx, cw, seed, offset)
    torch.cuda.synchronize()
    _f32_equal(cx, _colmax_ref(xb), "X column absmax from its row pass")
    _f32_equal(cw, _colmax_ref(wb), "W column absmax from its row pass")
    qxr, sxr = oracle.quantize(xb, 0, stream_id=oracle.STREAM_FWD_X, **kw)
    _f32_equal(sx, sxr, "forward X scales")
    _codes_equal(qx, qxr, "forward X codes")
    qwr, swr = oracle.quantize(wb, 0, stream_id=oracle.STREAM_FWD_W, **kw)
    _f32_equal(sw, swr, "forward W scales")
    _codes_equal(qw, qwr, "forward W codes")
    ref_y = oracle.scaled_mm(qxr[rows_t], sxr[rows_t], qwr, swr, len(rows_t), N, K)
    del qxr, qwr

    # grad input: dY by rows (with its column maxima), W by columns from its maxima
    qg, sg = step._q(l["dY"], 0, m.INT8MP_STREAM_GI_DY, step.qa, step.sa, seed, offset, cg)
    torch.cuda.synchronize()
    _f32_equal(cg, _colmax_ref(gb), "dY column absmax from its row pass")
    qgr, sgr = oracle.quantize(gb, 0, stream_id=oracle.STREAM_GI_DY, **kw)
    _f32_equal(sg, sgr, "grad-input dY scales")
    _codes_equal(qg, qgr, "grad-input dY codes")
    qwc, swc = step._q(l["W"], 2, m.INT8MP_STREAM_GI_W, step.qb, step.sb, seed, offset, cw)
    torch.cuda.synchronize()
    qwtr, swtr = oracle.quantize(wb, 1, stream_id=oracle.STREAM_GI_W, **kw)  # [K, N]
    _f32_equal(swc, swtr, "grad-input W column scales")
    _codes_equal(qwc, np.ascontiguousarray(qwtr.T), "grad-input W column codes")
    ref_dx = oracle.scaled_mm(qgr[rows_t], sgr[rows_t], qwtr, swtr, len(rows_t), K, N)
    del qgr, qwtr

    # grad weight: dY and X by columns from their maxima
    qgc, sgc = step._q(l["dY"], 2, m.INT8MP_STREAM_GW_DY, step.qa, step.sa, seed, offset, cg)
    torch.cuda.synchronize()
    qgtr, sgtr = oracle.quantize(gb, 1, stream_id=oracle.STREAM_GW_DY, **kw)  # [N, T]
    _f32_equal(sgc, sgtr, "grad-weight dY column scales")
    _codes_equal(qgc, np.ascontiguousarray(qgtr.T), "grad-weight dY column codes")
    qxc, sxc = step._q(l["X"], 2, m.INT8MP_STREAM_GW_X, step.qb, step.sb, seed, offset, cx)
    torch.cuda.synchronize()
    qxtr, sxtr = oracle.quantize(xb, 1, stream_id=oracle.STREAM_GW_X, **kw)  # [K, T]
    _f32_equal(sxc, sxtr, "grad-weight X column scales")
    _codes_equal(qxc, np.ascontiguousarray(qxtr.T), "grad-weight X column codes")
    ref_dw = oracle.scaled_mm(qgtr[rows_n], sgtr[rows_n], qxtr, sxtr, len(rows_n), K, T)
    del qgtr, qxtr

    # the whole timed step, as the benchmark runs it
    step.run(seed=seed, offset=offset)
    torch.cuda.synchronize()
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    _rows_equal(l["Y"], rows_t, ref_y, f"{name} forward")
    _rows_equal(l["dX"], rows_t, ref_dx, f"{name} grad input")
    _rows_equal(l["dW"], rows_n, ref_dw, f"{name} grad weight")


SAVED_CASES = [("down", oracle.RNE), ("q", oracle.SR)]


@pytest.mark.parametrize("name,mode", SAVED_CASES)
def test_layer_entry_points_with_saved_absmax_full_size(name, mode):
    """int8mp_linear_fwd_save / int8mp_linear_bwd_saved at T = 32768: the
    saved column absmax in full, sampled rows of Y, dX and dW."""
    X, W, dY = synth.linear_inputs(synth.LLAMA2_1B, name)
    T, K = X.shape
    N = W.shape[0]
    seed, offset = 9, 1 << 33
    cfg = m.linear_cfg(mode=mode, seed=seed, offset=offset)
    Xd, Wd, dYd = X.to(DEV), W.to(DEV), dY.to(DEV)
    absmax = torch.full((2 * K,), -1.0, dtype=torch.float32, device=DEV)
    Y = m.int8mp_linear_fwd_save(Xd, Wd, absmax, cfg)
    dX, dW = m.int8mp_linear_bwd_saved(dYd, Xd, Wd, absmax, cfg)
    torch.cuda.synchronize()
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    del Xd, Wd, dYd
    xb, wb, gb = bf16_bits(X), bf16_bits(W), bf16_bits(dY)
    _f32_equal(absmax[:K], _colmax_ref(xb), "saved X column absmax")
    _f32_equal(absmax[K:], _colmax_ref(wb), "saved W column absmax")
    kw = dict(mode=mode, seed=seed, offset=offset)
    rows_t = _sample(T, 6, 21)
    rows_n = _sample(N, 4, 22)
    qx, sx = oracle.quantize(xb, 0, stream_id=oracle.STREAM_FWD_X, **kw)
    qw, sw = oracle.quantize(wb, 0, stream_id=oracle.STREAM_FWD_W, **kw)
    _rows_equal(Y, rows_t, oracle.scaled_mm(qx[rows_t], sx[rows_t], qw, sw, len(rows_t), N, K),
                f"{name} forward (saved absmax)")
    del qx, qw
    qg, sg = oracle.quantize(gb, 0, stream_id=oracle.STREAM_GI_DY, **kw)
    qwt, swt = oracle.quantize(wb, 1, stream_id=oracle.STREAM_GI_W, **kw)
    _rows_equal(dX, rows_t, oracle.scaled_mm(qg[rows_t], sg[rows_t], qwt, swt, len(rows_t), K, N),
                f"{name} grad input (saved absmax)")
    del qg, qwt
    qgt, sgt = oracle.quantize(gb, 1, stream_id=oracle.STREAM_GW_DY, **kw)
    qxt, sxt = oracle.quantize(xb, 1, stream_id=oracle.STREAM_GW_X, **kw)
    _rows_equal(dW, rows_n, oracle.scaled_mm(qgt[rows_n], sgt[rows_n], qxt, sxt, len(rows_n), K, T),
                f"{name} grad weight (saved absmax)")
