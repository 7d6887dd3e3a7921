"""Parity at the benchmark's full sizes.

The Llama2-1B layer linears at T = 16 x 2048 (nearest-even and stochastic
rounding) and the Llama-3-8B ones at T = 16384 run through
int8mp_linear_fwd / int8mp_linear_bwd, and the 4096^3 square problem in
the three layouts through int8mp_quantize_rowwise + int8mp_scaled_mm: the
kernels and launch shapes the benchmark times.  The oracle quantizes every
operand in full and computes a sample of output rows (each output row
depends only on its own row of the first operand and all of the second, so
a sampled row is exact); those rows must match bit for bit.
"""
import numpy as np
import pytest
import torch

import int8_mixed_precision_row_gb300 as m
import oracle
from helpers import bf16_bits, bf16_pass_close
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


def _rows_equal(got_t, idx, ref, what):
    got = bf16_bits(got_t[torch.from_numpy(idx).to(got_t.device)].cpu())
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        pytest.fail(f"{what}: {len(bad)} of {ref.size} sampled outputs differ, first at {bad[0]}")


CASES = [
    ("llama2-1b", "q", oracle.RNE),
    ("llama2-1b", "down", oracle.RNE),
    ("llama2-1b", "gate", oracle.SR),
    ("llama3-8b", "k", oracle.RNE),
    ("llama3-8b", "down", oracle.RNE),
]


@pytest.mark.parametrize("spec_name,name,mode", CASES)
def test_full_size_linear_sampled_rows(spec_name, name, mode):
    spec = {"llama2-1b": synth.LLAMA2_1B, "llama3-8b": synth.LLAMA3_8B}[spec_name]
    X, W, dY = synth.linear_inputs(spec, name)
    T, K = X.shape
    N = W.shape[0]
    seed, offset = 0, 0
    cfg = m.linear_cfg(mode=mode, seed=seed, offset=offset)
    Xd, Wd, dYd = X.to(DEV), W.to(DEV), dY.to(DEV)
    Y = m.int8mp_linear_fwd(Xd, Wd, cfg)
    dX, dW = m.int8mp_linear_bwd(dYd, Xd, Wd, cfg)
    torch.cuda.synchronize()
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    del Xd, Wd, dYd

    xb, wb, gb = bf16_bits(X), bf16_bits(W), bf16_bits(dY)
    del X, W, dY
    kw = dict(mode=mode, seed=seed, offset=offset)
    rows_t = _sample(T, 8, 1)
    rows_n = _sample(N, 4, 2)
    # forward: X and W along K
    qx, sx = oracle.quantize(xb, 0, stream_id=oracle.STREAM_FWD_X, **kw)
    qw, sw = oracle.quantize(wb, 0, stream_id=oracle.STREAM_FWD_W, **kw)
    ref = oracle.scaled_mm(qx[rows_t], sx[rows_t], qw, sw, len(rows_t), N, K)
    _rows_equal(Y, rows_t, ref, f"{spec_name} {name} forward")
    del qx, qw
    # grad input: dY along N (rows), W along N (columns)
    qg, sg = oracle.quantize(gb, 0, stream_id=oracle.STREAM_GI_DY, **kw)
    qwt, swt = oracle.quantize(wb, 1, stream_id=oracle.STREAM_GI_W, **kw)
    ref = oracle.scaled_mm(qg[rows_t], sg[rows_t], qwt, swt, len(rows_t), K, N)
    _rows_equal(dX, rows_t, ref, f"{spec_name} {name} grad input")
    del qg, qwt
    # grad weight: dY and X along T (columns)
    qgt, sgt = oracle.quantize(gb, 1, stream_id=oracle.STREAM_GW_DY, **kw)
    qxt, sxt = oracle.quantize(xb, 1, stream_id=oracle.STREAM_GW_X, **kw)
    ref = oracle.scaled_mm(qgt[rows_n], sgt[rows_n], qxt, sxt, len(rows_n), K, T)
    _rows_equal(dW, rows_n, ref, f"{spec_name} {name} grad weight")


@pytest.mark.parametrize("layout", ["AxBT", "AxB", "ATxB"])
def test_square_4096_sampled_rows(layout):
    # as the benchmark runs it: operands stored K-first are quantized by
    # columns with their codes left in place and multiplied in that layout
    S = 4096
    A, B = synth.square_inputs(S, layout)
    a_cols = layout == "ATxB"
    b_cols = layout != "AxBT"
    ax = lambda cols: m.INT8MP_GROUP_COLS if cols else m.INT8MP_GROUP_ROWS
    lay = {"AxBT": m.INT8MP_AxBT, "AxB": m.INT8MP_AxB, "ATxB": m.INT8MP_ATxB}[layout]
    qa, sa = m.int8mp_quantize_rowwise(A.to(DEV), axis=ax(a_cols), codes=m.INT8MP_CODES_F16)
    qb, sb = m.int8mp_quantize_rowwise(B.to(DEV), axis=ax(b_cols), codes=m.INT8MP_CODES_F16)
    out = m.int8mp_scaled_mm(qa, sa, qb, sb, layout=lay)
    torch.cuda.synchronize()
    # the oracle returns K-major codes (column groups transposed)
    qar, sar = oracle.quantize(bf16_bits(A), axis=1 if a_cols else 0)
    qbr, sbr = oracle.quantize(bf16_bits(B), axis=1 if b_cols else 0)
    # the quantized operands themselves, in full, in the stored layout
    stored = lambda q, cols: np.ascontiguousarray(q.T) if cols else q
    np.testing.assert_array_equal(sa.cpu().numpy().view(np.int32), sar.view(np.int32))
    np.testing.assert_array_equal(qa.cpu().float().to(torch.int8).numpy(), stored(qar, a_cols))
    np.testing.assert_array_equal(sb.cpu().numpy().view(np.int32), sbr.view(np.int32))
    np.testing.assert_array_equal(qb.cpu().float().to(torch.int8).numpy(), stored(qbr, b_cols))
    rows = _sample(S, 8, 3)
    ref = oracle.scaled_mm(qar[rows], sar[rows], qbr, sbr, len(rows), S, S)  # K-major codes
    _rows_equal(out, rows, ref, f"square 4096 {layout}")


@pytest.mark.parametrize("name", ["q", "down"])
def test_full_size_bf16_passes_sampled_rows(name):
    """The pages' BF16 training-table row at full size: all three passes in
    BF16 (bf16 operands, fp32 accumulation in the tcgen05 kernels; the down
    projection's forward pass splits its last wave), sampled output rows
    against the oracle's bf16 product within the fp32 accumulation bound."""
    X, W, dY = synth.linear_inputs(synth.LLAMA2_1B, name)
    T, K = X.shape
    N = W.shape[0]
    cfg = m.linear_cfg(int8_fwd=0, int8_grad_in=0, int8_grad_w=0)
    Xd, Wd, dYd = X.to(DEV), W.to(DEV), dY.to(DEV)
    Y = m.int8mp_linear_fwd(Xd, Wd, cfg)
    dX, dW = m.int8mp_linear_bwd(dYd, Xd, Wd, cfg)
    torch.cuda.synchronize()
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    del Xd, Wd, dYd
    xb, wb, gb = bf16_bits(X), bf16_bits(W), bf16_bits(dY)
    rows_t = _sample(T, 8, 5)
    rows_n = _sample(N, 4, 6)
    it, in_ = torch.from_numpy(rows_t), torch.from_numpy(rows_n)
    ref = oracle.matmul_bf16(xb[rows_t], wb, len(rows_t), N, K, layout=oracle.AxBT)
    bf16_pass_close(Y[it.to(DEV)], ref, X[it].float(), W.float(), f"{name} BF16 forward")
    ref = oracle.matmul_bf16(gb[rows_t], wb, len(rows_t), K, N, layout=oracle.AxB)
    bf16_pass_close(dX[it.to(DEV)], ref, dY[it].float(), W.float().T.contiguous(),
                    f"{name} BF16 grad input")
    ref = oracle.matmul_bf16(np.ascontiguousarray(gb[:, rows_n]), xb, len(rows_n), K, T,
                             layout=oracle.ATxB)
    bf16_pass_close(dW[in_.to(DEV)], ref, dY[:, in_].float().T.contiguous(),
                    X.float().T.contiguous(), f"{name} BF16 grad weight")
