"""GPU parity: the CUDA path (through the C ABI) against the oracle on the
same seeded bf16 inputs.

Bar: INT8 codes, fp32 scales (bit patterns) and int32 accumulators must be
bit-exact; bf16 outputs are allowed 1 ulp by the method's reading of the
rescale, but the kernels perform the same IEEE operations in the same order
as the oracle, so the tests require exact equality and report the ulp
distance if it ever differs.
"""
import numpy as np
import pytest
import torch

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


def _dev(t):
    return t.to(DEV)


def _codes_np(q):
    q = q.cpu()
    if q.dtype == torch.float16:
        f = q.float()
        assert torch.equal(f, f.round()) and f.abs().max() <= 127
        return f.to(torch.int8).numpy()
    return q.numpy()


def _f32_bits(t):
    return t.cpu().contiguous().view(torch.int32).numpy()


def _bf16_ulp_dist(a_bits, b_bits):
    def ordered(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + (b & 0x7FFF))
    return np.abs(ordered(a_bits) - ordered(b_bits))


def assert_bf16_equal(got_t, ref_bits, what):
    got = bf16_bits(got_t.cpu())
    if not np.array_equal(got, ref_bits):
        d = _bf16_ulp_dist(got, ref_bits)
        pytest.fail(f"{what}: {np.count_nonzero(d)} of {d.size} bf16 outputs differ, max {d.max()} ulp")


def _edge_input(rows, cols, seed):
    x = synth.bf16_normal((rows, cols), seed, outlier_frac=0.01, outlier_scale=20.0).float()
    if rows >= 8:
        x[1] = 0.0
        x[2] = -x[2].abs() * 3.0
        x[3] = x[3] * 1e-38
        x[4] = 0.0
        x[4, min(5, cols - 1)] = 1e-40
        x[5] = x[5] * 1e36  # large but finite: inf/NaN inputs are outside the contract
        x[6, 0] = 127.0
        x[6, 1:] = torch.arange(1, cols) * 0.5 - 40
    return x.to(torch.bfloat16)


ROW_SHAPES = [(256, 512), (8, 8), (77, 136), (300, 5632), (40, 14336), (9, 24576), (1, 2048),
              (3, 53248)]
COL_SHAPES = [(256, 512), (8, 8), (264, 136), (1032, 64), (520, 2048), (16, 4096)]


@pytest.mark.parametrize("codes", [m.INT8MP_CODES_S8, m.INT8MP_CODES_F16])
@pytest.mark.parametrize("mode", [m.INT8MP_RNE, m.INT8MP_SR])
@pytest.mark.parametrize("shape", ROW_SHAPES)
def test_quantize_rows_bit_exact(shape, mode, codes):
    rows, cols = shape
    x = _edge_input(rows, cols, seed=rows + cols)
    seed, off, sid = 1234567, 13, 3
    q, s = m.int8mp_quantize_rowwise(_dev(x), axis=0, mode=mode, seed=seed, offset=off,
                                     stream_id=sid, codes=codes)
    qr, sr = oracle.quantize(bf16_bits(x), axis=0, mode=mode, seed=seed, offset=off, stream_id=sid)
    np.testing.assert_array_equal(_f32_bits(s), sr.view(np.int32))
    np.testing.assert_array_equal(_codes_np(q), qr)


@pytest.mark.parametrize("codes", [m.INT8MP_CODES_S8, m.INT8MP_CODES_F16])
@pytest.mark.parametrize("mode", [m.INT8MP_RNE, m.INT8MP_SR])
@pytest.mark.parametrize("shape", COL_SHAPES)
def test_quantize_cols_bit_exact(shape, mode, codes):
    rows, cols = shape
    x = _edge_input(rows, cols, seed=7 * rows + cols)
    seed, off, sid = 99, 2**33 + 1, 5
    q, s = m.int8mp_quantize_rowwise(_dev(x), axis=1, mode=mode, seed=seed, offset=off,
                                     stream_id=sid, codes=codes)
    qr, sr = oracle.quantize(bf16_bits(x), axis=1, mode=mode, seed=seed, offset=off, stream_id=sid)
    np.testing.assert_array_equal(_f32_bits(s), sr.view(np.int32))
    np.testing.assert_array_equal(_codes_np(q), qr)


def test_quantize_with_padded_leading_dimension():
    base = _edge_input(64, 160, seed=3)
    view = _dev(base)[:, :136]  # ld 160 > cols 136
    q, s = m.int8mp_quantize_rowwise(view, axis=0, codes=m.INT8MP_CODES_F16)
    qr, sr = oracle.quantize(bf16_bits(base), axis=0, cols=136)
    np.testing.assert_array_equal(_codes_np(q), qr)
    q1, s1 = m.int8mp_quantize_rowwise(view, axis=1, codes=m.INT8MP_CODES_S8)
    qr1, sr1 = oracle.quantize(bf16_bits(base[:, :136].contiguous()), axis=1)
    np.testing.assert_array_equal(_codes_np(q1), qr1)
    np.testing.assert_array_equal(_f32_bits(s1), sr1.view(np.int32))


def _rand_codes(M, K, seed, extreme=False):
    g = torch.Generator().manual_seed(seed)
    if extreme:
        sign = torch.randint(0, 2, (M, K), generator=g) * 2 - 1
        return (sign * 127).to(torch.int8)
    return torch.randint(-127, 128, (M, K), generator=g, dtype=torch.int32).to(torch.int8)


MM_SHAPES = [(256, 256, 512), (128, 256, 16), (200, 264, 144), (130, 520, 1040),
             (256, 512, 3072), (64, 96, 4096), (1000, 776, 2096), (100, 1024, 64)]


@pytest.mark.parametrize("shape", MM_SHAPES)
def test_mm_s32_bit_exact(shape):
    M, N, K = shape
    a, b = _rand_codes(M, K, 1), _rand_codes(N, K, 2)
    acc = m.int8mp_mm_s32(_dev(a.half()), _dev(b.half()))
    ref = oracle.mm_s32(a.numpy(), b.numpy(), M, N, K)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref)


@pytest.mark.parametrize("M", [128, 256])  # single-CTA and CTA-pair kernels
def test_mm_s32_chunking_keeps_large_sums_exact(M):
    # all codes +-127 with K = 8192: partial sums reach 127^2 * 8192 = 1.3e8,
    # far above 2^24, so a single fp32 accumulation would round
    N, K = 256, 8192
    a = _rand_codes(M, K, 3, extreme=True)
    b = _rand_codes(N, K, 4, extreme=True)
    b[0] = a[0]          # row 0 of the output hits 127^2 * K exactly
    b[1] = -a[1]
    acc = m.int8mp_mm_s32(_dev(a.half()), _dev(b.half())).cpu().numpy()
    ref = oracle.mm_s32(a.numpy(), b.numpy(), M, N, K)
    assert ref[0, 0] == 127 * 127 * K and ref[1, 1] == -127 * 127 * K
    np.testing.assert_array_equal(acc, ref)


@pytest.mark.parametrize("shape", [(256, 256, 512), (200, 264, 144), (384, 512, 2048)])
def test_scaled_mm_bit_exact(shape):
    M, N, K = shape
    A = synth.bf16_normal((M, K), 0, outlier_frac=0.01, outlier_scale=20.0)
    B = synth.bf16_normal((N, K), 1, outlier_frac=0.01, outlier_scale=20.0)
    qa, sa = m.int8mp_quantize_rowwise(_dev(A), axis=0, codes=m.INT8MP_CODES_F16)
    qb, sb = m.int8mp_quantize_rowwise(_dev(B), axis=0, codes=m.INT8MP_CODES_F16)
    out = m.int8mp_scaled_mm(qa, sa, qb, sb)
    qar, sar = oracle.quantize(bf16_bits(A), axis=0)
    qbr, sbr = oracle.quantize(bf16_bits(B), axis=0)
    ref = oracle.scaled_mm(qar, sar, qbr, sbr, M, N, K)
    assert_bf16_equal(out, ref, "scaled_mm")


@pytest.mark.parametrize("layout", ["AxBT", "AxB", "ATxB"])
def test_square_layouts_through_quantize_side_transpose(layout):
    # A @ B: B [K,N] quantized along K = its columns (axis 1 writes [N,K]);
    # A.T @ B: A [K,M] likewise.  The matmul then always reads K-major codes.
    S = 256
    A, B = synth.square_inputs(S, layout)
    a_axis = 1 if layout == "ATxB" else 0
    b_axis = 0 if layout == "AxBT" else 1
    qa, sa = m.int8mp_quantize_rowwise(_dev(A), axis=a_axis, codes=m.INT8MP_CODES_F16)
    qb, sb = m.int8mp_quantize_rowwise(_dev(B), axis=b_axis, codes=m.INT8MP_CODES_F16)
    out = m.int8mp_scaled_mm(qa, sa, qb, sb)
    lay = {"AxBT": oracle.AxBT, "AxB": oracle.AxB, "ATxB": oracle.ATxB}[layout]
    qar, sar = oracle.quantize(bf16_bits(A), axis=a_axis)
    qbr, sbr = oracle.quantize(bf16_bits(B), axis=b_axis)
    # the oracle multiplies in the stored layout: hand it the codes as stored
    qa_st = qar if layout != "ATxB" else np.ascontiguousarray(qar.T)
    qb_st = qbr if layout == "AxBT" else np.ascontiguousarray(qbr.T)
    ref = oracle.scaled_mm(qa_st, sar, qb_st, sbr, S, S, S, layout=lay)
    assert_bf16_equal(out, ref, f"square {layout}")


LINEAR_SHAPES = [(256, 256, 512), (128, 96, 160), (48, 32, 1056), (1040, 64, 48)]


@pytest.mark.parametrize("mode", [m.INT8MP_RNE, m.INT8MP_SR])
@pytest.mark.parametrize("shape", LINEAR_SHAPES)
def test_linear_fwd_bwd_bit_exact(shape, mode):
    T, N, K = shape
    X = synth.bf16_normal((T, K), 10, outlier_frac=0.005, outlier_scale=30.0)
    W = synth.bf16_normal((N, K), 20, std=0.02)
    dY = synth.bf16_normal((T, N), 30, std=1e-3)
    cfg = m.linear_cfg(mode=mode, seed=2024, offset=64)
    Y = m.int8mp_linear_fwd(_dev(X), _dev(W), cfg)
    dX, dW = m.int8mp_linear_bwd(_dev(dY), _dev(X), _dev(W), cfg)
    Yr = oracle.linear_fwd(bf16_bits(X), bf16_bits(W), mode=mode, seed=2024, offset=64)
    dXr, dWr = oracle.linear_bwd(bf16_bits(dY), bf16_bits(X), bf16_bits(W), mode=mode, seed=2024,
                                 offset=64)
    assert_bf16_equal(Y, Yr, "fwd")
    assert_bf16_equal(dX, dXr, "grad_input")
    assert_bf16_equal(dW, dWr, "grad_weight")


def test_single_forward_matmul_256x512():
    X, W = synth.single_matmul_inputs()
    Y = m.int8mp_linear_fwd(_dev(X), _dev(W))
    assert_bf16_equal(Y, oracle.linear_fwd(bf16_bits(X), bf16_bits(W)), "256x512 forward")


def test_bwd_skips_passes_on_null_outputs():
    T, N, K = 64, 48, 32
    X = synth.bf16_normal((T, K), 1)
    W = synth.bf16_normal((N, K), 2, std=0.02)
    dY = synth.bf16_normal((T, N), 3, std=1e-3)
    dX, dW = m.int8mp_linear_bwd(_dev(dY), _dev(X), _dev(W), want_dw=False)
    assert dW is None
    dXr, _ = oracle.linear_bwd(bf16_bits(dY), bf16_bits(X), bf16_bits(W), want_dw=False)
    assert_bf16_equal(dX, dXr, "grad_input only")


def test_empty_and_zero_contraction():
    z = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    q, s = m.int8mp_quantize_rowwise(z, axis=0)
    assert q.shape == (0, 64)
    a = torch.empty((32, 0), dtype=torch.float16, device=DEV)
    b = torch.empty((16, 0), dtype=torch.float16, device=DEV)
    out = torch.full((32, 16), 7.0, dtype=torch.bfloat16, device=DEV)
    sa = torch.ones(32, device=DEV)
    sb = torch.ones(16, device=DEV)
    m.int8mp_scaled_mm(a, sa, b, sb, out=out)
    assert torch.count_nonzero(out) == 0


def test_bounded_wait_reports_timeout_and_context_survives():
    M, N, K = 256, 512, 256
    a, b = _rand_codes(M, K, 5), _rand_codes(N, K, 6)
    ad, bd = _dev(a.half()), _dev(b.half())
    out = torch.zeros((M, N), dtype=torch.int32, device=DEV)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    st = m.int8mp_debug_mm_s32_drop_first_load(ad, bd, out, wait_limit_ms=100)
    assert st == m.INT8MP_OK
    assert m.int8mp_poll_device_status() == m.INT8MP_ERR_TIMEOUT
    assert m.int8mp_poll_device_status() == m.INT8MP_OK  # the word was cleared
    # the CUDA context is intact: a normal launch still runs and is exact
    acc = m.int8mp_mm_s32(ad, bd).cpu().numpy()
    np.testing.assert_array_equal(acc, oracle.mm_s32(a.numpy(), b.numpy(), M, N, K))
    assert m.int8mp_poll_device_status() == m.INT8MP_OK


def test_division_gives_ieee_codes_for_every_bf16_pair():
    # codes from the quantizers' reciprocal-and-FMA quotient against codes
    # from __fdiv_rn on every (absmax, x) pair of bf16 values with absmax > 0
    # finite and |x| <= absmax: nearest-even bit for bit, stochastic for
    # every possible draw
    bad, pairs, fast, qdiff, first = m.int8mp_debug_check_division()
    print(f"division check: {pairs} pairs, {fast} on the fast path, {qdiff} quotients differ "
          f"in some bit, {bad} codes differ")
    assert pairs > 1_000_000_000
    assert fast > 200_000_000  # the fast path is exercised (scales in [2^-60, 2^10])
    assert bad == 0, f"{bad} codes differ; first at bf16 bits (absmax, x) = {first}"


@pytest.mark.parametrize("axis", [0, 1])
def test_quantize_division_ties_bit_exact(axis):
    # bf16 pairs where x / s sits on (or within rounding of) k + 1/2 and a
    # reciprocal multiply would round the other way than IEEE division
    from test_oracle_quantize import DIVISION_TIES
    rows = np.zeros((len(DIVISION_TIES), 8), dtype=np.float32)
    for i, (amax, xv) in enumerate(DIVISION_TIES):
        rows[i, 0], rows[i, 1] = amax, xv
        rows[i, 2:] = np.float32(xv) * np.array([1, -1, 0.5, -0.5, 0.25, 3], dtype=np.float32)
    x = torch.from_numpy(rows).to(torch.bfloat16)
    if axis == 1:
        x = x.t().contiguous()
    for codes in (m.INT8MP_CODES_S8, m.INT8MP_CODES_F16):
        q, s = m.int8mp_quantize_rowwise(_dev(x), axis=axis, codes=codes)
        qr, sr = oracle.quantize(bf16_bits(x), axis=axis)
        np.testing.assert_array_equal(_f32_bits(s), sr.view(np.int32))
        np.testing.assert_array_equal(_codes_np(q), qr)


def _bf16_pass_close(got_t, ref_bits, a, b, what):
    """BF16 pass: cuBLASLt accumulates in fp32 in its own order, the oracle
    in fp64; allow two bf16 ulps plus the fp32 accumulation bound
    K 2^-23 sum |a||b| per output."""
    got = got_t.cpu().float().double()
    ref = torch.from_numpy(bits_to_f32(ref_bits).astype(np.float64))
    K = a.shape[1]
    bound = 2.0 ** -7 * ref.abs() + K * 2.0 ** -23 * (a.abs().double() @ b.abs().double().T)
    bad = (got - ref).abs() > bound
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} outputs outside the bound"


@pytest.mark.parametrize("flags", [(0, 0, 0), (1, 0, 0), (1, 1, 0), (0, 1, 1), (1, 0, 1)])
def test_linear_per_pass_switches(flags):
    T, N, K = 256, 192, 320
    X = synth.bf16_normal((T, K), 40)
    W = synth.bf16_normal((N, K), 41, std=0.02)
    dY = synth.bf16_normal((T, N), 42, std=1e-3)
    f, gi, gw = flags
    cfg = m.linear_cfg(mode=m.INT8MP_SR, seed=3, offset=7, int8_fwd=f, int8_grad_in=gi,
                       int8_grad_w=gw)
    Y = m.int8mp_linear_fwd(_dev(X), _dev(W), cfg)
    dX, dW = m.int8mp_linear_bwd(_dev(dY), _dev(X), _dev(W), cfg)
    kw = dict(mode=oracle.SR, seed=3, offset=7)
    Yr = oracle.linear_fwd_cfg(bf16_bits(X), bf16_bits(W), int8_fwd=f, **kw)
    dXr, dWr = oracle.linear_bwd_cfg(bf16_bits(dY), bf16_bits(X), bf16_bits(W), int8_grad_in=gi,
                                     int8_grad_w=gw, **kw)
    xf, wf, gf = X.float(), W.float(), dY.float()
    if f:
        assert_bf16_equal(Y, Yr, "INT8 forward")
    else:
        _bf16_pass_close(Y, Yr, xf, wf, "BF16 forward")
    if gi:
        assert_bf16_equal(dX, dXr, "INT8 grad input")
    else:
        _bf16_pass_close(dX, dXr, gf, wf.T.contiguous(), "BF16 grad input")
    if gw:
        assert_bf16_equal(dW, dWr, "INT8 grad weight")
    else:
        _bf16_pass_close(dW, dWr, gf.T.contiguous(), xf.T.contiguous(), "BF16 grad weight")
