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
from helpers import bf16_bits, bf16_pass_close, bits_to_f32
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


# up to 2048 rows: the one-launch kernel (1024 or 2048 rows per register
# share); more rows: the absmax, scale and code passes
COL_NAT_SHAPES = [(256, 512), (8, 8), (77, 136), (1032, 64), (520, 2048), (16, 4096),
                  (3001, 264), (1, 5632), (2048, 40), (2056, 72), (8200, 24)]


@pytest.mark.parametrize("off", [2**35 + 3, 2**35 + 4])
@pytest.mark.parametrize("codes", [m.INT8MP_CODES_S8, m.INT8MP_CODES_F16])
@pytest.mark.parametrize("mode", [m.INT8MP_RNE, m.INT8MP_SR])
@pytest.mark.parametrize("shape", COL_NAT_SHAPES)
def test_quantize_cols_in_input_layout_bit_exact(shape, mode, codes, off):
    # column groups with the codes left in x's layout: the same numbers as
    # the oracle's column quantization, which it returns transposed (an
    # offset that is a multiple of 4 starts every group of eight at a Philox
    # block, the stochastic kernel's two-rows-at-a-time path)
    rows, cols = shape
    x = _edge_input(rows, cols, seed=5 * rows + cols)
    seed, sid = 4242, 4
    q, s = m.int8mp_quantize_rowwise(_dev(x), axis=m.INT8MP_GROUP_COLS, mode=mode, seed=seed,
                                     offset=off, stream_id=sid, codes=codes)
    assert tuple(q.shape) == (rows, cols)
    qr, sr = oracle.quantize(bf16_bits(x), axis=1, mode=mode, seed=seed, offset=off, stream_id=sid)
    np.testing.assert_array_equal(_f32_bits(s), sr.view(np.int32))
    np.testing.assert_array_equal(_codes_np(q), np.ascontiguousarray(qr.T))


# Plain inputs (every column's scale in the division's fast range, as in a
# real operand), on both sides of the one-launch kernel's 2048-row limit
COL_NAT_PLAIN_SHAPES = [(1024, 1024), (2048, 264), (2049, 64), (4096, 136), (9, 8)]


@pytest.mark.parametrize("off", [3, 2**20])
@pytest.mark.parametrize("codes", [m.INT8MP_CODES_S8, m.INT8MP_CODES_F16])
@pytest.mark.parametrize("mode", [m.INT8MP_RNE, m.INT8MP_SR])
@pytest.mark.parametrize("shape", COL_NAT_PLAIN_SHAPES)
def test_quantize_cols_in_input_layout_plain_inputs(shape, mode, codes, off):
    rows, cols = shape
    x = synth.bf16_normal((rows, cols), 3 * rows + cols, outlier_frac=0.01, outlier_scale=20.0)
    seed, sid = 31337, 2
    q, s = m.int8mp_quantize_rowwise(_dev(x), axis=m.INT8MP_GROUP_COLS, mode=mode, seed=seed,
                                     offset=off, stream_id=sid, codes=codes)
    qr, sr = oracle.quantize(bf16_bits(x), axis=1, mode=mode, seed=seed, offset=off, stream_id=sid)
    np.testing.assert_array_equal(_f32_bits(s), sr.view(np.int32))
    np.testing.assert_array_equal(_codes_np(q), np.ascontiguousarray(qr.T))


def _col_absmax_bits(x):
    """Each column's absmax as fp32 bits: the plain definition, max |x|."""
    return np.abs(bits_to_f32(bf16_bits(x))).max(axis=0).astype(np.float32).view(np.int32)


# cols 2048 / 4096 / 5632 / 14336 take the fused pass; 24576 (more vectors
# per thread than registers hold) and 53248 (the long-row kernel) fall back
# to a separate column pass
COLMAX_SHAPES = [(256, 512), (8, 8), (77, 136), (520, 2048), (300, 5632), (33, 4096),
                 (40, 14336), (9, 24576), (3, 53248), (4099, 1024)]


@pytest.mark.parametrize("mode", [m.INT8MP_RNE, m.INT8MP_SR])
@pytest.mark.parametrize("shape", COLMAX_SHAPES)
def test_rows_with_column_absmax_then_columns(shape, mode):
    rows, cols = shape
    x = _edge_input(rows, cols, seed=11 * rows + cols)
    xd = _dev(x)
    seed, off = 77, 5
    colmax = torch.zeros(cols, dtype=torch.float32, device=DEV)
    q, s = m.int8mp_quantize_rows_colmax(xd, colmax, mode=mode, seed=seed, offset=off, stream_id=2,
                                         codes=m.INT8MP_CODES_F16)
    qr, sr = oracle.quantize(bf16_bits(x), axis=0, mode=mode, seed=seed, offset=off, stream_id=2)
    np.testing.assert_array_equal(_f32_bits(s), sr.view(np.int32))
    np.testing.assert_array_equal(_codes_np(q), qr)
    np.testing.assert_array_equal(_f32_bits(colmax), _col_absmax_bits(x))
    # the column groups fed by that absmax: the oracle's column quantization
    qc, sc = m.int8mp_quantize_cols_absmax(xd, colmax, mode=mode, seed=seed, offset=off,
                                           stream_id=4, codes=m.INT8MP_CODES_F16)
    qcr, scr = oracle.quantize(bf16_bits(x), axis=1, mode=mode, seed=seed, offset=off, stream_id=4)
    np.testing.assert_array_equal(_f32_bits(sc), scr.view(np.int32))
    np.testing.assert_array_equal(_codes_np(qc), np.ascontiguousarray(qcr.T))


# Two matrices with the same row length in one launch (int8mp_quantize_rows_batch):
# ragged rows, a split of the launch's blocks that is not proportional
# (3 and 300 rows), rows longer than a team's share (5632 columns)
ROWS_BATCH_SHAPES = [((1040, 2048), (264, 2048)), ((77, 136), (9, 136)), ((3, 5632), (300, 5632)),
                     ((16384, 1024), (1024, 1024))]


@pytest.mark.parametrize("with_colmax", [False, True])
@pytest.mark.parametrize("codes", [m.INT8MP_CODES_S8, m.INT8MP_CODES_F16])
@pytest.mark.parametrize("mode", [m.INT8MP_RNE, m.INT8MP_SR])
@pytest.mark.parametrize("shapes", ROWS_BATCH_SHAPES)
def test_rows_batch_matches_the_oracle_per_matrix(shapes, mode, codes, with_colmax):
    (r0, cols), (r1, _) = shapes
    xs = [_edge_input(r0, cols, seed=r0 + 3), _edge_input(r1, cols, seed=r1 + 5)]
    offs, sids, seed = [5, (1 << 33) + 4], [m.INT8MP_STREAM_FWD_X, m.INT8MP_STREAM_FWD_W], 19
    cms = [torch.zeros(cols, dtype=torch.float32, device=DEV) for _ in xs] if with_colmax else None
    got = m.int8mp_quantize_rows_batch([_dev(x) for x in xs], mode=mode, seed=seed, offsets=offs,
                                       stream_ids=sids, codes=codes, colmaxes=cms)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    for i, x in enumerate(xs):
        q, sc = got[i]
        qr, sr = oracle.quantize(bf16_bits(x), axis=0, mode=mode, seed=seed, offset=offs[i],
                                 stream_id=sids[i])
        np.testing.assert_array_equal(_f32_bits(sc), sr.view(np.int32), err_msg=str(i))
        np.testing.assert_array_equal(_codes_np(q), qr, err_msg=str(i))
        if with_colmax:
            np.testing.assert_array_equal(_f32_bits(cms[i]), _col_absmax_bits(x), err_msg=str(i))


# Two matrices' column groups in one launch (int8mp_quantize_cols_batch):
# rows of each size class of the one-launch kernel (a different one per
# matrix), ragged column strips, plain operands and edge rows; a pair with a
# matrix over 2048 rows takes each matrix's passes.
COLS_BATCH_SHAPES = [((1024, 1024), (1024, 1024)), ((77, 136), (2048, 136)),
                     ((2048, 264), (9, 264)), ((3001, 64), (100, 64))]


@pytest.mark.parametrize("codes", [m.INT8MP_CODES_S8, m.INT8MP_CODES_F16])
@pytest.mark.parametrize("mode", [m.INT8MP_RNE, m.INT8MP_SR])
@pytest.mark.parametrize("shapes", COLS_BATCH_SHAPES)
def test_cols_batch_matches_the_oracle_per_matrix(shapes, mode, codes):
    (r0, cols), (r1, _) = shapes
    xs = [synth.bf16_normal((r0, cols), r0 + 7, outlier_frac=0.01, outlier_scale=20.0),
          _edge_input(r1, cols, seed=r1 + 9)]
    offs, sids, seed = [4, (1 << 33) + 1], [m.INT8MP_STREAM_GW_DY, m.INT8MP_STREAM_GW_X], 23
    got = m.int8mp_quantize_cols_batch([_dev(x) for x in xs], mode=mode, seed=seed, offsets=offs,
                                       stream_ids=sids, codes=codes)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    for i, x in enumerate(xs):
        q, sc = got[i]
        qr, sr = oracle.quantize(bf16_bits(x), axis=1, mode=mode, seed=seed, offset=offs[i],
                                 stream_id=sids[i])
        np.testing.assert_array_equal(_f32_bits(sc), sr.view(np.int32), err_msg=str(i))
        np.testing.assert_array_equal(_codes_np(q), np.ascontiguousarray(qr.T), err_msg=str(i))


@pytest.mark.parametrize("mode", [m.INT8MP_RNE, m.INT8MP_SR])
def test_columns_from_absmax_int8_codes(mode):
    rows, cols = 1000, 2056
    x = _edge_input(rows, cols, seed=17)
    xd = _dev(x)
    colmax = torch.zeros(cols, dtype=torch.float32, device=DEV)
    m.int8mp_quantize_rows_colmax(xd, colmax, codes=m.INT8MP_CODES_S8)
    q, s = m.int8mp_quantize_cols_absmax(xd, colmax, mode=mode, seed=5, offset=9, stream_id=4,
                                         codes=m.INT8MP_CODES_S8)
    qr, sr = oracle.quantize(bf16_bits(x), axis=1, mode=mode, seed=5, offset=9, stream_id=4)
    np.testing.assert_array_equal(_f32_bits(s), sr.view(np.int32))
    np.testing.assert_array_equal(_codes_np(q), np.ascontiguousarray(qr.T))


@pytest.mark.parametrize("codes", [m.INT8MP_CODES_S8, m.INT8MP_CODES_F16])
def test_columns_from_a_too_small_absmax_are_clamped(codes):
    # a caller's absmax below the true one: scale = claim / 127 and every
    # code still lies in [-127, 127], equal to the clamped nearest-even code
    rows, cols = 256, 512
    x = synth.bf16_normal((rows, cols), 18)
    xd = _dev(x)
    true_max = xd.float().abs().amax(dim=0)
    claim = (true_max * 0.5).contiguous()
    q, s = m.int8mp_quantize_cols_absmax(xd, claim, codes=codes)
    codes_np = _codes_np(q).astype(np.int64)
    assert np.abs(codes_np).max() == 127
    sc = (claim.cpu().double() / 127).float().double().numpy()      # fp32 scale, as stored
    np.testing.assert_array_equal(_f32_bits(s), (claim.cpu() / 127).numpy().view(np.int32))
    v = bits_to_f32(bf16_bits(x)).astype(np.float64) / sc[None, :]
    far = np.abs(np.abs(v) - np.floor(np.abs(v)) - 0.5) > 1e-3    # away from ties
    expect = np.clip(np.rint(v), -127, 127)
    np.testing.assert_array_equal(codes_np[far], expect[far])


def test_column_absmax_accumulates_over_row_blocks():
    x = _edge_input(640, 2048, seed=91)
    xd = _dev(x)
    colmax = torch.zeros(2048, dtype=torch.float32, device=DEV)
    m.int8mp_quantize_rows_colmax(xd[:320], colmax, codes=m.INT8MP_CODES_S8)
    m.int8mp_quantize_rows_colmax(xd[320:], colmax, codes=m.INT8MP_CODES_S8)
    np.testing.assert_array_equal(_f32_bits(colmax), _col_absmax_bits(x))
    # an initial value above every column's absmax survives (the input's
    # largest entries are about 1e38: its row 5 is scaled by 1e36)
    big = torch.finfo(torch.float32).max
    colmax.fill_(big)
    m.int8mp_quantize_rows_colmax(xd, colmax, codes=m.INT8MP_CODES_S8)
    assert bool((colmax == big).all())


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
    q2, s2 = m.int8mp_quantize_rowwise(view, axis=m.INT8MP_GROUP_COLS, mode=m.INT8MP_SR, seed=8,
                                       codes=m.INT8MP_CODES_F16)
    qr2, sr2 = oracle.quantize(bf16_bits(base[:, :136].contiguous()), axis=1, mode=oracle.SR,
                               seed=8)
    np.testing.assert_array_equal(_codes_np(q2), np.ascontiguousarray(qr2.T))
    np.testing.assert_array_equal(_f32_bits(s2), sr2.view(np.int32))


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


# M-major / N-major operands: A stored [K,M] (A.T @ B), B stored [K,N] (A @ B
# and A.T @ B).  Shapes reach the single-CTA kernel (M <= 128, or few tiles)
# and the CTA-pair kernel (>= 76 pair tiles, or K >= 8192), ragged M and N.
LAYOUT_MM_SHAPES = [(128, 256, 512), (200, 264, 144), (64, 776, 1040), (2560, 2048, 128),
                    (256, 264, 8192), (1000, 520, 2096)]


@pytest.mark.parametrize("layout", [m.INT8MP_AxB, m.INT8MP_ATxB])
@pytest.mark.parametrize("shape", LAYOUT_MM_SHAPES)
def test_mm_s32_mn_major_layouts_bit_exact(shape, layout):
    M, N, K = shape
    a = _rand_codes(M, K, 5) if layout == m.INT8MP_AxB else _rand_codes(K, M, 5)
    b = _rand_codes(K, N, 6)
    acc = m.int8mp_mm_s32(_dev(a.half()), _dev(b.half()), layout=layout)
    ref = oracle.mm_s32(a.numpy(), b.numpy(), M, N, K, layout=layout)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref)


@pytest.mark.parametrize("layout", [m.INT8MP_AxB, m.INT8MP_ATxB])
def test_mm_s32_mn_major_large_sums_exact(layout):
    M, N, K = 256, 256, 8192
    a = _rand_codes(M, K, 7, extreme=True)
    b = _rand_codes(N, K, 8, extreme=True)
    b[0] = a[0]
    b[1] = -a[1]
    a_st = a if layout == m.INT8MP_AxB else a.T.contiguous()
    b_st = b.T.contiguous()
    acc = m.int8mp_mm_s32(_dev(a_st.half()), _dev(b_st.half()), layout=layout).cpu().numpy()
    assert acc[0, 0] == 127 * 127 * K and acc[1, 1] == -127 * 127 * K
    np.testing.assert_array_equal(acc, oracle.mm_s32(a.numpy(), b.numpy(), M, N, K))


@pytest.mark.parametrize("layout", [m.INT8MP_AxBT, m.INT8MP_ATxB])
def test_mm_s32_at_the_int32_limit_of_k(layout):
    # K = 133,136, the largest multiple of 16 within the API's bound: with
    # every code +-127, sums reach 127^2 K = 2,147,350,544, 133,104 below
    # 2^31; 131 exact fp32 chunks per output, on the CTA-pair kernel
    M, N, K = 256, 256, 133136
    assert K <= m.INT8MP_MAX_K < K + 16
    a = _rand_codes(M, K, 61, extreme=True)
    b = _rand_codes(N, K, 62, extreme=True)
    b[0] = a[0]
    b[1] = -a[1]
    a_st = a if layout == m.INT8MP_AxBT else a.T.contiguous()
    b_st = b if layout == m.INT8MP_AxBT else b.T.contiguous()
    acc = m.int8mp_mm_s32(_dev(a_st.half()), _dev(b_st.half()), layout=layout).cpu().numpy()
    assert acc[0, 0] == 127 * 127 * K and acc[1, 1] == -127 * 127 * K
    np.testing.assert_array_equal(acc, oracle.mm_s32(a.numpy(), b.numpy(), M, N, K))


# Split last wave: with a workspace, the CTA-pair kernel splits the R tiles
# of a partial last wave into s = min(pairs / R, 4) k-parts each, added as
# int32 totals: one tile of K = 8192, 80 tiles (4 left over: 4 parts of 16
# to 33 k-blocks), 90 tiles (14 left, 4 parts), 12 tiles (4 parts); 64
# tiles on 76 pairs are left whole.
SPLIT_TAIL_SHAPES = [(256, 256, 8192, m.INT8MP_AxBT), (2048, 2048, 8192, m.INT8MP_AxBT),
                  (2560, 2048, 4096, m.INT8MP_AxBT), (2312, 2056, 8192, m.INT8MP_AxB),
                  (2312, 1800, 8256, m.INT8MP_ATxB), (768, 776, 16384, m.INT8MP_ATxB)]


def _stored(codes, layout, which, M, N, K, seed):
    """Random codes for operand `which` stored as `layout` wants."""
    if which == "A":
        return _rand_codes(K, M, seed) if layout == m.INT8MP_ATxB else _rand_codes(M, K, seed)
    return _rand_codes(N, K, seed) if layout == m.INT8MP_AxBT else _rand_codes(K, N, seed)


# Shapes that take each tile width of the single-CTA GEMM (on 152 SMs): 128 x
# 256 when its tiles fill half of the SMs or more, else 128 x 128, else
# 128 x 64 (the CTA-pair kernel takes neither: fewer than 76 pair tiles and
# K < 8192).  Every width in every layout and output mode.
SINGLE_TILE_SHAPES = [(2048, 2048, 256),    # 128 tiles of 128 x 256
                      (1024, 1280, 1040),   # 80 tiles of 128 x 128 (40 of 128 x 256)
                      (512, 528, 1040)]     # 36 tiles of 128 x 64 (20 of 128 x 128)


@pytest.mark.parametrize("layout", [m.INT8MP_AxBT, m.INT8MP_AxB, m.INT8MP_ATxB])
@pytest.mark.parametrize("shape", SINGLE_TILE_SHAPES)
def test_single_cta_tile_widths_all_outputs(shape, layout):
    M, N, K = shape
    a = _stored(None, layout, "A", M, N, K, 31)
    b = _stored(None, layout, "B", M, N, K, 32)
    g = torch.Generator().manual_seed(33)
    sa = (torch.rand(M, generator=g) * 2.0 ** -6).float()
    sb = (torch.rand(N, generator=g) * 2.0 ** -3).float()
    ad, bd = _dev(a.half()), _dev(b.half())
    acc = m.int8mp_mm_s32(ad, bd, layout=layout)
    y = m.int8mp_scaled_mm(ad, _dev(sa), bd, _dev(sb), layout=layout)
    y32 = m.int8mp_scaled_mm_f32(ad, _dev(sa), bd, _dev(sb), layout=layout)
    torch.cuda.synchronize()
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    an, bn = a.numpy(), b.numpy()
    np.testing.assert_array_equal(acc.cpu().numpy(), oracle.mm_s32(an, bn, M, N, K, layout=layout))
    assert_bf16_equal(y, oracle.scaled_mm(an, sa.numpy(), bn, sb.numpy(), M, N, K, layout=layout),
                      "scaled_mm")
    np.testing.assert_array_equal(
        y32.cpu().numpy().view(np.int32),
        oracle.scaled_mm_f32(an, sa.numpy(), bn, sb.numpy(), M, N, K, layout=layout).view(np.int32))


@pytest.mark.parametrize("shape", SINGLE_TILE_SHAPES)
def test_single_cta_tile_widths_bf16_pass(shape):
    # the plain-bf16 mode of the same kernels: the forward matmul of a linear
    # layer with its pass in BF16
    T, N, K = shape
    X = synth.bf16_normal((T, K), 41)
    W = synth.bf16_normal((N, K), 42, std=0.02)
    Y = m.int8mp_linear_fwd(_dev(X), _dev(W), cfg=m.linear_cfg(int8_fwd=0))
    torch.cuda.synchronize()
    ref = oracle.matmul_bf16(bf16_bits(X), bf16_bits(W), T, N, K)
    _bf16_pass_close(Y, ref, X.float(), W.float(), "BF16 forward")


@pytest.mark.parametrize("shape", SPLIT_TAIL_SHAPES)
def test_mm_s32_split_tail_bit_exact(shape):
    M, N, K, layout = shape
    a = _stored(None, layout, "A", M, N, K, 21)
    b = _stored(None, layout, "B", M, N, K, 22)
    ad, bd = _dev(a.half()), _dev(b.half())
    ws = torch.empty(m.int8mp_mm_workspace_size(), dtype=torch.uint8, device=DEV)
    acc = m.int8mp_mm_s32(ad, bd, layout=layout, workspace=ws)
    acc2 = m.int8mp_mm_s32(ad, bd, layout=layout, workspace=ws)  # the scratch is reusable as is
    plain = m.int8mp_mm_s32(ad, bd, layout=layout)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    assert torch.equal(acc, acc2) and torch.equal(acc, plain)
    ref = oracle.mm_s32(a.numpy(), b.numpy(), M, N, K, layout=layout)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref)


def test_mm_s32_split_tail_extreme_sums():
    # +-127 everywhere with K = 16384, 4 tiles split 4 ways: every part and
    # the total stay exact
    M, N, K = 512, 512, 16384
    a = _rand_codes(M, K, 23, extreme=True)
    b = _rand_codes(N, K, 24, extreme=True)
    b[0] = a[0]
    b[300] = -a[300]
    acc = m.int8mp_mm_s32(_dev(a.half()), _dev(b.half()), workspace=True).cpu().numpy()
    assert acc[0, 0] == 127 * 127 * K and acc[300, 300] == -127 * 127 * K
    np.testing.assert_array_equal(acc, oracle.mm_s32(a.numpy(), b.numpy(), M, N, K))


def test_scaled_mm_split_tail_bit_exact():
    M, N, K = 2048, 2312, 4096
    A = synth.bf16_normal((M, K), 31, outlier_frac=0.01, outlier_scale=20.0)
    B = synth.bf16_normal((N, K), 32, outlier_frac=0.01, outlier_scale=20.0)
    qa, sa = m.int8mp_quantize_rowwise(_dev(A), axis=0, codes=m.INT8MP_CODES_F16)
    qb, sb = m.int8mp_quantize_rowwise(_dev(B), axis=0, codes=m.INT8MP_CODES_F16)
    out = m.int8mp_scaled_mm(qa, sa, qb, sb, workspace=True)
    plain = m.int8mp_scaled_mm(qa, sa, qb, sb)
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))
    qar, sar = oracle.quantize(bf16_bits(A), axis=0)
    qbr, sbr = oracle.quantize(bf16_bits(B), axis=0)
    ref = oracle.scaled_mm(qar, sar, qbr, sbr, M, N, K)
    assert_bf16_equal(out, ref, "scaled_mm split tail")


def test_split_tail_gemm_replays_in_a_cuda_graph():
    # a captured launch keeps its counter epoch; the last part of each split
    # tile clears its counter, so every replay finalizes every tile
    M, N, K = 2048, 2312, 4096            # 80 tiles: 4 split 4 ways on 76 SM pairs
    g = torch.Generator().manual_seed(40)
    a = torch.empty((M, K), dtype=torch.float16, device=DEV)
    b = torch.empty((N, K), dtype=torch.float16, device=DEV)
    sa = torch.rand(M, generator=g).to(DEV)
    sb = torch.rand(N, generator=g).to(DEV)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    acc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    ws = torch.empty(m.int8mp_mm_workspace_size(), dtype=torch.uint8, device=DEV)

    def refill():
        a.copy_(_rand_codes(M, K, int(torch.randint(0, 1 << 30, (1,), generator=g))).half())
        b.copy_(_rand_codes(N, K, int(torch.randint(0, 1 << 30, (1,), generator=g))).half())

    refill()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # first calls outside the capture
        m.int8mp_scaled_mm(a, sa, b, sb, out=out, workspace=ws)
        m.int8mp_mm_s32(a, b, out=acc, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        m.int8mp_scaled_mm(a, sa, b, sb, out=out, workspace=ws)
        m.int8mp_mm_s32(a, b, out=acc, workspace=ws)
    for _ in range(3):
        refill()
        graph.replay()
        ref_out = m.int8mp_scaled_mm(a, sa, b, sb)
        ref_acc = m.int8mp_mm_s32(a, b)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(acc, ref_acc)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    rows = np.array([0, 1000, 2047])
    ref = oracle.mm_s32(a.cpu().to(torch.int8).numpy()[rows], b.cpu().to(torch.int8).numpy(),
                        len(rows), N, K)
    np.testing.assert_array_equal(acc.cpu().numpy()[rows], ref)


def test_linear_layer_replays_in_a_cuda_graph():
    # forward with saved absmax and backward, captured once and replayed on
    # fresh inputs: the absmax zeroing, the dependent launches and the split
    # last wave (80 tiles of grad input) must give the eager calls' results
    # (which the other tests hold to the oracle) bit for bit each time
    T, N, K = 2560, 2048, 2048
    cfg = m.linear_cfg(mode=m.INT8MP_SR, seed=5, offset=3)
    X = torch.empty((T, K), dtype=torch.bfloat16, device=DEV)
    W = torch.empty((N, K), dtype=torch.bfloat16, device=DEV)
    dY = torch.empty((T, N), dtype=torch.bfloat16, device=DEV)
    Y = torch.empty((T, N), dtype=torch.bfloat16, device=DEV)
    dX = torch.empty((T, K), dtype=torch.bfloat16, device=DEV)
    dW = torch.empty((N, K), dtype=torch.bfloat16, device=DEV)
    absmax = torch.empty(2 * K, dtype=torch.float32, device=DEV)
    ws = torch.empty(m.int8mp_linear_workspace_size(T, N, K, cfg), dtype=torch.uint8, device=DEV)

    def step():
        m.int8mp_linear_fwd_save(X, W, absmax, cfg, Y=Y, workspace=ws)
        m.int8mp_linear_bwd_saved(dY, X, W, absmax, cfg, dX=dX, dW=dW, workspace=ws)

    def refill(i):
        X.copy_(synth.bf16_normal((T, K), 70 + i))
        W.copy_(synth.bf16_normal((N, K), 80 + i, std=0.02))
        dY.copy_(synth.bf16_normal((T, N), 90 + i, std=1e-3))

    refill(0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for i in range(1, 4):
        refill(i)
        graph.replay()
        got = [t.clone() for t in (Y, dX, dW)]
        step()
        torch.cuda.synchronize()
        for g_, e_ in zip(got, (Y, dX, dW)):
            assert torch.equal(g_.view(torch.int16), e_.view(torch.int16)), i
    assert m.int8mp_poll_device_status() == m.INT8MP_OK


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


@pytest.mark.parametrize("s32", [False, True])
@pytest.mark.parametrize("M", [2600, 8200])
def test_pair_gemm_writes_only_its_strided_output(s32, M):
    # CTA-pair kernel, ragged M and N: the tile stores must land at row
    # stride ldo and column offset 8 of a larger buffer, clip at row M and
    # column N, and leave every other element as it was; sB at a 4-byte (not
    # 16-byte) aligned address.  M = 2600: 99 tiles, at most two per SM pair
    # (scales loaded when a tile starts); M = 8200: 297 tiles (scales loaded
    # by the store, scalar loads for the misaligned sB)
    N, K, ldo = 2056, 144, 2088
    a, b = _rand_codes(M, K, 41), _rand_codes(N, K, 42)
    ad, bd = _dev(a.half()), _dev(b.half())
    g = torch.Generator().manual_seed(43)
    sa = torch.rand(M, generator=g) + 0.5
    sb_store = torch.rand(N + 1, generator=g) + 0.5
    dtype = torch.int32 if s32 else torch.bfloat16
    big = torch.full((M + 3, ldo), -7, dtype=torch.int32).to(dtype).to(DEV)
    sentinel = big.clone()
    view = big[1:M + 1, 8:8 + N]
    if s32:
        m.int8mp_mm_s32(ad, bd, out=view)
    else:
        m.int8mp_scaled_mm(ad, _dev(sa), bd, _dev(sb_store)[1:], out=view)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    outside = torch.ones(big.shape, dtype=torch.bool)
    outside[1:M + 1, 8:8 + N] = False
    assert torch.equal(big.cpu()[outside], sentinel.cpu()[outside])
    rows = np.r_[0:40, M // 2 - 7:M // 2 + 9, M - 40:M]  # first, middle and ragged last tiles
    got = view.cpu()[torch.from_numpy(rows)]
    an = a.numpy()[rows]
    if s32:
        np.testing.assert_array_equal(got.numpy(), oracle.mm_s32(an, b.numpy(), len(rows), N, K))
    else:
        ref = oracle.scaled_mm(an, sa.numpy()[rows], b.numpy(), sb_store[1:].numpy(), len(rows), N, K)
        assert_bf16_equal(got, ref, "scaled_mm into a strided output")


def test_matmul_rejects_an_output_with_strided_columns():
    a = _dev(_rand_codes(256, 64, 44).half())
    out = torch.empty((256, 512), dtype=torch.int32, device=DEV)[:, ::2]
    with pytest.raises(ValueError):
        m.int8mp_mm_s32(a, a, out=out)


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


@pytest.mark.parametrize("layout", ["AxB", "ATxB"])
@pytest.mark.parametrize("S", [256, 2560])
def test_square_layouts_with_column_codes_in_place(layout, S):
    # the K-first operand quantized by columns with its codes left in place,
    # multiplied in the stored layout (no transposition anywhere)
    A, B = synth.square_inputs(S, layout)
    a_axis = m.INT8MP_GROUP_COLS if layout == "ATxB" else m.INT8MP_GROUP_ROWS
    qa, sa = m.int8mp_quantize_rowwise(_dev(A), axis=a_axis, codes=m.INT8MP_CODES_F16)
    qb, sb = m.int8mp_quantize_rowwise(_dev(B), axis=m.INT8MP_GROUP_COLS, codes=m.INT8MP_CODES_F16)
    lay = {"AxB": m.INT8MP_AxB, "ATxB": m.INT8MP_ATxB}[layout]
    out = m.int8mp_scaled_mm(qa, sa, qb, sb, layout=lay)
    qar, sar = oracle.quantize(bf16_bits(A), axis=1 if layout == "ATxB" else 0)
    qbr, sbr = oracle.quantize(bf16_bits(B), axis=1)
    qa_st = qar if layout == "AxB" else np.ascontiguousarray(qar.T)
    qb_st = np.ascontiguousarray(qbr.T)
    if S == 256:
        ref = oracle.scaled_mm(qa_st, sar, qb_st, sbr, S, S, S, layout=lay)
        assert_bf16_equal(out, ref, f"square {layout}")
    else:
        # sampled output rows: each is exact on its own
        rows = np.random.default_rng(S).choice(S, 8, replace=False)
        acc = oracle.mm_s32(np.ascontiguousarray(qar[rows]), qbr, 8, S, S)
        ref = oracle.rescale_bf16(acc, sar[rows], sbr)
        assert_bf16_equal(out[torch.from_numpy(rows).to(DEV)], ref, f"square {layout} rows")


@pytest.mark.parametrize("layout", ["AxBT", "AxB", "ATxB"])
@pytest.mark.parametrize("S", [1024, 2048])
def test_square_sweep_sizes(layout, S):
    # the square quant+scaled-mm configuration at 1024 and 2048 (4096 is in
    # the full-size tests), run as the benchmark runs it: K-first operands
    # quantized by columns in place, the matmul in the stored layout, with
    # the split-last-wave workspace
    A, B = synth.square_inputs(S, layout)
    a_cols, b_cols = layout == "ATxB", layout != "AxBT"
    ax = lambda cols: m.INT8MP_GROUP_COLS if cols else m.INT8MP_GROUP_ROWS
    lay = {"AxBT": m.INT8MP_AxBT, "AxB": m.INT8MP_AxB, "ATxB": m.INT8MP_ATxB}[layout]
    qa, sa = m.int8mp_quantize_rowwise(_dev(A), axis=ax(a_cols), codes=m.INT8MP_CODES_F16)
    qb, sb = m.int8mp_quantize_rowwise(_dev(B), axis=ax(b_cols), codes=m.INT8MP_CODES_F16)
    out = m.int8mp_scaled_mm(qa, sa, qb, sb, layout=lay, workspace=True)
    qar, sar = oracle.quantize(bf16_bits(A), axis=1 if a_cols else 0)
    qbr, sbr = oracle.quantize(bf16_bits(B), axis=1 if b_cols else 0)
    rows = np.random.default_rng(S + len(layout)).choice(S, 16, replace=False)
    ref = oracle.scaled_mm(np.ascontiguousarray(qar[rows]), sar[rows], qbr, sbr, len(rows), S, S)
    assert_bf16_equal(out[torch.from_numpy(rows).to(DEV)], ref, f"square {S} {layout}")


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


@pytest.mark.parametrize("flags", [(1, 1, 1), (1, 0, 1), (1, 1, 0), (0, 1, 1)])
@pytest.mark.parametrize("shape", [(256, 256, 512), (1040, 64, 48), (48, 5632, 2048)])
def test_linear_with_saved_absmax_matches_plain_passes(shape, flags):
    T, N, K = shape
    X = synth.bf16_normal((T, K), 14, outlier_frac=0.005, outlier_scale=30.0)
    W = synth.bf16_normal((N, K), 24, std=0.02)
    dY = synth.bf16_normal((T, N), 34, std=1e-3)
    f, gi, gw = flags
    cfg = m.linear_cfg(mode=m.INT8MP_SR, seed=9, offset=3, int8_fwd=f, int8_grad_in=gi,
                       int8_grad_w=gw)
    Xd, Wd, dYd = _dev(X), _dev(W), _dev(dY)
    absmax = torch.full((2 * K,), -1.0, dtype=torch.float32, device=DEV)  # overwritten
    Y1 = m.int8mp_linear_fwd_save(Xd, Wd, absmax, cfg)
    dX1, dW1 = m.int8mp_linear_bwd_saved(dYd, Xd, Wd, absmax, cfg)
    Y0 = m.int8mp_linear_fwd(Xd, Wd, cfg)
    dX0, dW0 = m.int8mp_linear_bwd(dYd, Xd, Wd, cfg)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    zero = np.zeros(K, dtype=np.int32)
    np.testing.assert_array_equal(_f32_bits(absmax[:K]), _col_absmax_bits(X) if gw else zero)
    np.testing.assert_array_equal(_f32_bits(absmax[K:]), _col_absmax_bits(W) if gi else zero)
    for a, b, what in ((Y1, Y0, "Y"), (dX1, dX0, "dX"), (dW1, dW0, "dW")):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), what
    if f and gi and gw:
        Yr = oracle.linear_fwd(bf16_bits(X), bf16_bits(W), mode=oracle.SR, seed=9, offset=3)
        dXr, dWr = oracle.linear_bwd(bf16_bits(dY), bf16_bits(X), bf16_bits(W), mode=oracle.SR,
                                     seed=9, offset=3)
        assert_bf16_equal(Y1, Yr, "saved forward")
        assert_bf16_equal(dX1, dXr, "saved grad input")
        assert_bf16_equal(dW1, dWr, "saved grad weight")


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
    """BF16 pass: the tensor core accumulates in fp32 in its own order, the
    oracle in fp64 (helpers.bf16_pass_close gives the bound)."""
    bf16_pass_close(got_t, ref_bits, a, b, what)


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
