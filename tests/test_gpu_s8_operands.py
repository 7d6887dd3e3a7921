"""The matmul on int8 codes (INT8MP_CODES_S8).

"Integrate INT8 mixed-precision from torchao 0.7", discussion: weights and
activations are quantized dynamically to INT8 so that the matmul runs on
INT8 operands.  int8mp_scaled_mm / int8mp_mm_s32 (and their _ws forms) take
`const int8_t*` codes as the quantizer writes them by default; the CTA-pair
kernel brings the int8 tiles in with TMA and widens them to f16 in shared
memory before the tensor core reads them.

Every result is compared with the oracle (the int32 product is pinned to
int64 brute force on the CPU) bit for bit, and with the same matmul on f16
containers of the same codes: ragged M and N, contractions that cross the
1024-term chunks, all three layouts, sums far above 2^24 and at the int32
limit of K, the split last wave, and codes from the quantizer itself.
"""
import numpy as np
import pytest
import torch

import int8_mixed_precision_row_gb300 as m
import oracle
from helpers import bf16_bits
from int8_mixed_precision_row_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int8_mixed_precision_row_gb300 import build
    build.build()
    m.load()


def _rand_codes(rows, cols, seed, extreme=False):
    g = torch.Generator().manual_seed(seed)
    if extreme:
        sign = torch.randint(0, 2, (rows, cols), generator=g) * 2 - 1
        return (sign * 127).to(torch.int8)
    return torch.randint(-127, 128, (rows, cols), generator=g, dtype=torch.int32).to(torch.int8)


def _operands(layout, M, N, K, seed, extreme=False):
    """Codes as `layout` stores them, and the K-major [M,K] / [N,K] views
    the oracle takes."""
    a = _rand_codes(M, K, seed, extreme)
    b = _rand_codes(N, K, seed + 1, extreme)
    a_st = a.T.contiguous() if layout == m.INT8MP_ATxB else a
    b_st = b if layout == m.INT8MP_AxBT else b.T.contiguous()
    return a, b, a_st, b_st


# (M, N, K): ragged M and N (multiples of 16 where an int8 operand is stored
# [K, M] or [K, N]), K from one k-block to several exact chunks, few tiles and
# more than a wave of 76 CTA pairs
S8_SHAPES = [(256, 256, 512), (16, 16, 16), (112, 48, 1040), (208, 272, 144),
             (1008, 784, 2096), (2560, 2048, 128), (256, 512, 3072)]
LAYOUTS = [m.INT8MP_AxBT, m.INT8MP_AxB, m.INT8MP_ATxB]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape", S8_SHAPES)
def test_mm_s32_int8_operands_bit_exact(shape, layout):
    M, N, K = shape
    a, b, a_st, b_st = _operands(layout, M, N, K, 100 + M + K)
    ad, bd = a_st.to(DEV), b_st.to(DEV)
    acc = m.int8mp_mm_s32(ad, bd, layout=layout)
    assert acc.dtype == torch.int32
    via_f16 = m.int8mp_mm_s32(ad.half(), bd.half(), layout=layout)
    torch.cuda.synchronize()
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    ref = oracle.mm_s32(a.numpy(), b.numpy(), M, N, K)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref)
    assert torch.equal(acc, via_f16)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_mm_s32_int8_operands_large_sums(layout):
    # +-127 everywhere, K = 8192: partial sums far above 2^24 stay exact
    M, N, K = 256, 256, 8192
    a, b, _, _ = _operands(layout, M, N, K, 7, extreme=True)
    b[0] = a[0]
    b[1] = -a[1]
    a_st = a.T.contiguous() if layout == m.INT8MP_ATxB else a
    b_st = b if layout == m.INT8MP_AxBT else b.T.contiguous()
    acc = m.int8mp_mm_s32(a_st.to(DEV), b_st.to(DEV), layout=layout).cpu().numpy()
    assert acc[0, 0] == 127 * 127 * K and acc[1, 1] == -127 * 127 * K
    np.testing.assert_array_equal(acc, oracle.mm_s32(a.numpy(), b.numpy(), M, N, K))


def test_mm_s32_int8_operands_at_the_int32_limit_of_k():
    # K = 133,136: 127^2 K = 2,147,350,544, 133,104 below 2^31
    M, N, K = 256, 256, 133136
    a = _rand_codes(M, K, 61, extreme=True)
    b = _rand_codes(N, K, 62, extreme=True)
    b[0] = a[0]
    b[1] = -a[1]
    acc = m.int8mp_mm_s32(a.to(DEV), b.to(DEV)).cpu().numpy()
    assert acc[0, 0] == 127 * 127 * K and acc[1, 1] == -127 * 127 * K
    np.testing.assert_array_equal(acc, oracle.mm_s32(a.numpy(), b.numpy(), M, N, K))


# the split last wave: 80 tiles (4 split 4 ways), 90 tiles (14 split), 4 tiles
S8_SPLIT_SHAPES = [(2048, 2048, 8192, m.INT8MP_AxBT), (2304, 2064, 8192, m.INT8MP_AxB),
                   (2320, 1808, 8256, m.INT8MP_ATxB), (512, 512, 16384, m.INT8MP_ATxB)]


@pytest.mark.parametrize("shape", S8_SPLIT_SHAPES)
def test_mm_s32_int8_operands_split_tail(shape):
    M, N, K, layout = shape
    a, b, a_st, b_st = _operands(layout, M, N, K, 21)
    ad, bd = a_st.to(DEV), b_st.to(DEV)
    ws = torch.empty(m.int8mp_mm_workspace_size(), dtype=torch.uint8, device=DEV)
    acc = m.int8mp_mm_s32(ad, bd, layout=layout, workspace=ws)
    plain = m.int8mp_mm_s32(ad, bd, layout=layout)
    assert m.int8mp_poll_device_status() == m.INT8MP_OK
    assert torch.equal(acc, plain)
    np.testing.assert_array_equal(acc.cpu().numpy(),
                                  oracle.mm_s32(a.numpy(), b.numpy(), M, N, K))


@pytest.mark.parametrize("layout", ["AxBT", "AxB", "ATxB"])
@pytest.mark.parametrize("S", [256, 1040, 2560])
def test_scaled_mm_on_quantizer_int8_codes(layout, S):
    """The square problem of the README's matmul tables with the
    quantizer's own int8 codes: operands stored K-first quantized by columns
    with their codes left in place."""
    A, B = synth.square_inputs(S, layout)
    a_cols = layout == "ATxB"
    b_cols = layout != "AxBT"
    ax = lambda cols: m.INT8MP_GROUP_COLS if cols else m.INT8MP_GROUP_ROWS
    lay = {"AxBT": m.INT8MP_AxBT, "AxB": m.INT8MP_AxB, "ATxB": m.INT8MP_ATxB}[layout]
    qa, sa = m.int8mp_quantize_rowwise(A.to(DEV), axis=ax(a_cols), codes=m.INT8MP_CODES_S8)
    qb, sb = m.int8mp_quantize_rowwise(B.to(DEV), axis=ax(b_cols), codes=m.INT8MP_CODES_S8)
    assert qa.dtype == torch.int8
    out = m.int8mp_scaled_mm(qa, sa, qb, sb, layout=lay, workspace=True)
    via_f16 = m.int8mp_scaled_mm(qa.half(), sa, qb.half(), sb, layout=lay)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), via_f16.view(torch.int16))
    qar, sar = oracle.quantize(bf16_bits(A), axis=1 if a_cols else 0)   # K-major codes
    qbr, sbr = oracle.quantize(bf16_bits(B), axis=1 if b_cols else 0)
    rows = np.unique(np.linspace(0, S - 1, 9).astype(np.int64))
    ref = oracle.scaled_mm(qar[rows], sar[rows], qbr, sbr, len(rows), S, S)
    got = bf16_bits(out[torch.from_numpy(rows).to(DEV)].cpu())
    np.testing.assert_array_equal(got, ref)
