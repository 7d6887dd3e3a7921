"""Pins of the oracle's quantizer against what the pages and arithmetic fix.

Method: "Quantized model training" README, section "INT8 mixed precision
training" (dynamic row-wise quantization); quantizer x_q = clamp(x / scale +
zp) from "Add QAT support for distributed finetuning", summary (zp = 0).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from helpers import (bf16_bits, bits_to_f32, f32_to_bf16_bits_exact, read_golden, rn_f32,
                     round_half_even_int)
from int8_mixed_precision_row_gb300 import synth


def test_golden_4x8_rows_and_columns():
    g = read_golden("quantize_4x8.txt")
    x = f32_to_bf16_bits_exact(g["x"].astype(np.float32))
    q, s = oracle.quantize(x, axis=0)
    np.testing.assert_array_equal(s, g["scale"].reshape(-1).astype(np.float32))
    np.testing.assert_array_equal(q, g["q"].astype(np.int8))
    # the same groups as columns of the transposed matrix; codes come out
    # transposed, i.e. identical to the row-wise codes above
    qt, st = oracle.quantize(np.ascontiguousarray(x.T), axis=1)
    np.testing.assert_array_equal(st, s)
    np.testing.assert_array_equal(qt, q)


def _edge_matrix(rows, cols, seed):
    x = synth.bf16_normal((rows, cols), seed).float()
    x[1] = 0.0                                  # all-zero group
    x[2] = -x[2].abs() * 3.0                    # absmax attained by a negative value
    x[3] = x[3] * 1e-38                         # subnormal-range values and scale
    x[4, :] = 0.0
    x[4, 5] = 1e-40                             # one subnormal, rest zero
    x[5] = x[5] * 3e37                          # near the top of the range
    x[6, 0] = 127.0
    x[6, 1:] = torch.arange(1, cols) * 0.5 - 40  # many exact ties
    return bf16_bits(x.to(torch.bfloat16))


def _exact_rne_codes(xf, s):
    """Expected codes from the definition: v = RN_f32(x / s) computed in
    exact rationals, then the nearest integer (ties to even), clamped."""
    out = []
    for xv in xf:
        if s == 0:
            out.append(0)
            continue
        v = rn_f32(Fraction(float(xv)) / Fraction(float(s)))
        out.append(max(-127, min(127, round_half_even_int(v))))
    return np.array(out, dtype=np.int8)


@pytest.mark.parametrize("axis", [0, 1])
def test_rne_matches_exact_rational_definition(axis):
    x = _edge_matrix(8, 24, seed=3)
    q, s = oracle.quantize(x, axis=axis)
    xf = bits_to_f32(x)
    groups = xf if axis == 0 else xf.T
    for g in range(groups.shape[0]):
        amax = float(np.max(np.abs(groups[g])))
        # the scale is the correctly rounded absmax / 127
        assert Fraction(float(s[g])) == rn_f32(Fraction(amax) / 127), g
        np.testing.assert_array_equal(q[g], _exact_rne_codes(groups[g], s[g]), err_msg=f"group {g}")


def test_ld_larger_than_cols_is_ignored_padding():
    x = _edge_matrix(8, 32, seed=5)
    q_ref, s_ref = oracle.quantize(x[:, :24], axis=0)
    q, s = oracle.quantize(x, axis=0, cols=24)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(s, s_ref)


@pytest.mark.parametrize("shape,frac,scale", [((64, 512), 0.0, 1.0), ((48, 256), 0.01, 20.0),
                                              ((32, 2048), 0.005, 30.0)])
@pytest.mark.parametrize("axis", [0, 1])
def test_rne_invariants(shape, frac, scale, axis):
    x = bf16_bits(synth.bf16_normal(shape, 11, outlier_frac=frac, outlier_scale=scale))
    q, s = oracle.quantize(x, axis=axis)
    xf = bits_to_f32(x).astype(np.float64)
    groups = xf if axis == 0 else xf.T
    assert q.min() >= -127 and q.max() <= 127
    for g in range(groups.shape[0]):
        if s[g] == 0:
            assert np.all(q[g] == 0)
            continue
        assert np.max(np.abs(q[g].astype(np.int32))) == 127  # the absmax element maps to +-127
        err = np.abs(groups[g] - q[g].astype(np.float64) * float(s[g]))
        # |x - q s| <= s (1/2 + 2^-17): rounding of x/s (v < 128) plus half a code
        assert np.all(err <= float(s[g]) * (0.5 + 2.0 ** -17))


def test_sr_brackets_and_changes_with_seed_offset_stream():
    x = bf16_bits(synth.bf16_normal((16, 256), 4))
    qr, s = oracle.quantize(x, axis=0)
    xf = bits_to_f32(x)
    seen = []
    for seed, off, sid in [(0, 0, 0), (1, 0, 0), (0, 4, 0), (0, 0, 1), (2**64 - 1, 2**40, 5)]:
        q, s2 = oracle.quantize(x, axis=0, mode=oracle.SR, seed=seed, offset=off, stream_id=sid)
        np.testing.assert_array_equal(s2, s)
        v = (xf / s[:, None]).astype(np.float32)
        lo = np.floor(v)
        assert np.all((q == lo) | (q == lo + 1) | (np.abs(q) == 127))
        assert np.all(np.abs(xf - q * s[:, None]) < s[:, None] * (1 + 2.0 ** -16))
        seen.append(q)
    for a in range(len(seen)):
        for b in range(a + 1, len(seen)):
            assert not np.array_equal(seen[a], seen[b])


def test_sr_offset_shifts_the_stream_by_elements():
    # n = offset + index: element e under offset o draws what element e+1
    # draws under offset o-1; check with a row whose values are all equal
    row = np.full((1, 64), 0x3F90, dtype=np.uint16)  # 1.125
    row[0, 0] = 0x42FE                               # 127 -> scale 1, v = 1.125
    q_a, _ = oracle.quantize(row, axis=0, mode=oracle.SR, seed=9, offset=8)
    q_b, _ = oracle.quantize(row, axis=0, mode=oracle.SR, seed=9, offset=7)
    np.testing.assert_array_equal(q_a[0, 1:-1], q_b[0, 2:])


def test_sr_is_unbiased():
    # E[q s] = x: average over many seeds; tolerance 4.5 standard errors
    x = bf16_bits(synth.bf16_normal((2, 64), 8))
    _, s = oracle.quantize(x, axis=0)
    xf = bits_to_f32(x).astype(np.float64)
    n = 3000
    acc = np.zeros_like(xf)
    for seed in range(n):
        q, _ = oracle.quantize(x, axis=0, mode=oracle.SR, seed=seed)
        acc += q.astype(np.float64)
    mean = acc / n * s[:, None]
    v = xf / s[:, None]
    p = v - np.floor(v)
    sd = np.sqrt(p * (1 - p)) * s[:, None] / np.sqrt(n)
    assert np.all(np.abs(mean - xf) <= 4.5 * sd + 1e-7 * s[:, None])
    # rounding nearest would be biased on this data; SR must not be
    qr, _ = oracle.quantize(x, axis=0)
    assert np.abs((qr * s[:, None] - xf)).mean() > np.abs(mean - xf).mean()


def test_sr_exact_values_are_never_moved():
    # integer x/s: fractional part 0, so u < 0 never holds and q = x/s
    vals = np.array([[127, -3, 5, 0, 64, -127, 1, 2]], dtype=np.float32)
    x = f32_to_bf16_bits_exact(vals)
    for seed in range(50):
        q, s = oracle.quantize(x, axis=0, mode=oracle.SR, seed=seed)
        np.testing.assert_array_equal(q, vals.astype(np.int8))


def test_invalid_arguments_are_rejected():
    x = np.zeros((4, 8), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.quantize(x, axis=2)
    with pytest.raises(ValueError):
        oracle.quantize(x, axis=0, mode=7)


# x = absmax / 2 lands exactly on the tie 63.5 in exact arithmetic; with
# s = RN(absmax / 127) the quotient x / s rounds to 63.5 or just below it,
# and multiplying by RN(1 / s) instead of dividing lands on the other side
# for every pair below (found by a search over bf16 values).
DIVISION_TIES = [(2.734375, -1.3671875), (0.68359375, -0.341796875), (3.734375, 1.8671875),
                 (2.4375, -1.21875), (3.375, -1.6875), (3.515625, 1.7578125),
                 (1.8828125, 0.94140625), (0.82421875, 0.412109375)]


def test_codes_use_ieee_division_not_reciprocal():
    rows = np.zeros((len(DIVISION_TIES), 8), dtype=np.float32)
    for i, (amax, xv) in enumerate(DIVISION_TIES):
        rows[i, 0], rows[i, 1] = amax, xv
    x = f32_to_bf16_bits_exact(rows)
    q, s = oracle.quantize(x, axis=0)
    disagree = 0
    for i, (amax, xv) in enumerate(DIVISION_TIES):
        assert Fraction(float(s[i])) == rn_f32(Fraction(amax) / 127)
        np.testing.assert_array_equal(q[i], _exact_rne_codes(bits_to_f32(x[i]), s[i]))
        recip = np.rint(np.float32(xv) * (np.float32(1) / s[i]))
        disagree += int(recip != q[i, 1])
    assert disagree == len(DIVISION_TIES)
