"""Pins of the oracle's Philox4x32-10, integer matmul and rescale.

Philox4x32-10: Salmon et al., "Parallel random numbers: as easy as 1, 2, 3"
(SC'11), checked against cuRAND's host generator (a library routine).
Integer matmul and rescale: "Quantized model training" README (scaled INT8
matmul in the layouts A @ B.T, A @ B, A.T @ B); "Integrate INT8
mixed-precision from torchao 0.7" (the result is scaled back to BF16).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from helpers import curand_host_philox_words, rn_bf16, bits_to_f32


@pytest.mark.parametrize("seed", [0, 1, 42, 0x123456789ABCDEF, 2**64 - 1])
def test_philox_matches_curand_host_generator(seed):
    words = curand_host_philox_words(seed, 4 * 65541)
    if words is None:
        pytest.skip("cuRAND host generator unavailable")
    blocks = words.reshape(-1, 4)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for b in list(range(0, 40)) + [65535, 65536, 65537, 65540]:
        ctr = [b >> 16, 0, b & 0xFFFF, 0]
        np.testing.assert_array_equal(oracle.philox4x32_10(ctr, key), blocks[b], err_msg=str(ctr))


def test_philox_is_injective_on_a_sample():
    key = [0xDEADBEEF, 0x12345678]
    seen = {tuple(oracle.philox4x32_10([i, i >> 3, 7, 0], key)) for i in range(2048)}
    assert len(seen) == 2048


def _int_operands(rng, M, N, K, layout):
    a = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    b = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    A = a if layout != oracle.ATxB else np.ascontiguousarray(a.T)
    B = b if layout == oracle.AxBT else np.ascontiguousarray(b.T)
    return a, b, A, B


@pytest.mark.parametrize("layout", [oracle.AxBT, oracle.AxB, oracle.ATxB])
def test_mm_s32_equals_int64_brute_force(layout):
    rng = np.random.default_rng(1)
    for M, N, K in [(1, 1, 1), (3, 5, 16), (17, 9, 33), (8, 17, 64), (5, 4, 0), (2, 3, 127)]:
        a, b, A, B = _int_operands(rng, M, N, K, layout)
        acc = oracle.mm_s32(A, B, M, N, K, layout=layout, nthreads=3)
        ref = a.astype(np.int64) @ b.astype(np.int64).T
        np.testing.assert_array_equal(acc.astype(np.int64), ref, err_msg=f"{M}x{N}x{K}")


def test_mm_identity_returns_codes():
    rng = np.random.default_rng(2)
    a = rng.integers(-127, 128, size=(7, 32)).astype(np.int8)
    eye = np.eye(32, dtype=np.int8)
    np.testing.assert_array_equal(oracle.mm_s32(a, eye, 7, 32, 32), a.astype(np.int32))


def test_mm_extreme_magnitude_stays_in_int32():
    K = 133143  # largest K with 127*127*K < 2^31
    a = np.full((1, K), 127, dtype=np.int8)
    b = np.full((1, K), -127, dtype=np.int8)
    assert oracle.mm_s32(a, b, 1, 1, K)[0, 0] == -127 * 127 * K
    with pytest.raises(ValueError):
        oracle.mm_s32(np.zeros((1, K + 1), np.int8), np.zeros((1, K + 1), np.int8), 1, 1, K + 1)


def test_rescale_closed_forms_and_ties():
    # powers of two: exact; 257/256 and 259/256 are bf16 ties (even wins);
    # 2^24 + 1 rounds to 2^24 when converted to fp32
    acc = np.array([[4, -6, 257, 259, 2**24 + 1, 0]], dtype=np.int32)
    sA = np.array([2.0 ** -8], dtype=np.float32)
    sB = np.array([2.0 ** 3, 0.5, 1.0, 1.0, 2.0 ** 8, 3.0], dtype=np.float32)
    out = bits_to_f32(oracle.rescale_bf16(acc, sA, sB))[0]
    np.testing.assert_array_equal(out, np.array([0.125, -0.01171875, 1.0, 1.015625, 2.0 ** 24, 0.0],
                                                dtype=np.float32))


def test_rescale_within_rounding_bound_of_exact_product():
    rng = np.random.default_rng(3)
    acc = rng.integers(-2**30, 2**30, size=(6, 7)).astype(np.int32)
    acc[0, :3] = [0, 1, -1]
    sA = (rng.random(6) * 1e-2).astype(np.float32)
    sB = (rng.random(7) * 1e-3).astype(np.float32)
    out = bits_to_f32(oracle.rescale_bf16(acc, sA, sB))
    for i in range(6):
        for j in range(7):
            exact = Fraction(int(acc[i, j])) * Fraction(float(sA[i])) * Fraction(float(sB[j]))
            got = Fraction(float(out[i, j]))
            # three fp32 roundings (2^-24 each) then one bf16 rounding (2^-8)
            bound = abs(exact) * (Fraction(1, 2**8) * (1 + Fraction(4, 2**24)) + Fraction(4, 2**24))
            assert abs(got - exact) <= bound, (i, j)
            # and the result is a bf16 value nearest to its fp32 pre-image
            assert got == rn_bf16(got)
