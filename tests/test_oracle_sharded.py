"""Pins of the oracle's fp32 rescale and of its token-sharded grad-weight.

The sharded grad-weight is the reading of data-parallel INT8 training
("Integrate INT8 mixed-precision from torchao 0.7", discussion: FSDP2 on two
A100s; torchao issue 1887: gradients reduce-scattered across ranks): each
rank quantizes its own token rows of dY and X along T with its own column
scales, forms an fp32 partial (acc * sA) * sB, the partials are summed in fp32
and rounded once to bf16.  Pinned by: the exact-rational statement of the
unrounded rescale; one shard being the single-device grad-weight (itself
pinned in test_oracle_linear.py); operands that every shard quantizes
losslessly, whose sharded result must be the exact integer product rounded
once -- which fails if the shards used global column scales, or if each
partial were rounded to bf16 before the sum.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from helpers import bits_to_f32, f32_to_bf16_bits_exact, rn_bf16, rn_f32


def test_rescale_f32_is_step_five_without_its_rounding():
    rng = np.random.default_rng(3)
    acc = rng.integers(-(2 ** 31) + 1, 2 ** 31 - 1, size=(6, 7), dtype=np.int64).astype(np.int32)
    acc[0, :3] = [2 ** 24 + 1, -(2 ** 24) - 3, 0]
    sA = (rng.random(6) * 2.0 ** rng.integers(-30, 4, 6)).astype(np.float32)
    sB = (rng.random(7) * 2.0 ** rng.integers(-30, 4, 7)).astype(np.float32)
    got = oracle.rescale_f32(acc, sA, sB)
    for i in range(6):
        for j in range(7):
            f = rn_f32(Fraction(int(acc[i, j])))
            t = rn_f32(f * Fraction(float(sA[i])))
            o = rn_f32(t * Fraction(float(sB[j])))
            assert Fraction(float(got[i, j])) == o, (i, j)


def test_scaled_mm_f32_rounds_to_scaled_mm():
    rng = np.random.default_rng(4)
    M, N, K = 9, 17, 48
    A = rng.integers(-127, 128, size=(M, K), dtype=np.int64).astype(np.int8)
    B = rng.integers(-127, 128, size=(N, K), dtype=np.int64).astype(np.int8)
    sA = rng.random(M).astype(np.float32) * 0.01
    sB = rng.random(N).astype(np.float32) * 0.3
    f32 = oracle.scaled_mm_f32(A, sA, B, sB, M, N, K)
    bf = oracle.scaled_mm(A, sA, B, sB, M, N, K)
    rounded = np.array([[oracle.bf16_rne(v) for v in row] for row in f32], dtype=np.uint16)
    np.testing.assert_array_equal(rounded, bf)


@pytest.mark.parametrize("mode", [oracle.RNE, oracle.SR])
def test_one_shard_is_the_single_device_grad_weight(mode):
    rng = np.random.default_rng(5)
    T, N, K = 48, 24, 40
    g = (rng.standard_normal((T, N)) * 1e-3).astype(np.float32)
    x = rng.standard_normal((T, K)).astype(np.float32)
    gb = (g.view(np.uint32) >> 16).astype(np.uint16)   # truncated to bf16: any bf16 will do
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    W = np.zeros((N, K), dtype=np.uint16)
    _, dW = oracle.linear_bwd(gb, xb, W, mode=mode, seed=7, offset=11, want_dx=False)
    got = oracle.grad_weight_sharded(gb, xb, 1, [11], mode=mode, seed=7)
    np.testing.assert_array_equal(got, dW)


def _lossless_shard_operand(rng, rows, cols, exps):
    """Integer multiples of 2^e (per column, this shard's e) with |v| <= 127
    2^e and 127 2^e attained: quantized along its rows exactly, scale 2^e."""
    v = rng.integers(-127, 128, size=(rows, cols)).astype(np.int64)
    v[0, :] = 127 * np.where(rng.random(cols) < 0.5, 1, -1)
    return v * (2.0 ** np.asarray(exps))[None, :]


def test_shards_of_lossless_operands_sum_exactly_then_round_once():
    rng = np.random.default_rng(6)
    nshards, Ts, N, K = 2, 16, 8, 12
    g_parts, x_parts = [], []
    for r in range(nshards):
        # each shard's columns have their own power-of-two scale, different
        # from the other shard's
        g_parts.append(_lossless_shard_operand(rng, Ts, N, rng.integers(-3, 1, N) - 2 * r))
        x_parts.append(_lossless_shard_operand(rng, Ts, K, rng.integers(-2, 2, K) + r))
    g = np.concatenate(g_parts)
    x = np.concatenate(x_parts)
    gb = f32_to_bf16_bits_exact(g.astype(np.float32))
    xb = f32_to_bf16_bits_exact(x.astype(np.float32))
    got = oracle.grad_weight_sharded(gb, xb, nshards, [0, 1 << 40])
    exact = [[rn_bf16(sum(Fraction(float(g[t, n])) * Fraction(float(x[t, k]))
                          for t in range(nshards * Ts))) for k in range(K)] for n in range(N)]
    assert np.array_equal(bits_to_f32(got).astype(np.float64),
                          np.array([[float(v) for v in row] for row in exact]))
    # the shards' scales matter: one shard (global column scales) is lossy here
    one = oracle.grad_weight_sharded(gb, xb, 1, [0])
    assert not np.array_equal(one, got)
    # and the partials are summed before the one rounding: rounding each
    # shard's partial to bf16 first gives other values here
    def part(r, n, k):
        return sum(Fraction(float(g[t, n])) * Fraction(float(x[t, k]))
                   for t in range(r * Ts, (r + 1) * Ts))
    twice = [[float(rn_bf16(rn_bf16(part(0, n, k)) + rn_bf16(part(1, n, k)))) for k in range(K)]
             for n in range(N)]
    assert not np.array_equal(bits_to_f32(got).astype(np.float64), np.array(twice))
