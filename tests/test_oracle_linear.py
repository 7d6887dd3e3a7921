"""Pins of the oracle's linear forward / backward.

"Quantized model training" README, section "INT8 mixed precision training":
forward, backward grad-input and backward grad-weight each run as a dynamic
row-wise quantization plus a scaled INT8 matmul, quantizing along the
matmul's contraction axis.

Closed forms: operands built as integer matrices (entries in [-127, 127])
whose groups along the contraction axis are scaled by distinct powers of two
and each contain a +-127 are quantized without loss, so the pass equals the
exact integer product times the powers of two, rounded once to bf16.  The
same matrices grouped along the other axis are lossy (the power-of-two spread
is 2^11), so quantizing along the wrong axis, or transposing an operand,
changes the result.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from helpers import bits_to_f32, f32_to_bf16_bits_exact, rn_bf16
from int8_mixed_precision_row_gb300 import synth
from helpers import bf16_bits


def _int_matrix(rng, R, C, full_axis):
    """Integers in [-127, 127]; every row (full_axis=0) or column (1) holds a
    +-127 so that its absmax is 127 times its power of two."""
    m = rng.integers(-127, 128, size=(R, C))
    if full_axis == 0:
        m[np.arange(R), rng.integers(0, C, size=R)] = 127 * rng.choice([-1, 1], size=R)
    else:
        m[rng.integers(0, R, size=C), np.arange(C)] = 127 * rng.choice([-1, 1], size=C)
    return m


def _scaled(m, row_exp=None, col_exp=None):
    e = np.zeros(m.shape, dtype=np.int64)
    if row_exp is not None:
        e += row_exp[:, None]
    if col_exp is not None:
        e += col_exp[None, :]
    vals = np.ldexp(m.astype(np.float64), e).astype(np.float32)
    return f32_to_bf16_bits_exact(vals)


def _expected(int_prod, exp_rows, exp_cols):
    out = np.zeros(int_prod.shape, dtype=np.float64)
    for i in range(int_prod.shape[0]):
        for j in range(int_prod.shape[1]):
            v = Fraction(int(int_prod[i, j])) * Fraction(2) ** int(exp_rows[i] + exp_cols[j])
            out[i, j] = float(rn_bf16(v))
    return out


@pytest.mark.parametrize("mode", [oracle.RNE, oracle.SR])
def test_forward_closed_form(mode):
    rng = np.random.default_rng(10)
    T, N, K = 24, 16, 40
    Ix, Iw = _int_matrix(rng, T, K, 0), _int_matrix(rng, N, K, 0)
    a = rng.integers(-8, 4, size=T)
    b = rng.integers(-10, 2, size=N)
    X, W = _scaled(Ix, row_exp=a), _scaled(Iw, row_exp=b)
    Y = bits_to_f32(oracle.linear_fwd(X, W, mode=mode, seed=5, nthreads=2))
    np.testing.assert_array_equal(Y, _expected(Ix @ Iw.T, a, b))


@pytest.mark.parametrize("mode", [oracle.RNE, oracle.SR])
def test_grad_input_closed_form(mode):
    rng = np.random.default_rng(11)
    T, N, K = 24, 32, 16
    Idy = _int_matrix(rng, T, N, 0)           # dY grouped by rows (along N)
    Iw = _int_matrix(rng, N, K, 1)            # W grouped by columns (along N)
    c = rng.integers(-12, -1, size=T)
    d = np.linspace(-11, 0, K).astype(np.int64)  # 2^11 spread across a row of W
    dY, W = _scaled(Idy, row_exp=c), _scaled(Iw, col_exp=d)
    X = np.zeros((T, K), dtype=np.uint16)
    dX, _ = oracle.linear_bwd(dY, X, W, mode=mode, seed=3, want_dw=False)
    np.testing.assert_array_equal(bits_to_f32(dX), _expected(Idy @ Iw, c, d))


@pytest.mark.parametrize("mode", [oracle.RNE, oracle.SR])
def test_grad_weight_closed_form(mode):
    rng = np.random.default_rng(12)
    T, N, K = 48, 16, 24
    Idy = _int_matrix(rng, T, N, 1)           # dY grouped by columns (along T)
    Ix = _int_matrix(rng, T, K, 1)            # X grouped by columns (along T)
    e = np.linspace(-11, 0, N).astype(np.int64)
    f = rng.integers(-6, 3, size=K)
    dY, X = _scaled(Idy, col_exp=e), _scaled(Ix, col_exp=f)
    W = np.zeros((N, K), dtype=np.uint16)
    _, dW = oracle.linear_bwd(dY, X, W, mode=mode, seed=4, want_dx=False)
    np.testing.assert_array_equal(bits_to_f32(dW), _expected(Idy.T @ Ix, e, f))


def test_wrong_axis_would_be_detected():
    # the grad-input operands above, quantized along K instead of N, lose
    # information: the closed form is sensitive to the grouping axis
    rng = np.random.default_rng(11)
    T, N, K = 24, 32, 16
    Iw = _int_matrix(rng, N, K, 1)
    d = np.linspace(-11, 0, K).astype(np.int64)
    W = _scaled(Iw, col_exp=d)
    q_rows, s_rows = oracle.quantize(W, axis=0)
    deq = q_rows.astype(np.float64) * s_rows[:, None]
    assert not np.array_equal(deq, bits_to_f32(W).astype(np.float64))


def test_relative_error_against_fp64_product():
    """Reported accuracy (not a parity pin): relative Frobenius error of the
    three passes against fp64 products of the same bf16 inputs."""
    T, N, K = 128, 96, 256
    X = bf16_bits(synth.bf16_normal((T, K), 1))
    W = bf16_bits(synth.bf16_normal((N, K), 2, std=0.02))
    dY = bf16_bits(synth.bf16_normal((T, N), 3, std=1e-3))
    xf, wf, gf = (bits_to_f32(a).astype(np.float64) for a in (X, W, dY))
    Y = bits_to_f32(oracle.linear_fwd(X, W)).astype(np.float64)
    dX, dW = oracle.linear_bwd(dY, X, W)
    errs = {}
    for name, got, ref in (("fwd", Y, xf @ wf.T), ("grad_in", bits_to_f32(dX), gf @ wf),
                           ("grad_w", bits_to_f32(dW), gf.T @ xf)):
        errs[name] = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    print("relative Frobenius error", errs)
    for name, e in errs.items():
        # about 0.9% expected for N(0,1)-like rows (s/sqrt(12) per operand)
        assert 0.002 < e < 0.03, (name, e)


# ------------------------------------------------------------ BF16 passes
# "BF16" entries of the INT8 mixed precision training table ("Quantized
# model training" README): the pass is the plain bf16 product.

def _exact_bf16_product(a, b):
    """bf16_RNE(fp32_RN(exact sum)) of a @ b.T, exact rationals."""
    from fractions import Fraction
    from helpers import rn_f32, rn_bf16
    M, K = a.shape
    N = b.shape[0]
    out = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(float(a[i, k])) * Fraction(float(b[j, k])) for k in range(K))
            out[i, j] = float(rn_bf16(rn_f32(s)))
    return out


@pytest.mark.parametrize("layout", [oracle.AxBT, oracle.AxB, oracle.ATxB])
def test_bf16_matmul_matches_exact_rational_product(layout):
    M, N, K = 5, 7, 33
    A = bf16_bits(synth.bf16_normal((M, K), 5))
    B = bf16_bits(synth.bf16_normal((N, K), 6))
    a, bb = bits_to_f32(A), bits_to_f32(B)
    As = A if layout != oracle.ATxB else np.ascontiguousarray(A.T)
    Bs = B if layout == oracle.AxBT else np.ascontiguousarray(B.T)
    got = bits_to_f32(oracle.matmul_bf16(As, Bs, M, N, K, layout=layout, nthreads=2))
    np.testing.assert_array_equal(got, _exact_bf16_product(a, bb))


def test_bf16_passes_in_the_linear_layer():
    T, N, K = 16, 8, 24
    X = bf16_bits(synth.bf16_normal((T, K), 7))
    W = bf16_bits(synth.bf16_normal((N, K), 8, std=0.02))
    dY = bf16_bits(synth.bf16_normal((T, N), 9, std=1e-3))
    x, w, g = bits_to_f32(X), bits_to_f32(W), bits_to_f32(dY)
    np.testing.assert_array_equal(bits_to_f32(oracle.linear_fwd_cfg(X, W, int8_fwd=0)),
                                  _exact_bf16_product(x, w))
    dX, dW = oracle.linear_bwd_cfg(dY, X, W, int8_grad_in=0, int8_grad_w=0)
    np.testing.assert_array_equal(bits_to_f32(dX), _exact_bf16_product(g, np.ascontiguousarray(w.T)))
    np.testing.assert_array_equal(bits_to_f32(dW), _exact_bf16_product(np.ascontiguousarray(g.T),
                                                                       np.ascontiguousarray(x.T)))
    # switches are per pass: INT8 grad-input with BF16 grad-weight
    dX8, dWb = oracle.linear_bwd_cfg(dY, X, W, int8_grad_in=1, int8_grad_w=0)
    np.testing.assert_array_equal(dX8, oracle.linear_bwd(dY, X, W, want_dw=False)[0])
    np.testing.assert_array_equal(dWb, dW)
