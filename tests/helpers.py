"""Test helpers: bf16 <-> bit conversions, exact-rational rounding used by
the pins, a golden-file reader, and a wrapper of cuRAND's host Philox
generator (a library routine used as an independent reference)."""
import ctypes
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bf16_bits(t):
    """bf16 torch tensor (CPU) -> numpy uint16 bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits_exact(values):
    """fp32 values that are exactly representable in bf16 -> bits."""
    v = np.asarray(values, dtype=np.float32)
    bits = v.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def read_golden(name):
    sections, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = line.strip("[]")
                sections[cur] = []
                continue
            sections[cur].append([float(v) for v in line.split()])
    return {k: np.array(v) for k, v in sections.items()}


# ---- exact rational rounding (independent of the oracle's C arithmetic) ----
def _round_half_even(fr):
    fl = math.floor(fr)
    rem = fr - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def round_to_float(fr, mant_bits, emin):
    """Round a Fraction to the nearest binary float with `mant_bits`
    significand bits (incl. the implicit one) and minimum normal exponent
    `emin`, ties to even.  Subnormals are kept.  No overflow handling."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - (mant_bits - 1))
    return sign * _round_half_even(a / ulp) * ulp


def rn_f32(fr):
    return round_to_float(Fraction(fr), 24, -126)


def rn_bf16(fr):
    return round_to_float(Fraction(fr), 8, -126)


def round_half_even_int(fr):
    return _round_half_even(Fraction(fr))


# ---- cuRAND host Philox4x32-10 generator ----------------------------------
CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


def curand_lib():
    for path in ("/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"):
        try:
            return ctypes.CDLL(path)
        except OSError:
            continue
    return None


def curand_host_philox_words(seed, n):
    """n 32-bit outputs of cuRAND's host Philox4x32-10 generator.  Its
    default ordering emits block b = Philox(counter (b >> 16, 0, b & 0xFFFF,
    0), key (lo32(seed), hi32(seed)))."""
    cur = curand_lib()
    if cur is None:
        return None
    g = ctypes.c_void_p()
    if cur.curandCreateGeneratorHost(ctypes.byref(g), CURAND_RNG_PSEUDO_PHILOX4_32_10) != 0:
        return None
    try:
        assert cur.curandSetPseudoRandomGeneratorSeed(g, ctypes.c_ulonglong(seed)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert cur.curandGenerate(g, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        cur.curandDestroyGenerator(g)
    return out


# ---- BF16 passes: tolerance of an fp32-accumulated bf16 product ----------
def bf16_pass_close(got_t, ref_bits, a, b, what):
    """A BF16 pass (plain bf16 product, fp32 accumulation in the tensor
    core's order) against the oracle's (fp64 sum, rounded to fp32 then
    bf16): within two bf16 ulps of the reference plus the fp32 accumulation
    bound K 2^-23 sum_k |a_ik||b_jk| per output.  a [M, K], b [N, K] as
    float tensors (CPU); got_t bf16 [M, N]."""
    got = got_t.cpu().float().double()
    ref = torch.from_numpy(bits_to_f32(ref_bits).astype(np.float64))
    K = a.shape[1]
    bound = 2.0 ** -7 * ref.abs() + K * 2.0 ** -23 * (a.abs().double() @ b.abs().double().T)
    bad = (got - ref).abs() > bound
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} of {bad.numel()} outputs outside the bound"
