// divide.cuh -- x / s for a fixed per-group scale s, rounded exactly like an
// IEEE round-to-nearest division, in three fused operations.
//
// Method: Markstein's correction (P. W. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop.
// 34(1), 1990).  With r = RN(1/s) and q0 = RN(x r) within an ulp of x/s, the
// remainder x - q0 s is exactly representable and an FMA computes it
// exactly; q = RN(q0 + rem r) is then the correctly rounded quotient, as long
// as nothing over- or underflows.  The remainder is a multiple of about
// |x| 2^-46, so it stays exact only while that quantum is not below the
// smallest subnormal 2^-149.
//
// Domain used by the quantizers: s = RN(absmax / 127) for a bf16 absmax and
// |x| <= absmax.  The fast path is taken when 2^-100 <= s <= 2^10 (group
// flag) and x = 0 or |x| >= 2^-100 (element test); then |x/s| >= 2^-110 and
// every intermediate is a normal number.  Otherwise IEEE division is used.
// div_scale() is that rule for one element; int8mp_debug_check_division()
// compares it with __fdiv_rn over every such (x, absmax) pair of bf16 values.
// The vector forms below give, element by element, the same results: a batch
// of elements takes the fast path only if every element of it qualifies, and
// is otherwise recomputed with IEEE division.
#pragma once

namespace int8mp {

struct ScaleDiv {
  float s;
  float r;
  bool fast;
};

__device__ __forceinline__ bool scale_is_fast(float s) { return s >= 0x1p-100f && s <= 0x1p10f; }

__device__ __forceinline__ ScaleDiv make_scale_div(float s) {
  ScaleDiv d;
  d.s = s;
  d.fast = scale_is_fast(s);
  d.r = d.fast ? __frcp_rn(s) : 0.0f;
  return d;
}

// element test of the fast path: 0 or at least 2^-100 in magnitude
__device__ __forceinline__ bool fast_element(float x) {
  const float a = fabsf(x);
  return a >= 0x1p-100f || a == 0.0f;
}

__device__ __forceinline__ float div_fast(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float rem = __fmaf_rn(-q0, s, x);
  return __fmaf_rn(rem, r, q0);
}

// x / s for s > 0, equal to __fdiv_rn(x, s)
__device__ __forceinline__ float div_scale(float x, const ScaleDiv& d) {
  if (d.fast && fast_element(x)) return div_fast(x, d.s, d.r);
  return __fdiv_rn(x, d.s);
}

// Fast quotients of eight elements of one group; returns whether all of them
// took the fast path (otherwise redo them with div8_ieee).
__device__ __forceinline__ bool div8_try(const float (&x)[8], const ScaleDiv& d, float (&v)[8]) {
  bool ok = d.fast;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = div_fast(x[i], d.s, d.r);
    ok = ok && fast_element(x[i]);
  }
  return ok;
}

// Same for eight elements of eight groups (scales s[i], reciprocals r[i]).
__device__ __forceinline__ bool div8_each_try(const float (&x)[8], const float (&s)[8],
                                              const float (&r)[8], bool all_fast,
                                              float (&v)[8]) {
  bool ok = all_fast;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = div_fast(x[i], s[i], r[i]);
    ok = ok && fast_element(x[i]);
  }
  return ok;
}

// IEEE quotients (a zero scale gives 0: the group is all zero).
__device__ __forceinline__ void div8_ieee(const float (&x)[8], float s, float (&v)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = s != 0.0f ? __fdiv_rn(x[i], s) : 0.0f;
}
__device__ __forceinline__ void div8_each_ieee(const float (&x)[8], const float (&s)[8],
                                               float (&v)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = s[i] != 0.0f ? __fdiv_rn(x[i], s[i]) : 0.0f;
}

__device__ __forceinline__ bool scale_is_normal(float s) { return s >= 0x1p-126f; }

}  // namespace int8mp
