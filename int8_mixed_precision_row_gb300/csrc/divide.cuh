// divide.cuh -- x / s for a fixed per-group scale s, in three fused
// operations (two lanes per instruction), for the quantizers' codes.
//
// Method: Markstein's correction (P. W. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop.
// 34(1), 1990).  With r = RN(1/s) and q0 = RN(x r) within an ulp of x/s, the
// remainder x - q0 s is exactly representable and an FMA computes it
// exactly; q = RN(q0 + rem r) is then the correctly rounded quotient, as long
// as nothing over- or underflows.  The remainder is a multiple of about
// |x| 2^-46, so the quotient is exact while |x| >= 2^-103.
//
// The quantizers use the fast form for every element of a group whose scale
// s = RN(absmax / 127) lies in [2^-60, 2^10], and IEEE division otherwise.
// Below |x| = 2^-103 the fast quotient may differ from the IEEE one in its
// last bits, but then |x/s| < 2^-43 and both have the same sign and are
// nonzero together, so every code is the same: nearest-even gives 0, and the
// stochastic draw floor(v) + (u < v - floor(v)) with u a multiple of 2^-24
// gives the same result for every u.  int8mp_debug_check_division() verifies
// that the codes agree -- the nearest-even code bit for bit, and for the
// stochastic code floor(v) and the number of draws u below v - floor(v) --
// over every (x, absmax) pair of bf16 values.
#pragma once

namespace int8mp {

struct ScaleDiv {
  float s;
  float r;
  bool fast;
};

__device__ __forceinline__ bool scale_is_fast(float s) { return s >= 0x1p-60f && s <= 0x1p10f; }

__device__ __forceinline__ ScaleDiv make_scale_div(float s) {
  ScaleDiv d;
  d.s = s;
  d.fast = scale_is_fast(s);
  d.r = d.fast ? __frcp_rn(s) : 0.0f;
  return d;
}

// The fast form for two quotients at once, with the packed two-lane fp32
// instructions of sm_100+ (FMUL2 / FFMA2): each lane is rounded exactly as
// its scalar counterpart, so every quotient equals the scalar three-operation
// result.  The division certificate runs both forms over every bf16 pair and
// requires them to agree.
__device__ __forceinline__ float2 div2_fast(float2 x, float2 s, float2 r) {
  const float2 q0 = __fmul2_rn(x, r);
  const float2 rem = __ffma2_rn(make_float2(-q0.x, -q0.y), s, x);
  return __ffma2_rn(rem, r, q0);
}

// Fast quotients of eight elements of one group; returns d.fast (otherwise
// redo them with div8_ieee).
__device__ __forceinline__ bool div8_try(const float (&x)[8], const ScaleDiv& d, float (&v)[8]) {
  const float2 s2 = make_float2(d.s, d.s), r2 = make_float2(d.r, d.r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = div2_fast(make_float2(x[2 * i], x[2 * i + 1]), s2, r2);
    v[2 * i] = q.x;
    v[2 * i + 1] = q.y;
  }
  return d.fast;
}

// The same three operations for one quotient.
__device__ __forceinline__ float div_fast(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float rem = __fmaf_rn(-q0, s, x);
  return __fmaf_rn(rem, r, q0);
}

// Same for eight elements of eight groups (scales s[i], reciprocals r[i]);
// all_fast: every s[i] is in the fast range.  Scalar: pairing eight
// different scales into two-lane operands costs more than it saves.
__device__ __forceinline__ bool div8_each_try(const float (&x)[8], const float (&s)[8],
                                              const float (&r)[8], bool all_fast,
                                              float (&v)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = div_fast(x[i], s[i], r[i]);
  return all_fast;
}

// The same with the two-lane instructions, pairing the scales of columns
// 2i and 2i+1 (for the stochastic column codes, whose kernels are bound by
// instruction issue rather than memory).
__device__ __forceinline__ bool div8_each_try2(const float (&x)[8], const float (&s)[8],
                                               const float (&r)[8], bool all_fast,
                                               float (&v)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = div2_fast(make_float2(x[2 * i], x[2 * i + 1]),
                               make_float2(s[2 * i], s[2 * i + 1]),
                               make_float2(r[2 * i], r[2 * i + 1]));
    v[2 * i] = q.x;
    v[2 * i + 1] = q.y;
  }
  return all_fast;
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
