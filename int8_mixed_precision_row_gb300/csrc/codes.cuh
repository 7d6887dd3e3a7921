// codes.cuh -- per-element steps shared by the quantizers (quantize.cu) and
// the GEMM's prologue quantization of a bf16 operand (gemm.cu): bf16 values
// out of their packed words, and the nearest-even code of an exact quotient.
// Both places therefore form the same codes from the same quotients.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace int8mp {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// the eight bf16 values of a 16-byte vector, in order, as floats (exact)
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Code from an exact quotient v: an exact float in [-127, 127] (a zero code
// may come out as -0; both containers hold the integer 0 for it).
__device__ __forceinline__ float code_rne(float v) {
  return fminf(fmaxf(rintf(v), -127.0f), 127.0f);
}
// When the group scale is a normal number s = RN(absmax / 127),
// s >= (absmax / 127)(1 - 2^-24), so |v| <= 127 (1 + 2^-23) < 127.5 and
// rounding cannot leave [-127, 127]: the clamp is dropped, and two codes
// take two packed fp32 adds: for |v| < 2^22, v + 1.5 * 2^23
// lies in [2^23, 2^24), where the spacing of floats is 1, so the nearest-even
// rounding of the sum is 1.5 * 2^23 plus the nearest-even integer to v (the
// constant is even), and subtracting the constant back is exact.
__device__ __forceinline__ float2 code_rne_normal_scale2(float2 v) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  const float2 t = __fadd2_rn(v, make_float2(kMagic, kMagic));
  return __fadd2_rn(t, make_float2(-kMagic, -kMagic));
}

}  // namespace int8mp
