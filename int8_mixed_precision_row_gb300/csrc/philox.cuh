// philox.cuh -- device Philox4x32-10 and the stochastic-rounding draw.
//
// Philox4x32 with 10 rounds as published by Salmon, Moraes, Dror and Shaw,
// "Parallel random numbers: as easy as 1, 2, 3" (SC'11): each round
// multiplies counter words 0 and 2 by two fixed odd constants (32x32 -> 64),
// mixes the high halves with the other two words and the round key, and the
// key advances by a Weyl sequence between rounds.
#pragma once

#include <stdint.h>

namespace int8mp {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
  constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
  constexpr uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round != 0) {
      k.x += kWeylA;
      k.y += kWeylB;
    }
    const uint32_t hiA = __umulhi(kMulA, c.x), loA = kMulA * c.x;
    const uint32_t hiB = __umulhi(kMulB, c.z), loB = kMulB * c.z;
    c = make_uint4(hiB ^ c.y ^ k.x, loB, hiA ^ c.w ^ k.y, loA);
  }
  return c;
}

// The eight random words for logical elements n0 .. n0+7, n0 = offset + e0.
// Word for element n is word (n & 3) of philox at counter block n >> 2.
__device__ __forceinline__ void philox_words8(uint64_t seed, uint64_t n0, uint32_t stream_id,
                                              uint32_t (&w)[8]) {
  const uint2 key = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
  const uint64_t blk = n0 >> 2;
  const uint32_t shift = (uint32_t)(n0 & 3u);
  uint32_t all[12];
#pragma unroll
  for (int b = 0; b < 3; ++b) {
    if (b < 2 || shift != 0) {
      const uint64_t cb = blk + (uint64_t)b;
      const uint4 r = philox4x32_10(make_uint4((uint32_t)cb, (uint32_t)(cb >> 32), stream_id, 0u), key);
      all[4 * b + 0] = r.x;
      all[4 * b + 1] = r.y;
      all[4 * b + 2] = r.z;
      all[4 * b + 3] = r.w;
    } else {
      all[4 * b + 0] = all[4 * b + 1] = all[4 * b + 2] = all[4 * b + 3] = 0u;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a0 = all[i], a1 = all[i + 1], a2 = all[i + 2], a3 = all[i + 3];
    w[i] = shift == 0 ? a0 : shift == 1 ? a1 : shift == 2 ? a2 : a3;
  }
}

// u in [0, 1) carrying the word's top 24 bits (exact in fp32).
__device__ __forceinline__ float sr_uniform(uint32_t word) {
  return __uint2float_rn(word >> 8) * 0x1p-24f;
}

}  // namespace int8mp
