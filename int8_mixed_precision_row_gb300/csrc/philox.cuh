// philox.cuh -- device Philox4x32-10: the random words of stochastic rounding.
//
// Philox4x32 with 10 rounds as published by Salmon, Moraes, Dror and Shaw,
// "Parallel random numbers: as easy as 1, 2, 3" (SC'11): each round
// multiplies counter words 0 and 2 by two fixed odd constants (32x32 -> 64),
// mixes the high halves with the other two words and the round key, and the
// key advances by a Weyl sequence between rounds.
//
// The key is the same for every element of a launch, so the host computes
// the ten round keys once (PhiloxKeys) and the kernels read them from their
// parameters: each round is then two multiplies of each kind and two
// three-input XORs.  Counter word 2 is the stream id and word 3 is 0, so
// round 0's second product is a constant of the stream too (PhiloxStream).
#pragma once

#include <stdint.h>

namespace int8mp {

constexpr uint32_t kPhiloxMulA = 0xD2511F53u, kPhiloxMulB = 0xCD9E8D57u;
constexpr uint32_t kPhiloxWeylA = 0x9E3779B9u, kPhiloxWeylB = 0xBB67AE85u;

struct PhiloxKeys {
  uint32_t k[20];  // round r uses key words k[2r], k[2r + 1]
};
struct PhiloxStream {
  uint32_t z_hi, z_lo;  // round 0: kPhiloxMulB * stream id, high and low words
};

// Host side: the round keys of key (lo32(seed), hi32(seed)).
inline PhiloxKeys philox_keys(uint64_t seed) {
  PhiloxKeys p;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    p.k[2 * r] = k0;
    p.k[2 * r + 1] = k1;
    k0 += kPhiloxWeylA;
    k1 += kPhiloxWeylB;
  }
  return p;
}
// Host side: the round-0 product for counter word 2 = stream_id.
inline PhiloxStream philox_stream(uint32_t stream_id) {
  const uint64_t z = static_cast<uint64_t>(kPhiloxMulB) * stream_id;
  return PhiloxStream{static_cast<uint32_t>(z >> 32), static_cast<uint32_t>(z)};
}

// The four words of Philox4x32-10 at counter (c0, c1, stream id, 0).
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, const PhiloxKeys& pk,
                                               PhiloxStream st) {
  // round 0: word 2 * B is the stream's constant (z_hi, z_lo), word 3 is 0
  uint4 c = make_uint4(st.z_hi ^ c1 ^ pk.k[0], st.z_lo, __umulhi(kPhiloxMulA, c0) ^ pk.k[1],
                       kPhiloxMulA * c0);
#pragma unroll
  for (int round = 1; round < 10; ++round) {
    const uint32_t hiA = __umulhi(kPhiloxMulA, c.x), loA = kPhiloxMulA * c.x;
    const uint32_t hiB = __umulhi(kPhiloxMulB, c.z), loB = kPhiloxMulB * c.z;
    c = make_uint4(hiB ^ c.y ^ pk.k[2 * round], loB, hiA ^ c.w ^ pk.k[2 * round + 1], loA);
  }
  return c;
}

// The eight random words for logical elements n0 .. n0+7.  Word for element
// n is word (n & 3) of philox at counter block n >> 2.  When n0 is a
// multiple of 4 (the usual case: every group and vector starts there) the
// eight words are two whole blocks.
__device__ __forceinline__ void philox_words8(const PhiloxKeys& pk, PhiloxStream st, uint64_t n0,
                                              uint32_t (&w)[8]) {
  const uint64_t blk = n0 >> 2;
  const uint32_t shift = static_cast<uint32_t>(n0 & 3u);
  const uint4 r0 =
      philox4x32_10(static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32), pk, st);
  const uint4 r1 = philox4x32_10(static_cast<uint32_t>(blk + 1),
                                 static_cast<uint32_t>((blk + 1) >> 32), pk, st);
  if (shift == 0) {
    w[0] = r0.x, w[1] = r0.y, w[2] = r0.z, w[3] = r0.w;
    w[4] = r1.x, w[5] = r1.y, w[6] = r1.z, w[7] = r1.w;
    return;
  }
  const uint4 r2 = philox4x32_10(static_cast<uint32_t>(blk + 2),
                                 static_cast<uint32_t>((blk + 2) >> 32), pk, st);
  const uint32_t all[12] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w, r2.x, r2.y, r2.z, r2.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a1 = all[i + 1], a2 = all[i + 2], a3 = all[i + 3];
    w[i] = shift == 1 ? a1 : shift == 2 ? a2 : a3;
  }
}

// The words of two groups of eight elements at na and nb, both multiples of
// 4: four whole blocks, computed round by round so that the four
// independent chains of multiplies overlap each other's latency.
__device__ __forceinline__ void philox_words8x2(const PhiloxKeys& pk, PhiloxStream st,
                                                uint64_t na, uint64_t nb, uint32_t (&wa)[8],
                                                uint32_t (&wb)[8]) {
  const uint64_t blk[4] = {na >> 2, (na >> 2) + 1, nb >> 2, (nb >> 2) + 1};
  uint4 c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c0 = static_cast<uint32_t>(blk[i]), c1 = static_cast<uint32_t>(blk[i] >> 32);
    c[i] = make_uint4(st.z_hi ^ c1 ^ pk.k[0], st.z_lo, __umulhi(kPhiloxMulA, c0) ^ pk.k[1],
                      kPhiloxMulA * c0);
  }
#pragma unroll
  for (int round = 1; round < 10; ++round) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t hiA = __umulhi(kPhiloxMulA, c[i].x), loA = kPhiloxMulA * c[i].x;
      const uint32_t hiB = __umulhi(kPhiloxMulB, c[i].z), loB = kPhiloxMulB * c[i].z;
      c[i] = make_uint4(hiB ^ c[i].y ^ pk.k[2 * round], loB, hiA ^ c[i].w ^ pk.k[2 * round + 1],
                        loA);
    }
  }
  wa[0] = c[0].x, wa[1] = c[0].y, wa[2] = c[0].z, wa[3] = c[0].w;
  wa[4] = c[1].x, wa[5] = c[1].y, wa[6] = c[1].z, wa[7] = c[1].w;
  wb[0] = c[2].x, wb[1] = c[2].y, wb[2] = c[2].z, wb[3] = c[2].w;
  wb[4] = c[3].x, wb[5] = c[3].y, wb[6] = c[3].z, wb[7] = c[3].w;
}

}  // namespace int8mp
