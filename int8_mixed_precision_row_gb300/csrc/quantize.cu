// quantize.cu -- dynamic symmetric INT8 quantization of bf16 matrices.
//
// "Quantized model training" README, section "INT8 mixed precision
// training": each matmul operand is quantized dynamically and row-wise (one
// scale per row of the contraction).  "Add QAT support for distributed
// finetuning", summary: x_q = clamp(x / scale + zp) -- here zp = 0 and
// scale = absmax / 127.
//
// Two groupings, both HBM-bound and both fed by TMA:
//   rows    one group per row of x [rows, cols] (the contraction axis is
//           contiguous).  Teams of warps stream whole rows into a ring of
//           2-4 shared-memory slots with bulk copies (cp.async.bulk), reduce
//           the absmax from shared memory and write the codes; a slot is
//           refilled as soon as every warp of the team has left it.  One
//           variant also keeps each column's absmax on the way (for the
//           column groups of the same matrix).
//   columns one group per column (the contraction axis is the leading one):
//           the column absmax comes from that row pass, or from a pass of
//           its own (atomic max on the fp32 bit pattern, valid for values
//           >= 0); the codes are written either in the input's layout
//           [rows, cols] (each thread streams one 8-column vector down its
//           rows with the 8 scales in registers) or transposed [cols, rows]
//           (each warp streams 32x64 sub-tiles through its own two-slot ring
//           of 2-D TMA loads and writes them through its own staging tile).
//
// Arithmetic per element (identical to the header of int8mp.h):
//   v = x / s rounded as an IEEE division (div8_*: a reciprocal and two FMAs,
//   certified against IEEE division over all bf16 inputs), then
//   q = clamp(rint(v)) or, stochastically, q = clamp(floor(v) + (u < v -
//   floor(v))) with u from Philox4x32-10.
// Every wait on a copy is bounded; a wait that runs out sets the device
// status word and the warp or block stops after its copies have landed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>
#include <type_traits>

#include "check.cuh"
#include "codes.cuh"
#include "common.cuh"
#include "divide.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace int8mp {
namespace ptx {
// The two halves of a cluster-wide barrier, for threads that need not be
// converged: arrive (ordering this thread's earlier shared-memory accesses
// before the peers' later ones) and wait for every thread of the cluster.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// 16 bytes from a shared::cluster address (any CTA of the cluster).
__device__ __forceinline__ uint4 ld_shared_cluster_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
}  // namespace ptx

namespace {

constexpr int kThreads = 256;


// |v| of eight bf16 values, bit patterns still packed two per word
__device__ __forceinline__ uint4 abs_bits8(const uint4& v) {
  return make_uint4(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu, v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
}
// Running max of |bf16| kept as a packed pair: non-negative bf16 bit
// patterns order as unsigned integers, so a per-halfword unsigned max is the
// max (one instruction per two values).
__device__ __forceinline__ uint32_t absmax8_bits(uint32_t m2, const uint4& a) {
  return __vmaxu2(m2, __vmaxu2(__vmaxu2(a.x, a.y), __vmaxu2(a.z, a.w)));
}
// the float value of the larger half of a packed pair (bf16 bits shifted up)
__device__ __forceinline__ float unpack_max(uint32_t m2) {
  return __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
}

// max(m, |v_0|, ..., |v_7|) as a tree: a dependency depth of 4, not 8
__device__ __forceinline__ float absmax8(float m, const uint4& v) {
  const float a = fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x)));
  const float b = fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)));
  const float c = fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z)));
  const float d = fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)));
  return fmaxf(m, fmaxf(fmaxf(a, b), fmaxf(c, d)));
}


// Stochastic codes of two quotients v from their random words w:
// floor(v) + (u < v - floor(v)) with u = (w >> 8) 2^-24, computed as
// ceil(v - u).  With f = floor(v) and fr = v - f in [0, 1), fr - u lies in
// (-1, 1) and its ceiling is 1 exactly when u < fr, so ceil(v - u) =
// f + (u < fr).  One fused multiply-add rounded upwards gives y = RU(v - u)
// (u's product is exact), and ceil(y) = ceil(v - u) because that integer is
// a float at least v - u, and rounding upwards never passes it.  The ceiling
// itself is y + 1.5 * 2^23 rounded upwards (for |y| < 2^22 the sum lies in
// [2^23, 2^24), where floats are the integers) minus the constant again,
// exactly; a zero code comes out as +0.  |v| stays below 128 for every group
// scale, so the codes lie in [-128, 128] before the clamp.
// kClamp false: the caller clamps afterwards (f16 codes, as packed half2
// min/max: every unclamped code is an integer in [-128, 128], exact in f16).
template <bool kClamp>
__device__ __forceinline__ float2 code_sr2(float v0, float v1, uint32_t w0, uint32_t w1) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  const float2 k = make_float2(__uint2float_rn(w0 >> 8), __uint2float_rn(w1 >> 8));
  const float2 y = __ffma2_ru(k, make_float2(-0x1p-24f, -0x1p-24f), make_float2(v0, v1));
  const float2 t = __fadd2_ru(y, make_float2(kMagic, kMagic));
  const float2 q = __fadd2_rn(t, make_float2(-kMagic, -kMagic));
  if (!kClamp) return q;
  return make_float2(fminf(fmaxf(q.x, -127.0f), 127.0f), fminf(fmaxf(q.y, -127.0f), 127.0f));
}

// Eight stochastic codes from eight quotients and their random words.
template <bool kSrClamp>
__device__ __forceinline__ void codes_sr8(const float (&v)[8], const uint32_t (&w)[8],
                                          float (&c)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = code_sr2<kSrClamp>(v[2 * i], v[2 * i + 1], w[2 * i], w[2 * i + 1]);
    c[2 * i] = q.x;
    c[2 * i + 1] = q.y;
  }
}

// Eight codes from eight quotients (elements n0 .. n0+7 of the SR stream).
// normal_scales: every element's group scale is at least 2^-126.
// kSrClamp false: stochastic codes are left unclamped for a later half2 clamp.
template <bool SR, bool kSrClamp = true>
__device__ __forceinline__ void codes_of(const float (&v)[8], const PhiloxKeys& keys,
                                         PhiloxStream st, uint64_t n0, bool normal_scales,
                                         float (&c)[8]) {
  if (SR) {
    uint32_t w[8];
    philox_words8(keys, st, n0, w);
    codes_sr8<kSrClamp>(v, w, c);
  } else if (normal_scales) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 q = code_rne_normal_scale2(make_float2(v[2 * i], v[2 * i + 1]));
      c[2 * i] = q.x;
      c[2 * i + 1] = q.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = code_rne(v[i]);
  }
}

// eight f16 codes (one uint4) clamped to [-127, 127]
__device__ __forceinline__ uint4 clamp_half8(uint4 v) {
  const __half2 lo = __float2half2_rn(-127.0f), hi = __float2half2_rn(127.0f);
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    h = __hmin2(__hmax2(h, lo), hi);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint2 clamp_half8(uint2 v) { return v; }  // int8 codes: clamped before

template <typename CodeT>
struct Pack8;

template <>
struct Pack8<int8_t> {
  using Vec = uint2;
  __device__ __forceinline__ static Vec pack(const float (&c)[8]) {
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = static_cast<uint32_t>(__float2int_rn(c[i])) & 0xFFu;
    return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                      b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
  }
};

template <>
struct Pack8<__half> {
  using Vec = uint4;
  __device__ __forceinline__ static uint32_t h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  __device__ __forceinline__ static Vec pack(const float (&c)[8]) {
    return make_uint4(h2(c[0], c[1]), h2(c[2], c[3]), h2(c[4], c[5]), h2(c[6], c[7]));
  }
};

// ------------------------------------------------------------ row groups
// The block's warps form teams of T warps (T = 1, 2, 4 or 8).  Each team owns
// a ring of S row slots of `slot_bytes` in dynamic shared memory and walks the rows
// g, g + n, ... (g = its global team index, n = teams in the grid).  The
// team's first lane issues the bulk copies, waits for them and publishes the
// outcome; each warp of the team reduces and quantizes a strided share of the
// row's 16-byte vectors, and the partial absmax values meet in shared memory.
// The copy of row it + S - 1 starts as soon as every warp of the team has
// left row it - 1.
__device__ __forceinline__ void team_sync(int team, int T) {
  if (T == 1) {
    __syncwarp();
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(T * 32) : "memory");
  }
}

// Codes of two 16-byte vectors a, b of one row (b absent when !has_b): exact
// quotients (fast form, or IEEE division for both vectors if either has an
// element outside the fast form's range), then the rounding.
template <typename CodeT, bool SR>
__device__ __forceinline__ void quantize_two(const uint4& a, const uint4& b, bool has_b,
                                             const ScaleDiv& d, bool normal,
                                             const PhiloxKeys& keys, PhiloxStream st,
                                             uint64_t na, uint64_t nb,
                                             typename Pack8<CodeT>::Vec* qa,
                                             typename Pack8<CodeT>::Vec* qb) {
  float fa[8], fb[8], va[8], vb[8], c[8];
  unpack8(a, fa);
  unpack8(b, fb);
  const bool ok_a = div8_try(fa, d, va);
  const bool ok_b = div8_try(fb, d, vb);
  if (!(ok_a && ok_b)) {
    div8_ieee(fa, d.s, va);
    div8_ieee(fb, d.s, vb);
  }
  // f16 stochastic codes: clamped as packed half2 after the conversion
  constexpr bool kHalfClamp = SR && std::is_same<CodeT, __half>::value;
  if (SR && has_b && ((na | nb) & 3u) == 0) {
    // both groups start a Philox block: their four blocks side by side
    uint32_t wa[8], wb[8];
    philox_words8x2(keys, st, na, nb, wa, wb);
    codes_sr8<!kHalfClamp>(va, wa, c);
    *qa = Pack8<CodeT>::pack(c);
    if (kHalfClamp) *qa = clamp_half8(*qa);
    codes_sr8<!kHalfClamp>(vb, wb, c);
    *qb = Pack8<CodeT>::pack(c);
    if (kHalfClamp) *qb = clamp_half8(*qb);
    return;
  }
  codes_of<SR, !kHalfClamp>(va, keys, st, na, normal, c);
  *qa = Pack8<CodeT>::pack(c);
  if (kHalfClamp) *qa = clamp_half8(*qa);
  if (has_b) {
    codes_of<SR, !kHalfClamp>(vb, keys, st, nb, normal, c);
    *qb = Pack8<CodeT>::pack(c);
    if (kHalfClamp) *qb = clamp_half8(*qb);
  }
}

// The same for a row whose scale is in the fast range of the division (so
// also a normal number), with the stochastic words' blocks aligned (na, nb
// multiples of 4): no branch inside, so that the generator, the divisions
// and the codes of the two vectors form one block of independent work.
template <typename CodeT, bool SR>
__device__ __forceinline__ void quantize_two_fast(const uint4& a, const uint4& b, bool has_b,
                                                  const ScaleDiv& d, const PhiloxKeys& keys,
                                                  PhiloxStream st, uint64_t na, uint64_t nb,
                                                  typename Pack8<CodeT>::Vec* qa,
                                                  typename Pack8<CodeT>::Vec* qb) {
  constexpr bool kHalfClamp = SR && std::is_same<CodeT, __half>::value;
  float fa[8], fb[8], va[8], vb[8], c[8];
  uint32_t wa[8], wb[8];
  if (SR) philox_words8x2(keys, st, na, nb, wa, wb);
  unpack8(a, fa);
  unpack8(b, fb);
  (void)div8_try(fa, d, va);
  (void)div8_try(fb, d, vb);
  if (SR) {
    codes_sr8<!kHalfClamp>(va, wa, c);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 qv = code_rne_normal_scale2(make_float2(va[2 * i], va[2 * i + 1]));
      c[2 * i] = qv.x;
      c[2 * i + 1] = qv.y;
    }
  }
  *qa = Pack8<CodeT>::pack(c);
  if (kHalfClamp) *qa = clamp_half8(*qa);
  if (SR) {
    codes_sr8<!kHalfClamp>(vb, wb, c);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 qv = code_rne_normal_scale2(make_float2(vb[2 * i], vb[2 * i + 1]));
      c[2 * i] = qv.x;
      c[2 * i + 1] = qv.y;
    }
  }
  typename Pack8<CodeT>::Vec pb = Pack8<CodeT>::pack(c);
  if (kHalfClamp) pb = clamp_half8(pb);
  if (has_b) *qb = pb;
}

// Column absmax alongside the row groups (kColMax): each thread owns the same
// vectors first + k*step, k < kColVecs, of every row it sees and keeps their
// running |x| maxima as packed bf16 pairs (|x| of a bf16 is a bf16, and
// non-negative bf16 bit patterns order as unsigned integers, so a per-halfword
// unsigned max is the max).  At the end the teams of a block merge theirs in
// shared memory and the block merges into colmax[] by atomic max on the fp32
// bit pattern (the bf16 bits shifted up: the same value).
constexpr int kColVecs = 8;

__device__ __forceinline__ void colmax_acc(uint4& m, const uint4& a) {  // a = abs_bits8(v)
  m.x = __vmaxu2(m.x, a.x);
  m.y = __vmaxu2(m.y, a.y);
  m.z = __vmaxu2(m.z, a.z);
  m.w = __vmaxu2(m.w, a.w);
}

constexpr int kMaxSlots = 4;

// A second matrix of the same row length, quantized by blocks split ..
// gridDim.x - 1 of the same launch (split = gridDim.x: none).
struct RowsJob2 {
  const uint16_t* x;
  int64_t rows, ld;
  void* q;
  float* scale;
  unsigned int* colmax;
  uint64_t offset;
  PhiloxStream stream;
  int split;
};

template <typename CodeT, bool SR, bool kColMax>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(
    const uint16_t* __restrict__ x1, int64_t rows1, int64_t cols, int64_t ld1,
    CodeT* __restrict__ q1, float* __restrict__ scale1, SrArgs sr, uint32_t slot_bytes, int T,
    int S, unsigned int* status, uint64_t limit_ns, unsigned int* __restrict__ colmax1,
    RowsJob2 job2) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[kThreads / 32][kMaxSlots];
  __shared__ float red[kThreads / 32];
  __shared__ int got_row[kThreads / 32];
  // this block's matrix: the first one, or job2 from block job2.split on
  const bool second = static_cast<int>(blockIdx.x) >= job2.split;
  const uint16_t* __restrict__ x = second ? job2.x : x1;
  const int64_t rows = second ? job2.rows : rows1;
  const int64_t ld = second ? job2.ld : ld1;
  CodeT* __restrict__ q = second ? static_cast<CodeT*>(job2.q) : q1;
  float* __restrict__ scale = second ? job2.scale : scale1;
  unsigned int* __restrict__ colmax = second ? job2.colmax : colmax1;
  const uint64_t sr_offset = second ? job2.offset : sr.offset;
  const PhiloxStream sr_stream = second ? job2.stream : sr.stream;
  const int64_t block = second ? blockIdx.x - job2.split : blockIdx.x;
  const int64_t blocks = second ? gridDim.x - job2.split : job2.split;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / T, wt = warp % T;
  const int teams = (blockDim.x >> 5) / T;
  const bool leader = wt == 0 && lane == 0;
  const uint32_t row_bytes = static_cast<uint32_t>(cols) * 2u;
  const int nvec = static_cast<int>(cols >> 3);
  const uint8_t* slots = smem + static_cast<size_t>(team) * S * slot_bytes;
  const uint32_t slot_addr = ptx::smem_addr(slots);
  const uint32_t bar0 = ptx::smem_addr(&bars[team][0]);  // slot k's barrier: bar0 + 8k
  const int64_t g = block * teams + team;
  const int64_t n = blocks * teams;
  using P = Pack8<CodeT>;
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();

  uint32_t pending = 0u, pend_par = 0u;  // leader: copies in flight per slot, their parity
  if (leader) {
    for (int k = 0; k < S; ++k) ptx::mbar_init(bar0 + 8u * k, 1);
    ptx::fence_mbar_init();
    for (int k = 0; k < S; ++k) {
      const int64_t r = g + k * n;
      if (r < rows && in_bounds(r >= 0 && (k + 1) * slot_bytes <= S * slot_bytes, status)) {
        ptx::mbar_arrive_expect_tx(bar0 + 8u * k, row_bytes);
        ptx::bulk_load(slot_addr + k * slot_bytes, x + r * ld, row_bytes, bar0 + 8u * k);
        pending |= 1u << k;
      }
    }
  }
  const int first = wt * 32 + lane, step = T * 32;  // this thread's vectors of a row
  uint4 cm[kColMax ? kColVecs : 1];
#pragma unroll
  for (int k = 0; k < (kColMax ? kColVecs : 1); ++k) cm[k] = make_uint4(0u, 0u, 0u, 0u);
  // row it of the team sits in slot it % S; its wait parity is (it / S) & 1
  int it = 0, b = 0;
  uint32_t phase = 0u;
  for (int64_t r = g; r < rows; r += n, ++it) {
    if (leader) {
      const bool ok = ptx::mbar_wait_timeout(bar0 + 8u * b, phase, limit_ns);
      got_row[team] = ok ? 1 : 0;
      if (ok) pending &= ~(1u << b);
      else atomicOr(status, 1u);
    }
    team_sync(team, T);  // the row has landed; every warp has left row it-1
    if (!got_row[team]) break;
    if (leader && it >= 1 && r + (S - 1) * n < rows && in_bounds(r >= 0, status)) {
      // row it+S-1 goes to the slot of row it-1, which every warp has left
      const int nb = b == 0 ? S - 1 : b - 1;
      const int j = it + S - 1;
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive_expect_tx(bar0 + 8u * nb, row_bytes);
      ptx::bulk_load(slot_addr + nb * slot_bytes, x + (r + (S - 1) * n) * ld, row_bytes,
                     bar0 + 8u * nb);
      pending |= 1u << nb;
      pend_par = (pend_par & ~(1u << nb)) | (static_cast<uint32_t>((j / S) & 1) << nb);
    }
    const uint4* rowv = reinterpret_cast<const uint4*>(slots + b * slot_bytes);
    if (++b == S) {
      b = 0;
      phase ^= 1u;
    }
    uint32_t am2 = 0u;  // packed pair of |x| maxima
    if (kColMax) {
#pragma unroll
      for (int k = 0; k < kColVecs; ++k) {
        const int v = first + k * step;
        if (v < nvec && in_bounds((v + 1) * 16u <= slot_bytes, status)) {
          const uint4 a = abs_bits8(rowv[v]);
          am2 = absmax8_bits(am2, a);
          colmax_acc(cm[k], a);
        }
      }
    } else {
      for (int v = first; v < nvec; v += step)
        if (in_bounds((v + 1) * 16u <= slot_bytes, status))
          am2 = absmax8_bits(am2, abs_bits8(rowv[v]));
    }
    float amax = unpack_max(am2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (T > 1) {
      if (lane == 0) red[warp] = amax;
      team_sync(team, T);
      amax = red[team * T];
      for (int w = 1; w < T; ++w) amax = fmaxf(amax, red[team * T + w]);
    }
    const float s = __fdiv_rn(amax, 127.0f);
    if (leader && in_bounds(r < rows, status)) scale[r] = s;
    const ScaleDiv d = make_scale_div(s);
    const bool normal = scale_is_normal(s);
    typename P::Vec* qr = reinterpret_cast<typename P::Vec*>(q + r * cols);
    const uint64_t nrow = sr_offset + static_cast<uint64_t>(r * cols);
    if (d.fast && (nrow & 3u) == 0) {
      for (int v = first; v < nvec; v += 2 * step) {
        const int v2 = v + step;
        const bool has2 = v2 < nvec;
        if (!in_bounds(r < rows && (has2 ? v2 : v) < nvec &&
                           ((has2 ? v2 : v) + 1) * 16u <= slot_bytes, status))
          continue;
        const uint4 a = rowv[v];
        const uint4 bb = has2 ? rowv[v2] : make_uint4(0u, 0u, 0u, 0u);
        quantize_two_fast<CodeT, SR>(a, bb, has2, d, sr.keys, sr_stream, nrow + 8u * v,
                                     nrow + 8u * v2, qr + v, qr + (has2 ? v2 : v));
      }
      continue;
    }
    for (int v = first; v < nvec; v += 2 * step) {
      const int v2 = v + step;
      const bool has2 = v2 < nvec;
      if (!in_bounds(r < rows && (has2 ? v2 : v) < nvec &&
                         ((has2 ? v2 : v) + 1) * 16u <= slot_bytes, status))
        continue;
      const uint4 a = rowv[v];
      const uint4 bb = has2 ? rowv[v2] : make_uint4(0u, 0u, 0u, 0u);
      quantize_two<CodeT, SR>(a, bb, has2, d, normal, sr.keys, sr_stream, nrow + 8u * v,
                              nrow + 8u * v2, qr + v, qr + (has2 ? v2 : v));
    }
  }
  // after a timeout: never leave a copy in flight into this block's memory
  bool copies_done = true;
  if (leader) {
    for (int k = 0; k < S; ++k)
      if (pending & (1u << k))
        if (!ptx::mbar_wait_timeout(bar0 + 8u * k, (pend_par >> k) & 1u, limit_ns)) {
          atomicOr(status, 1u);
          copies_done = false;
        }
  }
  if (kColMax) {
    // every team's maxima into its own first slot (cols bf16 values), then
    // the block's maximum over teams, one atomic per column
    __shared__ int all_done;
    if (threadIdx.x == 0) all_done = 1;
    __syncthreads();
    if (leader && !copies_done) all_done = 0;
    __syncthreads();
    if (!all_done) return;  // a copy may still land in the slots: leave them alone
    uint4* mine = reinterpret_cast<uint4*>(smem + static_cast<size_t>(team) * S * slot_bytes);
#pragma unroll
    for (int k = 0; k < kColVecs; ++k) {
      const int v = first + k * step;
      if (v < nvec && in_bounds((v + 1) * 16u <= S * slot_bytes, status)) mine[v] = cm[k];
    }
    __syncthreads();
    const uint16_t* all = reinterpret_cast<const uint16_t*>(smem);
    const size_t team_stride = static_cast<size_t>(S) * slot_bytes / 2;  // in uint16
    for (int c = threadIdx.x; c < cols; c += kThreads) {
      uint32_t mx = 0u;
      for (int t = 0; t < teams; ++t)
        if (in_bounds(t * team_stride + c < teams * team_stride, status))
          mx = max(mx, static_cast<uint32_t>(all[t * team_stride + c]));
      if (mx != 0u) atomicMax(colmax + c, mx << 16);
    }
  }
}

// Rows of at most 256 kV columns with no column maxima: one warp per row,
// the row in registers (kV 16-byte vectors per lane, loaded right after the
// grid dependency wait), no shared memory, no barrier and no bulk copy to
// set up -- for the small matrices whose launches are latency-bound.
// Blocks job2.split .. gridDim.x - 1 take the second matrix, as in
// quant_rows_kernel.  Faster than the ring of bulk copies at every size it
// takes (A and B of 1024^2: 3.5 -> 2.8 us; X of 32768 x 2048: 38.0 -> 36.4
// us), slower at 4096 columns (16 vectors per lane), which keep the ring.
// (Blocks of 128 threads capped at 85 registers, small enough to sit beside
// a GEMM CTA, measured slower: 2048^2 A and B 10.6 -> 12.2 us.)
constexpr int kRegMaxV = 8;
constexpr int kRegThreads = kThreads;

template <typename CodeT, bool SR, int kV>
__global__ void __launch_bounds__(kRegThreads) quant_rows_reg_kernel(
    const uint16_t* __restrict__ x1, int64_t rows1, int64_t cols, int64_t ld1,
    CodeT* __restrict__ q1, float* __restrict__ scale1, SrArgs sr, unsigned int* status,
    RowsJob2 job2) {
  const bool second = static_cast<int>(blockIdx.x) >= job2.split;
  const uint16_t* __restrict__ x = second ? job2.x : x1;
  const int64_t rows = second ? job2.rows : rows1;
  const int64_t ld = second ? job2.ld : ld1;
  CodeT* __restrict__ q = second ? static_cast<CodeT*>(job2.q) : q1;
  float* __restrict__ scale = second ? job2.scale : scale1;
  const uint64_t sr_offset = second ? job2.offset : sr.offset;
  const PhiloxStream sr_stream = second ? job2.stream : sr.stream;
  const int64_t block = second ? blockIdx.x - job2.split : blockIdx.x;
  const int64_t blocks = second ? gridDim.x - job2.split : job2.split;
  constexpr int kWarps = kRegThreads / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = static_cast<int>(cols >> 3);
  using P = Pack8<CodeT>;
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();
  if (!in_bounds(nvec <= 32 * kV && cols <= ld, status)) return;
  for (int64_t r = block * kWarps + warp; r < rows; r += blocks * kWarps) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + r * ld);
    uint4 a[kV];
    uint32_t am2 = 0u;  // packed pair of |x| maxima
#pragma unroll
    for (int i = 0; i < kV; ++i) {
      const int v = lane + 32 * i;
      a[i] = v < nvec ? __ldg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
      am2 = absmax8_bits(am2, abs_bits8(a[i]));
    }
    float amax = unpack_max(am2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = __fdiv_rn(amax, 127.0f);
    if (lane == 0) scale[r] = s;
    const ScaleDiv d = make_scale_div(s);
    const bool normal = scale_is_normal(s);
    typename P::Vec* qr = reinterpret_cast<typename P::Vec*>(q + r * cols);
    const uint64_t nrow = sr_offset + static_cast<uint64_t>(r * cols);
    const bool fast = d.fast && (nrow & 3u) == 0;
#pragma unroll
    for (int i = 0; i < kV; i += 2) {
      const int v = lane + 32 * i, v2 = v + 32;
      if (v < nvec) {
        const bool has2 = i + 1 < kV && v2 < nvec;
        const uint4 b = i + 1 < kV ? a[i + 1 < kV ? i + 1 : i] : make_uint4(0u, 0u, 0u, 0u);
        if (fast)
          quantize_two_fast<CodeT, SR>(a[i], b, has2, d, sr.keys, sr_stream, nrow + 8u * v,
                                       nrow + 8u * v2, qr + v, qr + (has2 ? v2 : v));
        else
          quantize_two<CodeT, SR>(a[i], b, has2, d, normal, sr.keys, sr_stream, nrow + 8u * v,
                                  nrow + 8u * v2, qr + v, qr + (has2 ? v2 : v));
      }
    }
  }
}

// Rows too long for two shared-memory slots: one block per row, two sweeps
// over global memory (the second hits L2).
template <typename CodeT, bool SR>
__global__ void __launch_bounds__(kThreads) quant_rows_long_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, CodeT* __restrict__ q,
    float* __restrict__ scale, SrArgs sr, unsigned int* status) {
  __shared__ float red[kThreads / 32];
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  if (row >= rows || !in_bounds(cols <= ld, status)) return;
  const int64_t nvec = cols >> 3;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * ld);
  float amax = 0.0f;
  for (int64_t vi = threadIdx.x; vi < nvec; vi += kThreads) amax = absmax8(amax, __ldg(xr + vi));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
  for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const float s = __fdiv_rn(amax, 127.0f);
  if (threadIdx.x == 0) scale[row] = s;
  const ScaleDiv d = make_scale_div(s);
  const bool normal = scale_is_normal(s);
  using P = Pack8<CodeT>;
  typename P::Vec* qr = reinterpret_cast<typename P::Vec*>(q + row * cols);
  for (int64_t vi = threadIdx.x; vi < nvec; vi += kThreads) {
    const uint64_t n0 = sr.offset + static_cast<uint64_t>(row * cols + vi * 8);
    quantize_two<CodeT, SR>(__ldg(xr + vi), make_uint4(0u, 0u, 0u, 0u), false, d, normal, sr.keys,
                            sr.stream, n0, n0, qr + vi, qr + vi);
  }
}

// --------------------------------------------------------- column groups
// Pass 1: absmax of each column over this block's rows, merged by atomic max
// on the bit pattern (absolute values are >= +0, whose bits order as
// unsigned integers).  Lane = one 8-column vector, warp = row phase; eight
// rows in flight per thread.
__global__ void __launch_bounds__(kThreads) col_absmax_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
    int64_t rows_per_block, unsigned int* __restrict__ amax_bits, unsigned int* status) {
  __shared__ float red[kThreads / 32][32][9];
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nvec = cols >> 3;
  const int64_t vi = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_block;
  const int64_t r1 = min(rows, r0 + rows_per_block);
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = 0.0f;
  if (vi < nvec && in_bounds(vi * 8 + 8 <= cols && r1 <= rows, status)) {
    const uint16_t* base = x + vi * 8;
    int64_t r = r0 + warp;
    constexpr int U = 8;
    for (; r + (U - 1) * 8 < r1; r += U * 8) {
      uint4 a[U];
#pragma unroll
      for (int u = 0; u < U; ++u) a[u] = __ldg(reinterpret_cast<const uint4*>(base + (r + u * 8) * ld));
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[8];
        unpack8(a[u], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) m[i] = fmaxf(m[i], fabsf(f[i]));
      }
    }
    for (; r < r1; r += 8) {
      float f[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(base + r * ld)), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) m[i] = fmaxf(m[i], fabsf(f[i]));
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[warp][lane][i] = m[i];
  __syncthreads();
  if (warp == 0 && vi < nvec) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float mm = red[0][lane][i];
#pragma unroll
      for (int w = 1; w < kThreads / 32; ++w) mm = fmaxf(mm, red[w][lane][i]);
      atomicMax(amax_bits + vi * 8 + i, __float_as_uint(mm));
    }
  }
}

// Zeroes n 32-bit words (absmax buffers before an atomic-max merge); a kernel
// rather than a memset so that it keeps the stream's dependent launches.
__global__ void zero_words_kernel(unsigned int* __restrict__ p, int64_t n) {
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    p[i] = 0u;
}

// y[i] = bf16_RNE(x[i]): eight values per thread and step (two 16-byte
// loads, one 16-byte store), the remainder one at a time.
__global__ void round_bf16_kernel(const float* __restrict__ x, uint16_t* __restrict__ y,
                                  int64_t n) {
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n8 = n / 8;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  uint4* y8 = reinterpret_cast<uint4*>(y);
  auto pack = [](float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  };
  for (int64_t i = t; i < n8; i += stride) {
    const float4 a = __ldg(x4 + 2 * i), b = __ldg(x4 + 2 * i + 1);
    y8[i] = make_uint4(pack(a.x, a.y), pack(a.z, a.w), pack(b.x, b.y), pack(b.z, b.w));
  }
  for (int64_t i = n8 * 8 + t; i < n; i += stride) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x[i]);
    y[i] = *reinterpret_cast<const uint16_t*>(&h);
  }
}

// Pass 2: scale = absmax / 127, in place, before any code is computed.
__global__ void col_scale_kernel(unsigned int* __restrict__ amax_bits, int64_t cols) {
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c < cols) amax_bits[c] = __float_as_uint(__fdiv_rn(__uint_as_float(amax_bits[c]), 127.0f));
}

// Pass 3, codes in the input's layout q [rows, cols]: lane = one 8-column
// vector (16-byte loads and stores), warp = row phase, four rows in flight
// per thread; the thread's eight column scales and their reciprocals stay in
// registers for all of its rows.  kFromAbsmax: `in` holds the columns'
// absmax (computed elsewhere, e.g. alongside a row quantization of x); the
// kernel forms the scales, the blocks of the first row band store them, and
// the codes keep their clamp (the absmax is the caller's claim).  Otherwise
// `in` is the scale array itself.
constexpr int kNatUnroll = 4;
static_assert(kNatUnroll % 2 == 0, "stochastic codes go two rows at a time");

template <typename CodeT, bool SR, bool kFromAbsmax>
__global__ void __launch_bounds__(kThreads, SR ? 2 : 3) quant_cols_nat_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
    int64_t rows_per_block, const float* __restrict__ in, float* __restrict__ scale_out,
    CodeT* __restrict__ q, SrArgs sr, unsigned int* status) {
  using P = Pack8<CodeT>;
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t vi = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  if (vi >= (cols >> 3) || !in_bounds(vi * 8 + 8 <= cols && cols <= ld, status)) return;
  const int64_t c = vi * 8;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_block;
  const int64_t r1 = min(rows, r0 + rows_per_block);
  // f16 codes from a given absmax keep their clamp as a packed half2 min/max
  // after rounding (a caller's absmax below the true one would otherwise let
  // a code leave [-127, 127]), and so do f16 stochastic codes; int8 codes
  // clamp before packing
  constexpr bool kHalfClamp = (kFromAbsmax || SR) && std::is_same<CodeT, __half>::value;
  float s[8], r[8];
  bool all_fast = true, normal = !kFromAbsmax || kHalfClamp;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    s[j] = kFromAbsmax ? __fdiv_rn(__ldg(in + c + j), 127.0f) : __ldg(in + c + j);
    all_fast = all_fast && scale_is_fast(s[j]);
    normal = normal && scale_is_normal(s[j]);
    r[j] = __frcp_rn(s[j]);
  }
  if (kFromAbsmax && blockIdx.y == 0 && warp == 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j) scale_out[c + j] = s[j];
  }
  const uint16_t* xc = x + c;
  auto put = [&](int64_t row, const float (&cd)[8]) {
    typename P::Vec out = P::pack(cd);
    if (kHalfClamp) out = clamp_half8(out);
    if (in_bounds(row < rows, status))
      *reinterpret_cast<typename P::Vec*>(q + row * cols + c) = out;
  };
  auto load_row = [&](int64_t row) {
    return row < r1 && in_bounds(row < rows, status)
               ? __ldg(reinterpret_cast<const uint4*>(xc + row * ld))
               : make_uint4(0u, 0u, 0u, 0u);
  };
  if (SR && (sr.offset & 3u) == 0) {
    // Stochastic codes, every group of eight starting a Philox block: two
    // rows at a time, the next two rows' loads issued before this pair's
    // generator and codes, so that the long computation per pair hides the
    // load latency instead of waiting for it.  Input and code pointers and
    // the element counter of row rr advance by additions.
    const int64_t row0 = r0 + warp;
    const uint16_t* xp = xc + row0 * ld;
    typename P::Vec* qp = reinterpret_cast<typename P::Vec*>(q + row0 * cols + c);
    uint64_t n = sr.offset + static_cast<uint64_t>(row0 * cols + c);
    const int64_t xstep = 8 * ld, qstep = cols;  // 8 rows of input; 8 rows of codes, in vectors
    const uint64_t nstep = 8u * static_cast<uint64_t>(cols);
    auto ld_at = [&](const uint16_t* ptr, int64_t row) {
      return row < r1 && in_bounds(row < rows, status)
                 ? __ldg(reinterpret_cast<const uint4*>(ptr))
                 : make_uint4(0u, 0u, 0u, 0u);
    };
    auto put_at = [&](typename P::Vec* dst, int64_t row, const float (&cd)[8]) {
      typename P::Vec out = P::pack(cd);
      if (kHalfClamp) out = clamp_half8(out);
      if (in_bounds(row < rows, status)) *dst = out;
    };
    // (every scale in the division's fast range, the usual case: a loop with
    // no fallback branch in it)
    auto run = [&](auto fast_tag) {
      constexpr bool kFast = decltype(fast_tag)::value;
      auto divide = [&](const float (&f)[8], float (&v)[8]) {
        if (kFast)
          (void)div8_each_try2(f, s, r, true, v);
        else if (!div8_each_try2(f, s, r, all_fast, v))
          div8_each_ieee(f, s, v);
      };
      uint4 cur0 = ld_at(xp, row0), cur1 = ld_at(xp + xstep, row0 + 8);
      uint4 nxt0 = ld_at(xp + 2 * xstep, row0 + 16), nxt1 = ld_at(xp + 3 * xstep, row0 + 24);
#pragma unroll 2
      for (int64_t rr = row0; rr < r1; rr += 16) {
        // the loads of the pair after next: two pairs of rows in flight
        const uint4 nn0 = ld_at(xp + 4 * xstep, rr + 32), nn1 = ld_at(xp + 5 * xstep, rr + 40);
        uint32_t w_a[8], w_b[8];
        philox_words8x2(sr.keys, sr.stream, n, n + nstep, w_a, w_b);
        float f[8], v[8], cd[8];
        unpack8(cur0, f);
        divide(f, v);
        codes_sr8<!kHalfClamp>(v, w_a, cd);
        put_at(qp, rr, cd);
        if (rr + 8 < r1) {
          unpack8(cur1, f);
          divide(f, v);
          codes_sr8<!kHalfClamp>(v, w_b, cd);
          put_at(qp + qstep, rr + 8, cd);
        }
        cur0 = nxt0;
        cur1 = nxt1;
        nxt0 = nn0;
        nxt1 = nn1;
        xp += 2 * xstep;
        qp += 2 * qstep;
        n += 2 * nstep;
      }
    };
    if (all_fast)
      run(std::true_type{});
    else
      run(std::false_type{});
    return;
  }
  if (!SR && all_fast && normal) {
    // nearest-even codes, every scale in the division's fast range (and a
    // normal number): no branch per row
    for (int64_t rr = r0 + warp; rr < r1; rr += kNatUnroll * 8) {
      uint4 a[kNatUnroll];
#pragma unroll
      for (int u = 0; u < kNatUnroll; ++u) a[u] = load_row(rr + u * 8);
#pragma unroll
      for (int u = 0; u < kNatUnroll; ++u) {
        const int64_t row = rr + u * 8;
        if (row < r1) {
          float f[8], v[8], cd[8];
          unpack8(a[u], f);
          (void)div8_each_try(f, s, r, true, v);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 qv = code_rne_normal_scale2(make_float2(v[2 * i], v[2 * i + 1]));
            cd[2 * i] = qv.x;
            cd[2 * i + 1] = qv.y;
          }
          put(row, cd);
        }
      }
    }
    return;
  }
  for (int64_t rr = r0 + warp; rr < r1; rr += kNatUnroll * 8) {
    uint4 a[kNatUnroll];
#pragma unroll
    for (int u = 0; u < kNatUnroll; ++u) a[u] = load_row(rr + u * 8);
#pragma unroll
    for (int u = 0; u < kNatUnroll; u += 2) {
      const int64_t row_a = rr + u * 8, row_b = row_a + 8;
      const uint64_t n_a = sr.offset + static_cast<uint64_t>(row_a * cols + c);
      const uint64_t n_b = sr.offset + static_cast<uint64_t>(row_b * cols + c);
      if (SR && row_b < r1 && ((n_a | n_b) & 3u) == 0) {
        // stochastic codes of two rows: their four Philox blocks side by side
        float f_a[8], f_b[8], v_a[8], v_b[8], cd[8];
        unpack8(a[u], f_a);
        unpack8(a[u + 1], f_b);
        if (!div8_each_try(f_a, s, r, all_fast, v_a)) div8_each_ieee(f_a, s, v_a);
        if (!div8_each_try(f_b, s, r, all_fast, v_b)) div8_each_ieee(f_b, s, v_b);
        uint32_t w_a[8], w_b[8];
        philox_words8x2(sr.keys, sr.stream, n_a, n_b, w_a, w_b);
        codes_sr8<!kHalfClamp>(v_a, w_a, cd);
        put(row_a, cd);
        codes_sr8<!kHalfClamp>(v_b, w_b, cd);
        put(row_b, cd);
        continue;
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t row = row_a + 8 * e;
        if (row < r1) {
          float f[8], v[8], cd[8];
          unpack8(a[u + e], f);
          if (!div8_each_try(f, s, r, all_fast, v)) div8_each_ieee(f, s, v);
          codes_of<SR, !kHalfClamp>(v, sr.keys, sr.stream,
                                    sr.offset + static_cast<uint64_t>(row * cols + c), normal, cd);
          put(row, cd);
        }
      }
    }
  }
}

// Column groups of a matrix of at most kClMaxRows (2048) rows in ONE launch, codes
// in the input's layout (instead of zero, absmax, scale and codes as four).
// A cluster of kClCtas CTAs owns a strip of 64 columns; CTA k of it holds
// the rows (p kClCtas + k) 32 + t/8, p < kU, in registers (thread t: the
// 16-byte vector t % 8 of the strip; eight lanes read a row's whole 128-byte
// segment).  Each CTA reduces its maxima, the cluster exchanges the eight
// partial maxima through distributed shared memory, and every CTA forms the
// strip's scales and codes its own rows without reading x again: the same
// numbers as the three passes.
constexpr int kClCtas = 8;                          // CTAs of a cluster
constexpr int kClVecs = 8;                          // 16-byte vectors per strip row
constexpr int kClRows = kThreads / kClVecs;         // rows per CTA and pass
constexpr int kClMaxU = 8;                          // passes (16-byte loads) per thread
constexpr int64_t kClMaxRows = static_cast<int64_t>(kClCtas) * kClRows * kClMaxU;  // 2048

// One matrix of a launch of the kernel below (x bf16 [rows, cols], stride
// ld; codes q [rows, cols]; scale [cols]; SR counters from offset on stream).
struct ColsJob {
  const uint16_t* x;
  int64_t rows, ld;
  void* q;
  float* scale;
  uint64_t offset;
  PhiloxStream stream;
};

// Strips 0 .. split - 1 (blockIdx.x) belong to matrix j0, the rest to j1:
// every CTA of a cluster shares blockIdx.x, so a cluster stays within one
// matrix.
template <typename CodeT, bool SR, int kU>
__global__ void __cluster_dims__(1, kClCtas, 1) __launch_bounds__(kThreads)
    quant_cols_cluster_kernel(ColsJob j0, ColsJob j1, int split, int64_t cols, PhiloxKeys keys,
                              unsigned int* status) {
  using P = Pack8<CodeT>;
  __shared__ uint4 red[kThreads / 32][kClVecs];
  __shared__ uint4 part[kClVecs];  // this CTA's maxima of the strip's 64 columns
  const bool second = static_cast<int>(blockIdx.x) >= split;
  const uint16_t* __restrict__ x = second ? j1.x : j0.x;
  const int64_t rows = second ? j1.rows : j0.rows;
  const int64_t ld = second ? j1.ld : j0.ld;
  CodeT* __restrict__ q = static_cast<CodeT*>(second ? j1.q : j0.q);
  float* __restrict__ scale = second ? j1.scale : j0.scale;
  const uint64_t offset = second ? j1.offset : j0.offset;
  const PhiloxStream st = second ? j1.stream : j0.stream;
  const int64_t strip = second ? blockIdx.x - split : blockIdx.x;
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int vec = threadIdx.x % kClVecs, rsub = threadIdx.x / kClVecs;
  const int64_t k = blockIdx.y;  // the CTA's rank in its cluster (grid y = kClCtas)
  const int64_t c = strip * (8 * kClVecs) + 8 * vec;
  // no thread leaves early: every one reaches the cluster barriers
  const bool col_ok =
      c + 8 <= cols && in_bounds(cols <= ld && rows <= static_cast<int64_t>(kClCtas) * kClRows * kU,
                                 status);
  const int64_t pass_rows = static_cast<int64_t>(kClCtas) * kClRows;  // rows between p and p+1
  const int64_t row0 = k * kClRows + rsub;
  uint4 a[kU];
  uint4 m = make_uint4(0u, 0u, 0u, 0u);  // packed |x| maxima (bf16 bits), columns 2i, 2i+1
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int64_t r = row0 + u * pass_rows;
    a[u] = col_ok && r < rows ? __ldg(reinterpret_cast<const uint4*>(x + r * ld + c))
                              : make_uint4(0u, 0u, 0u, 0u);
    colmax_acc(m, abs_bits8(a[u]));
  }
  // lanes with the same vector differ in lane bits 3 and 4
#pragma unroll
  for (int o = kClVecs; o < 32; o <<= 1) {
    m.x = __vmaxu2(m.x, __shfl_xor_sync(0xFFFFFFFFu, m.x, o));
    m.y = __vmaxu2(m.y, __shfl_xor_sync(0xFFFFFFFFu, m.y, o));
    m.z = __vmaxu2(m.z, __shfl_xor_sync(0xFFFFFFFFu, m.z, o));
    m.w = __vmaxu2(m.w, __shfl_xor_sync(0xFFFFFFFFu, m.w, o));
  }
  if (lane < kClVecs) red[warp][lane] = m;
  __syncthreads();
  if (threadIdx.x < kClVecs) {
    uint4 t = red[0][threadIdx.x];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) colmax_acc(t, red[w][threadIdx.x]);
    part[threadIdx.x] = t;
  }
  ptx::cluster_arrive_release();
  ptx::cluster_wait_acquire();  // every CTA's part[] is written
  m = make_uint4(0u, 0u, 0u, 0u);
  const uint32_t mine = ptx::smem_addr(&part[vec]);
#pragma unroll
  for (int j = 0; j < kClCtas; ++j) colmax_acc(m, ptx::ld_shared_cluster_v4(ptx::mapa_shared(mine, j)));
  ptx::cluster_arrive_release();  // done reading the peers' part[]
  const uint32_t mw[4] = {m.x, m.y, m.z, m.w};
  float s[8], r[8];
  bool all_fast = true, normal = true;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t bits = (j & 1) ? (mw[j >> 1] & 0xFFFF0000u) : (mw[j >> 1] << 16);
    s[j] = __fdiv_rn(__uint_as_float(bits), 127.0f);
    all_fast = all_fast && scale_is_fast(s[j]);
    normal = normal && scale_is_normal(s[j]);
    r[j] = __frcp_rn(s[j]);
  }
  if (k == 0 && rsub == 0 && col_ok) {
#pragma unroll
    for (int j = 0; j < 8; ++j) scale[c + j] = s[j];
  }
  // f16 stochastic codes are clamped as packed half2 after the conversion
  constexpr bool kHalfClamp = SR && std::is_same<CodeT, __half>::value;
  const uint64_t n0 = offset + static_cast<uint64_t>(c);  // SR counter of (row 0, column c)
  auto put = [&](int64_t row, const float (&cd)[8]) {
    typename P::Vec out = P::pack(cd);
    if (kHalfClamp) out = clamp_half8(out);
    if (in_bounds(row < rows, status))
      *reinterpret_cast<typename P::Vec*>(q + row * cols + c) = out;
  };
  auto divide = [&](const uint4& in, float (&v)[8]) {
    float f[8];
    unpack8(in, f);
    if (!div8_each_try2(f, s, r, all_fast, v)) div8_each_ieee(f, s, v);
  };
  if (col_ok) {
    if (SR && (offset & 3u) == 0) {
      // every group of eight starts a Philox block: two rows' blocks side by side
#pragma unroll
      for (int u = 0; u < kU; u += 2) {
        const int64_t ra = row0 + u * pass_rows, rb = ra + pass_rows;
        if (ra < rows) {
          uint32_t wa[8], wb[8];
          philox_words8x2(keys, st, n0 + static_cast<uint64_t>(ra * cols),
                          n0 + static_cast<uint64_t>(rb * cols), wa, wb);
          float v[8], cd[8];
          divide(a[u], v);
          codes_sr8<!kHalfClamp>(v, wa, cd);
          put(ra, cd);
          if (rb < rows) {
            divide(a[u + 1], v);
            codes_sr8<!kHalfClamp>(v, wb, cd);
            put(rb, cd);
          }
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t row = row0 + u * pass_rows;
        if (row < rows) {
          float v[8], cd[8];
          divide(a[u], v);
          if (!SR && all_fast && normal) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 qv = code_rne_normal_scale2(make_float2(v[2 * i], v[2 * i + 1]));
              cd[2 * i] = qv.x;
              cd[2 * i + 1] = qv.y;
            }
          } else {
            codes_of<SR, !kHalfClamp>(v, keys, st, n0 + static_cast<uint64_t>(row * cols),
                                      normal, cd);
          }
          put(row, cd);
        }
      }
    }
  }
  ptx::cluster_wait_acquire();  // no CTA exits while a peer may still read its part[]
}

// Pass 3: codes, one warp per 32-row x 64-column sub-tile at a time.  Each
// warp keeps its own two-slot ring of sub-tiles filled by 2-D TMA loads
// (rows of 128 bytes, no swizzle) and its own staging tile for the
// transposed codes, so warps never wait for one another.  Lane (rg, cg)
// reads rows rg*8 .. rg*8+7 of column group cg (8 columns, one 16-byte
// vector per row), quantizes the 8x8 block, packs the codes column by
// column, and writes the 8 column vectors to staging rows cg*8 .. cg*8+7
// (one per column of x, i.e. per row of the transposed output).  Shared
// memory serves 16-byte accesses eight lanes at a time and 8-byte accesses
// sixteen at a time; the staging row and slot permutations below give every
// such group distinct banks, for the writes and for the row-wise read-out.
// The read-out stores 8-code vectors of the transposed rows.
constexpr int kCwRows = 32, kCwCols = 64;
constexpr uint32_t kCwInBytes = kCwRows * kCwCols * 2;

template <typename CodeT>
struct ColPack;
template <>
struct ColPack<int8_t> {
  using Vec = uint2;
  // rows 2p, 2p+1 of the 8-row block: bytes 2p, 2p+1 of the column vector
  __device__ __forceinline__ static void put2(Vec& v, int p, float a, float b) {
    const uint32_t two = (static_cast<uint32_t>(__float2int_rn(a)) & 0xFFu) |
                         ((static_cast<uint32_t>(__float2int_rn(b)) & 0xFFu) << 8);
    if (p < 2) v.x |= two << (16 * p); else v.y |= two << (16 * (p - 2));
  }
};
template <>
struct ColPack<__half> {
  using Vec = uint4;
  __device__ __forceinline__ static void put2(Vec& v, int p, float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    const uint32_t u = *reinterpret_cast<const uint32_t*>(&h);
    switch (p) {
      case 0: v.x = u; break;
      case 1: v.y = u; break;
      case 2: v.z = u; break;
      default: v.w = u; break;
    }
  }
};

template <typename CodeT>
__host__ __device__ constexpr uint32_t col_warp_bytes() {
  return 2 * kCwInBytes + 64 * 4 * static_cast<uint32_t>(sizeof(typename ColPack<CodeT>::Vec));
}

// staging position of (row rho, slot) of the transposed output
template <typename CodeT>
struct Staging;
template <>
struct Staging<__half> {  // 64-byte rows of four 16-byte slots
  __device__ __forceinline__ static int row(int rho) { return rho ^ ((rho >> 3) & 1); }
  __device__ __forceinline__ static int slot(int rho, int sl) { return sl ^ ((rho >> 4) & 3); }
};
template <>
struct Staging<int8_t> {  // 32-byte rows of four 8-byte slots
  __device__ __forceinline__ static int row(int rho) { return rho ^ ((rho >> 3) & 3); }
  __device__ __forceinline__ static int slot(int rho, int sl) { return sl ^ (((rho >> 5) & 1) << 1); }
};

template <typename CodeT, bool SR>
__global__ void __launch_bounds__(kThreads, 2) quant_cols_kernel(
    const __grid_constant__ CUtensorMap tmx, int64_t rows, int64_t cols,
    const float* __restrict__ scale, CodeT* __restrict__ q, int64_t col_tiles, int64_t tiles,
    SrArgs sr, unsigned int* status, uint64_t limit_ns) {
  using CP = ColPack<CodeT>;
  using Vec = typename CP::Vec;
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ uint64_t bars[kThreads / 32][2];
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cg = lane & 7, rg = lane >> 3;
  uint8_t* in = smem + warp * col_warp_bytes<CodeT>();
  const uint32_t in_addr = ptx::smem_addr(in);
  Vec(*out)[4] = reinterpret_cast<Vec(*)[4]>(in + 2 * kCwInBytes);
  const uint32_t bar[2] = {ptx::smem_addr(&bars[warp][0]), ptx::smem_addr(&bars[warp][1])};
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + warp;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * (kThreads / 32);

  uint32_t pending = 0u, pend_par = 0u;  // lane 0 only
  auto issue = [&](int b, int64_t t) {
    ptx::mbar_arrive_expect_tx(bar[b], kCwInBytes);
    ptx::tma_load_2d(in_addr + b * kCwInBytes, &tmx, bar[b],
                     static_cast<int32_t>((t % col_tiles) * kCwCols),
                     static_cast<int32_t>((t / col_tiles) * kCwRows));
  };
  if (lane == 0) {
    ptx::mbar_init(bar[0], 1);
    ptx::mbar_init(bar[1], 1);
    ptx::fence_mbar_init();
    for (int k = 0; k < 2; ++k) {
      const int64_t t = gw + k * nw;
      if (t < tiles) {
        issue(k, t);
        pending |= 1u << k;
      }
    }
  }
  __syncwarp();
  int64_t cur_cb = -1;
  float s[8], r[8];
  bool all_fast = false, normal = false;
  int it = 0;
  for (int64_t t = gw; t < tiles; t += nw, ++it) {
    const int b = it & 1;
    int got = 1;
    if (lane == 0) {
      got = ptx::mbar_wait_timeout(bar[b], (it >> 1) & 1, limit_ns) ? 1 : 0;
      if (got) pending &= ~(1u << b);
      else atomicOr(status, 1u);
    }
    got = __shfl_sync(0xFFFFFFFFu, got, 0);
    if (!got) break;
    const int64_t cb = t % col_tiles, r0 = (t / col_tiles) * kCwRows, c0 = cb * kCwCols;
    const int64_t c = c0 + cg * 8, rb = r0 + rg * 8;
    if (cb != cur_cb) {
      cur_cb = cb;
      all_fast = true;
      normal = true;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s[j] = c < cols ? __ldg(scale + c + j) : 1.0f;
        all_fast = all_fast && scale_is_fast(s[j]);
        normal = normal && scale_is_normal(s[j]);
        r[j] = __frcp_rn(s[j]);
      }
    }
    Vec colv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) colv[j] = Vec{};
    if (c < cols) {
      const uint8_t* src = in + b * kCwInBytes + (rg * 8) * 128 + cg * 16;
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // rows 4h .. 4h+3 of the 8-row block
        float quo[4][8];             // [row][column]
        bool ok = true;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float f[8];
          unpack8(*reinterpret_cast<const uint4*>(src + (4 * h + i) * 128), f);
          ok = div8_each_try(f, s, r, all_fast, quo[i]) && ok;
        }
        if (!ok) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float f[8];
            unpack8(*reinterpret_cast<const uint4*>(src + (4 * h + i) * 128), f);
            div8_each_ieee(f, s, quo[i]);
          }
        }
#pragma unroll
        for (int p = 0; p < 2; ++p) {  // row pairs (4h+2p, 4h+2p+1)
          float cd[2][8];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = 4 * h + 2 * p + e;
            codes_of<SR>(quo[2 * p + e], sr.keys, sr.stream,
                         sr.offset + static_cast<uint64_t>((rb + i) * cols + c), normal, cd[e]);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) CP::put2(colv[j], 2 * h + p, cd[0][j], cd[1][j]);
        }
      }
    }
    __syncwarp();  // every lane has read slot b
    if (lane == 0) {
      const int64_t nt = t + 2 * nw;
      if (nt < tiles) {
        ptx::fence_proxy_async_smem();
        issue(b, nt);
        pending |= 1u << b;
        pend_par = (pend_par & ~(1u << b)) | (static_cast<uint32_t>(((it + 2) >> 1) & 1) << b);
      }
    }
    using SG = Staging<CodeT>;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int rho = cg * 8 + j;
      out[SG::row(rho)][SG::slot(rho, rg)] = colv[j];
    }
    __syncwarp();
    // read-out: 8 staging rows per step, 4 lanes (32 codes) per row
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int rho = k * 8 + (lane >> 2), slot = lane & 3;
      const int64_t cc = c0 + rho, rr = r0 + slot * 8;
      if (cc < cols && rr < rows && in_bounds(rr + 8 <= rows, status))
        *reinterpret_cast<Vec*>(q + cc * rows + rr) = out[SG::row(rho)][SG::slot(rho, slot)];
    }
    __syncwarp();  // the staging tile may be rewritten
  }
  if (lane == 0) {
    for (int k = 0; k < 2; ++k)
      if (pending & (1u << k))
        if (!ptx::mbar_wait_timeout(bar[k], (pend_par >> k) & 1u, limit_ns)) atomicOr(status, 1u);
  }
}

// ------------------------------------------------------------------ host
// Resident blocks per SM of a kernel at a given dynamic shared-memory size.
template <typename Kernel>
int blocks_per_sm(Kernel k, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess || n < 1)
    n = 1;
  return n;
}

constexpr size_t kMaxDynSmem = 200 * 1024;

// per-device "dynamic shared memory attribute set" flags, one set per kernel
template <typename Kernel>
cudaError_t allow_smem(Kernel k, bool* done) {
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMaxDynSmem));
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

// One wave of blocks of 32 8-column vectors x rows_per_block rows (a
// multiple of `row_quantum`), for the passes that walk columns.
struct ColGrid {
  unsigned gx, gy;
  int64_t rows_per_block;
};
ColGrid col_grid(int64_t rows, int64_t cols, int64_t blocks_target, int64_t row_quantum) {
  const int64_t gx = ((cols >> 3) + 31) / 32;
  int64_t gy = blocks_target / gx;
  const int64_t max_gy = (rows + 63) / 64;
  if (gy > max_gy) gy = max_gy;
  if (gy < 1) gy = 1;
  if (gy > 65535) gy = 65535;
  int64_t rpb = (rows + gy - 1) / gy;
  rpb = (rpb + row_quantum - 1) / row_quantum * row_quantum;
  gy = (rows + rpb - 1) / rpb;
  return ColGrid{static_cast<unsigned>(gx), static_cast<unsigned>(gy), rpb};
}

// column absmax merged into amax_bits (atomic max), pass 1 of the columns
cudaError_t launch_col_absmax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                              unsigned int* amax_bits, const DeviceInfo& dev, cudaStream_t stream) {
  static const int occ1 = blocks_per_sm(col_absmax_kernel, kThreads, 0);
  const int sms = dev.sms > 0 ? dev.sms : 148;
  const ColGrid g1 = col_grid(rows, cols, static_cast<int64_t>(sms) * occ1, 1);
  return launch_overlapped(col_absmax_kernel, dim3(g1.gx, g1.gy), dim3(kThreads), 0, stream, x,
                           rows, cols, ld, g1.rows_per_block, amax_bits, dev.status_word);
}

// Row groups; with colmax != nullptr also max-merge each column's absmax
// into colmax (in the same pass when every thread's share of a row fits
// its registers, else by a separate column pass).
template <typename CodeT, bool SR>
cudaError_t rows_dispatch(const RowsJob* jobs, int njobs, int64_t cols, const SrArgs& base,
                          const DeviceInfo& dev, cudaStream_t stream) {
  const bool cm = jobs[0].colmax != nullptr;
  const int sms = dev.sms > 0 ? dev.sms : 148;
  const uint32_t slot = static_cast<uint32_t>((cols * 2 + 127) / 128 * 128);
  // the stochastic-rounding parameters of job j: the seed's keys, its own
  // offset and stream
  auto sr_of = [&](const RowsJob& j) {
    SrArgs s = base;
    s.offset = j.offset;
    s.stream_id = j.stream_id;
    s.stream = philox_stream(j.stream_id);
    return s;
  };
  auto col_pass = [&](const RowsJob& j) {
    return launch_col_absmax(static_cast<const uint16_t*>(j.x), j.rows, cols, j.ld,
                             reinterpret_cast<unsigned int*>(j.colmax), dev, stream);
  };
  // blocks [0, split) take job 0 and [split, blocks) job 1, in proportion
  // to their rows when the two need more than one wave of blocks (`per`:
  // rows a block takes at a time; `cap`: blocks of one wave)
  auto plan = [&](int64_t per, int64_t cap, int64_t* split, int64_t* blocks) {
    auto need = [&](const RowsJob& j) { return (j.rows + per - 1) / per; };
    if (njobs == 1) {
      *split = *blocks = need(jobs[0]) < cap ? need(jobs[0]) : cap;
    } else if (need(jobs[0]) + need(jobs[1]) <= cap) {
      *split = need(jobs[0]);
      *blocks = *split + need(jobs[1]);
    } else {
      *blocks = cap;
      const double share = static_cast<double>(jobs[0].rows) / (jobs[0].rows + jobs[1].rows);
      *split = static_cast<int64_t>(share * cap + 0.5);
      if (*split < 1) *split = 1;
      if (*split > cap - 1) *split = cap - 1;
    }
  };
  auto second_job = [&](int64_t split, bool with_colmax) {
    RowsJob2 j2{nullptr, 0, 0, nullptr, nullptr, nullptr, 0, PhiloxStream{0u, 0u},
                static_cast<int>(split)};
    if (njobs > 1) {
      const RowsJob& j1 = jobs[1];
      j2 = RowsJob2{static_cast<const uint16_t*>(j1.x), j1.rows, j1.ld, j1.q, j1.scale,
                    with_colmax ? reinterpret_cast<unsigned int*>(j1.colmax) : nullptr,
                    j1.offset, philox_stream(j1.stream_id), static_cast<int>(split)};
    }
    return j2;
  };
  if (!cm && cols <= 256 * kRegMaxV) {
    // short rows, no column maxima: one warp per row, the row in registers
    auto kernel = cols <= 256   ? quant_rows_reg_kernel<CodeT, SR, 1>
                  : cols <= 512 ? quant_rows_reg_kernel<CodeT, SR, 2>
                  : cols <= 1024 ? quant_rows_reg_kernel<CodeT, SR, 4>
                                 : quant_rows_reg_kernel<CodeT, SR, kRegMaxV>;
    const int occ = blocks_per_sm(kernel, kRegThreads, 0);
    int64_t split, blocks;
    plan(kRegThreads / 32, static_cast<int64_t>(sms) * occ, &split, &blocks);
    const RowsJob& j0 = jobs[0];
    return launch_overlapped(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kRegThreads), 0,
                             stream, static_cast<const uint16_t*>(j0.x), j0.rows, cols, j0.ld,
                             static_cast<CodeT*>(j0.q), j0.scale, sr_of(j0), dev.status_word,
                             second_job(split, false));
  }
  if (2ull * slot > kMaxDynSmem) {
    for (int i = 0; i < njobs; ++i) {
      const RowsJob& j = jobs[i];
      cudaError_t e = launch_overlapped(quant_rows_long_kernel<CodeT, SR>,
                                        dim3(static_cast<unsigned>(j.rows)), dim3(kThreads), 0,
                                        stream, static_cast<const uint16_t*>(j.x), j.rows, cols,
                                        j.ld, static_cast<CodeT*>(j.q), j.scale, sr_of(j),
                                        dev.status_word);
      if (e == cudaSuccess && cm) e = col_pass(j);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  // 8 warps per block in teams of T, each team with a ring of S row slots
  // (S - 1 rows in flight while it works on one).  Shared memory per block:
  // 72 KB, so that three blocks share an SM, or 108 KB for the variant that
  // also keeps column maxima (its registers allow two blocks per SM).  T is
  // the smallest whose two slots per team fit (and, for the column maxima,
  // whose threads' share of a row fits their registers); S fills the rest.
  const int warps = kThreads / 32;
  const size_t budget = cm ? 108u * 1024u : 72u * 1024u;
  int T = 1;
  while (T < 8 && (static_cast<size_t>(warps / T) * 2 * slot > budget ||
                   (cm && (cols >> 3) > static_cast<int64_t>(kColVecs) * 32 * T)))
    T <<= 1;
  const bool fused = cm && (cols >> 3) <= static_cast<int64_t>(kColVecs) * 32 * T &&
                     static_cast<size_t>(warps / T) * 2 * slot <= budget;
  if (cm && !fused) {  // the plain ring and a separate column pass
    T = 1;
    while (T < 8 && static_cast<size_t>(warps / T) * 2 * slot > 72u * 1024u) T <<= 1;
  }
  const size_t team_bytes = static_cast<size_t>(warps / T) * slot;
  int S = static_cast<int>((fused ? budget : 72u * 1024u) / team_bytes);
  if (S > kMaxSlots) S = kMaxSlots;
  if (S < 2) S = 2;
  const size_t smem = team_bytes * S;
  const int64_t teams = warps / T;
  auto kernel = fused ? quant_rows_kernel<CodeT, SR, true> : quant_rows_kernel<CodeT, SR, false>;
  static bool attr_fused[64] = {}, attr_plain[64] = {};
  cudaError_t e = allow_smem(kernel, fused ? attr_fused : attr_plain);
  if (e != cudaSuccess) return e;
  const int occ = blocks_per_sm(kernel, kThreads, smem);
  int64_t split, blocks;
  plan(teams, static_cast<int64_t>(sms) * occ, &split, &blocks);
  const RowsJob& j0 = jobs[0];
  const RowsJob2 j2 = second_job(split, fused);
  e = launch_overlapped(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), smem, stream,
                        static_cast<const uint16_t*>(j0.x), j0.rows, cols, j0.ld,
                        static_cast<CodeT*>(j0.q), j0.scale, sr_of(j0), slot, T, S,
                        dev.status_word, kWaitLimitNs,
                        fused ? reinterpret_cast<unsigned int*>(j0.colmax) : nullptr, j2);
  if (e != cudaSuccess || !cm || fused) return e;
  for (int i = 0; i < njobs && e == cudaSuccess; ++i) e = col_pass(jobs[i]);
  return e;
}

template <typename CodeT, bool SR, bool kFromAbsmax>
cudaError_t launch_cols_nat(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                            const float* in, float* scale_out, CodeT* q, const SrArgs& sr,
                            const DeviceInfo& dev, cudaStream_t stream) {
  static const int occ = blocks_per_sm(quant_cols_nat_kernel<CodeT, SR, kFromAbsmax>, kThreads, 0);
  const int sms = dev.sms > 0 ? dev.sms : 148;
  const ColGrid g = col_grid(rows, cols, static_cast<int64_t>(sms) * occ, 8 * kNatUnroll);
  return launch_overlapped(quant_cols_nat_kernel<CodeT, SR, kFromAbsmax>, dim3(g.gx, g.gy),
                           dim3(kThreads), 0, stream, x, rows, cols, ld, g.rows_per_block, in,
                           scale_out, q, sr, dev.status_word);
}

// The cluster kernel over njobs (1 or 2) matrices of at most kClMaxRows rows
// and `cols` columns each, in one launch.
template <typename CodeT, bool SR>
cudaError_t launch_cols_cluster(const ColsJob& j0, const ColsJob& j1, int njobs, int64_t cols,
                                const PhiloxKeys& keys, const DeviceInfo& dev,
                                cudaStream_t stream) {
  const int64_t strips = (cols + 8 * kClVecs - 1) / (8 * kClVecs);
  const dim3 grid(static_cast<unsigned>(strips * njobs), kClCtas);
  const int64_t rows = njobs > 1 && j1.rows > j0.rows ? j1.rows : j0.rows;
  const int64_t per_u = static_cast<int64_t>(kClCtas) * kClRows;  // 256 rows
  const int split = static_cast<int>(strips);
  return rows <= per_u * 4
             ? launch_overlapped(quant_cols_cluster_kernel<CodeT, SR, 4>, grid, dim3(kThreads), 0,
                                 stream, j0, j1, split, cols, keys, dev.status_word)
             : launch_overlapped(quant_cols_cluster_kernel<CodeT, SR, kClMaxU>, grid,
                                 dim3(kThreads), 0, stream, j0, j1, split, cols, keys,
                                 dev.status_word);
}

template <typename CodeT, bool SR>
cudaError_t cols_dispatch(const void* x, int64_t rows, int64_t cols, int64_t ld, void* q,
                          float* scale, bool transposed, const SrArgs& sr, const DeviceInfo& dev,
                          cudaStream_t stream) {
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  if (!transposed && rows <= kClMaxRows) {
    // up to 2048 rows: one launch, each column strip's rows held in the
    // registers of one cluster (at 4096 rows the three passes were faster:
    // 4096^2 operands 41 us instead of 37)
    const ColsJob j{xp, rows, ld, q, scale, sr.offset, sr.stream};
    const cudaError_t e = launch_cols_cluster<CodeT, SR>(j, j, 1, cols, sr.keys, dev, stream);
    if (e == cudaSuccess) return e;
    // the cluster launch was refused (e.g. no eight-CTA cluster fits the
    // stream's SM partition): clear that error and take the passes, whose
    // launches report any error that persists
    (void)cudaGetLastError();
  }
  unsigned int* amax = reinterpret_cast<unsigned int*>(scale);
  cudaError_t err = launch_zero_words(amax, cols, dev, stream);
  if (err != cudaSuccess) return err;
  const int sms = dev.sms > 0 ? dev.sms : 148;
  // pass 1: one wave of blocks
  err = launch_col_absmax(xp, rows, cols, ld, amax, dev, stream);
  if (err != cudaSuccess) return err;
  err = launch_overlapped(col_scale_kernel, dim3(static_cast<unsigned>((cols + 255) / 256)),
                          dim3(256), 0, stream, amax, cols);
  if (err != cudaSuccess) return err;
  if (!transposed) {
    // pass 3 in the input's layout: one wave, whole 32-row steps per block
    return launch_cols_nat<CodeT, SR, false>(xp, rows, cols, ld, scale, nullptr,
                                             static_cast<CodeT*>(q), sr, dev, stream);
  }
  CUtensorMap tmx;
  if (!encode_tensor_map_2d(&tmx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, cols, ld,
                            kCwCols, kCwRows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  static bool attr[64] = {};
  err = allow_smem(quant_cols_kernel<CodeT, SR>, attr);
  if (err != cudaSuccess) return err;
  // pass 3 transposed: persistent warps over 32x64 sub-tiles, column-block fastest
  const int64_t col_tiles = (cols + kCwCols - 1) / kCwCols;
  const int64_t tiles = col_tiles * ((rows + kCwRows - 1) / kCwRows);
  const size_t smem = 1024 + (kThreads / 32) * col_warp_bytes<CodeT>();
  static const int occ3 = blocks_per_sm(quant_cols_kernel<CodeT, SR>, kThreads, smem);
  const int64_t need = (tiles + kThreads / 32 - 1) / (kThreads / 32);
  const int64_t cap = static_cast<int64_t>(sms) * occ3;
  int64_t blocks = need < cap ? need : cap;
  // a warp count that is a multiple of the column blocks keeps every warp on
  // one column block (its scales are loaded once)
  const int64_t wpb = kThreads / 32;
  if (blocks * wpb >= col_tiles) {
    const int64_t warps = blocks * wpb / col_tiles * col_tiles;
    blocks = (warps + wpb - 1) / wpb;
    if (blocks * wpb != warps) {
      // round down to whole blocks whose warp count is still a multiple
      int64_t b = blocks;
      while (b > 1 && (b * wpb) % col_tiles != 0) --b;
      if ((b * wpb) % col_tiles == 0) blocks = b;
    }
  }
  return launch_overlapped(quant_cols_kernel<CodeT, SR>, dim3(static_cast<unsigned>(blocks)),
                           dim3(kThreads), smem, stream, tmx, rows, cols, scale,
                           static_cast<CodeT*>(q), col_tiles, tiles, sr, dev.status_word,
                           kWaitLimitNs);
}

}  // namespace

namespace {
cudaError_t rows_jobs(const RowsJob* jobs, int njobs, int64_t cols, int8mp_round mode,
                      const SrArgs& base, int8mp_codes codes, const DeviceInfo& dev,
                      cudaStream_t stream) {
  const bool s = mode == INT8MP_SR;
  if (codes == INT8MP_CODES_S8)
    return s ? rows_dispatch<int8_t, true>(jobs, njobs, cols, base, dev, stream)
             : rows_dispatch<int8_t, false>(jobs, njobs, cols, base, dev, stream);
  return s ? rows_dispatch<__half, true>(jobs, njobs, cols, base, dev, stream)
           : rows_dispatch<__half, false>(jobs, njobs, cols, base, dev, stream);
}
}  // namespace

cudaError_t launch_quantize_rows(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                 int8mp_round mode, const SrArgs& sr, void* q,
                                 int8mp_codes codes, float* scale, float* colmax,
                                 const DeviceInfo& dev, cudaStream_t stream) {
  const RowsJob job{x, rows, ld, q, scale, colmax, sr.offset, sr.stream_id};
  return rows_jobs(&job, 1, cols, mode, sr, codes, dev, stream);
}

cudaError_t launch_quantize_rows_jobs(const RowsJob* jobs, int njobs, int64_t cols,
                                      int8mp_round mode, uint64_t seed, int8mp_codes codes,
                                      const DeviceInfo& dev, cudaStream_t stream) {
  if (njobs < 1 || njobs > kMaxRowsJobs) return cudaErrorInvalidValue;
  return rows_jobs(jobs, njobs, cols, mode, make_sr(seed, 0, 0), codes, dev, stream);
}

cudaError_t launch_zero_words(void* p, int64_t n, const DeviceInfo& dev, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int sms = dev.sms > 0 ? dev.sms : 148;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4 * sms) blocks = 4 * sms;
  return launch_overlapped(zero_words_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                           stream, static_cast<unsigned int*>(p), n);
}

cudaError_t launch_round_bf16(const float* x, void* y, int64_t n, const DeviceInfo& dev,
                              cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int sms = dev.sms > 0 ? dev.sms : 148;
  int64_t blocks = (n / 8 + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 8 * sms) blocks = 8 * sms;
  return launch_overlapped(round_bf16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                           stream, x, static_cast<uint16_t*>(y), n);
}

cudaError_t launch_column_absmax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                 float* colmax, const DeviceInfo& dev, cudaStream_t stream) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  return launch_col_absmax(static_cast<const uint16_t*>(x), rows, cols, ld,
                           reinterpret_cast<unsigned int*>(colmax), dev, stream);
}

cudaError_t launch_quantize_cols_from_absmax(const void* x, int64_t rows, int64_t cols,
                                             int64_t ld, const float* absmax, int8mp_round mode,
                                             const SrArgs& sr, void* q, int8mp_codes codes,
                                             float* scale, const DeviceInfo& dev,
                                             cudaStream_t stream) {
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  const bool s = mode == INT8MP_SR;
  if (codes == INT8MP_CODES_S8) {
    int8_t* qp = static_cast<int8_t*>(q);
    return s ? launch_cols_nat<int8_t, true, true>(xp, rows, cols, ld, absmax, scale, qp, sr, dev, stream)
             : launch_cols_nat<int8_t, false, true>(xp, rows, cols, ld, absmax, scale, qp, sr, dev, stream);
  }
  __half* qp = static_cast<__half*>(q);
  return s ? launch_cols_nat<__half, true, true>(xp, rows, cols, ld, absmax, scale, qp, sr, dev, stream)
           : launch_cols_nat<__half, false, true>(xp, rows, cols, ld, absmax, scale, qp, sr, dev, stream);
}

cudaError_t launch_quantize_cols(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                 int8mp_round mode, const SrArgs& sr, void* q,
                                 int8mp_codes codes, float* scale, bool transposed,
                                 const DeviceInfo& dev, cudaStream_t stream) {
  const bool s = mode == INT8MP_SR;
  const bool t = transposed;
  if (codes == INT8MP_CODES_S8)
    return s ? cols_dispatch<int8_t, true>(x, rows, cols, ld, q, scale, t, sr, dev, stream)
             : cols_dispatch<int8_t, false>(x, rows, cols, ld, q, scale, t, sr, dev, stream);
  return s ? cols_dispatch<__half, true>(x, rows, cols, ld, q, scale, t, sr, dev, stream)
           : cols_dispatch<__half, false>(x, rows, cols, ld, q, scale, t, sr, dev, stream);
}

namespace {
template <typename CodeT, bool SR>
cudaError_t cols_jobs(const RowsJob* jobs, int njobs, int64_t cols, uint64_t seed,
                      const DeviceInfo& dev, cudaStream_t stream) {
  bool small = true;
  for (int i = 0; i < njobs; ++i) small = small && jobs[i].rows <= kClMaxRows;
  if (small) {
    ColsJob cj[kMaxRowsJobs];
    for (int i = 0; i < njobs; ++i) {
      const RowsJob& j = jobs[i];
      cj[i] = ColsJob{static_cast<const uint16_t*>(j.x), j.rows, j.ld, j.q, j.scale, j.offset,
                      philox_stream(j.stream_id)};
    }
    const cudaError_t e = launch_cols_cluster<CodeT, SR>(cj[0], cj[njobs > 1 ? 1 : 0], njobs, cols,
                                                         philox_keys(seed), dev, stream);
    if (e == cudaSuccess) return e;
    (void)cudaGetLastError();  // refused: the passes below
  }
  for (int i = 0; i < njobs; ++i) {
    const RowsJob& j = jobs[i];
    const cudaError_t e =
        cols_dispatch<CodeT, SR>(j.x, j.rows, cols, j.ld, j.q, j.scale, false,
                                 make_sr(seed, j.offset, j.stream_id), dev, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_quantize_cols_jobs(const RowsJob* jobs, int njobs, int64_t cols,
                                      int8mp_round mode, uint64_t seed, int8mp_codes codes,
                                      const DeviceInfo& dev, cudaStream_t stream) {
  if (njobs < 1 || njobs > kMaxRowsJobs) return cudaErrorInvalidValue;
  const bool s = mode == INT8MP_SR;
  if (codes == INT8MP_CODES_S8)
    return s ? cols_jobs<int8_t, true>(jobs, njobs, cols, seed, dev, stream)
             : cols_jobs<int8_t, false>(jobs, njobs, cols, seed, dev, stream);
  return s ? cols_jobs<__half, true>(jobs, njobs, cols, seed, dev, stream)
           : cols_jobs<__half, false>(jobs, njobs, cols, seed, dev, stream);
}

}  // namespace int8mp
