// gemm.cu -- scaled INT8 matmul on the sm_103a tensor cores.
//
// What it computes ("Quantized model training" README, INT8 mixed precision
// training: a scaled INT8 matmul; "Integrate INT8 mixed-precision from
// torchao 0.7": the product is scaled back to BF16):
//   acc[i,j] = sum_k qA[i,k] * qB[j,k]                 (exact int32)
//   out[i,j] = bf16_RNE((fp32_RN(acc) * sA[i]) * sB[j])  or acc itself.
// The same kernels also run the BF16 passes of the training table's mixed
// rows (a matmul left in BF16): bf16 operands, one fp32 accumulation over
// the whole contraction in tensor memory, out = bf16_RNE(acc).
//
// How: sm_103a has no INT8 tcgen05 MMA, so the codes arrive as f16 values
// (exact for |q| <= 127) and the contraction runs on tcgen05.mma.kind::f16
// with fp32 accumulation in tensor memory.  Every product is exact
// (|q q'| <= 16129) and so is every fp32 partial sum while its magnitude is
// below 2^24, which holds for any 1024 consecutive terms (127^2 * 1024 =
// 16,516,096 < 16,777,216).  The K loop therefore runs in chunks of at most
// 1024; each chunk lands in one of two TMEM accumulators, and the epilogue
// warps convert it (exactly) to int32 and add it into per-thread int32
// totals while the tensor core fills the other accumulator.
//
// Operands are K-major (contraction innermost: A [M,K], B [N,K]) or
// MN-major (A stored [K,M], B stored [K,N]); an MN-major operand arrives in
// 64-column TMA boxes and is described to the tensor core as such, so that
// column-grouped codes need no transposition.
//
// Structure (one persistent CTA per SM, 320 threads; tiles of 128 x 256, or
// 128 x 128 or 128 x 64 for launches with few tiles):
//   warp 0      TMA producer (one thread): 4-stage ring of 128x64 A and
//               256x64 B f16 tiles (6 and 8 stages with 128- and 64-row B
//               tiles), 128-byte swizzled, one mbarrier per stage
//   warp 1      TMEM allocator + MMA issuer (one thread): 4 MMAs of
//               128 x N x 16 per stage, commit frees the stage; commit after
//               each K-chunk hands the accumulator to the epilogue
//   warps 2-9   epilogue: warp w reads TMEM lanes 32*(w%4).. and one half
//               of the tile's columns (warps 2-5 the whole of a 64-column
//               tile), keeps an int32 total per column and thread, and writes
//               the finished tile through a 4 KB shared-memory staging
//               buffer with TMA tensor stores
// Every mbarrier wait is bounded (wall clock); a wait that runs out raises
// the CTA abort flag and the device status word, every role winds down,
// outstanding copies and MMAs are waited for (bounded), TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <mutex>

#include "check.cuh"
#include "codes.cuh"
#include "common.cuh"
#include "divide.cuh"
#include "ptx.cuh"

namespace int8mp {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;  // kBK f16 = 128 bytes per row
constexpr int kChunkBlocks = 16;  // 16 * 64 = 1024 terms per exact fp32 chunk
constexpr int kABytes = kBM * kBK * 2;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;  // CTA pair: two 128x256 fp32 accumulators per CTA
constexpr int kBarrierBytes = 256;
constexpr int kMnBlockBytes = 64 * kBK * 2;  // one 64 (M or N) x 64 (K) MN-major box
// each epilogue warp stages its outputs in 4 KB: one 32-row x 128-byte box
constexpr int kStoreBoxBytes = 32 * 128;
constexpr int kStagingBytes = kEpiWarps * kStoreBoxBytes;

struct GemmParams {
  const float* sA;
  const float* sB;
  void* out;
  int64_t ldo;
  int M, N, K;
  int m_tiles, n_tiles, k_blocks;
  int mode;  // 0: bf16 scaled, 1: int32 accumulators, 2: plain bf16 (fp32 accumulator),
             // 3: fp32 scaled (not rounded to bf16)
  uint32_t ab_format;   // operand-format bits of the instruction descriptor (bf16 or f16)
  int chunk_blocks;     // k-blocks per accumulator hand-off (exact chunks, or all of K)
  unsigned int* status;
  uint64_t wait_limit_ns;
  int drop_first_load;
  int32_t* partials;             // split tail: a 256 x 256 int32 slot per pair
  unsigned long long* counters;  // split tail: 2 x 8 counters per tail tile
  uint64_t epoch;                // split tail: tags this launch's counts (40 bits)
  int dp_tiles;                  // tiles computed whole (all of them without a split tail)
  int sk_tail, sk_split;         // split tail: its tiles, and the parts of each
  int m_fastest;                 // tile order: 1 = consecutive tiles down a column of tiles
};

// Row and column block of a tile.  Consecutive tiles (the CTAs of one wave)
// share a row block (and its A k-slices) -- or, with m_fastest, a column
// block: each wave then streams all of A's k-slices instead of all of B's,
// which re-reads less from DRAM when A is the smaller operand (M < N).
__device__ __forceinline__ void tile_mn(const GemmParams& p, int tile, int& mb, int& nb) {
  if (p.m_fastest) {
    mb = tile % p.m_tiles;
    nb = tile / p.m_tiles;
  } else {
    mb = tile / p.n_tiles;
    nb = tile % p.n_tiles;
  }
}

__device__ __forceinline__ void raise_abort(volatile int* abort, unsigned int* status) {
  *abort = 1;
  atomicOr(status, 1u);
}

// TMA of one operand's k-block: kRows rows (M or N) x 64 k.  K-major: one
// box of 64 k x kRows rows.  MN-major: kRows / 64 boxes of 64 (M or N) x 64
// k, each a 8 KB block of 64 swizzled 128-byte rows, one per k.
template <bool kMN, int kRows>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                             int kb, int mn0) {
  if (kMN) {
#pragma unroll
    for (int j = 0; j < kRows / 64; ++j)
      ptx::tma_load_2d(dst + j * kMnBlockBytes, map, bar, mn0 + 64 * j, kb * kBK);
  } else {
    ptx::tma_load_2d(dst, map, bar, kb * kBK, mn0);
  }
}
template <bool kMN, int kRows>
__device__ __forceinline__ void load_operand_pair(uint32_t dst, const CUtensorMap* map,
                                                  uint32_t bar, int kb, int mn0) {
  if (kMN) {
#pragma unroll
    for (int j = 0; j < kRows / 64; ++j)
      ptx::tma_load_2d_pair(dst + j * kMnBlockBytes, map, bar, mn0 + 64 * j, kb * kBK);
  } else {
    ptx::tma_load_2d_pair(dst, map, bar, kb * kBK, mn0);
  }
}

// Descriptor of an operand's stage tile and its advance per MMA (16 k):
// 32 bytes along a K-major row, two 8-row groups (2048 bytes) MN-major.
template <bool kMN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t addr) {
  return kMN ? ptx::smem_desc_mnmajor_sw128(addr, kMnBlockBytes) : ptx::smem_desc_kmajor_sw128(addr);
}
template <bool kMN>
__host__ __device__ constexpr uint64_t k_step() {
  return kMN ? (16u * 128u) >> 4 : 32u >> 4;
}

// Eight outputs of row `row`, columns col .. col+7 (N % 8 == 0, so all or
// none are inside), from their int32 totals.  bf16: (fp32(acc) * sA[row]) *
// sB[col], round to nearest even; fp32: the same product, not rounded to
// bf16; int32: the totals themselves.
__device__ __forceinline__ void store_vec8(const GemmParams& p, int64_t row, int64_t col, float sa,
                                           const int32_t* t) {
  if (col >= p.N) return;
  if (!in_bounds(row < p.M && col + 8 <= p.ldo, p.status)) return;
  if (p.mode == 1) {
    int4* o = reinterpret_cast<int4*>(static_cast<int32_t*>(p.out) + row * p.ldo + col);
    o[0] = make_int4(t[0], t[1], t[2], t[3]);
    o[1] = make_int4(t[4], t[5], t[6], t[7]);
    return;
  }
  if (p.mode == 3) {
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      o[e] = __fmul_rn(__fmul_rn(__int2float_rn(t[e]), sa), __ldg(p.sB + col + e));
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(p.out) + row * p.ldo + col);
    d[0] = make_float4(o[0], o[1], o[2], o[3]);
    d[1] = make_float4(o[4], o[5], o[6], o[7]);
    return;
  }
  uint32_t w[4];
  if (p.mode == 2) {  // t holds fp32 bit patterns
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 h =
          __floats2bfloat162_rn(__int_as_float(t[2 * e]), __int_as_float(t[2 * e + 1]));
      w[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * p.ldo + col) =
        make_uint4(w[0], w[1], w[2], w[3]);
    return;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float o0 = __fmul_rn(__fmul_rn(__int2float_rn(t[2 * e]), sa), __ldg(p.sB + col + 2 * e));
    const float o1 =
        __fmul_rn(__fmul_rn(__int2float_rn(t[2 * e + 1]), sa), __ldg(p.sB + col + 2 * e + 1));
    const __nv_bfloat162 h = __floats2bfloat162_rn(o0, o1);
    w[e] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * p.ldo + col) =
      make_uint4(w[0], w[1], w[2], w[3]);
}

// Drain one 128-column half of a chunk accumulator (this warp's 32 lanes)
// from tensor memory into the int32 totals; every fp32 value is an exact
// integer below 2^24 in magnitude.  Plain bf16 launches (one chunk per tile)
// keep the fp32 bit patterns themselves.
template <int kCols>
__device__ __forceinline__ void drain_chunk(uint32_t taddr, int32_t (&tot)[kCols], bool plain) {
  if (plain) {
#pragma unroll
    for (int sub = 0; sub < kCols / 16; ++sub) {
      uint32_t r[16];
      ptx::tmem_ld_16cols(taddr + sub * 16, r);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) tot[sub * 16 + i] = static_cast<int32_t>(r[i]);
    }
    return;
  }
#pragma unroll
  for (int sub = 0; sub < kCols / 16; ++sub) {
    uint32_t r[16];
    ptx::tmem_ld_16cols(taddr + sub * 16, r);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) tot[sub * 16 + i] += __float2int_rn(__uint_as_float(r[i]));
  }
}

// Scales of an epilogue warp's part of a tile (rows row0 .. row0+31,
// columns col0 .. col0+127) for launches whose CTAs have at most two tiles
// each (kRegScales), where the store's own scale loads -- a DRAM round trip
// per 64 columns -- would add straight to the kernel's time: loaded when the
// tile starts, so that their latency hides behind its MMAs.  Lane l holds
// its row's scale and the column scales col0 + 32 q + l in sb[q].  Outside
// the output they are 0; int32 outputs need none.  Launches with more tiles
// per CTA hide the store's latency behind the next tile's MMAs instead and
// load nothing here.
struct TileScales {
  float sa;
  float sb[4];
};
template <bool kRegScales, int kCols = 128>
__device__ __forceinline__ TileScales load_tile_scales(const GemmParams& p, int64_t row0,
                                                       int64_t col0) {
  TileScales t{0.0f, {0.0f, 0.0f, 0.0f, 0.0f}};
  if (!kRegScales || p.mode != 0) return t;
  const int lane = threadIdx.x & 31;
  if (row0 + lane < p.M) t.sa = __ldg(p.sA + row0 + lane);
#pragma unroll
  for (int q = 0; q < kCols / 32; ++q)
    if (col0 + 32 * q + lane < p.N) t.sb[q] = __ldg(p.sB + col0 + 32 * q + lane);
  return t;
}

// Output of one epilogue warp's part of a whole tile (rows row0 ..
// row0+31, columns col0 .. col0+127) by TMA tensor stores, one 128-byte-wide
// box at a time (64 bf16 or 32 int32 columns x 32 rows).  Lane l converts
// row row0 + l and writes it into the warp's 4 KB staging buffer in the
// 128-byte swizzled layout of the store map -- 16-byte chunk c of row r at
// r * 128 + (c ^ (r % 8)) * 16 -- so each group of eight lanes covers all 32
// banks.  The scales come from ts (kRegScales: the column scales by shuffles
// from the lanes holding them) or from global memory.  The store clips rows
// and columns outside the output; a box that starts at or past column N is
// not stored.  Before the buffer is rewritten, lane 0 waits until the
// previous store has read it.
template <bool kRegScales, int kCols>
__device__ __forceinline__ void store_tile_tma(const GemmParams& p, const CUtensorMap* map,
                                               uint32_t buf, int64_t row0, int64_t col0,
                                               const TileScales& ts, const int32_t (&tot)[kCols]) {
  if (row0 >= p.M) return;
  const int lane = threadIdx.x & 31;
  const int64_t row = row0 + lane;
  const uint32_t dst = buf + static_cast<uint32_t>(lane) * 128u;
  const uint32_t sw = static_cast<uint32_t>(lane & 7);
  auto publish = [&](int64_t c0) {
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(map, buf, static_cast<int32_t>(c0), static_cast<int32_t>(row0));
      ptx::bulk_commit_group();
    }
  };
  auto reuse = [&]() {
    if (lane == 0) ptx::bulk_wait_group_read0();
    __syncwarp();
  };
  if (p.mode == 1) {
#pragma unroll
    for (int j = 0; j < kCols / 32; ++j) {
      const int64_t c0 = col0 + 32 * j;
      if (c0 >= p.N) break;
      reuse();
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int32_t* t = tot + 32 * j + 4 * c;
        ptx::st_shared_v4(dst + ((static_cast<uint32_t>(c) ^ sw) << 4), t[0], t[1], t[2], t[3]);
      }
      publish(c0);
    }
    return;
  }
  if (!kRegScales && p.mode == 3) {  // fp32 scaled: 32-column boxes, like the int32 totals
    // (a data-parallel partial, off the training step's hot path: launched
    // without tile-start scales, and the column scales come from global
    // memory, which keeps this branch out of the other epilogues' registers)
    const float sa = row < p.M ? __ldg(p.sA + row) : 0.0f;
#pragma unroll
    for (int j = 0; j < kCols / 32; ++j) {
      const int64_t c0 = col0 + 32 * j;
      if (c0 >= p.N) break;
      reuse();
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int k0 = 32 * j + 4 * c;  // columns col0 + k0 .. col0 + k0 + 3
        float sb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t col = col0 + k0 + e;
          sb[e] = col < p.N ? __ldg(p.sB + col) : 0.0f;
        }
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = __float_as_uint(__fmul_rn(__fmul_rn(__int2float_rn(tot[k0 + e]), sa), sb[e]));
        ptx::st_shared_v4(dst + ((static_cast<uint32_t>(c) ^ sw) << 4), w[0], w[1], w[2], w[3]);
      }
      publish(c0);
    }
    return;
  }
  if (p.mode == 2) {  // plain bf16: tot holds fp32 bit patterns
#pragma unroll
    for (int j = 0; j < kCols / 64; ++j) {
      const int64_t c0 = col0 + 64 * j;
      if (c0 >= p.N) break;
      reuse();
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int32_t* t = tot + 64 * j + 8 * c;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 h =
              __floats2bfloat162_rn(__int_as_float(t[2 * e]), __int_as_float(t[2 * e + 1]));
          w[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
        ptx::st_shared_v4(dst + ((static_cast<uint32_t>(c) ^ sw) << 4), w[0], w[1], w[2], w[3]);
      }
      publish(c0);
    }
    return;
  }
  const float sa = kRegScales ? ts.sa : row < p.M ? __ldg(p.sA + row) : 0.0f;
  const bool sb_vec4 = (reinterpret_cast<uintptr_t>(p.sB) & 15u) == 0;
#pragma unroll
  for (int j = 0; j < kCols / 64; ++j) {
    const int64_t c0 = col0 + 64 * j;
    if (c0 >= p.N) break;
    reuse();
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int64_t col = c0 + 8 * c;
      float sb[8];
      if (kRegScales) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int k = 64 * j + 8 * c + e;  // column col0 + k
          sb[e] = __shfl_sync(0xFFFFFFFFu, ts.sb[k >> 5], k & 31);
        }
      } else if (col + 8 <= p.N && sb_vec4) {
        const float4 lo = __ldg(reinterpret_cast<const float4*>(p.sB + col));
        const float4 hi = __ldg(reinterpret_cast<const float4*>(p.sB + col) + 1);
        sb[0] = lo.x, sb[1] = lo.y, sb[2] = lo.z, sb[3] = lo.w;
        sb[4] = hi.x, sb[5] = hi.y, sb[6] = hi.z, sb[7] = hi.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) sb[e] = col + 8 <= p.N ? __ldg(p.sB + col + e) : 0.0f;
      }
      const int32_t* t = tot + 64 * j + 8 * c;
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float o0 = __fmul_rn(__fmul_rn(__int2float_rn(t[2 * e]), sa), sb[2 * e]);
        const float o1 = __fmul_rn(__fmul_rn(__int2float_rn(t[2 * e + 1]), sa), sb[2 * e + 1]);
        const __nv_bfloat162 h = __floats2bfloat162_rn(o0, o1);
        w[e] = *reinterpret_cast<const uint32_t*>(&h);
      }
      ptx::st_shared_v4(dst + ((static_cast<uint32_t>(c) ^ sw) << 4), w[0], w[1], w[2], w[3]);
    }
    publish(c0);
  }
}

// Single-CTA tiles of 128 x kTileN: 256 (four stages of 48 KB, two 256-column
// accumulators) or, for launches with few tiles, 128 (six stages of 32 KB,
// two 128-column accumulators) or 64 (eight stages of 24 KB, two 64-column
// accumulators), so that more SMs share the work.  kEpi epilogue warps drain
// a tile, each 32 rows x kCols columns: all eight with two column halves, or
// the first four with whole 64-column tiles.
template <int kTileN>
struct SingleTile {
  static constexpr int kStages = kTileN == 256 ? 4 : kTileN == 128 ? 6 : 8;
  static constexpr int kCols = kTileN == 64 ? 64 : kTileN / 2;
  static constexpr int kEpi = kTileN == 64 ? kEpiWarps / 2 : kEpiWarps;
  static constexpr int kBBytes = kTileN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2u * kTileN;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStagingBytes + kBarrierBytes;
  static_assert(kSmemBytes <= 227 * 1024, "single-CTA kernel shared memory");
  static_assert((2 * kStages + 5) * 8 + 12 <= kBarrierBytes, "barrier area");
};

template <bool kAmn, bool kBmn, bool kRegScales, int kTileN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_s8f16_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmO, const GemmParams p) {
  using Cfg = SingleTile<kTileN>;
  constexpr int kStages = Cfg::kStages;
  constexpr int kBBytes = Cfg::kBBytes;
  constexpr int kStageBytes = Cfg::kStageBytes;
  constexpr uint32_t kTmemCols = Cfg::kTmemCols;
  constexpr int kCols = Cfg::kCols;  // columns of a tile per epilogue warp
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t a_base = sbase;
  const uint32_t b_base = sbase + kStages * kABytes;
  const uint32_t staging = sbase + kStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kStagingBytes);
  const uint32_t bar0 = ptx::smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never = reinterpret_cast<volatile int*>(tmem_slot + 2);  // stays 0

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), Cfg::kEpi);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort = 0;
    *never = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    ptx::tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();

  const int num_tiles = p.m_tiles * p.n_tiles;
  const uint64_t limit = p.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0;
      uint32_t armed = 0u, armed_par = 0u;  // per-stage outstanding copy + its parity
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tile_mn(p, tile, mb, nb);
        const int m0 = mb * kBM;
        const int n0 = nb * kTileN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!ptx::mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort, limit)) {
            ok = false;
            break;
          }
          armed &= ~(1u << stage);  // the previous copy into this stage was consumed
          const bool drop = p.drop_first_load && tile == static_cast<int>(blockIdx.x) && kb == 0;
          if (!drop) {
            ptx::mbar_arrive_expect_tx(full_bar(stage), kStageBytes);
            load_operand<kAmn, kBM>(a_base + stage * kABytes, &tmA, full_bar(stage), kb, m0);
            load_operand<kBmn, kTileN>(b_base + stage * kBBytes, &tmB, full_bar(stage), kb, n0);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) raise_abort(abort, p.status);
      // never leave a copy in flight into shared memory of an exiting CTA
      for (int s = 0; s < kStages; ++s)
        if (armed & (1u << s))
          if (!ptx::mbar_wait_bounded(full_bar(s), (armed_par >> s) & 1u, never, limit))
            raise_abort(abort, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA
      const uint32_t idesc = ptx::idesc_f16_f32(kBM, kTileN, kAmn, kBmn) | p.ab_format;
      uint32_t stage = 0, phase = 0, chunk = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        for (int kb0 = 0; kb0 < p.k_blocks && ok; kb0 += p.chunk_blocks) {
          const uint32_t buf = chunk & 1u, aph = (chunk >> 1) & 1u;
          if (!ptx::mbar_wait_bounded(tempty_bar(buf), aph ^ 1u, abort, limit)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * kTileN;
          const int kb_end = min(kb0 + p.chunk_blocks, p.k_blocks);
          for (int kb = kb0; kb < kb_end; ++kb) {
            if (!ptx::mbar_wait_bounded(full_bar(stage), phase, abort, limit)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t adesc = operand_desc<kAmn>(a_base + stage * kABytes);
            const uint64_t bdesc = operand_desc<kBmn>(b_base + stage * kBBytes);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              ptx::mma_f16(d_tmem, adesc + k_step<kAmn>() * kk, bdesc + k_step<kBmn>() * kk, idesc,
                           (kb > kb0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(empty_bar(stage));
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          ptx::mma_commit(tfull_bar(buf));
          ++chunk;
        }
      }
      if (!ok) raise_abort(abort, p.status);
      // every MMA issued above completes before TMEM is released
      ptx::mma_commit(drain_bar);
      if (!ptx::mbar_wait_bounded(drain_bar, 0u, never, limit)) raise_abort(abort, p.status);
    }
  } else if (warp - 2 < Cfg::kEpi) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;           // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;    // which half of the tile's columns
    uint32_t chunk = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      int mb, nb;
      tile_mn(p, tile, mb, nb);
      const int m0 = mb * kBM;
      const int n0 = nb * kTileN;
      const TileScales ts = load_tile_scales<kRegScales, kCols>(
          p, static_cast<int64_t>(m0) + quad * 32, static_cast<int64_t>(n0) + half * kCols);
      int32_t tot[kCols];
#pragma unroll
      for (int i = 0; i < kCols; ++i) tot[i] = 0;
      for (int kb0 = 0; kb0 < p.k_blocks; kb0 += p.chunk_blocks) {
        const uint32_t buf = chunk & 1u, aph = (chunk >> 1) & 1u;
        int got = 1;
        if (lane == 0) got = ptx::mbar_wait_bounded(tfull_bar(buf), aph, abort, limit) ? 1 : 0;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * kTileN +
                               static_cast<uint32_t>(half * kCols);
        drain_chunk(taddr, tot, p.mode == 2);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty_bar(buf));
        ++chunk;
      }
      if (!ok) break;
      store_tile_tma<kRegScales, kCols>(p, &tmO, staging + (warp - 2) * kStoreBoxBytes,
                                        static_cast<int64_t>(m0) + quad * 32,
                                        static_cast<int64_t>(n0) + half * kCols, ts, tot);
    }
    if (!ok && lane == 0) raise_abort(abort, p.status);
    if (lane == 0) ptx::bulk_wait_group0();  // the tile stores are complete
  }

  // ------------------------------------------------------------ teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------ CTA-pair kernel
// Same computation on 256x256 tiles by a cluster of two CTAs (one per SM of
// a pair).  CTA r loads rows r*128 .. r*128+127 of the tile's A block and
// columns r*128 .. r*128+127 of its B block (32 KB per stage instead of
// 48 KB, so six stages fit); the even CTA's MMA thread issues
// tcgen05.mma.cta_group::2, which reads both CTAs' shared memory and writes
// each CTA's 128 accumulator rows into that CTA's tensor memory.  Both CTAs'
// loads complete on the even CTA's full barrier; the MMA commits arrive on
// both CTAs' empty and accumulator-full barriers; the odd CTA's epilogue warps
// arrive on the even CTA's accumulator-empty barrier.  K runs in exact
// 1024-term chunks drained into int32 totals, as in the single-CTA kernel.
//
// Work split.  Pair p takes tiles p, p + P, ... (P pairs), so that the pairs
// of a wave work on neighbouring tiles at the same k and share their A and B
// k-slices in L2.  When the tiles leave a partial last wave of R < P tiles
// and a scratch is given, those R tiles are instead split into s equal
// k-parts (s = min(P / R, 4)) computed by otherwise idle pairs, still in step
// with one another.  Each part stores its int32 totals in the pair's slot and
// counts itself in on the tile's counters; whichever part arrives last sums
// the s parts and writes the tile.  No CTA waits for another: the last
// arrival finds every other part stored.
constexpr int kPairStages = 6;
constexpr int kPairABytes = 128 * kBK * 2;
constexpr int kPairBBytes = 128 * kBK * 2;
constexpr int kPairStageBytes = kPairABytes + kPairBBytes;
constexpr int kPairSmemBytes =
    1024 + kPairStages * kPairStageBytes + kStagingBytes + kBarrierBytes;
static_assert(kPairSmemBytes <= 227 * 1024, "pair kernel shared memory");
// Converter stage (kConv != 0): TMA brings each CTA's raw k-block into a
// ring of its own, and six converter warps turn it into the f16 stage the
// tensor core reads -- fewer f16 stages, more raw ones (the raw ring covers
// the DRAM latency, the f16 ring only decouples the converters from the MMA).
//   kConvWiden (1): int8 codes of A and of B (128 x 64 each, 16 KB), widened.
//   kConvQuantB (2): the bf16 B operand (128 x 64, 16 KB) quantized with its
//                    given row scales, as the row quantizer would (A arrives
//                    as f16 codes by TMA, as in the plain kernel).
// The kernel runs four warpgroups: warpgroup 0 (producer, MMA, converters
// 0-1) and 3 (converters 2-5) give up registers, warpgroups 1-2 (the
// epilogue, warps 4-11) take them: 256 x kConvRegsEpi + 256 x kConvRegsOther
// = 65,536, the launch's registers.
constexpr int kConvNone = 0, kConvWiden = 1, kConvQuantB = 2;
constexpr int kS8Stages = 4;
constexpr int kRawStages = 4;
constexpr int kRawOperandBytes = 128 * kBK;  // 128 rows x 64 k, one byte each
constexpr int kRawStageBytes = 2 * kRawOperandBytes;
constexpr int kConvWarps = 6;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kS8Threads = 512;
constexpr int kS8RegsEpi = 184, kS8RegsOther = 72;
static_assert(256 * kS8RegsEpi + 256 * kS8RegsOther <= 65536, "register split of the S8 kernel");
static_assert(kS8Threads * 128 == 65536, "the S8 kernel launches with 128 registers a thread");
constexpr int kS8SmemBytes = 1024 + kS8Stages * kPairStageBytes + kRawStages * kRawStageBytes +
                             kStagingBytes + kBarrierBytes;
static_assert(kS8SmemBytes <= 227 * 1024, "int8-operand pair kernel shared memory");
static_assert((3 * kS8Stages + 5 + 2 * kRawStages) * 8 + 12 <= kBarrierBytes, "barrier area");
constexpr int kCasLimit = 4096;  // bound on the counter's compare-and-swap retries
constexpr int kMaxSplit = 4;     // most parts a tile of the last wave is split into
static_assert(static_cast<size_t>(kSplitTailMaxPairs) * 256 * 256 * 4 +
                      kSplitTailMaxPairs * 2 * kEpiWarps * 8 <= kSplitTailScratchBytes,
              "split-tail scratch layout");

// TMA of one operand's int8 k-block (128 rows of M or N x 64 k) into the
// CTA's raw ring, unswizzled: K-major [128][64] (a 64-byte row per M/N),
// MN-major [64][128] (a 128-byte row per k).  Completion on this CTA's own
// barrier.
template <bool kMN>
__device__ __forceinline__ void load_raw(uint32_t dst, const CUtensorMap* map, uint32_t bar, int kb,
                                         int mn0) {
  if (kMN)
    ptx::tma_load_2d(dst, map, bar, mn0, kb * kBK);
  else
    ptx::tma_load_2d(dst, map, bar, kb * kBK, mn0);
}

// Four int8 codes (one word) as two f16x2 words holding the same integers:
// the biased byte u = q + 128 becomes the f16 0x6400 | u = 1024 + u, and
// subtracting 1152 leaves q exactly (every value involved is an integer
// below 2048, exact in f16).
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// Widen one operand's raw int8 k-block (8 KB at `raw`) into its f16 stage
// tile at `dst`, in the 128-byte swizzled layout a TMA load would have
// written: K-major, row m (128 bytes: 64 k) at m * 128; MN-major, 64-wide
// block b, row k at b * 8192 + k * 128; 16-byte chunk c of row r at
// (c ^ (r % 8)) * 16.  Converter thread ct (of kConvThreads) takes 16-byte
// raw chunks ct, ct + kConvThreads, ...; each becomes 32 bytes (two chunks)
// of one f16 row.
// Bank conflicts: eight consecutive raw chunks (a quarter warp) are 128
// contiguous bytes.  K-major, they fill two f16 rows with different
// swizzles, so the first (and the second) stores of the quarter warp land in
// complementary chunk sets.  MN-major, they are one k of both 64-wide blocks
// (same swizzle): the threads of block 1 store their second chunk first.
// Quantize one CTA's bf16 B k-block (128 rows x 64 k at `raw`, unswizzled
// 128-byte rows) into its f16 stage tile at `dst` (K-major, 128-byte
// swizzle): row n's codes with its scale sB[n] (rows at or past `nrows` are
// the zero fill, code 0), exactly as the row quantizer forms them -- the
// certified three-operation quotient when the scale allows it, else IEEE
// division; nearest even by the packed magic-number add when the scale is
// normal, else rint and clamp.  Each 16-byte raw chunk (eight values of one
// row) becomes one 16-byte chunk of codes; a quarter warp covers one row.
__device__ __forceinline__ void quant_tile_b(uint32_t raw, uint32_t dst, int ct,
                                             const float* __restrict__ sB, int nrows) {
#pragma unroll 2
  for (int c = ct; c < 128 * 8; c += kConvThreads) {
    const int row = c >> 3, j = c & 7;
    const uint4 v = ptx::ld_shared_v4(raw + static_cast<uint32_t>(c) * 16u);
    const float sc = row < nrows ? __ldg(sB + row) : 0.0f;
    const ScaleDiv d = make_scale_div(sc);
    float f[8], q[8];
    unpack8(v, f);
    if (!div8_try(f, d, q)) div8_ieee(f, sc, q);
    uint32_t h[4];
    if (scale_is_normal(sc)) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 cc = code_rne_normal_scale2(make_float2(q[2 * i], q[2 * i + 1]));
        const __half2 hh = __floats2half2_rn(cc.x, cc.y);
        h[i] = *reinterpret_cast<const uint32_t*>(&hh);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 hh = __floats2half2_rn(code_rne(q[2 * i]), code_rne(q[2 * i + 1]));
        h[i] = *reinterpret_cast<const uint32_t*>(&hh);
      }
    }
    const uint32_t sw = static_cast<uint32_t>(row & 7);
    ptx::st_shared_v4(dst + static_cast<uint32_t>(row) * 128u + ((static_cast<uint32_t>(j) ^ sw) << 4),
                      h[0], h[1], h[2], h[3]);
  }
}

template <bool kMN>
__device__ __forceinline__ void widen_tile(uint32_t raw, uint32_t dst, int ct) {
  static_assert(kConvThreads % 8 == 0, "a thread's chunks keep their bit 2");
  const int swap = kMN ? (ct >> 2) & 1 : 0;  // the same for every chunk of this thread
#pragma unroll 3
  for (int c = ct; c < kRawOperandBytes / 16; c += kConvThreads) {
    const int row = kMN ? ((c >> 2) & 1) * 64 + (c >> 3) : c >> 2;
    const int chunk = (c & 3) * 2;  // first of the row's two 16-byte chunks
    uint4 v = ptx::ld_shared_v4(raw + static_cast<uint32_t>(c) * 16u);
    if (swap) {
      const uint32_t x = v.x, y = v.y;
      v.x = v.z, v.y = v.w, v.z = x, v.w = y;
    }
    uint32_t h[8];
    widen4(v.x, h[0], h[1]);
    widen4(v.y, h[2], h[3]);
    widen4(v.z, h[4], h[5]);
    widen4(v.w, h[6], h[7]);
    const uint32_t rowaddr = dst + static_cast<uint32_t>(row) * 128u;
    const uint32_t sw = static_cast<uint32_t>(row & 7);
    const uint32_t c0 = static_cast<uint32_t>(chunk + swap), c1 = static_cast<uint32_t>(chunk + 1 - swap);
    ptx::st_shared_v4(rowaddr + ((c0 ^ sw) << 4), h[0], h[1], h[2], h[3]);
    ptx::st_shared_v4(rowaddr + ((c1 ^ sw) << 4), h[4], h[5], h[6], h[7]);
  }
}

// The fragments (tile, k-blocks [kb0, kb1)) one pair computes, in order:
// whole tiles pair, pair + P, ... below p.dp_tiles (P pairs), then, when
// the last wave is split, unit `pair` of the tail: tile dp_tiles + pair / s,
// k-part pair % s of s equal parts (pairs from tail * s on have no unit).
struct FragIter {
  int g;
  bool tail_done;
  __device__ FragIter(const GemmParams&, int pair) : g(pair), tail_done(false) {}
  __device__ bool next(const GemmParams& p, int pair, int npairs, int& tile, int& kb0, int& kb1) {
    if (g < p.dp_tiles) {
      tile = g;
      kb0 = 0;
      kb1 = p.k_blocks;
      g += npairs;
      return true;
    }
    if (tail_done || pair >= p.sk_tail * p.sk_split) return false;
    tail_done = true;
    tile = p.dp_tiles + pair / p.sk_split;
    const int j = pair % p.sk_split;
    kb0 = j * p.k_blocks / p.sk_split;
    kb1 = (j + 1) * p.k_blocks / p.sk_split;
    return true;
  }
};

// Counts one contributor in on a split tile's counter for this launch and
// tells whether it was the last of n.  The counter holds the launch's epoch
// in its high 40 bits and the count in the low 24; a word left by another
// launch (or never written) carries another epoch and counts as 0, so the
// counters need no clearing before a launch.  The last arrival clears the
// word (0 is no launch's tag), so that a launch replayed with the same epoch
// -- a captured CUDA graph -- starts from 0 too.  Returns -1 if the
// compare-and-swap kept failing.
__device__ __forceinline__ int sk_arrive(unsigned long long* ctr, uint64_t epoch, int n) {
  const unsigned long long tag = (epoch & 0xFFFFFFFFFFull) << 24;
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ctr);
  for (int i = 0; i < kCasLimit; ++i) {
    const unsigned long long cnt = (old & ~0xFFFFFFull) == tag ? (old & 0xFFFFFFull) : 0ull;
    const unsigned long long seen = atomicCAS(ctr, old, tag | (cnt + 1ull));
    if (seen == old) {
      if (static_cast<int>(cnt + 1ull) != n) return 0;
      atomicExch(ctr, 0ull);  // every part has arrived: nothing else touches it
      return 1;
    }
    old = seen;
  }
  return -1;
}

// Epilogue of a tail unit (part of a split tile), per epilogue warp (32
// tile rows x 128 columns) with its own counter.  A slot holds the pair's
// 256 x 256 int32 totals warp-coalesced: vector v (columns 4v .. 4v+3 of the
// lane's 128) of lane l of epilogue warp w of CTA r at int4 index
// ((r * 8 + w) * 32 + v) * 32 + l, so each store or load instruction of a
// warp moves 512 contiguous bytes.  The warp stores its totals, counts itself
// in, and the last of the tile's s parts sums all s parts' totals (its own
// read back) and stores the outputs.
__device__ __forceinline__ const int4* sk_warp_slot(const GemmParams& p, int slot, int rank,
                                                    int ewarp) {
  return reinterpret_cast<const int4*>(p.partials + static_cast<size_t>(slot) * (256u * 256u)) +
         (rank * kEpiWarps + ewarp) * 32 * 32 + (threadIdx.x & 31);
}

__device__ __forceinline__ void sk_store_part(const GemmParams& p, int pair, int rank, int ewarp,
                                              const int32_t (&tot)[128]) {
  if (!in_bounds(pair < kSplitTailMaxPairs, p.status)) return;
  int4* dst = const_cast<int4*>(sk_warp_slot(p, pair, rank, ewarp));
#pragma unroll
  for (int v = 0; v < 32; ++v)
    __stcg(dst + v * 32, make_int4(tot[4 * v], tot[4 * v + 1], tot[4 * v + 2], tot[4 * v + 3]));
  __threadfence();
  __syncwarp();
}

// fp32 sum of two fp32 bit patterns, as a bit pattern
__device__ __forceinline__ int32_t fadd_bits(int32_t a, int32_t b) {
  return __float_as_int(__fadd_rn(__int_as_float(a), __int_as_float(b)));
}

__device__ __forceinline__ void sk_complete(const GemmParams& p, int rank, int ewarp, int tile,
                                            int64_t row, int64_t col0, volatile int* abort) {
  const int t = tile - p.dp_tiles;  // tail tile: parts come from pairs t*s .. t*s+s-1
  if (!in_bounds(t >= 0 && t * p.sk_split + p.sk_split <= kSplitTailMaxPairs &&
                     (2 * t + rank) * kEpiWarps + ewarp < 2 * kSplitTailMaxPairs * kEpiWarps,
                 p.status))
    return;
  int r = 0;
  if ((threadIdx.x & 31) == 0)
    r = sk_arrive(p.counters + (2 * t + rank) * kEpiWarps + ewarp, p.epoch, p.sk_split);
  r = __shfl_sync(0xFFFFFFFFu, r, 0);
  if (r < 0) {
    if ((threadIdx.x & 31) == 0) raise_abort(abort, p.status);
    return;
  }
  if (r == 0 || row >= p.M) return;
  __threadfence();
  const float sa = (p.mode == 0 || p.mode == 3) ? __ldg(p.sA + row) : 0.0f;
  // 32 columns at a time: each part's 8 vectors are loaded together
  for (int h = 0; h < 4; ++h) {
    int32_t acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0;
    for (int j = 0; j < p.sk_split; ++j) {
      const int4* src = sk_warp_slot(p, t * p.sk_split + j, rank, ewarp) + h * 8 * 32;
      int4 x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __ldcg(src + i * 32);
      if (p.mode == 2) {  // fp32 partial sums, added in part order
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[4 * i] = fadd_bits(acc[4 * i], x[i].x);
          acc[4 * i + 1] = fadd_bits(acc[4 * i + 1], x[i].y);
          acc[4 * i + 2] = fadd_bits(acc[4 * i + 2], x[i].z);
          acc[4 * i + 3] = fadd_bits(acc[4 * i + 3], x[i].w);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[4 * i] += x[i].x;
          acc[4 * i + 1] += x[i].y;
          acc[4 * i + 2] += x[i].z;
          acc[4 * i + 3] += x[i].w;
        }
      }
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) store_vec8(p, row, col0 + h * 32 + v * 8, sa, acc + v * 8);
  }
}

// kConv != 0: a converter stage.  Each CTA's producer brings its raw
// k-blocks into a raw ring (its own barriers); converter warps 2-3 and 12-15
// of both CTAs turn them into the f16 stages and arrive on the even CTA's
// full barrier (release at cluster scope, after a proxy fence so that the
// tensor core sees the stores), which the MMA thread waits on at cluster
// scope; the epilogue is warps 4-11.  kConvWiden: both operands are int8
// codes (INT8MP_CODES_S8).  kConvQuantB: A is f16 codes loaded by TMA into
// the f16 stage as in the plain kernel (the even CTA's arrive carries their
// bytes), B is bf16, quantized by the converters.  Everything else is the
// f16 kernel.
template <bool kAmn, bool kBmn, bool kRegScales, int kConv>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kConv != kConvNone ? kS8Threads : kThreads, 1)
    gemm_s8f16_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmO, const GemmParams p) {
  constexpr bool kS8 = kConv != kConvNone;  // a converter stage (any kind)
  constexpr int kStagesHere = kS8 ? kS8Stages : kPairStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t a_base = sbase;
  const uint32_t b_base = sbase + kStagesHere * kPairABytes;
  const uint32_t rawring = sbase + kStagesHere * kPairStageBytes;  // kS8 only
  constexpr int kRawBytesHere = kS8 ? kRawStages * kRawStageBytes : 0;
  const uint32_t staging = sbase + kStagesHere * kPairStageBytes + kRawBytesHere;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStagesHere * kPairStageBytes +
                                               kRawBytesHere + kStagingBytes);
  const uint32_t bar0 = ptx::smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStagesHere + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kStagesHere + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kStagesHere + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStagesHere + 4);
  auto rfull_bar = [&](int s) { return bar0 + 8u * (2 * kStagesHere + 5 + s); };
  auto rempty_bar = [&](int s) { return bar0 + 8u * (2 * kStagesHere + 5 + kRawStages + s); };
  // odd CTA: its converters' stage done, forwarded to the even CTA by one thread
  auto cdone_bar = [&](int s) { return bar0 + 8u * (2 * kStagesHere + 5 + 2 * kRawStages + s); };
  constexpr int kBarsHere = 2 * kStagesHere + 5 + (kS8 ? 2 * kRawStages + kStagesHere : 0);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBarsHere);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool even = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesHere; ++s) {
      // converters: the even CTA's converter warps arrive, and one thread of
      // the odd CTA for all of its converters (and, quantizing B, the even
      // producer with A's bytes); f16: the TMA bytes
      ptx::mbar_init(full_bar(s), kConv == kConvWiden    ? kConvWarps + 1
                                  : kConv == kConvQuantB ? 1 + kConvWarps + 1
                                                         : 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull_bar(b), 1);
      ptx::mbar_init(tempty_bar(b), 2 * kEpiWarps);
    }
    ptx::mbar_init(drain_bar, 1);
    if constexpr (kS8) {
      for (int s = 0; s < kRawStages; ++s) {
        ptx::mbar_init(rfull_bar(s), 1);
        ptx::mbar_init(rempty_bar(s), kConvWarps);
      }
      for (int s = 0; s < kStagesHere; ++s) ptx::mbar_init(cdone_bar(s), kConvWarps);
    }
    *abort = 0;
    *never = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    ptx::tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // both CTAs' barriers exist before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  ptx::grid_dependency_wait();  // the previous kernel in the stream is done
  ptx::allow_dependents();

  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const uint64_t limit = p.wait_limit_ns;
  constexpr int kEpiFirst = kS8 ? 4 : 2;  // first epilogue warp

  auto s8_producer = [&]() {
    if (lane == 0) {
      // ------------------------------------------ producer (int8 operands)
      // each CTA fills its own raw ring with its 128 rows of A and of B
      uint32_t stage = 0, phase = 0;
      uint32_t armed = 0u, armed_par = 0u;  // raw stages with a copy in flight
      bool ok = true;
      FragIter it(p, pair);
      int tile, kb0, kb1;
      while (ok && it.next(p, pair, npairs, tile, kb0, kb1)) {
        int mb, nb;
        tile_mn(p, tile, mb, nb);
        const int m0 = mb * 256 + static_cast<int>(rank) * 128;
        const int n0 = nb * 256 + static_cast<int>(rank) * 128;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(rempty_bar(stage), phase ^ 1u, abort, limit)) {
            ok = false;
            break;
          }
          const uint32_t dst = rawring + stage * kRawStageBytes;
          ptx::mbar_arrive_expect_tx(rfull_bar(stage), kRawStageBytes);
          load_raw<kAmn>(dst, &tmA, rfull_bar(stage), kb, m0);
          load_raw<kBmn>(dst + kRawOperandBytes, &tmB, rfull_bar(stage), kb, n0);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kRawStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) raise_abort(abort, p.status);
      // never leave a copy in flight into shared memory of an exiting CTA:
      // wait for the last copy into every raw stage (the earlier ones were
      // consumed before the stage was refilled)
      for (int s = 0; s < kRawStages; ++s)
        if (armed & (1u << s))
          if (!ptx::mbar_wait_bounded(rfull_bar(s), (armed_par >> s) & 1u, never, limit))
            raise_abort(abort, p.status);
    }
  };
  auto qb_producer = [&]() {
    if (lane == 0) {
      // ------------------------------- producer (quantizing B in the prologue)
      // A's f16 codes by TMA into the f16 stage, completing on the even
      // CTA's full barrier (as in the plain kernel); B's bf16 rows into this
      // CTA's raw ring for the converters
      uint32_t stage = 0, phase = 0, rstage = 0, rphase = 0;
      uint32_t armed = 0u, armed_par = 0u, rarmed = 0u, rarmed_par = 0u;
      bool ok = true;
      FragIter it(p, pair);
      int tile, kb0, kb1;
      while (ok && it.next(p, pair, npairs, tile, kb0, kb1)) {
        int mb, nb;
        tile_mn(p, tile, mb, nb);
        const int m0 = mb * 256 + static_cast<int>(rank) * 128;
        const int n0 = nb * 256 + static_cast<int>(rank) * 128;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort, limit) ||
              !ptx::mbar_wait_bounded(rempty_bar(rstage), rphase ^ 1u, abort, limit)) {
            ok = false;
            break;
          }
          armed &= ~(1u << stage);
          const uint32_t fb = ptx::mapa_shared(full_bar(stage), 0);
          if (even) {
            ptx::mbar_arrive_expect_tx(full_bar(stage), 2 * kPairABytes);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          }
          load_operand_pair<kAmn, 128>(a_base + stage * kPairABytes, &tmA, fb, kb, m0);
          ptx::mbar_arrive_expect_tx(rfull_bar(rstage), kRawStageBytes);
          ptx::tma_load_2d(rawring + rstage * kRawStageBytes, &tmB, rfull_bar(rstage), kb * kBK,
                           n0);
          rarmed |= 1u << rstage;
          rarmed_par = (rarmed_par & ~(1u << rstage)) | (rphase << rstage);
          if (++stage == kStagesHere) {
            stage = 0;
            phase ^= 1u;
          }
          if (++rstage == kRawStages) {
            rstage = 0;
            rphase ^= 1u;
          }
        }
      }
      if (!ok) raise_abort(abort, p.status);
      // never leave a copy in flight into shared memory of an exiting CTA
      for (int s = 0; s < kRawStages; ++s)
        if (rarmed & (1u << s))
          if (!ptx::mbar_wait_bounded(rfull_bar(s), (rarmed_par >> s) & 1u, never, limit))
            raise_abort(abort, p.status);
      for (int s = 0; s < kStagesHere; ++s)
        if (armed & (1u << s))
          if (!ptx::mbar_wait_bounded_cluster(full_bar(s), (armed_par >> s) & 1u, never, limit))
            raise_abort(abort, p.status);
    }
  };
  auto converters = [&]() {
    // ------------------------------------------- converters (int8 operands)
    const int ct = warp < 4 ? threadIdx.x - 64 : threadIdx.x - 320;  // 0 .. kConvThreads-1
    uint32_t rstage = 0, rphase = 0, stage = 0, phase = 0;
    bool ok = true;
    FragIter it(p, pair);
    int tile, kb0, kb1;
    while (ok && it.next(p, pair, npairs, tile, kb0, kb1)) {
      for (int kb = kb0; kb < kb1; ++kb) {
        // every lane waits (each then reads the copied bytes itself); the
        // waits are bounded, so all lanes reach the vote and leave together
        bool got = ptx::mbar_wait_bounded(rfull_bar(rstage), rphase, abort, limit);
        got = got && ptx::mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort, limit);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        const uint32_t raw = rawring + rstage * kRawStageBytes;
        if constexpr (kConv == kConvQuantB) {
          int mb, nb;
          tile_mn(p, tile, mb, nb);
          const int n0 = nb * 256 + static_cast<int>(rank) * 128;
          quant_tile_b(raw, b_base + stage * kPairBBytes, ct, p.sB + n0, p.N - n0);
        } else {
          widen_tile<kAmn>(raw, a_base + stage * kPairABytes, ct);
          widen_tile<kBmn>(raw + kRawOperandBytes, b_base + stage * kPairBBytes, ct);
        }
        ptx::fence_proxy_async_smem();  // the tensor core reads these stores
        __syncwarp();
        if (lane == 0) {
          // CTA-scope arrivals only: on the even CTA's full barrier, or on
          // the odd CTA's stage-done barrier that its forwarder passes on
          ptx::mbar_arrive(rempty_bar(rstage));
          ptx::mbar_arrive(even ? full_bar(stage) : cdone_bar(stage));
        }
        if (++rstage == kRawStages) {
          rstage = 0;
          rphase ^= 1u;
        }
        if (++stage == kStagesHere) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) raise_abort(abort, p.status);
  };
  auto producer = [&]() {
    if (lane == 0) {
      // ------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0;
      uint32_t armed = 0u, armed_par = 0u;  // even CTA: stages whose full barrier it armed
      bool ok = true, first_load = true;
      FragIter it(p, pair);
      int tile, kb0, kb1;
      while (ok && it.next(p, pair, npairs, tile, kb0, kb1)) {
        int mb, nb;
        tile_mn(p, tile, mb, nb);
        const int m0 = mb * 256 + static_cast<int>(rank) * 128;
        const int n0 = nb * 256 + static_cast<int>(rank) * 128;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort, limit)) {
            ok = false;
            break;
          }
          armed &= ~(1u << stage);
          const bool drop = p.drop_first_load && even && first_load;
          first_load = false;
          if (!drop) {
            const uint32_t fb = ptx::mapa_shared(full_bar(stage), 0);
            if (even) {
              ptx::mbar_arrive_expect_tx(full_bar(stage), 2 * kPairStageBytes);
              armed |= 1u << stage;
              armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
            }
            load_operand_pair<kAmn, 128>(a_base + stage * kPairABytes, &tmA, fb, kb, m0);
            load_operand_pair<kBmn, 128>(b_base + stage * kPairBBytes, &tmB, fb, kb, n0);
          }
          if (++stage == kStagesHere) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) raise_abort(abort, p.status);
      for (int s = 0; s < kStagesHere; ++s)
        if (armed & (1u << s))
          if (!ptx::mbar_wait_bounded(full_bar(s), (armed_par >> s) & 1u, never, limit))
            raise_abort(abort, p.status);
    }
  };
  auto mma = [&]() {
    if (lane == 0 && even) {
      // ----------------------------------------------------------- MMA
      const uint32_t idesc = ptx::idesc_f16_f32(256, 256, kAmn, kBmn) | p.ab_format;
      uint32_t stage = 0, phase = 0, chunk = 0;
      bool ok = true;
      FragIter it(p, pair);
      int tile, kb0, kb1;
      while (ok && it.next(p, pair, npairs, tile, kb0, kb1)) {
        for (int kc = kb0; kc < kb1 && ok; kc += p.chunk_blocks) {
          const uint32_t buf = chunk & 1u, aph = (chunk >> 1) & 1u;
          if (!ptx::mbar_wait_bounded(tempty_bar(buf), aph ^ 1u, abort, limit)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * kBN;
          const int kc_end = min(kc + p.chunk_blocks, kb1);
          for (int kb = kc; kb < kc_end; ++kb) {
            const bool got = kS8 ? ptx::mbar_wait_bounded_cluster(full_bar(stage), phase, abort, limit)
                                 : ptx::mbar_wait_bounded(full_bar(stage), phase, abort, limit);
            if (!got) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t adesc = operand_desc<kAmn>(a_base + stage * kPairABytes);
            const uint64_t bdesc = operand_desc<kBmn>(b_base + stage * kPairBBytes);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              ptx::mma_f16_pair(d_tmem, adesc + k_step<kAmn>() * kk, bdesc + k_step<kBmn>() * kk,
                                idesc, (kb > kc || kk > 0) ? 1u : 0u);
            ptx::mma_commit_pair(empty_bar(stage), 0x3);
            if (++stage == kStagesHere) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          ptx::mma_commit_pair(tfull_bar(buf), 0x3);
          ++chunk;
        }
      }
      if (!ok) raise_abort(abort, p.status);
      ptx::mma_commit_pair(drain_bar, 0x1);
      if (!ptx::mbar_wait_bounded(drain_bar, 0u, never, limit)) raise_abort(abort, p.status);
    }
    if constexpr (kS8) {
      if (lane == 0 && !even) {
        // -------------------------- forwarder (odd CTA, converter stages)
        // once this CTA's converters are done with a stage, one arrival at
        // cluster scope on the even CTA's full barrier carries them all
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        FragIter it(p, pair);
        int tile, kb0, kb1;
        while (ok && it.next(p, pair, npairs, tile, kb0, kb1)) {
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!ptx::mbar_wait_bounded(cdone_bar(stage), phase, abort, limit)) {
              ok = false;
              break;
            }
            ptx::mbar_arrive_cluster(ptx::mapa_shared(full_bar(stage), 0));
            if (++stage == kStagesHere) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) raise_abort(abort, p.status);
      }
    }
  };
  auto epilogue = [&]() {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int half = (warp - kEpiFirst) >> 2;
    uint32_t chunk = 0;
    bool ok = true;
    FragIter it(p, pair);
    int tile, kb0, kb1;
    while (ok && it.next(p, pair, npairs, tile, kb0, kb1)) {
      int mb, nb;
      tile_mn(p, tile, mb, nb);
      const int m0 = mb * 256 + static_cast<int>(rank) * 128;
      const int n0 = nb * 256;
      const bool whole = kb0 == 0 && kb1 == p.k_blocks;
      TileScales ts{0.0f, {0.0f, 0.0f, 0.0f, 0.0f}};
      if (whole)
        ts = load_tile_scales<kRegScales>(p, static_cast<int64_t>(m0) + quad * 32,
                                          static_cast<int64_t>(n0) + half * 128);
      int32_t tot[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) tot[i] = 0;
      for (int kc = kb0; kc < kb1; kc += p.chunk_blocks) {
        const uint32_t buf = chunk & 1u, aph = (chunk >> 1) & 1u;
        int got = 1;
        if (lane == 0) got = ptx::mbar_wait_bounded(tfull_bar(buf), aph, abort, limit) ? 1 : 0;
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * kBN +
                               static_cast<uint32_t>(half * 128);
        drain_chunk(taddr, tot, p.mode == 2);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(buf), 0));
        ++chunk;
      }
      if (!ok) break;
      const int64_t row = static_cast<int64_t>(m0) + quad * 32 + lane;
      const int64_t col0 = static_cast<int64_t>(n0) + half * 128;
      if (whole) {
        store_tile_tma<kRegScales>(p, &tmO, staging + (warp - kEpiFirst) * kStoreBoxBytes, row - lane,
                                   col0, ts, tot);
      } else {
        sk_store_part(p, pair, static_cast<int>(rank), warp - kEpiFirst, tot);
        sk_complete(p, static_cast<int>(rank), warp - kEpiFirst, tile, row, col0, abort);
      }
    }
    if (!ok && lane == 0) raise_abort(abort, p.status);
    if (lane == 0) ptx::bulk_wait_group0();  // the tile stores are complete
  };

  if constexpr (kS8) {
    // register split by warpgroup: each warpgroup's four warps execute the
    // same adjustment at the top of their branch
    if (warp >= 4 && warp < 12) {
      ptx::setmaxnreg_inc<kS8RegsEpi>();
      epilogue();
    } else {
      ptx::setmaxnreg_dec<kS8RegsOther>();
      if (warp == 0) {
        if constexpr (kConv == kConvQuantB)
          qb_producer();
        else
          s8_producer();
      } else if (warp == 1)
        mma();
      else
        converters();
    }
  } else {
    if (warp == 0)
      producer();
    else if (warp == 1)
      mma();
    else
      epilogue();
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (threadIdx.x == 0 && *abort) {
    // after a timeout, give copies issued by either CTA time to land
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < 200000ull) {
    }
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // the pair's MMAs, copies and remote arrivals are done
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
// Operand map of 16-bit elements (f16 code containers, or bf16 for the plain
// passes), 128-byte swizzle, zero fill outside the tensor.
// K-major [mn, K] (row stride K): boxes of 64 k x box_mn rows.
// MN-major [K, mn] (row stride mn): boxes of 64 (M or N) x 64 k.
bool make_operand_map(CUtensorMap* map, const void* base, bool mn_major, int64_t mn, int64_t K,
                      int box_mn, bool bf16) {
  const CUtensorMapDataType t =
      bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (mn_major)
    return encode_tensor_map_2d(map, base, t, 2, K, mn, mn, 64, kBK, CU_TENSOR_MAP_SWIZZLE_128B);
  return encode_tensor_map_2d(map, base, t, 2, mn, K, K, kBK, box_mn, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Operand-format field of the kind::f16 instruction descriptor (bits 7-9 for
// A, 10-12 for B): 0 = f16, 1 = bf16.
constexpr uint32_t kFormatBf16 = (1u << 7) | (1u << 10);

// Operand map of int8 codes for the int8-operand pair kernel, no swizzle:
// K-major [mn, K]: boxes of 64 k x 128 rows; MN-major [K, mn]: boxes of 128
// (M or N) x 64 k.
bool make_raw_map(CUtensorMap* map, const void* base, bool mn_major, int64_t mn, int64_t K) {
  if (mn_major)
    return encode_tensor_map_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, mn, mn, 128, kBK,
                                CU_TENSOR_MAP_SWIZZLE_NONE);
  return encode_tensor_map_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, mn, K, K, kBK, 128,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Shared-memory size of a converter-stage kernel, and its launch register
// count: the register split assumes 128 registers a thread at launch; with
// fewer, its setmaxnreg.inc could never be satisfied, so such a build is
// refused instead of launched.
template <typename Kernel>
cudaError_t set_conv_attrs(Kernel kernel) {
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kS8SmemBytes);
  if (err != cudaSuccess) return err;
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, kernel);
  if (err == cudaSuccess && fa.numRegs != 128) err = cudaErrorInvalidDeviceFunction;
  return err;
}

template <bool kAmn, bool kBmn, bool kRegScales>
cudaError_t set_smem_attrs() {
  cudaError_t err =
      cudaFuncSetAttribute(gemm_s8f16_kernel<kAmn, kBmn, kRegScales, 256>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, SingleTile<256>::kSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(gemm_s8f16_kernel<kAmn, kBmn, kRegScales, 128>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SingleTile<128>::kSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(gemm_s8f16_kernel<kAmn, kBmn, kRegScales, 64>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SingleTile<64>::kSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(gemm_s8f16_pair_kernel<kAmn, kBmn, kRegScales, kConvNone>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemBytes);
  if (err == cudaSuccess)
    err = set_conv_attrs(gemm_s8f16_pair_kernel<kAmn, kBmn, kRegScales, kConvWiden>);
  if (err == cudaSuccess && !kAmn && !kBmn)
    err = set_conv_attrs(gemm_s8f16_pair_kernel<false, false, kRegScales, kConvQuantB>);
  return err;
}

// Launch epochs for the split-tail counters: 40 bits, never 0, distinct for
// 2^40 launches of the process.
uint64_t next_epoch() {
  static std::atomic<uint64_t> ctr{0};
  static const uint64_t base = [] {
    uint64_t x = static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count());
    x ^= reinterpret_cast<uintptr_t>(&ctr);
    x *= 0x9E3779B97F4A7C15ull;
    return x >> 24;
  }();
  uint64_t e = (base + ctr.fetch_add(1)) & 0xFFFFFFFFFFull;
  return e == 0 ? 1 : e;
}

// Output map for the tile stores: boxes of 128 bytes x 32 rows, 128-byte
// swizzle (bf16: 64 columns; int32 and fp32: 32).
bool make_output_map(CUtensorMap* map, void* out, GemmOut mode, int64_t M, int64_t N,
                     int64_t ldo) {
  if (mode == GemmOut::kS32)
    return encode_tensor_map_2d(map, out, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, M, N, ldo, 32, 32,
                                CU_TENSOR_MAP_SWIZZLE_128B);
  if (mode == GemmOut::kF32Scaled)
    return encode_tensor_map_2d(map, out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, M, N, ldo, 32, 32,
                                CU_TENSOR_MAP_SWIZZLE_128B);
  return encode_tensor_map_2d(map, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, N, ldo, 64, 32,
                              CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool kAmn, bool kBmn, bool kRegScales>
cudaError_t launch_kernel(bool pair, int conv, int tile_n, int grid, const CUtensorMap& mapA,
                          const CUtensorMap& mapB, const CUtensorMap& mapO, const GemmParams& p,
                          cudaStream_t stream) {
  if (conv == kConvWiden)
    return launch_overlapped(gemm_s8f16_pair_kernel<kAmn, kBmn, kRegScales, kConvWiden>,
                             dim3(grid), dim3(kS8Threads), kS8SmemBytes, stream, mapA, mapB, mapO,
                             p);
  if (conv == kConvQuantB) {
    if constexpr (!kAmn && !kBmn)
      return launch_overlapped(gemm_s8f16_pair_kernel<false, false, kRegScales, kConvQuantB>,
                               dim3(grid), dim3(kS8Threads), kS8SmemBytes, stream, mapA, mapB,
                               mapO, p);
    return cudaErrorInvalidValue;  // B quantized in the prologue: A @ B.T only
  }
  if (pair)
    return launch_overlapped(gemm_s8f16_pair_kernel<kAmn, kBmn, kRegScales, kConvNone>,
                             dim3(grid), dim3(kThreads), kPairSmemBytes, stream, mapA, mapB, mapO,
                             p);
  if (tile_n == 128)
    return launch_overlapped(gemm_s8f16_kernel<kAmn, kBmn, kRegScales, 128>, dim3(grid),
                             dim3(kThreads), SingleTile<128>::kSmemBytes, stream, mapA, mapB, mapO,
                             p);
  if (tile_n == 64)
    return launch_overlapped(gemm_s8f16_kernel<kAmn, kBmn, kRegScales, 64>, dim3(grid),
                             dim3(kThreads), SingleTile<64>::kSmemBytes, stream, mapA, mapB, mapO,
                             p);
  return launch_overlapped(gemm_s8f16_kernel<kAmn, kBmn, kRegScales, 256>, dim3(grid),
                           dim3(kThreads), SingleTile<256>::kSmemBytes, stream, mapA, mapB, mapO,
                           p);
}

template <bool kAmn, bool kBmn>
cudaError_t launch_layout(bool pair, int conv, int tile_n, bool reg_scales, int grid,
                          const CUtensorMap& mapA, const CUtensorMap& mapB,
                          const CUtensorMap& mapO, const GemmParams& p, cudaStream_t stream) {
  return reg_scales ? launch_kernel<kAmn, kBmn, true>(pair, conv, tile_n, grid, mapA, mapB, mapO,
                                                      p, stream)
                    : launch_kernel<kAmn, kBmn, false>(pair, conv, tile_n, grid, mapA, mapB, mapO,
                                                       p, stream);
}

}  // namespace

cudaError_t launch_gemm(const void* A, bool a_mn, const float* sA, const void* B, bool b_mn,
                        const float* sB, int64_t M, int64_t N, int64_t K, bool s8, GemmOut mode,
                        void* out, int64_t ldo, void* scratch, const DeviceInfo& dev,
                        const GemmDebug& dbg, cudaStream_t stream) {
  if (a_mn && !b_mn) return cudaErrorInvalidValue;  // no layout of the API needs it
  if (s8 && mode == GemmOut::kBf16Plain) return cudaErrorInvalidValue;
  // the converter stage: int8 codes widened, or (test only) the bf16 B
  // operand quantized in the prologue from its row scales sB
  const int conv = s8 ? kConvWiden : dbg.quant_b ? kConvQuantB : kConvNone;
  if (conv == kConvQuantB && (s8 || a_mn || b_mn || mode == GemmOut::kBf16Plain || !sB))
    return cudaErrorInvalidValue;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[device]) {
      err = set_smem_attrs<false, false, false>();
      if (err == cudaSuccess) err = set_smem_attrs<false, true, false>();
      if (err == cudaSuccess) err = set_smem_attrs<true, true, false>();
      if (err == cudaSuccess) err = set_smem_attrs<false, false, true>();
      if (err == cudaSuccess) err = set_smem_attrs<false, true, true>();
      if (err == cudaSuccess) err = set_smem_attrs<true, true, true>();
      if (err != cudaSuccess) return err;
      attr_set[device] = true;
    }
  }
  // CTA pairs (256x256 tiles) when they give every pair of SMs a tile or
  // the contraction is long (each tile then runs long enough for the pair's
  // per-tile efficiency to win); otherwise single CTAs (128x256 tiles)
  // int8 operands always take the CTA-pair kernel (the only one that widens)
  const int64_t pair_tiles = ((M + 255) / 256) * ((N + kBN - 1) / kBN);
  const bool pair = conv != kConvNone ||
                    (M > kBM && (pair_tiles >= dev.sms / 2 || K >= 8192) && !dbg.single_cta);
  const bool plain = mode == GemmOut::kBf16Plain;
  // single CTAs: 128-column tiles when the 256-column ones would leave more
  // than half of the SMs idle and the narrower tiles still fit in one wave
  int tile_n = kBN;
  if (!pair) {
    const int64_t mt = (M + kBM - 1) / kBM;
    const int64_t t256 = mt * ((N + 255) / 256), t128 = mt * ((N + 127) / 128);
    const int64_t t64 = mt * ((N + 63) / 64);
    if (t256 * 2 <= dev.sms && t128 <= dev.sms && t128 > t256) tile_n = 128;
    if (tile_n == 128 && t128 * 2 <= dev.sms && t64 <= dev.sms && t64 > t128) tile_n = 64;
  }
  CUtensorMap mapA, mapB, mapO;
  const bool maps_ok =
      conv == kConvWiden
          ? make_raw_map(&mapA, A, a_mn, M, K) && make_raw_map(&mapB, B, b_mn, N, K)
      : conv == kConvQuantB
          ? make_operand_map(&mapA, A, false, M, K, kBM, false) &&
                encode_tensor_map_2d(&mapB, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, N, K, K, kBK,
                                     128, CU_TENSOR_MAP_SWIZZLE_NONE)
          : make_operand_map(&mapA, A, a_mn, M, K, kBM, plain) &&
                make_operand_map(&mapB, B, b_mn, N, K, pair ? 128 : tile_n, plain);
  if (!maps_ok || !make_output_map(&mapO, out, mode, M, N, ldo))
    return cudaErrorInvalidValue;
  GemmParams p;
  p.sA = sA;
  p.sB = sB;
  p.out = out;
  p.ldo = ldo;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.m_tiles = static_cast<int>((M + (pair ? 255 : kBM - 1)) / (pair ? 256 : kBM));
  p.n_tiles = static_cast<int>((N + (pair ? kBN : tile_n) - 1) / (pair ? kBN : tile_n));
  p.m_fastest = M < N ? 1 : 0;
  p.k_blocks = static_cast<int>((K + kBK - 1) / kBK);
  p.mode = mode == GemmOut::kS32 ? 1 : plain ? 2 : mode == GemmOut::kF32Scaled ? 3 : 0;
  p.ab_format = plain ? kFormatBf16 : 0u;
  // integer codes: exact fp32 chunks of 1024 terms; bf16: all of K at once
  p.chunk_blocks = plain ? p.k_blocks : kChunkBlocks;
  p.status = dev.status_word;
  p.wait_limit_ns = dbg.wait_limit_ns;
  p.drop_first_load = dbg.drop_first_load;
  p.dp_tiles = static_cast<int>(p.m_tiles) * p.n_tiles;
  p.sk_tail = 0;
  p.sk_split = 1;
  p.partials = nullptr;
  p.counters = nullptr;
  p.epoch = 0;
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
  const int64_t slots = pair ? dev.sms / 2 : dev.sms;
  int grid = static_cast<int>((pair ? 2 : 1) * (tiles < slots ? tiles : slots));
  if (pair && scratch && !dbg.no_split_tail) {
    // the R tiles of a partial last wave split into s = min(P / R, 4)
    // k-parts each (P pairs): the wave then takes 1/s of a tile's time
    // instead of a whole one
    const int64_t npairs = slots < kSplitTailMaxPairs ? slots : kSplitTailMaxPairs;
    const int64_t tail = tiles % npairs;
    int64_t split = tail > 0 ? npairs / tail : 0;
    if (split > kMaxSplit) split = kMaxSplit;  // the last part reads all parts back
    if (split > p.k_blocks) split = p.k_blocks;
    // worth it when the wave shrinks by at least 32 k-blocks of MMA time,
    // about what storing and summing the parts costs (~10 us on GB300)
    const bool worth = split >= 2 && (split - 1) * p.k_blocks >= 32 * split;
    if (tail > 0 && worth) {
      p.dp_tiles = static_cast<int>(tiles - tail);
      p.sk_tail = static_cast<int>(tail);
      p.sk_split = static_cast<int>(split);
      p.partials = static_cast<int32_t*>(scratch);
      p.counters = reinterpret_cast<unsigned long long*>(static_cast<char*>(scratch) +
                                                         kSplitTailMaxPairs * 256 * 256 * 4);
      p.epoch = next_epoch();
      grid = static_cast<int>(2 * npairs);
    }
  }
  // at most two tiles per CTA (pair): the scales are loaded when a tile starts
  const int units = grid / (pair ? 2 : 1);
  const bool reg_scales =
      mode != GemmOut::kF32Scaled && static_cast<int64_t>(p.dp_tiles) <= 2 * units;
  if (!a_mn && !b_mn)
    return launch_layout<false, false>(pair, conv, tile_n, reg_scales, grid, mapA, mapB, mapO, p,
                                       stream);
  if (!a_mn)
    return launch_layout<false, true>(pair, conv, tile_n, reg_scales, grid, mapA, mapB, mapO, p,
                                      stream);
  return launch_layout<true, true>(pair, conv, tile_n, reg_scales, grid, mapA, mapB, mapO, p,
                                   stream);
}

}  // namespace int8mp
