// quantize.cu -- dynamic symmetric INT8 quantization of bf16 matrices.
//
// "Quantized model training" README, section "INT8 mixed precision
// training": each matmul operand is quantized dynamically and row-wise (one
// scale per row of the contraction).  "Add QAT support for distributed
// finetuning", summary: x_q = clamp(x / scale + zp) -- here zp = 0 and
// scale = absmax / 127.
//
// Two groupings:
//   rows    one group per row of x [rows, cols] (the contraction axis is
//           contiguous): the row is held in registers, reduced by warp
//           shuffles, and quantized without a second read.
//   columns one group per column (the contraction axis is the leading one):
//           pass 1 reduces column absmax over row blocks into the scale
//           buffer (atomic max on the fp32 bit pattern, valid for values
//           >= 0); pass 2 re-reads 256x64 tiles, quantizes, and writes the
//           codes transposed [cols, rows] through a swizzled shared-memory
//           tile; pass 3 turns the stored absmax into absmax / 127.
//
// Arithmetic per element (identical to the header of int8mp.h):
//   v = x / s (IEEE division), q = clamp(rint(v)) or, stochastically,
//   q = clamp(floor(v) + (u < v - floor(v))), u from Philox4x32-10.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "philox.cuh"

namespace int8mp {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float absmax8(float m, const uint4& v) {
  m = fmaxf(m, fabsf(bf16_lo(v.x)));
  m = fmaxf(m, fabsf(bf16_hi(v.x)));
  m = fmaxf(m, fabsf(bf16_lo(v.y)));
  m = fmaxf(m, fabsf(bf16_hi(v.y)));
  m = fmaxf(m, fabsf(bf16_lo(v.z)));
  m = fmaxf(m, fabsf(bf16_hi(v.z)));
  m = fmaxf(m, fabsf(bf16_lo(v.w)));
  m = fmaxf(m, fabsf(bf16_hi(v.w)));
  return m;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// One code as an exact float in [-127, 127] (never -0).  s > 0.
template <bool SR>
__device__ __forceinline__ float code_of(float x, float s, uint32_t word) {
  const float v = __fdiv_rn(x, s);
  float q;
  if (SR) {
    const float f = floorf(v);
    const float fr = __fsub_rn(v, f);
    q = (sr_uniform(word) < fr) ? __fadd_rn(f, 1.0f) : f;
  } else {
    q = rintf(v);
  }
  q = fminf(fmaxf(q, -127.0f), 127.0f);
  return __fadd_rn(q, 0.0f);  // -0 -> +0
}

// Eight codes of one vector (elements n0 .. n0+7 of the SR stream).
template <bool SR>
__device__ __forceinline__ void codes8(const float (&f)[8], float s, const SrArgs& sr, uint64_t n0,
                                       float (&c)[8]) {
  uint32_t w[8];
  if (SR) {
    philox_words8(sr.seed, n0, sr.stream_id, w);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0u;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = (s != 0.0f) ? code_of<SR>(f[i], s, w[i]) : 0.0f;
}

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
// A team of `wpr` warps owns one row; lane t of the team holds vectors
// t, t + 32*wpr, ... (VPL of them) in registers.
template <typename CodeT, int VPL, bool SR>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, CodeT* __restrict__ q,
    float* __restrict__ scale, int wpr, SrArgs sr) {
  __shared__ float red[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int teams = (kThreads / 32) / wpr;
  const int team = warp / wpr, wit = warp % wpr;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * teams + team;
  const bool active = row < rows;
  const int nvec = static_cast<int>(cols >> 3);
  const int tl = wit * 32 + lane, stride = wpr * 32;

  const uint4* xr = reinterpret_cast<const uint4*>(x + (active ? row : 0) * ld);
  uint4 v[VPL];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int vi = tl + j * stride;
    v[j] = (active && vi < nvec) ? __ldg(xr + vi) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int j = 0; j < VPL; ++j) amax = absmax8(amax, v[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if (wpr > 1) {
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[team * wpr];
    for (int w = 1; w < wpr; ++w) amax = fmaxf(amax, red[team * wpr + w]);
  }
  const float s = __fdiv_rn(amax, 127.0f);
  if (active && tl == 0) scale[row] = s;
  if (!active) return;

  using P = Pack8<CodeT>;
  typename P::Vec* qr = reinterpret_cast<typename P::Vec*>(q + row * cols);
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int vi = tl + j * stride;
    if (vi < nvec) {
      float f[8], c[8];
      unpack8(v[j], f);
      codes8<SR>(f, s, sr, sr.offset + static_cast<uint64_t>(row * cols + vi * 8), c);
      qr[vi] = P::pack(c);
    }
  }
}

// Rows too long for registers: one block per row, two sweeps (the second
// re-reads the row, which is still in L2).
template <typename CodeT, bool SR>
__global__ void __launch_bounds__(kThreads) quant_rows_long_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld, CodeT* __restrict__ q,
    float* __restrict__ scale, SrArgs sr) {
  __shared__ float red[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  if (row >= rows) return;
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
  using P = Pack8<CodeT>;
  typename P::Vec* qr = reinterpret_cast<typename P::Vec*>(q + row * cols);
  for (int64_t vi = threadIdx.x; vi < nvec; vi += kThreads) {
    float f[8], c[8];
    unpack8(__ldg(xr + vi), f);
    codes8<SR>(f, s, sr, sr.offset + static_cast<uint64_t>(row * cols + vi * 8), c);
    qr[vi] = P::pack(c);
  }
}

// --------------------------------------------------------- column groups
// Pass 1: absmax of each column over this block's rows, merged by atomic max
// on the bit pattern (absolute values are >= +0, whose bits order as
// unsigned integers).  Lane = one 8-column vector, warp = row phase.
__global__ void __launch_bounds__(kThreads) col_absmax_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
    int64_t rows_per_block, unsigned int* __restrict__ amax_bits) {
  __shared__ float red[kThreads / 32][32][9];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nvec = cols >> 3;
  const int64_t vi = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_block;
  const int64_t r1 = min(rows, r0 + rows_per_block);
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = 0.0f;
  if (vi < nvec) {
    const uint16_t* base = x + vi * 8;
    int64_t r = r0 + warp;
    for (; r + 3 * 8 < r1; r += 4 * 8) {
      uint4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = __ldg(reinterpret_cast<const uint4*>(base + (r + u * 8) * ld));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
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

// Pass 2: a 256-row x 64-column tile.  Thread (rg, cg) loads rows
// rg*8 .. rg*8+7 of column group cg (8 columns, one 16-byte vector each),
// quantizes the 8x8 block, transposes it in registers, and stores the 8
// column vectors into the shared tile [64 cols][256 rows]; the 16-byte (f16)
// or 8-byte (int8) slot of row group rg in column row rho is placed at slot
// rg ^ (rho / 8) so that both the writes and the row-wise read-out spread
// over the banks.  The read-out stores whole rows of the transposed codes.
template <typename CodeT, bool SR>
__global__ void __launch_bounds__(kThreads) quant_cols_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
    const unsigned int* __restrict__ amax_bits, CodeT* __restrict__ q, SrArgs sr) {
  using P = Pack8<CodeT>;
  using Vec = typename P::Vec;
  __shared__ Vec tile[64][32];
  const int t = threadIdx.x;
  const int cg = t & 7, rg = t >> 3;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 256;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 64;
  const int64_t c = c0 + cg * 8;
  const int64_t rb = r0 + rg * 8;
  if (c < cols) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      v[i] = (rb + i < rows) ? __ldg(reinterpret_cast<const uint4*>(x + (rb + i) * ld + c))
                             : make_uint4(0u, 0u, 0u, 0u);
    float s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = __fdiv_rn(__uint_as_float(__ldg(amax_bits + c + j)), 127.0f);
    float cd[8][8];  // [row i][col j]
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float f[8], out[8];
      unpack8(v[i], f);
      uint32_t w[8];
      if (SR) {
        philox_words8(sr.seed, sr.offset + static_cast<uint64_t>((rb + i) * cols + c), sr.stream_id, w);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = 0u;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) out[j] = (s[j] != 0.0f) ? code_of<SR>(f[j], s[j], w[j]) : 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) cd[i][j] = out[j];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float colv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) colv[i] = cd[i][j];
      const int rho = cg * 8 + j;
      tile[rho][rg ^ cg] = P::pack(colv);
    }
  }
  __syncthreads();
  // read-out: warp w handles rows rho = w, w+8, ..., lane = row-group slot
  const int warp = t >> 5, lane = t & 31;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int rho = warp + it * 8;
    const int64_t cc = c0 + rho;
    const int64_t rr = r0 + lane * 8;
    if (cc < cols && rr < rows) {
      Vec* dst = reinterpret_cast<Vec*>(q + cc * rows + rr);
      *dst = tile[rho][lane ^ (rho >> 3)];
    }
  }
}

// Pass 3: scale = absmax / 127, in place.
__global__ void col_scale_kernel(unsigned int* __restrict__ amax_bits, int64_t cols) {
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c < cols) {
    const float s = __fdiv_rn(__uint_as_float(amax_bits[c]), 127.0f);
    amax_bits[c] = __float_as_uint(s);
  }
}

template <typename CodeT, bool SR>
cudaError_t rows_dispatch(const void* x, int64_t rows, int64_t cols, int64_t ld, void* q,
                          float* scale, const SrArgs& sr, cudaStream_t stream) {
  const int64_t nvec = cols >> 3;
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  CodeT* qp = static_cast<CodeT*>(q);
  int wpr = 0, vpl = 0;
  for (int w = 1; w <= 8 && !wpr; w <<= 1)
    for (int p = 2; p <= 8; p <<= 1)
      if (static_cast<int64_t>(w) * 32 * p >= nvec) {
        wpr = w;
        vpl = p;
        break;
      }
  if (!wpr) {
    quant_rows_long_kernel<CodeT, SR><<<static_cast<unsigned>(rows), kThreads, 0, stream>>>(
        xp, rows, cols, ld, qp, scale, sr);
    return cudaGetLastError();
  }
  const int64_t teams = (kThreads / 32) / wpr;
  const unsigned blocks = static_cast<unsigned>((rows + teams - 1) / teams);
  switch (vpl) {
    case 2:
      quant_rows_kernel<CodeT, 2, SR><<<blocks, kThreads, 0, stream>>>(xp, rows, cols, ld, qp, scale, wpr, sr);
      break;
    case 4:
      quant_rows_kernel<CodeT, 4, SR><<<blocks, kThreads, 0, stream>>>(xp, rows, cols, ld, qp, scale, wpr, sr);
      break;
    default:
      quant_rows_kernel<CodeT, 8, SR><<<blocks, kThreads, 0, stream>>>(xp, rows, cols, ld, qp, scale, wpr, sr);
      break;
  }
  return cudaGetLastError();
}

template <typename CodeT, bool SR>
cudaError_t cols_dispatch(const void* x, int64_t rows, int64_t cols, int64_t ld, void* q,
                          float* scale, const SrArgs& sr, const DeviceInfo& dev,
                          cudaStream_t stream) {
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  unsigned int* amax = reinterpret_cast<unsigned int*>(scale);
  cudaError_t err = cudaMemsetAsync(amax, 0, static_cast<size_t>(cols) * sizeof(float), stream);
  if (err != cudaSuccess) return err;
  const int64_t nvec = cols >> 3;
  const int64_t gx = (nvec + 31) / 32;
  const int64_t target = static_cast<int64_t>(dev.sms > 0 ? dev.sms : 148) * 8;
  int64_t gy = target / gx;
  if (gy < 1) gy = 1;
  const int64_t max_gy = (rows + 63) / 64;
  if (gy > max_gy) gy = max_gy;
  if (gy > 65535) gy = 65535;
  const int64_t rpb = (rows + gy - 1) / gy;
  col_absmax_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), kThreads, 0, stream>>>(
      xp, rows, cols, ld, rpb, amax);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const dim3 grid2(static_cast<unsigned>((cols + 63) / 64), static_cast<unsigned>((rows + 255) / 256));
  quant_cols_kernel<CodeT, SR><<<grid2, kThreads, 0, stream>>>(xp, rows, cols, ld, amax,
                                                               static_cast<CodeT*>(q), sr);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  col_scale_kernel<<<static_cast<unsigned>((cols + 255) / 256), 256, 0, stream>>>(amax, cols);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_rows(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                 int8mp_round mode, const SrArgs& sr, void* q,
                                 int8mp_codes codes, float* scale, const DeviceInfo&,
                                 cudaStream_t stream) {
  const bool s = mode == INT8MP_SR;
  if (codes == INT8MP_CODES_S8)
    return s ? rows_dispatch<int8_t, true>(x, rows, cols, ld, q, scale, sr, stream)
             : rows_dispatch<int8_t, false>(x, rows, cols, ld, q, scale, sr, stream);
  return s ? rows_dispatch<__half, true>(x, rows, cols, ld, q, scale, sr, stream)
           : rows_dispatch<__half, false>(x, rows, cols, ld, q, scale, sr, stream);
}

cudaError_t launch_quantize_cols(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                 int8mp_round mode, const SrArgs& sr, void* q,
                                 int8mp_codes codes, float* scale, const DeviceInfo& dev,
                                 cudaStream_t stream) {
  const bool s = mode == INT8MP_SR;
  if (codes == INT8MP_CODES_S8)
    return s ? cols_dispatch<int8_t, true>(x, rows, cols, ld, q, scale, sr, dev, stream)
             : cols_dispatch<int8_t, false>(x, rows, cols, ld, q, scale, sr, dev, stream);
  return s ? cols_dispatch<__half, true>(x, rows, cols, ld, q, scale, sr, dev, stream)
           : cols_dispatch<__half, false>(x, rows, cols, ld, q, scale, sr, dev, stream);
}

}  // namespace int8mp
