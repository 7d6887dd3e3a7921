// common.cuh -- internal interface between the C-ABI layer (api.cu) and the
// kernel translation units (quantize.cu, gemm.cu).  Not installed, not part
// of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/int8mp.h"
#include "philox.cuh"

namespace int8mp {

// Everything a kernel needs to know about the device it runs on.
struct DeviceInfo {
  int sms = 0;
  unsigned int* status_word = nullptr;  // device address of the status word
};

// Stochastic-rounding parameters (header of int8mp.h gives the mapping),
// with the Philox round keys of the seed and the stream's round-0 product
// computed once on the host.
struct SrArgs {
  uint64_t seed;
  uint64_t offset;
  uint32_t stream_id;
  PhiloxKeys keys;
  PhiloxStream stream;
};

inline SrArgs make_sr(uint64_t seed, uint64_t offset, uint32_t stream_id) {
  return SrArgs{seed, offset, stream_id, philox_keys(seed), philox_stream(stream_id)};
}

// One matrix of a row-quantization launch (launch_quantize_rows_jobs):
// x [rows, cols] bf16 at row stride ld, codes q [rows, cols], scales
// [rows], column absmax colmax [cols] (updated) or null; offset and
// stream_id place its elements in the stochastic-rounding stream.
struct RowsJob {
  const void* x;
  int64_t rows, ld;
  void* q;
  float* scale;
  float* colmax;
  uint64_t offset;
  uint32_t stream_id;
};
constexpr int kMaxRowsJobs = 2;

// Wait limit for every bounded device-side wait, in nanoseconds of
// %globaltimer.  Long enough that no healthy wait reaches it.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---- launches ----------------------------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialization: its launch and set-up overlap the end of the kernel before
// it in the stream, and it waits (griddepcontrol.wait) before touching
// global memory, so stream order still holds for every byte.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- driver entry points (tma.cu) ------------------------------------------
// SMs of the green context (SM partition) `stream` belongs to; 0 if it
// belongs to none (then the device's count applies).
int stream_sm_count(cudaStream_t stream);

// ---- TMA tensor maps (tma.cu) -----------------------------------------------
// Row-major [rows, cols] matrix of `esize`-byte elements, row stride ld
// elements; boxes of box_rows x box_cols; zero fill outside the matrix.
bool encode_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                          int esize, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                          int box_rows, CUtensorMapSwizzle swizzle);

// ---- quantize (quantize.cu) ------------------------------------------------
// x bf16 [rows, cols] stride ld.  Row groups: q [rows, cols]; scale [rows].
// colmax (optional, fp32 [cols]): each column's absmax is max-merged into it.
// One launch for up to kMaxRowsJobs matrices with the same row length (two
// when their rows fit shared memory, one per matrix otherwise); every job
// has a colmax or none has.
cudaError_t launch_quantize_rows_jobs(const RowsJob* jobs, int njobs, int64_t cols,
                                      int8mp_round mode, uint64_t seed, int8mp_codes codes,
                                      const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_quantize_rows(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                 int8mp_round mode, const SrArgs& sr, void* q,
                                 int8mp_codes codes, float* scale, float* colmax,
                                 const DeviceInfo& dev, cudaStream_t stream);
// n 32-bit words at p set to 0 (a kernel: keeps dependent launches going).
cudaError_t launch_zero_words(void* p, int64_t n, const DeviceInfo& dev, cudaStream_t stream);
// y[i] = bf16_RNE(x[i]) for n fp32 values (x, y 16-byte aligned).
cudaError_t launch_round_bf16(const float* x, void* y, int64_t n, const DeviceInfo& dev,
                              cudaStream_t stream);
// colmax[c] = max(colmax[c], max_r |x[r,c]|) (fp32 [cols]), one pass.
cudaError_t launch_column_absmax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                 float* colmax, const DeviceInfo& dev, cudaStream_t stream);
// Column groups whose absmax is given (fp32 [cols]): scale [cols] =
// absmax / 127, codes q [rows, cols] (row stride cols).
cudaError_t launch_quantize_cols_from_absmax(const void* x, int64_t rows, int64_t cols,
                                             int64_t ld, const float* absmax, int8mp_round mode,
                                             const SrArgs& sr, void* q, int8mp_codes codes,
                                             float* scale, const DeviceInfo& dev,
                                             cudaStream_t stream);
// Column groups, scale [cols]; codes q [rows, cols] (row stride cols), or
// transposed q [cols, rows] (row stride rows) when `transposed`.
cudaError_t launch_quantize_cols(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                 int8mp_round mode, const SrArgs& sr, void* q,
                                 int8mp_codes codes, float* scale, bool transposed,
                                 const DeviceInfo& dev, cudaStream_t stream);
// Column groups (codes in the input's layout) of up to kMaxRowsJobs matrices
// with the same number of columns: one launch when every job has at most 2048
// rows, else each job's own passes.  Job colmax is unused.
cudaError_t launch_quantize_cols_jobs(const RowsJob* jobs, int njobs, int64_t cols,
                                      int8mp_round mode, uint64_t seed, int8mp_codes codes,
                                      const DeviceInfo& dev, cudaStream_t stream);

// ---- GEMM (gemm.cu) ---------------------------------------------------------
// kBf16Scaled: integer codes in f16 containers, out = bf16((acc * sA) * sB);
// kS32: the same codes, out = the int32 accumulator; kBf16Plain: bf16
// operands, out = bf16_RNE of their fp32-accumulated product (sA, sB unused);
// kF32Scaled: integer codes, out = the fp32 (acc * sA) * sB itself.
enum class GemmOut { kBf16Scaled = 0, kS32 = 1, kBf16Plain = 2, kF32Scaled = 3 };

struct GemmDebug {
  int drop_first_load = 0;        // test only: never issue the first TMA load
  int single_cta = 0;             // test only: use the single-CTA kernel for any M
  int no_split_tail = 0;            // test only: no split last wave even with scratch
  int quant_b = 0;  // test only: B is bf16, quantized in the GEMM's prologue with its scales sB
  uint64_t wait_limit_ns = kWaitLimitNs;
};

// Scratch of the CTA-pair GEMM's split last wave: a 256x256 int32 slot per
// pair and 16 64-bit counters per split tile, for up to kSplitTailMaxPairs
// pairs.  Needs no initialization; one scratch must not serve two GEMMs at
// the same time.
constexpr int kSplitTailMaxPairs = 80;
constexpr size_t kSplitTailScratchBytes =
    static_cast<size_t>(kSplitTailMaxPairs) * 256 * 256 * 4 + kSplitTailMaxPairs * 2 * 8 * 8;

// Integer codes in f16 containers, or as int8 (s8: widened to f16 inside the
// CTA-pair kernel), or bf16 values for kBf16Plain.  A is [M,K] (a_mn false,
// K contiguous) or [K,M] (a_mn true, M contiguous); B is [N,K] or [K,N]
// likewise.  Every combination but (a_mn, !b_mn) is served.  scratch: NULL,
// or kSplitTailScratchBytes (16-byte aligned) that lets the CTA-pair kernel
// split its last wave of tiles.
cudaError_t launch_gemm(const void* A, bool a_mn, const float* sA, const void* B, bool b_mn,
                        const float* sB, int64_t M, int64_t N, int64_t K, bool s8, GemmOut mode,
                        void* out, int64_t ldo, void* scratch, const DeviceInfo& dev,
                        const GemmDebug& dbg, cudaStream_t stream);

}  // namespace int8mp
