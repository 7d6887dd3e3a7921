// tma.cu -- host-side driver calls made through entry points resolved at run
// time (no link-time dependency on libcuda): encoding TMA tensor maps, and
// the SM count of a stream that belongs to a green context (an SM partition
// of the device), which sizes the persistent grids launched on it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace int8mp {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// CUdevResource as cuda.h lays it out (ABI version 1): type, padding, and a
// union whose SM member starts with smCount.
struct DevResource {
  int type;
  unsigned char pad[92];
  unsigned int sm_count, min_partition, coscheduled_alignment;
  unsigned char rest[48 - 12];
};
static_assert(sizeof(DevResource) == 144, "CUdevResource layout");

typedef CUresult (*StreamGetGreenCtxFn)(CUstream, CUgreenCtx*);
typedef CUresult (*GreenCtxGetDevResourceFn)(CUgreenCtx, DevResource*, int);

template <typename Fn>
Fn entry(const char* name, int version) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(f);
  return nullptr;
}

}  // namespace

int stream_sm_count(cudaStream_t stream) {
  static StreamGetGreenCtxFn get_ctx = nullptr;
  static GreenCtxGetDevResourceFn get_res = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_ctx = entry<StreamGetGreenCtxFn>("cuStreamGetGreenCtx", 12050);
    get_res = entry<GreenCtxGetDevResourceFn>("cuGreenCtxGetDevResource", 12040);
  });
  if (!stream || !get_ctx || !get_res) return 0;
  CUgreenCtx g = nullptr;
  if (get_ctx(reinterpret_cast<CUstream>(stream), &g) != CUDA_SUCCESS || !g) return 0;
  DevResource r{};
  if (get_res(g, &r, 1 /* CU_DEV_RESOURCE_TYPE_SM */) != CUDA_SUCCESS || r.type != 1) return 0;
  return static_cast<int>(r.sm_count);
}

bool encode_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                          int esize, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                          int box_rows, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * static_cast<cuuint64_t>(esize)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  return enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace int8mp
