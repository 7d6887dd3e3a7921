// api.cu -- the extern "C" entry points of libint8mp.so (declared in
// include/int8mp.h and include/int8mp_debug.h): argument validation,
// per-device state, workspace carving and the composition of the linear
// forward / backward passes out of the quantize and GEMM launchers.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/int8mp.h"
#include "../../include/int8mp_debug.h"
#include "common.cuh"

namespace {

using int8mp::DeviceInfo;

// Bit 0 set by any kernel whose bounded wait ran out; bit 1 by a failed
// bounds check (checked builds only).
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::once_flag once;
  int8mp_status status = INT8MP_OK;
  DeviceInfo info;
};
DeviceState g_devices[kMaxDevices];

int8mp_status current_device(DeviceInfo* info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return INT8MP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return INT8MP_ERR_UNSUPPORTED_DEVICE;
  DeviceState& st = g_devices[dev];
  std::call_once(st.once, [&st, dev] {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      st.status = INT8MP_ERR_CUDA;
      return;
    }
    if (major != 10 || minor != 3) {
      st.status = INT8MP_ERR_UNSUPPORTED_DEVICE;
      return;
    }
    void* word = nullptr;
    if (cudaGetSymbolAddress(&word, g_status_word) != cudaSuccess) {
      st.status = INT8MP_ERR_CUDA;
      return;
    }
    st.info.sms = sms;
    st.info.status_word = static_cast<unsigned int*>(word);
    st.status = INT8MP_OK;
  });
  if (st.status == INT8MP_OK) *info = st.info;
  return st.status;
}

// The device's info with the SM count of `stream`'s partition: kernels
// launched on a green-context stream see only that context's SMs, and the
// persistent grids are sized for them.
int8mp_status current_device(DeviceInfo* info, cudaStream_t stream) {
  const int8mp_status st = current_device(info);
  if (st != INT8MP_OK) return st;
  const int part = int8mp::stream_sm_count(stream);
  if (part > 0 && part < info->sms) info->sms = part;
  return INT8MP_OK;
}

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline int8mp_status from_cuda(cudaError_t e) { return e == cudaSuccess ? INT8MP_OK : INT8MP_ERR_CUDA; }

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// ------------------------------------------------------------ validation
int8mp_status check_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int axis,
                             int8mp_round mode, const void* q, int8mp_codes codes,
                             const float* scale) {
  if (axis != 0 && axis != 1 && axis != 2) return INT8MP_ERR_INVALID_ARG;
  if (mode != INT8MP_RNE && mode != INT8MP_SR) return INT8MP_ERR_INVALID_ARG;
  if (codes != INT8MP_CODES_S8 && codes != INT8MP_CODES_F16) return INT8MP_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ld < cols) return INT8MP_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return INT8MP_OK;
  if (!x || !q || !scale) return INT8MP_ERR_INVALID_ARG;
  if (axis == 1 && rows > 65535ll * 256) return INT8MP_ERR_INVALID_ARG;
  if (rows > (int64_t{1} << 31) - 1) return INT8MP_ERR_INVALID_ARG;
  if (cols % 8 || ld % 8 || !aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 4))
    return INT8MP_ERR_ALIGNMENT;
  if (axis == 1 && rows % 8) return INT8MP_ERR_ALIGNMENT;
  return INT8MP_OK;
}

int8mp_status check_mm(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                       int8mp_layout layout, int8mp_codes codes, const void* out, int64_t ldo) {
  if (layout != INT8MP_AxBT && layout != INT8MP_AxB && layout != INT8MP_ATxB)
    return INT8MP_ERR_INVALID_ARG;
  if (codes != INT8MP_CODES_S8 && codes != INT8MP_CODES_F16) return INT8MP_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || K > INT8MP_MAX_K || ldo < N) return INT8MP_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX) return INT8MP_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return INT8MP_OK;
  if (!out || (K > 0 && (!A || !B))) return INT8MP_ERR_INVALID_ARG;
  if (K % 16 || N % 8 || ldo % 8 || !aligned(out, 16)) return INT8MP_ERR_ALIGNMENT;
  if (layout == INT8MP_ATxB && M % 8) return INT8MP_ERR_ALIGNMENT;  // rows of A^T are M long
  // int8 rows of a [K, M] or [K, N] operand are 16-byte multiples (TMA strides)
  if (codes == INT8MP_CODES_S8 && ((layout != INT8MP_AxBT && N % 16) ||
                                   (layout == INT8MP_ATxB && M % 16)))
    return INT8MP_ERR_ALIGNMENT;
  if (K > 0 && (!aligned(A, 16) || !aligned(B, 16))) return INT8MP_ERR_ALIGNMENT;
  return INT8MP_OK;
}

// layout AxBT: both operands K-major; AxB: B MN-major ([K,N]); ATxB: both
// MN-major (A [K,M], B [K,N]).
// workspace of the *_ws matmuls: NULL (whole tiles), or at least
// int8mp_mm_workspace_size() bytes, 256-byte aligned
int8mp_status check_mm_workspace(const void* workspace, size_t ws_bytes) {
  if (!workspace) return INT8MP_OK;
  if (!aligned(workspace, 256)) return INT8MP_ERR_ALIGNMENT;
  if (ws_bytes < int8mp::kSplitTailScratchBytes) return INT8MP_ERR_WORKSPACE;
  return INT8MP_OK;
}

int8mp_status run_mm(const void* A, const float* sA, const void* B, const float* sB, int64_t M,
                     int64_t N, int64_t K, int8mp_layout layout, int8mp::GemmOut mode, void* out,
                     int64_t ldo, void* scratch, const int8mp::GemmDebug& dbg,
                     cudaStream_t stream, bool s8 = false) {
  if (M == 0 || N == 0) return INT8MP_OK;
  DeviceInfo dev;
  int8mp_status st = current_device(&dev, stream);
  if (st != INT8MP_OK) return st;
  const size_t esize = mode == int8mp::GemmOut::kS32 ? 4 : 2;
  if (K == 0)  // empty contraction: every accumulator is 0, and so is 0 * sA * sB
    return from_cuda(cudaMemset2DAsync(out, static_cast<size_t>(ldo) * esize, 0,
                                       static_cast<size_t>(N) * esize, static_cast<size_t>(M),
                                       stream));
  const bool a_mn = layout == INT8MP_ATxB, b_mn = layout != INT8MP_AxBT;
  return from_cuda(int8mp::launch_gemm(A, a_mn, sA, B, b_mn, sB, M, N, K, s8, mode, out, ldo,
                                       scratch, dev, dbg, stream));
}

// ------------------------------------------------------------- workspace
constexpr size_t kAlign = 256;
inline size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Carver {
  char* base;
  size_t used = 0;
  void* take(size_t bytes) {
    void* p = base ? base + used : nullptr;
    used += round_up(bytes);
    return p;
  }
};

// f16 codes + fp32 scales of one quantized operand
struct QOperand {
  void* q;
  float* s;
};
inline QOperand carve_operand(Carver& c, int64_t groups, int64_t glen) {
  QOperand o;
  o.q = c.take(static_cast<size_t>(groups) * static_cast<size_t>(glen) * 2);
  o.s = static_cast<float*>(c.take(static_cast<size_t>(groups) * 4));
  return o;
}

size_t fwd_bytes(int64_t T, int64_t N, int64_t K) {
  Carver c{nullptr};
  carve_operand(c, T, K);
  carve_operand(c, N, K);
  return c.used;
}
// backward codes: dY by rows [T,N] + s[T] (grad input, along N); W by
// columns [N,K] + s[K] (along N); dY by columns [T,N] + s[N] (grad weight,
// along T); X by columns [T,K] + s[K] (along T).  Column codes keep the
// input's layout and enter the matmul MN-major.  Then the column absmax of
// dY [N], X [K] and W [K] (contiguous, cleared by one memset).
struct BwdOperands {
  QOperand dy_rows, w_cols, dy_cols, x_cols;
  float* absmax;  // dY [N], then X [K], then W [K]
};
BwdOperands carve_bwd(Carver& c, int64_t T, int64_t N, int64_t K) {
  BwdOperands o;
  o.dy_rows = carve_operand(c, T, N);
  o.w_cols = carve_operand(c, K, N);
  o.dy_cols = carve_operand(c, N, T);
  o.x_cols = carve_operand(c, K, T);
  o.absmax = static_cast<float*>(c.take(static_cast<size_t>(N + 2 * K) * 4));
  return o;
}
size_t bwd_bytes(int64_t T, int64_t N, int64_t K) {
  Carver c{nullptr};
  carve_bwd(c, T, N, K);
  return c.used;
}

// The GEMM's last-wave scratch, when the workspace extends that far past the
// `used` bytes the pass needs (else NULL: whole-tile schedule).
void* gemm_scratch(void* workspace, size_t ws_bytes, size_t used) {
  if (!workspace || ws_bytes < used + int8mp::kSplitTailScratchBytes) return nullptr;
  return static_cast<char*>(workspace) + used;
}

int8mp_status check_linear(int64_t T, int64_t N, int64_t K, const int8mp_linear_cfg* cfg) {
  if (!cfg) return INT8MP_ERR_INVALID_ARG;
  auto flag = [](int v) { return v == 0 || v == 1; };
  if (!flag(cfg->int8_fwd) || !flag(cfg->int8_grad_in) || !flag(cfg->int8_grad_w))
    return INT8MP_ERR_INVALID_ARG;
  if (cfg->mode != INT8MP_RNE && cfg->mode != INT8MP_SR) return INT8MP_ERR_INVALID_ARG;
  if (T < 0 || N < 0 || K < 0) return INT8MP_ERR_INVALID_ARG;
  if (T > INT8MP_MAX_K || N > INT8MP_MAX_K || K > INT8MP_MAX_K) return INT8MP_ERR_INVALID_ARG;
  if (T % 16 || N % 16 || K % 16) return INT8MP_ERR_ALIGNMENT;
  return INT8MP_OK;
}

int8mp::SrArgs sr_of(const int8mp_linear_cfg* cfg, uint32_t stream_id) {
  return int8mp::make_sr(cfg->seed, cfg->offset, stream_id);
}

}  // namespace

extern "C" {

int8mp_status int8mp_quantize_rowwise(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                      int axis, int8mp_round mode, uint64_t seed,
                                      uint64_t offset, uint32_t stream_id, void* q,
                                      int8mp_codes codes, float* scale, void* stream) {
  int8mp_status st = check_quantize(x, rows, cols, ld, axis, mode, q, codes, scale);
  if (st != INT8MP_OK || rows == 0 || cols == 0) return st;
  DeviceInfo dev;
  st = current_device(&dev, as_stream(stream));
  if (st != INT8MP_OK) return st;
  const int8mp::SrArgs sr = int8mp::make_sr(seed, offset, stream_id);
  cudaError_t e = axis == 0
                      ? int8mp::launch_quantize_rows(x, rows, cols, ld, mode, sr, q, codes, scale,
                                                     nullptr, dev, as_stream(stream))
                      : int8mp::launch_quantize_cols(x, rows, cols, ld, mode, sr, q, codes, scale,
                                                     axis == 1, dev, as_stream(stream));
  return from_cuda(e);
}

int8mp_status int8mp_quantize_rows_colmax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                          int8mp_round mode, uint64_t seed, uint64_t offset,
                                          uint32_t stream_id, void* q, int8mp_codes codes,
                                          float* scale, float* colmax, void* stream) {
  int8mp_status st = check_quantize(x, rows, cols, ld, 0, mode, q, codes, scale);
  if (st != INT8MP_OK || rows == 0 || cols == 0) return st;
  if (!colmax) return INT8MP_ERR_INVALID_ARG;
  if (!aligned(colmax, 4)) return INT8MP_ERR_ALIGNMENT;
  DeviceInfo dev;
  st = current_device(&dev, as_stream(stream));
  if (st != INT8MP_OK) return st;
  const int8mp::SrArgs sr = int8mp::make_sr(seed, offset, stream_id);
  return from_cuda(int8mp::launch_quantize_rows(x, rows, cols, ld, mode, sr, q, codes, scale,
                                                colmax, dev, as_stream(stream)));
}

int8mp_status int8mp_quantize_rows_batch(const int8mp_rows_job* jobs, int njobs, int64_t cols,
                                         int8mp_round mode, uint64_t seed, int8mp_codes codes,
                                         void* stream) {
  if (!jobs || njobs < 1 || njobs > INT8MP_MAX_ROWS_JOBS) return INT8MP_ERR_INVALID_ARG;
  int8mp::RowsJob run[INT8MP_MAX_ROWS_JOBS];
  int nrun = 0;
  const bool cm = jobs[0].colmax != nullptr;
  for (int i = 0; i < njobs; ++i) {
    const int8mp_rows_job& j = jobs[i];
    int8mp_status st = check_quantize(j.x, j.rows, cols, j.ld, 0, mode, j.q, codes, j.scale);
    if (st != INT8MP_OK) return st;
    if ((j.colmax != nullptr) != cm) return INT8MP_ERR_INVALID_ARG;
    if (cm && !aligned(j.colmax, 4)) return INT8MP_ERR_ALIGNMENT;
    if (j.rows > 0 && cols > 0)
      run[nrun++] = int8mp::RowsJob{j.x, j.rows, j.ld, j.q, j.scale, j.colmax, j.offset,
                                    j.stream_id};
  }
  if (nrun == 0) return INT8MP_OK;
  DeviceInfo dev;
  int8mp_status st = current_device(&dev, as_stream(stream));
  if (st != INT8MP_OK) return st;
  return from_cuda(int8mp::launch_quantize_rows_jobs(run, nrun, cols, mode, seed, codes, dev,
                                                     as_stream(stream)));
}

int8mp_status int8mp_quantize_cols_batch(const int8mp_rows_job* jobs, int njobs, int64_t cols,
                                         int8mp_round mode, uint64_t seed, int8mp_codes codes,
                                         void* stream) {
  if (!jobs || njobs < 1 || njobs > INT8MP_MAX_ROWS_JOBS) return INT8MP_ERR_INVALID_ARG;
  int8mp::RowsJob run[INT8MP_MAX_ROWS_JOBS];
  int nrun = 0;
  for (int i = 0; i < njobs; ++i) {
    const int8mp_rows_job& j = jobs[i];
    int8mp_status st = check_quantize(j.x, j.rows, cols, j.ld, 2, mode, j.q, codes, j.scale);
    if (st != INT8MP_OK) return st;
    if (j.colmax != nullptr) return INT8MP_ERR_INVALID_ARG;
    if (j.rows > 0 && cols > 0)
      run[nrun++] = int8mp::RowsJob{j.x, j.rows, j.ld, j.q, j.scale, nullptr, j.offset,
                                    j.stream_id};
  }
  if (nrun == 0) return INT8MP_OK;
  DeviceInfo dev;
  int8mp_status st = current_device(&dev, as_stream(stream));
  if (st != INT8MP_OK) return st;
  return from_cuda(int8mp::launch_quantize_cols_jobs(run, nrun, cols, mode, seed, codes, dev,
                                                     as_stream(stream)));
}

int8mp_status int8mp_quantize_cols_absmax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                          const float* colmax, int8mp_round mode, uint64_t seed,
                                          uint64_t offset, uint32_t stream_id, void* q,
                                          int8mp_codes codes, float* scale, void* stream) {
  int8mp_status st = check_quantize(x, rows, cols, ld, 2, mode, q, codes, scale);
  if (st != INT8MP_OK || rows == 0 || cols == 0) return st;
  if (!colmax) return INT8MP_ERR_INVALID_ARG;
  if (!aligned(colmax, 4)) return INT8MP_ERR_ALIGNMENT;
  DeviceInfo dev;
  st = current_device(&dev, as_stream(stream));
  if (st != INT8MP_OK) return st;
  const int8mp::SrArgs sr = int8mp::make_sr(seed, offset, stream_id);
  return from_cuda(int8mp::launch_quantize_cols_from_absmax(x, rows, cols, ld, colmax, mode, sr,
                                                            q, codes, scale, dev,
                                                            as_stream(stream)));
}

size_t int8mp_mm_workspace_size(void) { return int8mp::kSplitTailScratchBytes; }

int8mp_status int8mp_scaled_mm(const void* A, const float* sA, const void* B, const float* sB,
                               int64_t M, int64_t N, int64_t K, int8mp_layout layout,
                               int8mp_codes codes, void* out, int64_t ldo, void* stream) {
  return int8mp_scaled_mm_ws(A, sA, B, sB, M, N, K, layout, codes, out, ldo, nullptr, 0, stream);
}

int8mp_status int8mp_scaled_mm_ws(const void* A, const float* sA, const void* B, const float* sB,
                                  int64_t M, int64_t N, int64_t K, int8mp_layout layout,
                                  int8mp_codes codes, void* out, int64_t ldo, void* workspace,
                                  size_t ws_bytes, void* stream) {
  int8mp_status st = check_mm(A, B, M, N, K, layout, codes, out, ldo);
  if (st != INT8MP_OK) return st;
  st = check_mm_workspace(workspace, ws_bytes);
  if (st != INT8MP_OK) return st;
  if (M > 0 && N > 0 && K > 0) {
    if (!sA || !sB) return INT8MP_ERR_INVALID_ARG;
    if (!aligned(sA, 4) || !aligned(sB, 4)) return INT8MP_ERR_ALIGNMENT;
  }
  return run_mm(A, sA, B, sB, M, N, K, layout, int8mp::GemmOut::kBf16Scaled, out, ldo,
                workspace, int8mp::GemmDebug{}, as_stream(stream), codes == INT8MP_CODES_S8);
}

int8mp_status int8mp_mm_s32(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                            int8mp_layout layout, int8mp_codes codes, int32_t* out, int64_t ldo,
                            void* stream) {
  return int8mp_mm_s32_ws(A, B, M, N, K, layout, codes, out, ldo, nullptr, 0, stream);
}

int8mp_status int8mp_mm_s32_ws(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                               int8mp_layout layout, int8mp_codes codes, int32_t* out, int64_t ldo,
                               void* workspace, size_t ws_bytes, void* stream) {
  int8mp_status st = check_mm(A, B, M, N, K, layout, codes, out, ldo);
  if (st != INT8MP_OK) return st;
  st = check_mm_workspace(workspace, ws_bytes);
  if (st != INT8MP_OK) return st;
  return run_mm(A, nullptr, B, nullptr, M, N, K, layout, int8mp::GemmOut::kS32, out, ldo,
                workspace, int8mp::GemmDebug{}, as_stream(stream), codes == INT8MP_CODES_S8);
}

int8mp_status int8mp_scaled_mm_f32(const void* A, const float* sA, const void* B, const float* sB,
                                   int64_t M, int64_t N, int64_t K, int8mp_layout layout,
                                   int8mp_codes codes, float* out, int64_t ldo, void* workspace,
                                   size_t ws_bytes, void* stream) {
  int8mp_status st = check_mm(A, B, M, N, K, layout, codes, out, ldo);
  if (st != INT8MP_OK) return st;
  st = check_mm_workspace(workspace, ws_bytes);
  if (st != INT8MP_OK) return st;
  if (M > 0 && N > 0 && K > 0) {
    if (!sA || !sB) return INT8MP_ERR_INVALID_ARG;
    if (!aligned(sA, 4) || !aligned(sB, 4)) return INT8MP_ERR_ALIGNMENT;
  }
  if (M == 0 || N == 0) return INT8MP_OK;
  if (K == 0) {  // an empty contraction: every product is 0 (the memset writes +0.0f)
    DeviceInfo dev;
    st = current_device(&dev, as_stream(stream));
    if (st != INT8MP_OK) return st;
    return from_cuda(cudaMemset2DAsync(out, static_cast<size_t>(ldo) * 4, 0,
                                       static_cast<size_t>(N) * 4, static_cast<size_t>(M),
                                       as_stream(stream)));
  }
  return run_mm(A, sA, B, sB, M, N, K, layout, int8mp::GemmOut::kF32Scaled, out, ldo, workspace,
                int8mp::GemmDebug{}, as_stream(stream), codes == INT8MP_CODES_S8);
}

int8mp_status int8mp_round_bf16(const float* x, void* y, int64_t n, void* stream) {
  if (n < 0) return INT8MP_ERR_INVALID_ARG;
  if (n == 0) return INT8MP_OK;
  if (!x || !y) return INT8MP_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return INT8MP_ERR_ALIGNMENT;
  DeviceInfo dev;
  int8mp_status st = current_device(&dev, as_stream(stream));
  if (st != INT8MP_OK) return st;
  return from_cuda(int8mp::launch_round_bf16(x, y, n, dev, as_stream(stream)));
}

size_t int8mp_linear_workspace_size(int64_t T, int64_t N, int64_t K, const int8mp_linear_cfg* cfg) {
  if (check_linear(T, N, K, cfg) != INT8MP_OK) return 0;
  const size_t f = fwd_bytes(T, N, K), b = bwd_bytes(T, N, K);
  return (f > b ? f : b) + int8mp::kSplitTailScratchBytes;
}

}  // extern "C"

namespace {

// Forward pass.  save_absmax (optional, fp32 [2K]): the column absmax of X
// (over T) and of W (over N), for a later backward pass over the same X, W;
// X's only when grad-weight runs in INT8, W's only when grad-input does (the
// other half stays 0).
int8mp_status linear_fwd_impl(const void* X, const void* W, void* Y, int64_t T, int64_t N,
                              int64_t K, const int8mp_linear_cfg* cfg, float* save_absmax,
                              void* workspace, size_t ws_bytes, void* stream) {
  int8mp_status st = check_linear(T, N, K, cfg);
  if (st != INT8MP_OK) return st;
  if (save_absmax && !aligned(save_absmax, 4)) return INT8MP_ERR_ALIGNMENT;
  if (T == 0 || N == 0) {
    if (save_absmax && K > 0)  // the absmax of an empty group is 0
      return from_cuda(cudaMemsetAsync(save_absmax, 0, static_cast<size_t>(2 * K) * 4,
                                       as_stream(stream)));
    return INT8MP_OK;
  }
  if (!Y || (K > 0 && (!X || !W || !workspace))) return INT8MP_ERR_INVALID_ARG;
  if (!aligned(Y, 16) || !aligned(X, 16) || !aligned(W, 16) || !aligned(workspace, 256))
    return INT8MP_ERR_ALIGNMENT;
  if (ws_bytes < fwd_bytes(T, N, K)) return INT8MP_ERR_WORKSPACE;
  DeviceInfo dev;
  st = current_device(&dev, as_stream(stream));
  if (st != INT8MP_OK) return st;
  cudaStream_t s = as_stream(stream);
  if (save_absmax && K > 0 && int8mp::launch_zero_words(save_absmax, 2 * K, dev, s) != cudaSuccess)
    return INT8MP_ERR_CUDA;
  float* x_absmax = save_absmax && K > 0 && cfg->int8_grad_w ? save_absmax : nullptr;
  float* w_absmax = save_absmax && K > 0 && cfg->int8_grad_in ? save_absmax + K : nullptr;
  if (!cfg->int8_fwd) {
    cudaError_t e = cudaSuccess;
    if (x_absmax) e = int8mp::launch_column_absmax(X, T, K, K, x_absmax, dev, s);
    if (e == cudaSuccess && w_absmax) e = int8mp::launch_column_absmax(W, N, K, K, w_absmax, dev, s);
    if (e != cudaSuccess) return INT8MP_ERR_CUDA;
    // BF16 pass: Y [T,N] = X W^T (A @ B.T), bf16 operands, fp32 accumulation
    return run_mm(X, nullptr, W, nullptr, T, N, K, INT8MP_AxBT, int8mp::GemmOut::kBf16Plain, Y, N,
                  gemm_scratch(workspace, ws_bytes, fwd_bytes(T, N, K)), int8mp::GemmDebug{}, s);
  }
  Carver c{static_cast<char*>(workspace)};
  const QOperand xq = carve_operand(c, T, K);
  const QOperand wq = carve_operand(c, N, K);
  if (K > 0) {
    // X and W by rows: one launch when both keep their column maxima or
    // neither does, else one each
    int8mp::RowsJob jobs[2];
    int n = 0;
    if (T > 0)
      jobs[n++] = int8mp::RowsJob{X, T, K, xq.q, xq.s, x_absmax, cfg->offset, INT8MP_STREAM_FWD_X};
    if (N > 0)
      jobs[n++] = int8mp::RowsJob{W, N, K, wq.q, wq.s, w_absmax, cfg->offset, INT8MP_STREAM_FWD_W};
    cudaError_t e = cudaSuccess;
    if (n == 2 && (x_absmax != nullptr) == (w_absmax != nullptr)) {
      e = int8mp::launch_quantize_rows_jobs(jobs, 2, K, cfg->mode, cfg->seed, INT8MP_CODES_F16,
                                            dev, s);
    } else {
      for (int i = 0; i < n && e == cudaSuccess; ++i)
        e = int8mp::launch_quantize_rows_jobs(jobs + i, 1, K, cfg->mode, cfg->seed,
                                              INT8MP_CODES_F16, dev, s);
    }
    if (e != cudaSuccess) return INT8MP_ERR_CUDA;
  }
  return run_mm(xq.q, xq.s, wq.q, wq.s, T, N, K, INT8MP_AxBT, int8mp::GemmOut::kBf16Scaled, Y, N,
                gemm_scratch(workspace, ws_bytes, fwd_bytes(T, N, K)), int8mp::GemmDebug{}, s);
}

// Backward pass.  saved_absmax (optional, fp32 [2K]): what the forward pass
// saved for these X and W; otherwise their column absmax is computed here.
int8mp_status linear_bwd_impl(const void* dY, const void* X, const void* W, void* dX, void* dW,
                              int64_t T, int64_t N, int64_t K, const int8mp_linear_cfg* cfg,
                              const float* saved_absmax, void* workspace, size_t ws_bytes,
                              void* stream) {
  int8mp_status st = check_linear(T, N, K, cfg);
  if (st != INT8MP_OK) return st;
  const bool want_dx = dX != nullptr && T > 0 && K > 0;
  const bool want_dw = dW != nullptr && N > 0 && K > 0;
  if (!want_dx && !want_dw) return INT8MP_OK;
  if (!dY || !W || !X || !workspace) return INT8MP_ERR_INVALID_ARG;
  if (!aligned(dY, 16) || !aligned(X, 16) || !aligned(W, 16) || !aligned(workspace, 256) ||
      (dX && !aligned(dX, 16)) || (dW && !aligned(dW, 16)) ||
      (saved_absmax && !aligned(saved_absmax, 4)))
    return INT8MP_ERR_ALIGNMENT;
  if (ws_bytes < bwd_bytes(T, N, K)) return INT8MP_ERR_WORKSPACE;
  DeviceInfo dev;
  st = current_device(&dev, as_stream(stream));
  if (st != INT8MP_OK) return st;
  cudaStream_t s = as_stream(stream);
  Carver c{static_cast<char*>(workspace)};
  const BwdOperands o = carve_bwd(c, T, N, K);
  void* scratch = gemm_scratch(workspace, ws_bytes, bwd_bytes(T, N, K));
  const bool int8_dx = want_dx && cfg->int8_grad_in && N > 0;
  const bool int8_dw = want_dw && cfg->int8_grad_w && T > 0;
  // column absmax: dY's (grad weight) comes with its row pass when grad
  // input runs in INT8; X's and W's are the forward's, or computed here
  float* dy_absmax = o.absmax;
  const float* x_absmax = saved_absmax ? saved_absmax : o.absmax + N;
  const float* w_absmax = saved_absmax ? saved_absmax + K : o.absmax + N + K;
  if ((int8_dx || int8_dw) && int8mp::launch_zero_words(o.absmax, N + 2 * K, dev, s) != cudaSuccess)
    return INT8MP_ERR_CUDA;
  if (!saved_absmax) {
    cudaError_t e = cudaSuccess;
    if (int8_dx) e = int8mp::launch_column_absmax(W, N, K, K, o.absmax + N + K, dev, s);
    if (e == cudaSuccess && int8_dw) e = int8mp::launch_column_absmax(X, T, K, K, o.absmax + N, dev, s);
    if (e != cudaSuccess) return INT8MP_ERR_CUDA;
  }
  if (int8_dw && !int8_dx &&
      int8mp::launch_column_absmax(dY, T, N, N, dy_absmax, dev, s) != cudaSuccess)
    return INT8MP_ERR_CUDA;

  if (want_dx && !cfg->int8_grad_in) {
    // BF16 pass: dX [T,K] = dY W (A @ B, W read N-major)
    st = run_mm(dY, nullptr, W, nullptr, T, K, N, INT8MP_AxB, int8mp::GemmOut::kBf16Plain, dX, K,
                scratch, int8mp::GemmDebug{}, s);
    if (st != INT8MP_OK) return st;
  } else if (want_dx) {
    // grad input: contraction over N; dY by rows, W by columns; dY W is A @ B
    if (N > 0) {
      cudaError_t e = int8mp::launch_quantize_rows(dY, T, N, N, cfg->mode,
                                                   sr_of(cfg, INT8MP_STREAM_GI_DY), o.dy_rows.q,
                                                   INT8MP_CODES_F16, o.dy_rows.s,
                                                   int8_dw ? dy_absmax : nullptr, dev, s);
      if (e == cudaSuccess)
        e = int8mp::launch_quantize_cols_from_absmax(W, N, K, K, w_absmax, cfg->mode,
                                                     sr_of(cfg, INT8MP_STREAM_GI_W), o.w_cols.q,
                                                     INT8MP_CODES_F16, o.w_cols.s, dev, s);
      if (e != cudaSuccess) return INT8MP_ERR_CUDA;
    }
    st = run_mm(o.dy_rows.q, o.dy_rows.s, o.w_cols.q, o.w_cols.s, T, K, N, INT8MP_AxB,
                int8mp::GemmOut::kBf16Scaled, dX, K, scratch, int8mp::GemmDebug{}, s);
    if (st != INT8MP_OK) return st;
  }
  if (want_dw && !cfg->int8_grad_w) {
    // BF16 pass: dW [N,K] = dY^T X (A.T @ B, both read T-major)
    st = run_mm(dY, nullptr, X, nullptr, N, K, T, INT8MP_ATxB, int8mp::GemmOut::kBf16Plain, dW, K,
                scratch, int8mp::GemmDebug{}, s);
  } else if (want_dw) {
    // grad weight: contraction over T; dY and X by columns; dY^T X is A.T @ B
    if (T > 0) {
      cudaError_t e = int8mp::launch_quantize_cols_from_absmax(
          dY, T, N, N, dy_absmax, cfg->mode, sr_of(cfg, INT8MP_STREAM_GW_DY), o.dy_cols.q,
          INT8MP_CODES_F16, o.dy_cols.s, dev, s);
      if (e == cudaSuccess)
        e = int8mp::launch_quantize_cols_from_absmax(X, T, K, K, x_absmax, cfg->mode,
                                                     sr_of(cfg, INT8MP_STREAM_GW_X), o.x_cols.q,
                                                     INT8MP_CODES_F16, o.x_cols.s, dev, s);
      if (e != cudaSuccess) return INT8MP_ERR_CUDA;
    }
    st = run_mm(o.dy_cols.q, o.dy_cols.s, o.x_cols.q, o.x_cols.s, N, K, T, INT8MP_ATxB,
                int8mp::GemmOut::kBf16Scaled, dW, K, scratch, int8mp::GemmDebug{}, s);
  }
  return st;
}

}  // namespace

extern "C" {

int8mp_status int8mp_linear_fwd(const void* X, const void* W, void* Y, int64_t T, int64_t N,
                                int64_t K, const int8mp_linear_cfg* cfg, void* workspace,
                                size_t ws_bytes, void* stream) {
  return linear_fwd_impl(X, W, Y, T, N, K, cfg, nullptr, workspace, ws_bytes, stream);
}

int8mp_status int8mp_linear_fwd_save(const void* X, const void* W, void* Y, int64_t T, int64_t N,
                                     int64_t K, const int8mp_linear_cfg* cfg, float* absmax,
                                     void* workspace, size_t ws_bytes, void* stream) {
  if (!absmax) return INT8MP_ERR_INVALID_ARG;
  return linear_fwd_impl(X, W, Y, T, N, K, cfg, absmax, workspace, ws_bytes, stream);
}

int8mp_status int8mp_linear_bwd(const void* dY, const void* X, const void* W, void* dX,
                                void* dW, int64_t T, int64_t N, int64_t K,
                                const int8mp_linear_cfg* cfg, void* workspace, size_t ws_bytes,
                                void* stream) {
  return linear_bwd_impl(dY, X, W, dX, dW, T, N, K, cfg, nullptr, workspace, ws_bytes, stream);
}

int8mp_status int8mp_linear_bwd_saved(const void* dY, const void* X, const void* W, void* dX,
                                      void* dW, int64_t T, int64_t N, int64_t K,
                                      const int8mp_linear_cfg* cfg, const float* absmax,
                                      void* workspace, size_t ws_bytes, void* stream) {
  if (!absmax) return INT8MP_ERR_INVALID_ARG;
  return linear_bwd_impl(dY, X, W, dX, dW, T, N, K, cfg, absmax, workspace, ws_bytes, stream);
}

int8mp_status int8mp_poll_device_status(void* stream) {
  DeviceInfo dev;
  int8mp_status st = current_device(&dev);
  if (st != INT8MP_OK) return st;
  cudaStream_t s = as_stream(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return INT8MP_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, dev.status_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return INT8MP_ERR_CUDA;
  if (word != 0) {
    if (cudaMemset(dev.status_word, 0, sizeof word) != cudaSuccess) return INT8MP_ERR_CUDA;
    return (word & 1u) ? INT8MP_ERR_TIMEOUT : INT8MP_ERR_BOUNDS;
  }
  return INT8MP_OK;
}

const char* int8mp_status_string(int8mp_status status) {
  switch (status) {
    case INT8MP_OK: return "ok";
    case INT8MP_ERR_INVALID_ARG: return "invalid argument";
    case INT8MP_ERR_ALIGNMENT: return "alignment or size-multiple requirement violated";
    case INT8MP_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103";
    case INT8MP_ERR_CUDA: return "CUDA runtime or launch error";
    case INT8MP_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case INT8MP_ERR_WORKSPACE: return "workspace too small";
    case INT8MP_ERR_BOUNDS: return "a bounds check of a checked build failed";
  }
  return "unknown status";
}

int int8mp_version(void) { return 100; }

int8mp_status int8mp_debug_mm_s32_drop_first_load(const void* A, const void* B, int64_t M,
                                                  int64_t N, int64_t K, int32_t* out,
                                                  int64_t ldo, int wait_limit_ms, void* stream) {
  int8mp_status st = check_mm(A, B, M, N, K, INT8MP_AxBT, INT8MP_CODES_F16, out, ldo);
  if (st != INT8MP_OK) return st;
  if (M == 0 || N == 0 || K == 0 || wait_limit_ms < 1 || wait_limit_ms > 5000)
    return INT8MP_ERR_INVALID_ARG;
  int8mp::GemmDebug dbg;
  dbg.drop_first_load = 1;
  dbg.wait_limit_ns = static_cast<uint64_t>(wait_limit_ms) * 1000000ull;
  return run_mm(A, nullptr, B, nullptr, M, N, K, INT8MP_AxBT, int8mp::GemmOut::kS32, out, ldo,
                nullptr, dbg, as_stream(stream));
}

int8mp_status int8mp_debug_scaled_mm_quant_b(const void* A, const float* sA, const void* B,
                                             const float* sB, int64_t M, int64_t N, int64_t K,
                                             void* out, int64_t ldo, void* stream) {
  int8mp_status st = check_mm(A, B, M, N, K, INT8MP_AxBT, INT8MP_CODES_F16, out, ldo);
  if (st != INT8MP_OK) return st;
  if (M == 0 || N == 0 || K == 0) return INT8MP_ERR_INVALID_ARG;
  if (!sA || !sB) return INT8MP_ERR_INVALID_ARG;
  if (!aligned(sA, 4) || !aligned(sB, 4)) return INT8MP_ERR_ALIGNMENT;
  int8mp::GemmDebug dbg;
  dbg.quant_b = 1;
  return run_mm(A, sA, B, sB, M, N, K, INT8MP_AxBT, int8mp::GemmOut::kBf16Scaled, out, ldo,
                nullptr, dbg, as_stream(stream));
}

}  // extern "C"
