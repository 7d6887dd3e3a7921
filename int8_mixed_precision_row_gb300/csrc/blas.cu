// blas.cu -- BF16 passes of the linear layer ("BF16" entries of the INT8
// mixed precision training table, "Quantized model training" README): a
// plain bf16 matmul with fp32 accumulation and bf16 output, which is a
// library GEMM, run by cuBLASLt.  The INT8 passes never come here.
#include <cublasLt.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace int8mp {
namespace {

constexpr int kMaxDevices = 64;

struct LtHandle {
  std::once_flag once;
  cublasLtHandle_t h = nullptr;
  bool ok = false;
};
LtHandle g_lt[kMaxDevices];

cublasLtHandle_t lt_handle() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  LtHandle& e = g_lt[dev];
  std::call_once(e.once, [&e] { e.ok = cublasLtCreate(&e.h) == CUBLAS_STATUS_SUCCESS; });
  return e.ok ? e.h : nullptr;
}

}  // namespace

// Column-major C [m, n] = op(A) [m, k] * op(B) [k, n]; A stored [m, k]
// (or [k, m] when transa), B stored [k, n] (or [n, k] when transb); all bf16.
cudaError_t bf16_gemm_colmajor(const void* A, const void* B, void* C, int64_t m, int64_t n,
                               int64_t k, bool transa, bool transb, int64_t lda, int64_t ldb,
                               int64_t ldc, cudaStream_t stream) {
  cublasLtHandle_t h = lt_handle();
  if (!h) return cudaErrorNotSupported;
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cudaError_t err = cudaErrorUnknown;
  const cublasOperation_t ta = transa ? CUBLAS_OP_T : CUBLAS_OP_N;
  const cublasOperation_t tb = transb ? CUBLAS_OP_T : CUBLAS_OP_N;
  const float alpha = 1.0f, beta = 0.0f;
  if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS &&
      cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof ta) ==
          CUBLAS_STATUS_SUCCESS &&
      cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof tb) ==
          CUBLAS_STATUS_SUCCESS &&
      cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, transa ? k : m, transa ? m : k, lda) ==
          CUBLAS_STATUS_SUCCESS &&
      cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, transb ? n : k, transb ? k : n, ldb) ==
          CUBLAS_STATUS_SUCCESS &&
      cublasLtMatrixLayoutCreate(&lc, CUDA_R_16BF, m, n, ldc) == CUBLAS_STATUS_SUCCESS &&
      cublasLtMatmul(h, op, &alpha, A, la, B, lb, &beta, C, lc, C, lc, nullptr, nullptr, 0,
                     stream) == CUBLAS_STATUS_SUCCESS)
    err = cudaSuccess;
  if (lc) cublasLtMatrixLayoutDestroy(lc);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  return err;
}

}  // namespace int8mp
