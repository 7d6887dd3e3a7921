/*
 * oracle.h -- plain CPU oracle for INT8 mixed-precision linear layers.
 *
 * TEST INFRASTRUCTURE ONLY.  This code is the slow, obviously-correct
 * definition that the CUDA path is checked against.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never calls it and shares no code, header or table with it.
 *
 * What it computes (sources are the pages' titles and sections):
 *   - "Quantized model training" README, section "INT8 mixed precision
 *     training": INT8 means dynamic row-wise quantization followed by a scaled
 *     INT8 matmul; forward, backward grad-input and backward grad-weight are the
 *     three matmuls, each switchable, plus a stochastic-rounding switch.
 *   - "Integrate INT8 mixed-precision from torchao 0.7", discussion: weights and
 *     activations are quantized dynamically to INT8 with a scale, multiplied in
 *     INT8, and the result is scaled back to BF16; weights and activations stay
 *     BF16 everywhere else.
 *   - "Add QAT support for distributed finetuning", summary: the quantizer is
 *     x_q = clamp(x / scale + zp); here zp = 0 (symmetric, row-wise absmax).
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): scale = fp32(absmax)/127 by IEEE division; code = clamp(RNE(x/s))
 * with x/s an IEEE fp32 division; an all-zero group gets s = 0 and codes 0;
 * int32 accumulation; out = bf16_RNE((fp32(acc) * sA[i]) * sB[j]);
 * stochastic rounding draws u from Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11) with
 * key = (lo32(seed), hi32(seed)), n = offset + (r*cols + c),
 * counter = (lo32(n>>2), hi32(n>>2), stream_id, 0), word n & 3,
 * u = (word >> 8) * 2^-24, q = floor(v) + (u < v - floor(v)).
 *
 * bf16 values are passed as their raw 16-bit patterns (uint16_t).
 * All matrices are row-major and contiguous unless a leading dimension is
 * given.  Every function returns 0 on success and a negative value on an
 * invalid argument.
 */
#ifndef INT8MP_ORACLE_H
#define INT8MP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_RNE = 0, ORC_SR = 1 };
/* Operand layouts of the scaled matmul, named as in the README's matmul
 * benchmark tables: A @ B.T (A [M,K], B [N,K]), A @ B (A [M,K], B [K,N]),
 * A.T @ B (A [K,M], B [K,N]). */
enum { ORC_AxBT = 0, ORC_AxB = 1, ORC_ATxB = 2 };

/* stochastic-rounding stream ids of the six quantizations in one linear step */
enum {
  ORC_STREAM_FWD_X = 0, ORC_STREAM_FWD_W = 1,
  ORC_STREAM_GI_DY = 2, ORC_STREAM_GI_W = 3,
  ORC_STREAM_GW_DY = 4, ORC_STREAM_GW_X = 5
};

float orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16_rne(float f);

/* Philox4x32 with 10 rounds, as published (SC'11): out = philox(ctr, key). */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Dynamic symmetric quantization of a bf16 matrix x [rows, cols] (row stride
 * ld elements).  axis 0: one group per row, q is [rows, cols], scale [rows].
 * axis 1: one group per column, q is written transposed [cols, rows],
 * scale [cols]. */
int orc_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int axis,
                 int mode, uint64_t seed, uint64_t offset, uint32_t stream_id,
                 int8_t* q, float* scale);

/* acc[i,j] = sum_k a(i,k) * b(j,k) in int32, operands stored per layout. */
int orc_mm_s32(const int8_t* A, const int8_t* B, int64_t M, int64_t N, int64_t K,
               int layout, int32_t* acc, int nthreads);

/* out[i,j] = bf16_RNE((float(acc[i,j]) * sA[i]) * sB[j]), out [M,N]. */
int orc_rescale_bf16(const int32_t* acc, const float* sA, const float* sB,
                     int64_t M, int64_t N, uint16_t* out);

/* int8 codes + scales -> bf16 [M,N]: orc_mm_s32 followed by orc_rescale_bf16. */
int orc_scaled_mm(const int8_t* A, const float* sA, const int8_t* B, const float* sB,
                  int64_t M, int64_t N, int64_t K, int layout, uint16_t* out, int nthreads);

/* Linear forward Y [T,N] = X [T,K] . W [N,K]^T with both operands quantized
 * along K (stream ids 0 and 1). */
int orc_linear_fwd(const uint16_t* X, const uint16_t* W, int64_t T, int64_t N, int64_t K,
                   int mode, uint64_t seed, uint64_t offset, uint16_t* Y, int nthreads);

/* Linear backward.  dX [T,K] = dY [T,N] . W [N,K] with dY quantized along N
 * (rows, stream 2) and W quantized along N (columns, stream 3).
 * dW [N,K] = dY^T . X with dY and X quantized along T (columns, streams 4
 * and 5).  dX or dW may be NULL to skip that pass. */
int orc_linear_bwd(const uint16_t* dY, const uint16_t* X, const uint16_t* W,
                   int64_t T, int64_t N, int64_t K, int mode, uint64_t seed,
                   uint64_t offset, uint16_t* dX, uint16_t* dW, int nthreads);

/* A BF16 pass (the "BF16" entries of the INT8 mixed precision training
 * table in the "Quantized model training" README): the plain product of the
 * bf16 operands, out[i,j] = bf16_RNE(fp32_RN(sum_k a(i,k) b(j,k))) with the
 * sum taken in fp64 (every product of two bf16 values is exact in fp64).
 * Operands stored per layout as in orc_mm_s32. */
int orc_matmul_bf16(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                    int layout, uint16_t* out, int nthreads);

/* Linear passes with per-pass switches: int8_* = 1 runs the pass as
 * orc_linear_fwd / orc_linear_bwd do, 0 runs it as a BF16 pass. */
int orc_linear_fwd_cfg(const uint16_t* X, const uint16_t* W, int64_t T, int64_t N, int64_t K,
                       int int8_fwd, int mode, uint64_t seed, uint64_t offset, uint16_t* Y,
                       int nthreads);
int orc_linear_bwd_cfg(const uint16_t* dY, const uint16_t* X, const uint16_t* W, int64_t T,
                       int64_t N, int64_t K, int int8_grad_in, int int8_grad_w, int mode,
                       uint64_t seed, uint64_t offset, uint16_t* dX, uint16_t* dW,
                       int nthreads);

/* Step 5 without the final bf16 rounding: out[i,j] = fp32 (fp32_RN(acc) *
 * sA[i]) * sB[j].  orc_scaled_mm_f32 = orc_mm_s32 + orc_rescale_f32. */
int orc_rescale_f32(const int32_t* acc, const float* sA, const float* sB, int64_t M, int64_t N,
                    float* out);
int orc_scaled_mm_f32(const int8_t* A, const float* sA, const int8_t* B, const float* sB,
                      int64_t M, int64_t N, int64_t K, int layout, float* out, int nthreads);

/* Grad-weight under token-sharded data parallelism (the reading of the
 * FSDP2 runs in "Integrate INT8 mixed-precision from torchao 0.7" and the
 * reduce-scatter of torchao issue 1887): shard r of nshards equal blocks of
 * consecutive token rows quantizes its dY and X rows by columns with its own
 * column scales (SR counters from offsets[r]), forms its fp32 partial
 * (orc_scaled_mm_f32), the partials are summed in fp32 in shard order and the
 * sum is rounded once: dW = bf16_RNE(P_0 + ... + P_{n-1}). */
int orc_grad_weight_sharded(const uint16_t* dY, const uint16_t* X, int64_t T, int64_t N, int64_t K,
                            int nshards, int mode, uint64_t seed, const uint64_t* offsets,
                            uint16_t* dW, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
