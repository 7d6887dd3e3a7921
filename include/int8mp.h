/*
 * int8mp.h -- C ABI of the GB300 (sm_103a) INT8 mixed-precision linear-layer
 * library (libint8mp.so).
 *
 * The method ("Quantized model training" README, section "INT8 mixed
 * precision training"; "Integrate INT8 mixed-precision from torchao 0.7",
 * discussion): every matmul of a linear layer -- forward, backward grad-input,
 * backward grad-weight -- dynamically quantizes both bf16 operands row-wise
 * along its contraction axis to INT8 codes with one fp32 scale per row,
 * multiplies the codes with int32 accumulation, and scales the product back to
 * bf16.  Weights and activations stay bf16 outside the matmul.
 *
 * Arithmetic (identical on every entry point):
 *   scale s   = fp32(max |x| over the group) / 127       (IEEE division)
 *   code q    = clamp(round(x / s), -127, 127)           (IEEE division)
 *               round = nearest-even (INT8MP_RNE) or stochastic (INT8MP_SR);
 *               an all-zero group has s = 0 and all codes 0
 *   acc[i,j]  = sum_k qA[i,k] * qB[j,k]                   (exact int32)
 *   out[i,j]  = bf16_RNE((fp32_RN(acc) * sA[i]) * sB[j])
 * Stochastic rounding: v = x/s, f = floor(v), q = f + (u < v - f) with
 *   u = (w >> 8) * 2^-24 and w word (n & 3) of Philox4x32-10 (Salmon et al.,
 *   SC'11) at counter (lo32(n>>2), hi32(n>>2), stream_id, 0) and key
 *   (lo32(seed), hi32(seed)), n = offset + (r * cols + c) for source element
 *   (r, c).  Results therefore do not depend on the kernels' tiling.
 *
 * Hardware note: sm_103a has no INT8 tcgen05 MMA, and its legacy INT8 tensor
 * path is an order of magnitude slower than its f16 path.  The library keeps
 * the INT8 codes and the exact int32 accumulator of the method, but performs
 * the contraction on the f16 tensor cores: codes in [-127, 127] are exact
 * fp16 values, every product is exact, and fp32 partial sums are exact while
 * below 2^24, so the reduction runs in chunks of at most 1024 and each
 * chunk's sum is added into an int32 total.
 *
 * Conventions for every entry point:
 *   - All pointers are device pointers unless stated; the caller owns every
 *     buffer.  Nothing here allocates device memory.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is
 *     enqueued asynchronously on it; no entry point synchronizes the host.
 *   - bf16 tensors are raw 16-bit bf16 arrays, row-major.
 *   - Host-detected errors return before anything is launched.  Errors of
 *     the launch itself return INT8MP_ERR_CUDA.  A device-side wait that ran
 *     out (every wait in the GEMM is bounded) is recorded in a device status
 *     word, read back by int8mp_poll_device_status().
 *   - Only sm_103 devices are accepted (INT8MP_ERR_UNSUPPORTED_DEVICE).
 *   - Entry points may be called from several host threads on different
 *     streams.
 */
#ifndef INT8MP_H
#define INT8MP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  INT8MP_OK = 0,
  INT8MP_ERR_INVALID_ARG = 1,        /* null pointer, bad enum, bad size     */
  INT8MP_ERR_ALIGNMENT = 2,          /* pointer / leading-dim / size rule    */
  INT8MP_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not sm_103         */
  INT8MP_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed    */
  INT8MP_ERR_TIMEOUT = 5,            /* a bounded device-side wait ran out   */
  INT8MP_ERR_WORKSPACE = 6,          /* workspace too small                  */
  INT8MP_ERR_BOUNDS = 7              /* a checked build caught an index out  */
                                     /* of its buffer (see below)            */
} int8mp_status;

typedef enum { INT8MP_RNE = 0, INT8MP_SR = 1 } int8mp_round;

/* Operand layouts, named as in the README's matmul benchmark tables. */
typedef enum {
  INT8MP_AxBT = 0, /* A [M,K] row-major, B [N,K] row-major  (A @ B.T) */
  INT8MP_AxB = 1,  /* A [M,K] row-major, B [K,N] row-major  (A @ B)   */
  INT8MP_ATxB = 2  /* A [K,M] row-major, B [K,N] row-major  (A.T @ B) */
} int8mp_layout;

/* Storage of INT8 codes.  INT8MP_CODES_S8: one int8_t per code.
 * INT8MP_CODES_F16: one IEEE binary16 per code holding the same integer
 * exactly (a zero code may be stored as -0); this is the container the
 * tensor-core GEMM reads directly. */
typedef enum { INT8MP_CODES_S8 = 0, INT8MP_CODES_F16 = 1 } int8mp_codes;

/* Stochastic-rounding stream ids used by the linear entry points, one per
 * quantization of a training step, so that the same tensor quantized in two
 * passes is rounded independently. */
enum {
  INT8MP_STREAM_FWD_X = 0, INT8MP_STREAM_FWD_W = 1,
  INT8MP_STREAM_GI_DY = 2, INT8MP_STREAM_GI_W = 3,
  INT8MP_STREAM_GW_DY = 4, INT8MP_STREAM_GW_X = 5
};

/* Groups and code layout of int8mp_quantize_rowwise (its `axis`). */
enum {
  INT8MP_GROUP_ROWS = 0,   /* one group per row; codes [rows, cols]               */
  INT8MP_GROUP_COLS_T = 1, /* one group per column; codes transposed [cols, rows] */
  INT8MP_GROUP_COLS = 2    /* one group per column; codes [rows, cols]            */
};

/* Largest contraction length: 127 * 127 * K must stay below 2^31. */
#define INT8MP_MAX_K 133143

/*
 * int8mp_quantize_rowwise -- dynamic symmetric row-wise quantization
 * ("Quantized model training" README, "INT8 mixed precision training":
 * dynamic row-wise quantization; "Add QAT support for distributed
 * finetuning", summary: x_q = clamp(x / scale + zp), here zp = 0).
 *
 *   x       bf16 [rows, cols], row stride `ld` elements (ld >= cols).
 *   axis    INT8MP_GROUP_ROWS (0): one group per row (along cols).  Codes
 *              q [rows, cols] (row stride cols), scale [rows].
 *           INT8MP_GROUP_COLS_T (1): one group per column (along rows).
 *              Codes written transposed, q [cols, rows] (row stride rows),
 *              scale [cols]: the contraction axis innermost (K-major).
 *           INT8MP_GROUP_COLS (2): one group per column (along rows).  Codes
 *              in the input's layout, q [rows, cols] (row stride cols), scale
 *              [cols]: the operand enters int8mp_scaled_mm as the [K, M] or
 *              [K, N] operand of the A @ B and A.T @ B layouts.
 *           The codes of 1 and 2 are the same numbers (the stochastic
 *           counter follows the source element), only their layout differs.
 *   mode    INT8MP_RNE or INT8MP_SR; seed, offset, stream_id are used by SR
 *           only (see the header comment for the counter mapping).
 *   q       output codes, int8_t or binary16 per `codes`.
 *   scale   output fp32 scales.
 * Requirements: rows, cols >= 0 (either may be 0: nothing is launched);
 * cols % 8 == 0, ld % 8 == 0 and x 16-byte aligned (128-bit loads); for
 * axis 1 also rows % 8 == 0 (128-bit stores of the transposed codes); q 16-byte
 * aligned; scale 4-byte aligned.  Violations return INT8MP_ERR_ALIGNMENT.  A
 * column-grouped call writes `scale` twice (absmax first, then the scale):
 * nothing else may read it until the call's work on `stream` is done.
 */
int8mp_status int8mp_quantize_rowwise(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                      int axis, int8mp_round mode, uint64_t seed,
                                      uint64_t offset, uint32_t stream_id, void* q,
                                      int8mp_codes codes, float* scale, void* stream);

/*
 * int8mp_quantize_rows_colmax -- row groups exactly as int8mp_quantize_rowwise
 * with INT8MP_GROUP_ROWS, and in the same pass over x the absmax of every
 * column merged into colmax:
 *   colmax[c] = max(colmax[c], max_r |x[r, c]|)      (fp32 [cols])
 * The caller initializes colmax with non-negative values (zeros for one
 * matrix; calls over row blocks of one matrix can accumulate into the same
 * array).  This is the
 * pass that feeds int8mp_quantize_cols_absmax when the same matrix is
 * quantized along both axes (the output gradient of a linear layer, whose
 * rows feed grad-input and whose columns feed grad-weight), so that the
 * column groups need no absmax pass of their own.
 * Requirements: those of INT8MP_GROUP_ROWS; colmax non-NULL, 4-byte aligned
 * (INT8MP_ERR_INVALID_ARG / INT8MP_ERR_ALIGNMENT).  While the call runs on
 * `stream`, colmax is updated by atomic max.
 */
int8mp_status int8mp_quantize_rows_colmax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                          int8mp_round mode, uint64_t seed, uint64_t offset,
                                          uint32_t stream_id, void* q, int8mp_codes codes,
                                          float* scale, float* colmax, void* stream);

/*
 * int8mp_quantize_rows_batch -- row groups (INT8MP_GROUP_ROWS) of up to two
 * matrices with the same row length in one launch, e.g. the activations and
 * the weight of a linear layer's forward pass.  The codes, scales and column
 * maxima are those of one int8mp_quantize_rows_colmax call per job (colmax
 * given) or one int8mp_quantize_rowwise call with INT8MP_GROUP_ROWS per job
 * (colmax NULL), with the mode, seed and codes given here and each job's own
 * offset and stream_id.
 *   jobs    njobs job descriptions (host memory, read during the call):
 *             x       bf16 [rows, cols], row stride ld elements
 *             rows, ld
 *             offset, stream_id   the job's place in the stochastic-rounding
 *                                 stream (as for int8mp_quantize_rowwise)
 *             q       codes [rows, cols] (container per `codes`)
 *             scale   fp32 [rows]
 *             colmax  fp32 [cols] column absmax, merged by atomic max, or
 *                     NULL -- the same for every job
 *   njobs   1 .. INT8MP_MAX_ROWS_JOBS.
 *   cols    the row length of every job.
 *   mode, seed, codes, stream   as for int8mp_quantize_rowwise, shared by
 *           all jobs; the caller owns every buffer and initializes colmax
 *           as for int8mp_quantize_rows_colmax.
 * Requirements: every job those of int8mp_quantize_rowwise with
 * INT8MP_GROUP_ROWS, and of int8mp_quantize_rows_colmax when colmax is
 * given; a job with rows == 0 is skipped.  jobs NULL, njobs out of range, or
 * colmax given for some jobs only: INT8MP_ERR_INVALID_ARG.
 */
#define INT8MP_MAX_ROWS_JOBS 2
typedef struct {
  const void* x;
  int64_t rows;
  int64_t ld;
  uint64_t offset;
  uint32_t stream_id;
  void* q;
  float* scale;
  float* colmax;
} int8mp_rows_job;
int8mp_status int8mp_quantize_rows_batch(const int8mp_rows_job* jobs, int njobs, int64_t cols,
                                         int8mp_round mode, uint64_t seed, int8mp_codes codes,
                                         void* stream);

/*
 * int8mp_quantize_cols_batch -- column groups with the codes in the input's
 * layout (INT8MP_GROUP_COLS) of up to two matrices with the same number of
 * columns, e.g. both K-first operands of A.T @ B.  The codes and scales are
 * those of one int8mp_quantize_rowwise call with INT8MP_GROUP_COLS per job,
 * with the mode, seed and codes given here and each job's own offset and
 * stream_id.  When every job has at most 2048 rows the jobs share one
 * launch; otherwise each job takes the passes of that call.
 *   jobs    as for int8mp_quantize_rows_batch, with scale fp32 [cols] and
 *           colmax NULL (INT8MP_ERR_INVALID_ARG otherwise).
 *   njobs   1 .. INT8MP_MAX_ROWS_JOBS.
 *   cols    the number of columns of every job.
 * Requirements: every job those of int8mp_quantize_rowwise with
 * INT8MP_GROUP_COLS; a job with rows == 0 is skipped.
 */
int8mp_status int8mp_quantize_cols_batch(const int8mp_rows_job* jobs, int njobs, int64_t cols,
                                         int8mp_round mode, uint64_t seed, int8mp_codes codes,
                                         void* stream);

/*
 * int8mp_quantize_cols_absmax -- column groups with the codes in the input's
 * layout (as INT8MP_GROUP_COLS), given each column's absmax (fp32 [cols],
 * e.g. from int8mp_quantize_rows_colmax over the same x): scale[c] =
 * colmax[c] / 127 and codes q [rows, cols].  When colmax holds the true
 * column absmax the results are those of int8mp_quantize_rowwise with
 * INT8MP_GROUP_COLS, bit for bit; otherwise codes are still clamped to
 * [-127, 127].  Requirements: those of INT8MP_GROUP_COLS; colmax non-NULL,
 * 4-byte aligned.
 */
int8mp_status int8mp_quantize_cols_absmax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                          const float* colmax, int8mp_round mode, uint64_t seed,
                                          uint64_t offset, uint32_t stream_id, void* q,
                                          int8mp_codes codes, float* scale, void* stream);

/*
 * int8mp_scaled_mm -- scaled INT8 matmul ("Quantized model training" README,
 * matmul benchmark tables A @ B.T, A @ B, A.T @ B; "Integrate INT8
 * mixed-precision from torchao 0.7": the INT8 product is scaled back to BF16).
 *
 *   out[i,j] = bf16_RNE((fp32_RN(sum_k a(i,k) b(j,k)) * sA[i]) * sB[j])
 *
 *   A, B    INT8 codes in the container `codes`, stored per `layout`
 *           (dense: row stride = row length): AxBT A [M,K], B [N,K]; AxB
 *           A [M,K], B [K,N]; ATxB A [K,M], B [K,N].  Operands quantized
 *           along K come from int8mp_quantize_rowwise: a [.., K] operand with
 *           INT8MP_GROUP_ROWS, a [K, ..] operand with INT8MP_GROUP_COLS (or
 *           with INT8MP_GROUP_COLS_T and the AxBT layout).
 *   sA      fp32 [M], sB fp32 [N].
 *   out     bf16 [M, N], row stride ldo elements (ldo >= N).
 * Requirements: M, N >= 0; 16 <= K <= INT8MP_MAX_K; K % 16 == 0 (when M or N
 * is 0 nothing is launched); A, B 16-byte aligned; N % 8 == 0, ldo % 8 == 0
 * and out 16-byte aligned (128-bit stores); for ATxB also M % 8 == 0.  M and
 * N need not be tile multiples.
 * codes: INT8MP_CODES_F16 containers are loaded by TMA straight into the
 * tensor core's operand tiles (the fast path: the linear entry points use
 * it).  INT8MP_CODES_S8 (`const int8_t*` codes in [-127, 127]) are loaded as
 * int8 and widened to f16 in shared memory inside the CTA-pair kernel; the
 * results are the same bit for bit, at roughly half the f16 path's speed.
 * With int8 codes an operand stored [K, N] (AxB, ATxB) also needs
 * N % 16 == 0 and one stored [K, M] (ATxB) M % 16 == 0 (16-byte row strides);
 * otherwise INT8MP_ERR_ALIGNMENT.  A code of -128 is outside the contract.
 */
int8mp_status int8mp_scaled_mm(const void* A, const float* sA, const void* B, const float* sB,
                               int64_t M, int64_t N, int64_t K, int8mp_layout layout,
                               int8mp_codes codes, void* out, int64_t ldo, void* stream);

/*
 * int8mp_mm_s32 -- the exact integer product alone: acc[i,j] = sum_k
 * a(i,k) b(j,k) as int32, out int32 [M, N] with row stride ldo.  Same operand
 * rules as int8mp_scaled_mm.  Exposes the int32 accumulator so that it can be
 * compared bit for bit.
 */
int8mp_status int8mp_mm_s32(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                            int8mp_layout layout, int8mp_codes codes, int32_t* out,
                            int64_t ldo, void* stream);

/*
 * int8mp_scaled_mm_ws / int8mp_mm_s32_ws -- the same matmuls with a
 * caller-provided device workspace of at least int8mp_mm_workspace_size()
 * bytes (256-byte aligned; no initialization needed).  With it, when the
 * output tiles leave a partial last wave on the GPU's SM pairs, the GEMM
 * splits the contraction of those last tiles into equal parts computed by
 * the otherwise idle pairs; the parts are added as exact int32 totals, so
 * the results are those of the plain calls bit for bit.  workspace may be NULL (the plain
 * schedule); a non-NULL one smaller than int8mp_mm_workspace_size() returns
 * INT8MP_ERR_WORKSPACE, a misaligned one INT8MP_ERR_ALIGNMENT.  One workspace
 * must not be used by two calls that may run at the same time.
 */
size_t int8mp_mm_workspace_size(void);
int8mp_status int8mp_scaled_mm_ws(const void* A, const float* sA, const void* B, const float* sB,
                                  int64_t M, int64_t N, int64_t K, int8mp_layout layout,
                                  int8mp_codes codes, void* out, int64_t ldo, void* workspace,
                                  size_t ws_bytes, void* stream);
int8mp_status int8mp_mm_s32_ws(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                               int8mp_layout layout, int8mp_codes codes, int32_t* out, int64_t ldo,
                               void* workspace, size_t ws_bytes, void* stream);

/*
 * int8mp_scaled_mm_f32 -- the scaled matmul with an fp32 result that is not
 * rounded to bf16:
 *   out[i,j] = (fp32_RN(sum_k a(i,k) b(j,k)) * sA[i]) * sB[j]     (fp32)
 * i.e. int8mp_scaled_mm before its final rounding.  This is the partial
 * grad-weight of one token shard in data-parallel training: each rank
 * quantizes its own rows of dY and X by columns (its own column scales),
 * multiplies them here, the ranks sum their partials (e.g. an all-reduce),
 * and int8mp_round_bf16 rounds the sum once ("Integrate INT8 mixed-precision
 * from torchao 0.7", discussion: FSDP2 training on two A100s; torchao issue
 * 1887: gradients reduce-scattered across ranks).
 *   out     fp32 [M, N], row stride ldo elements.
 *   workspace, ws_bytes   as for int8mp_scaled_mm_ws (NULL allowed).
 * Requirements and codes: those of int8mp_scaled_mm_ws.
 */
int8mp_status int8mp_scaled_mm_f32(const void* A, const float* sA, const void* B, const float* sB,
                                   int64_t M, int64_t N, int64_t K, int8mp_layout layout,
                                   int8mp_codes codes, float* out, int64_t ldo, void* workspace,
                                   size_t ws_bytes, void* stream);

/*
 * int8mp_round_bf16 -- y[i] = bf16_RNE(x[i]) for n fp32 values (round to
 * nearest, ties to even; the last step of a grad-weight whose fp32 partials
 * were summed across ranks).  x fp32 [n], y bf16 [n], both 16-byte aligned
 * (INT8MP_ERR_ALIGNMENT); n >= 0.
 */
int8mp_status int8mp_round_bf16(const float* x, void* y, int64_t n, void* stream);

/*
 * Per-pass configuration of a linear layer (the pages' per-matmul INT8
 * switches and stochastic-rounding switch; "Quantized model training"
 * README, INT8 mixed precision training table).  int8_* = 1 runs that pass
 * in INT8 as described above; 0 runs it in BF16: the plain product of the
 * bf16 operands, accumulated in fp32 by the same tcgen05 kernels (bf16
 * operand format, one accumulator over the whole contraction; a split last
 * wave adds its fp32 parts in a fixed order) and rounded once to bf16
 * (nearest even).  The fp32 summation order is the tensor core's, so a BF16
 * pass matches the plain product within fp32 accumulation error, not bit for
 * bit.  Other values return INT8MP_ERR_INVALID_ARG.  mode, seed and offset
 * apply to the INT8 passes.
 */
typedef struct {
  int int8_fwd;
  int int8_grad_in;
  int int8_grad_w;
  int8mp_round mode;
  uint64_t seed;
  uint64_t offset;
} int8mp_linear_cfg;

/* Bytes of device workspace int8mp_linear_fwd / int8mp_linear_bwd use for
 * these sizes: the codes and scales of the quantized operands (256-byte
 * aligned sub-buffers, required) followed by the matmul's last-wave scratch
 * (int8mp_mm_workspace_size() bytes; optional: a workspace that ends before
 * it gives the same results without splitting the last wave).  Returns 0
 * for invalid sizes. */
size_t int8mp_linear_workspace_size(int64_t T, int64_t N, int64_t K,
                                    const int8mp_linear_cfg* cfg);

/*
 * int8mp_linear_fwd -- Y [T,N] = X [T,K] . W [N,K]^T: X and W quantized
 * along K (SR streams 0 and 1), scaled matmul, bf16 out.
 * Requirements: T >= 0, N >= 0, K >= 16; K % 16 == 0, N % 16 == 0,
 * T % 16 == 0; all pointers 16-byte aligned; workspace (256-byte aligned)
 * of int8mp_linear_workspace_size() bytes, of which all but the trailing
 * int8mp_mm_workspace_size() are required (INT8MP_ERR_WORKSPACE otherwise).
 */
int8mp_status int8mp_linear_fwd(const void* X, const void* W, void* Y, int64_t T, int64_t N,
                                int64_t K, const int8mp_linear_cfg* cfg, void* workspace,
                                size_t ws_bytes, void* stream);

/*
 * int8mp_linear_bwd -- grad-input dX [T,K] = dY [T,N] . W [N,K] (dY along N
 * by rows, W along N by columns; SR streams 2 and 3) and grad-weight
 * dW [N,K] = dY^T . X (dY and X along T by columns; SR streams 4 and 5).
 * dX or dW may be NULL to skip that pass.  Nothing from the forward pass is
 * reused: both operands are re-quantized from bf16.  Same requirements as
 * int8mp_linear_fwd.
 */
int8mp_status int8mp_linear_bwd(const void* dY, const void* X, const void* W, void* dX,
                                void* dW, int64_t T, int64_t N, int64_t K,
                                const int8mp_linear_cfg* cfg, void* workspace, size_t ws_bytes,
                                void* stream);

/*
 * int8mp_linear_fwd_save / int8mp_linear_bwd_saved -- the same passes, with
 * the same results bit for bit, sharing one thing across them: the forward
 * pass, which reads X and W row by row anyway, also records their column
 * absmax -- absmax[0..K) for X over its T rows, absmax[K..2K) for W over its
 * N rows (fp32, 2K values, caller-owned) -- and the backward pass uses them
 * for the column groups of grad-weight (X along T) and grad-input (W along
 * N) instead of reading X and W once more.  X's half is filled only when
 * cfg->int8_grad_w is 1 and W's only when cfg->int8_grad_in is 1 (the other
 * half is set to 0); the backward pass must get the same cfg, X and W as the
 * forward pass that filled `absmax`.  Requirements:
 * those of int8mp_linear_fwd / int8mp_linear_bwd; absmax non-NULL and
 * 4-byte aligned.  (The 2K floats are the only state kept between the passes;
 * the INT8 codes are still recomputed from bf16.)
 */
int8mp_status int8mp_linear_fwd_save(const void* X, const void* W, void* Y, int64_t T, int64_t N,
                                     int64_t K, const int8mp_linear_cfg* cfg, float* absmax,
                                     void* workspace, size_t ws_bytes, void* stream);
int8mp_status int8mp_linear_bwd_saved(const void* dY, const void* X, const void* W, void* dX,
                                      void* dW, int64_t T, int64_t N, int64_t K,
                                      const int8mp_linear_cfg* cfg, const float* absmax,
                                      void* workspace, size_t ws_bytes, void* stream);

/*
 * int8mp_linear_fwd_noalloc -- the same forward pass as int8mp_linear_fwd
 * (same arguments, requirements and results, bit for bit) for callers that
 * cannot allocate device memory: programs that hand out all device memory
 * through their own pool or have reserved it up front, and latency-critical
 * code that may not call cudaMalloc/cudaFree (which can synchronize the
 * device).  The pages have no counterpart; this is a property of the library.
 *
 * The workspace is a library-owned array of INT8MP_NOALLOC_SCRATCH_BYTES on
 * every device that loads the library, held until the process exits.  Sizes
 * needing more, i.e. round256(2*T*K) + round256(4*T) + round256(2*N*K) +
 * round256(4*N) bytes above the maximum, return INT8MP_ERR_WORKSPACE before
 * anything is launched.  Nothing is allocated by the call.
 *
 * cfg->int8_fwd may be 0 (the BF16 forward pass needs no workspace).
 * The first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress); make that first call before
 * any stream capture.  All calls on a device share the array and it keeps the
 * last call's contents (nothing in it needs to start at zero: every byte a
 * call reads it has written first).  Calls that overlap on the GPU -- on
 * different streams, or from several host threads -- race on the array and
 * must be serialized by the caller.
 */
#define INT8MP_NOALLOC_SCRATCH_BYTES (32u << 20)
int8mp_status int8mp_linear_fwd_noalloc(const void* X, const void* W, void* Y, int64_t T,
                                        int64_t N, int64_t K, const int8mp_linear_cfg* cfg,
                                        void* stream);

/* Synchronizes `stream`, then returns and clears the device status word of
 * the current device: INT8MP_ERR_TIMEOUT if a bounded device wait ran out
 * since the last poll, INT8MP_ERR_BOUNDS if a bounds check of a checked
 * build failed (a library compiled with -DINT8MP_CHECK checks every global
 * index its kernels compute against its buffer and skips the access instead
 * of making it; the ordinary build has no checks), INT8MP_ERR_CUDA if the
 * stream reports an error, INT8MP_OK otherwise. */
int8mp_status int8mp_poll_device_status(void* stream);

/* Static, NUL-terminated description of a status code. */
const char* int8mp_status_string(int8mp_status status);

/* Library version as 10000 * major + 100 * minor + patch. */
int int8mp_version(void);

#ifdef __cplusplus
}
#endif
#endif /* INT8MP_H */
