/*
 * oracle.c -- plain CPU oracle for INT8 mixed-precision linear layers.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): loaded by the tests, the smoke
 * check and the benchmark's CPU-baseline leg, never by the product path.
 *
 * Built with -O2 -ffp-contract=off and without fast-math so that every fp32
 * operation below is one IEEE-754 operation rounded to nearest even.  Loops
 * are written in the order the definition states; the only parallelism is a
 * split of independent output rows of the integer matmul over threads.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

float orc_bf16_to_f32(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16; /* bf16 is the top half of an fp32 */
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

uint16_t orc_f32_to_bf16_rne(float f) {
  uint32_t bits;
  memcpy(&bits, &f, sizeof bits);
  if ((bits & 0x7f800000u) == 0x7f800000u && (bits & 0x007fffffu) != 0u)
    return (uint16_t)((bits >> 16) | 0x0040u); /* NaN stays a (quiet) NaN */
  /* round half to even on the 16 dropped bits */
  uint32_t lsb = (bits >> 16) & 1u;
  bits += 0x7fffu + lsb;
  return (uint16_t)(bits >> 16);
}

/* ---------------------------------------------------------------- Philox */
/* Philox4x32-10 (Salmon et al., SC'11, section 5): two 32x32->64 multiplies
 * per round with the published multipliers, a Weyl sequence on the key. */

static const uint32_t PHILOX_M0 = 0xD2511F53u;
static const uint32_t PHILOX_M1 = 0xCD9E8D57u;
static const uint32_t PHILOX_W0 = 0x9E3779B9u; /* golden ratio */
static const uint32_t PHILOX_W1 = 0xBB67AE85u; /* sqrt(3) - 1 */

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* uniform in [0, 1) with 24 random bits for logical element index e */
static float sr_uniform(uint64_t seed, uint64_t offset, uint32_t stream_id, uint64_t e) {
  uint64_t n = offset + e;
  uint64_t block = n >> 2;
  uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), stream_id, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t r[4];
  orc_philox4x32_10(ctr, key, r);
  uint32_t w = r[n & 3u];
  return (float)(w >> 8) * 0x1p-24f;
}

/* ------------------------------------------------------------- quantize */

static int8_t clamp_code(float q) {
  if (q > 127.0f) return 127;
  if (q < -127.0f) return -127;
  return (int8_t)q;
}

/* one code from x and the group scale s (s > 0) */
static int8_t quantize_one(float x, float s, int mode, uint64_t seed, uint64_t offset,
                           uint32_t stream_id, uint64_t e) {
  float v = x / s; /* IEEE division, as the QAT summary writes x / scale */
  if (mode == ORC_RNE) {
    return clamp_code(nearbyintf(v)); /* default rounding mode: half to even */
  }
  float f = floorf(v);
  float fr = v - f;
  float u = sr_uniform(seed, offset, stream_id, e);
  float q = (u < fr) ? f + 1.0f : f;
  return clamp_code(q);
}

int orc_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int axis,
                 int mode, uint64_t seed, uint64_t offset, uint32_t stream_id,
                 int8_t* q, float* scale) {
  if (rows < 0 || cols < 0 || ld < cols || (axis != 0 && axis != 1)) return -1;
  if (mode != ORC_RNE && mode != ORC_SR) return -1;
  if (rows == 0 || cols == 0) return 0;
  if (!x || !q || !scale) return -1;

  int64_t groups = axis == 0 ? rows : cols;
  int64_t glen = axis == 0 ? cols : rows;
  for (int64_t g = 0; g < groups; ++g) {
    /* step 1: absmax of the group in fp32 (exact: max is order-free) */
    float amax = 0.0f;
    for (int64_t i = 0; i < glen; ++i) {
      int64_t r = axis == 0 ? g : i, c = axis == 0 ? i : g;
      float a = fabsf(orc_bf16_to_f32(x[r * ld + c]));
      if (a > amax) amax = a;
    }
    /* step 2: scale = absmax / 127 */
    float s = amax / 127.0f;
    scale[g] = s;
    /* step 3: codes; an all-zero group has s = 0 and all codes 0 */
    for (int64_t i = 0; i < glen; ++i) {
      int64_t r = axis == 0 ? g : i, c = axis == 0 ? i : g;
      int8_t code = 0;
      if (s != 0.0f) {
        float xv = orc_bf16_to_f32(x[r * ld + c]);
        code = quantize_one(xv, s, mode, seed, offset, stream_id, (uint64_t)(r * cols + c));
      }
      q[g * glen + i] = code; /* axis 1 writes [cols, rows] */
    }
  }
  return 0;
}

/* ------------------------------------------------------- integer matmul */

typedef struct {
  const int8_t* A;
  const int8_t* B;
  int64_t M, N, K;
  int layout;
  int32_t* acc;
  int64_t i0, i1;
} mm_job;

static inline int32_t a_at(const mm_job* j, int64_t i, int64_t k) {
  return j->layout == ORC_ATxB ? j->A[k * j->M + i] : j->A[i * j->K + k];
}
static inline int32_t b_at(const mm_job* j, int64_t jn, int64_t k) {
  return j->layout == ORC_AxBT ? j->B[jn * j->K + k] : j->B[k * j->N + jn];
}

static void* mm_rows(void* arg) {
  mm_job* j = (mm_job*)arg;
  for (int64_t i = j->i0; i < j->i1; ++i) {
    for (int64_t n = 0; n < j->N; ++n) {
      int32_t s = 0;
      for (int64_t k = 0; k < j->K; ++k) s += a_at(j, i, k) * b_at(j, n, k);
      j->acc[i * j->N + n] = s;
    }
  }
  return NULL;
}

int orc_mm_s32(const int8_t* A, const int8_t* B, int64_t M, int64_t N, int64_t K,
               int layout, int32_t* acc, int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (layout != ORC_AxBT && layout != ORC_AxB && layout != ORC_ATxB) return -1;
  /* |acc| <= 127 * 127 * K must stay below 2^31 */
  if (K > 133143) return -1;
  if (M == 0 || N == 0) return 0;
  if (!A || !B || !acc) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > M) nthreads = (int)M;
  if (nthreads > 256) nthreads = 256;
  mm_job jobs[256];
  pthread_t tids[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (mm_job){A, B, M, N, K, layout, acc, M * t / nthreads, M * (t + 1) / nthreads};
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, mm_rows, &jobs[t]) != 0) break;
    started = t;
  }
  mm_rows(&jobs[0]);
  for (int t = started + 1; t < nthreads; ++t) mm_rows(&jobs[t]); /* not started */
  for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
  return 0;
}

/* --------------------------------------------------------------- rescale */

int orc_rescale_bf16(const int32_t* acc, const float* sA, const float* sB,
                     int64_t M, int64_t N, uint16_t* out) {
  if (M < 0 || N < 0) return -1;
  if (M == 0 || N == 0) return 0;
  if (!acc || !sA || !sB || !out) return -1;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      float f = (float)acc[i * N + j]; /* int32 -> fp32, round to nearest */
      float t = f * sA[i];
      float o = t * sB[j];
      out[i * N + j] = orc_f32_to_bf16_rne(o);
    }
  }
  return 0;
}

int orc_scaled_mm(const int8_t* A, const float* sA, const int8_t* B, const float* sB,
                  int64_t M, int64_t N, int64_t K, int layout, uint16_t* out, int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (M == 0 || N == 0) return 0;
  int32_t* acc = (int32_t*)malloc((size_t)(M * N) * sizeof(int32_t));
  if (!acc) return -2;
  int rc = orc_mm_s32(A, B, M, N, K, layout, acc, nthreads);
  if (rc == 0) rc = orc_rescale_bf16(acc, sA, sB, M, N, out);
  free(acc);
  return rc;
}

/* Step 5 without its final rounding: the fp32 value (acc * sA) * sB that a
 * token shard contributes to a data-parallel grad-weight before the shards'
 * values are summed. */
int orc_rescale_f32(const int32_t* acc, const float* sA, const float* sB, int64_t M, int64_t N,
                    float* out) {
  if (M < 0 || N < 0) return -1;
  if (M == 0 || N == 0) return 0;
  if (!acc || !sA || !sB || !out) return -1;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      float f = (float)acc[i * N + j]; /* int32 -> fp32, round to nearest */
      float t = f * sA[i];
      out[i * N + j] = t * sB[j];
    }
  }
  return 0;
}

int orc_scaled_mm_f32(const int8_t* A, const float* sA, const int8_t* B, const float* sB,
                      int64_t M, int64_t N, int64_t K, int layout, float* out, int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (M == 0 || N == 0) return 0;
  int32_t* acc = (int32_t*)malloc((size_t)(M * N) * sizeof(int32_t));
  if (!acc) return -2;
  int rc = orc_mm_s32(A, B, M, N, K, layout, acc, nthreads);
  if (rc == 0) rc = orc_rescale_f32(acc, sA, sB, M, N, out);
  free(acc);
  return rc;
}

/* ---------------------------------------------------------------- linear */

/* quantize X [R,C] along axis, multiply as A @ B.T with the codes, rescale */
static int quantized_product(const uint16_t* A, int64_t ar, int64_t ac, int a_axis, uint32_t a_stream,
                             const uint16_t* B, int64_t br, int64_t bc, int b_axis, uint32_t b_stream,
                             int64_t M, int64_t N, int64_t K, int mode, uint64_t seed,
                             uint64_t offset, uint16_t* out, int nthreads) {
  int8_t* qa = (int8_t*)malloc((size_t)(M * K) + 1);
  int8_t* qb = (int8_t*)malloc((size_t)(N * K) + 1);
  float* sa = (float*)malloc((size_t)M * sizeof(float) + 4);
  float* sb = (float*)malloc((size_t)N * sizeof(float) + 4);
  int rc = -2;
  if (qa && qb && sa && sb) {
    rc = orc_quantize(A, ar, ac, ac, a_axis, mode, seed, offset, a_stream, qa, sa);
    if (rc == 0) rc = orc_quantize(B, br, bc, bc, b_axis, mode, seed, offset, b_stream, qb, sb);
    if (rc == 0) rc = orc_scaled_mm(qa, sa, qb, sb, M, N, K, ORC_AxBT, out, nthreads);
  }
  free(qa); free(qb); free(sa); free(sb);
  return rc;
}

int orc_linear_fwd(const uint16_t* X, const uint16_t* W, int64_t T, int64_t N, int64_t K,
                   int mode, uint64_t seed, uint64_t offset, uint16_t* Y, int nthreads) {
  if (T < 0 || N < 0 || K < 0) return -1;
  /* X along K (its rows), W along K (its rows): Y = Xq . Wq^T */
  return quantized_product(X, T, K, 0, ORC_STREAM_FWD_X, W, N, K, 0, ORC_STREAM_FWD_W,
                           T, N, K, mode, seed, offset, Y, nthreads);
}

int orc_linear_bwd(const uint16_t* dY, const uint16_t* X, const uint16_t* W,
                   int64_t T, int64_t N, int64_t K, int mode, uint64_t seed,
                   uint64_t offset, uint16_t* dX, uint16_t* dW, int nthreads) {
  if (T < 0 || N < 0 || K < 0) return -1;
  int rc = 0;
  if (dX) {
    /* grad input: contraction over N.  dY along N = its rows; W along N =
     * its columns, written [K, N].  dX = dYq . (WqT)^T */
    rc = quantized_product(dY, T, N, 0, ORC_STREAM_GI_DY, W, N, K, 1, ORC_STREAM_GI_W,
                           T, K, N, mode, seed, offset, dX, nthreads);
    if (rc) return rc;
  }
  if (dW) {
    /* grad weight: contraction over T.  dY along T = its columns, written
     * [N, T]; X along T = its columns, written [K, T].  dW = dYqT . XqT^T */
    rc = quantized_product(dY, T, N, 1, ORC_STREAM_GW_DY, X, T, K, 1, ORC_STREAM_GW_X,
                           N, K, T, mode, seed, offset, dW, nthreads);
  }
  return rc;
}

/* ------------------------------------------------------------ BF16 passes */

typedef struct {
  const uint16_t* A;
  const uint16_t* B;
  int64_t M, N, K;
  int layout;
  uint16_t* out;
  int64_t i0, i1;
} bf_job;

static void* bf_rows(void* arg) {
  bf_job* j = (bf_job*)arg;
  for (int64_t i = j->i0; i < j->i1; ++i) {
    for (int64_t n = 0; n < j->N; ++n) {
      double s = 0.0;
      for (int64_t k = 0; k < j->K; ++k) {
        uint16_t a = j->layout == ORC_ATxB ? j->A[k * j->M + i] : j->A[i * j->K + k];
        uint16_t b = j->layout == ORC_AxBT ? j->B[n * j->K + k] : j->B[k * j->N + n];
        s += (double)orc_bf16_to_f32(a) * (double)orc_bf16_to_f32(b);
      }
      j->out[i * j->N + n] = orc_f32_to_bf16_rne((float)s);
    }
  }
  return NULL;
}

int orc_matmul_bf16(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                    int layout, uint16_t* out, int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (layout != ORC_AxBT && layout != ORC_AxB && layout != ORC_ATxB) return -1;
  if (M == 0 || N == 0) return 0;
  if (!out || (K > 0 && (!A || !B))) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > M) nthreads = (int)M;
  if (nthreads > 256) nthreads = 256;
  bf_job jobs[256];
  pthread_t tids[256];
  for (int t = 0; t < nthreads; ++t)
    jobs[t] = (bf_job){A, B, M, N, K, layout, out, M * t / nthreads, M * (t + 1) / nthreads};
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, bf_rows, &jobs[t]) != 0) break;
    started = t;
  }
  bf_rows(&jobs[0]);
  for (int t = started + 1; t < nthreads; ++t) bf_rows(&jobs[t]);
  for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
  return 0;
}

int orc_linear_fwd_cfg(const uint16_t* X, const uint16_t* W, int64_t T, int64_t N, int64_t K,
                       int int8_fwd, int mode, uint64_t seed, uint64_t offset, uint16_t* Y,
                       int nthreads) {
  if (int8_fwd) return orc_linear_fwd(X, W, T, N, K, mode, seed, offset, Y, nthreads);
  return orc_matmul_bf16(X, W, T, N, K, ORC_AxBT, Y, nthreads); /* Y = X . W^T */
}

int orc_linear_bwd_cfg(const uint16_t* dY, const uint16_t* X, const uint16_t* W, int64_t T,
                       int64_t N, int64_t K, int int8_grad_in, int int8_grad_w, int mode,
                       uint64_t seed, uint64_t offset, uint16_t* dX, uint16_t* dW,
                       int nthreads) {
  int rc = 0;
  if (dX) {
    rc = int8_grad_in
             ? orc_linear_bwd(dY, X, W, T, N, K, mode, seed, offset, dX, NULL, nthreads)
             : orc_matmul_bf16(dY, W, T, K, N, ORC_AxB, dX, nthreads); /* dX = dY . W */
    if (rc) return rc;
  }
  if (dW) {
    rc = int8_grad_w
             ? orc_linear_bwd(dY, X, W, T, N, K, mode, seed, offset, NULL, dW, nthreads)
             : orc_matmul_bf16(dY, X, N, K, T, ORC_ATxB, dW, nthreads); /* dW = dY^T . X */
  }
  return rc;
}

/* ------------------------------------------------- data-parallel grad weight */

/* Grad-weight of a linear layer whose T tokens are split into `nshards`
 * equal shards of consecutive rows (T % nshards == 0): shard r quantizes
 * its own rows of dY and X by columns (along T, its own column scales; SR
 * counters from offsets[r]), forms its fp32 partial with orc_scaled_mm_f32,
 * the partials are summed in fp32 in shard order, and the sum is rounded to
 * bf16 once:  dW = bf16_RNE(P_0 + P_1 + ... + P_{n-1}). */
int orc_grad_weight_sharded(const uint16_t* dY, const uint16_t* X, int64_t T, int64_t N, int64_t K,
                            int nshards, int mode, uint64_t seed, const uint64_t* offsets,
                            uint16_t* dW, int nthreads) {
  if (T < 0 || N < 0 || K < 0 || nshards < 1 || T % nshards != 0) return -1;
  if (N == 0 || K == 0) return 0;
  if (!dY || !X || !dW || !offsets) return -1;
  const int64_t Ts = T / nshards;
  float* sum = (float*)calloc((size_t)(N * K), sizeof(float));
  float* part = (float*)malloc((size_t)(N * K) * sizeof(float));
  int8_t* qg = (int8_t*)malloc((size_t)(N * Ts) + 1);
  int8_t* qx = (int8_t*)malloc((size_t)(K * Ts) + 1);
  float* sg = (float*)malloc((size_t)N * sizeof(float));
  float* sx = (float*)malloc((size_t)K * sizeof(float));
  int rc = (sum && part && qg && qx && sg && sx) ? 0 : -2;
  for (int r = 0; r < nshards && rc == 0; ++r) {
    const uint16_t* g = dY + (size_t)(r * Ts) * (size_t)N;
    const uint16_t* x = X + (size_t)(r * Ts) * (size_t)K;
    /* dY and X of this shard along T: column groups, codes [N, Ts] and [K, Ts] */
    rc = orc_quantize(g, Ts, N, N, 1, mode, seed, offsets[r], ORC_STREAM_GW_DY, qg, sg);
    if (rc == 0) rc = orc_quantize(x, Ts, K, K, 1, mode, seed, offsets[r], ORC_STREAM_GW_X, qx, sx);
    if (rc == 0) rc = orc_scaled_mm_f32(qg, sg, qx, sx, N, K, Ts, ORC_AxBT, part, nthreads);
    if (rc == 0)
      for (int64_t i = 0; i < N * K; ++i) sum[i] = sum[i] + part[i];
  }
  if (rc == 0)
    for (int64_t i = 0; i < N * K; ++i) dW[i] = orc_f32_to_bf16_rne(sum[i]);
  free(sum); free(part); free(qg); free(qx); free(sg); free(sx);
  return rc;
}
