/*
 * int8mp_debug.h -- test-only entry points of libint8mp.so.  Not needed to
 * use the library; they exist so that the failure paths can be exercised
 * without faulting or hanging a GPU, and so that a design choice can be
 * measured against its alternative.
 */
#ifndef INT8MP_DEBUG_H
#define INT8MP_DEBUG_H

#include "int8mp.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Runs the int32 product of int8mp_mm_s32 (INT8MP_AxBT, INT8MP_CODES_F16)
 * with one deliberate defect injected from the host: the first tile load of
 * the first CTA is never issued, so the tensor-core warp's bounded wait for
 * it runs out after `wait_limit_ms` milliseconds (1..5000).  The kernel then
 * records INT8MP_ERR_TIMEOUT in the device status word, lets its other warps
 * wind down, waits for its outstanding copies, frees its tensor memory and
 * returns; the CUDA context stays usable.  Returns INT8MP_OK if the launch
 * was enqueued; the timeout itself is reported by int8mp_poll_device_status.
 * Outputs of the first CTA's tiles are left unwritten.
 */
int8mp_status int8mp_debug_mm_s32_drop_first_load(const void* A, const void* B, int64_t M,
                                                  int64_t N, int64_t K, int32_t* out,
                                                  int64_t ldo, int wait_limit_ms, void* stream);

/*
 * Certifies the quantizers' division.  The quantizers compute x / s for the
 * group scale s = RN(absmax / 127) with a reciprocal and two FMAs
 * (Markstein's correction) when s is in [2^-60, 2^10], and by IEEE division
 * otherwise.  This runs that rule and IEEE division (__fdiv_rn) on every pair
 * of bf16 values with absmax > 0 finite and |x| <= absmax (about 1.07e9
 * pairs) and compares the codes the two quotients give: the nearest-even code
 * bit for bit, and for stochastic rounding floor(v) and the number of draws
 * u = k 2^-24 below v - floor(v), which fix the code for every u.
 * The fast rule has two forms, scalar (column quantizers) and packed two
 * lanes per instruction (row quantizers); a pair whose two fast quotients
 * differ counts as a mismatch too.
 * results[0] = pairs whose codes differ, [1] = pairs checked, [2] = pairs on
 * the fast path, [3] = pairs whose quotients differ in any bit (informative:
 * tiny x only).  first_bad[0..1] = bf16 bits (absmax, x) of one pair whose
 * codes differ.  Synchronizes the device.  Test use only.
 */
int8mp_status int8mp_debug_check_division(uint64_t* results, uint32_t* first_bad);

/*
 * The scaled matmul A @ B.T with the B operand quantized inside the GEMM's
 * prologue instead of by a separate pass ("Integrate INT8 mixed-precision
 * from torchao 0.7", limitations: the quantization must be compiled code to
 * pay off; here the alternative to the library's separate row pass, kept so
 * that the choice can be measured).  A: codes as f16 containers [M, K]
 * (INT8MP_GROUP_ROWS), sA fp32 [M].  B: the bf16 values [N, K] themselves,
 * with sB fp32 [N] their row scales (as int8mp_quantize_rowwise computes
 * them); six converter warps of the CTA-pair kernel quantize each bf16 tile
 * of B (nearest even) with its row scales as the row quantizer would, in
 * shared memory, before the tensor core reads it.  out: bf16 [M, N], row
 * stride ldo.  Results are those of int8mp_scaled_mm on B's codes, bit for
 * bit.  Requirements: those of int8mp_scaled_mm with INT8MP_AxBT and
 * INT8MP_CODES_F16.  Test use only.
 */
int8mp_status int8mp_debug_scaled_mm_quant_b(const void* A, const float* sA, const void* B,
                                             const float* sB, int64_t M, int64_t N, int64_t K,
                                             void* out, int64_t ldo, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* INT8MP_DEBUG_H */
