/*
 * int8mp_debug.h -- test-only entry points of libint8mp.so.  Not needed to
 * use the library; they exist so that the failure paths can be exercised
 * without faulting or hanging a GPU.
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
 * (Markstein's correction) instead of an IEEE division; this runs that
 * function and IEEE division (__fdiv_rn) on every pair of bf16 values with
 * absmax > 0 finite and |x| <= absmax (about 1.07e9 pairs) and reports how
 * many quotients differ (compared as floats, so +0 and -0 are equal: both
 * give code 0), how many pairs were checked, how many of them took the fast
 * path, the bf16 bit patterns (absmax, x) of one differing pair, and the
 * largest |x| bit pattern among differing pairs (first_bad has 3 entries).
 * Synchronizes the device.  Test use only.
 */
int8mp_status int8mp_debug_check_division(uint64_t* mismatches, uint64_t* pairs,
                                          uint64_t* fast_pairs, uint32_t* first_bad);

#ifdef __cplusplus
}
#endif
#endif /* INT8MP_DEBUG_H */
