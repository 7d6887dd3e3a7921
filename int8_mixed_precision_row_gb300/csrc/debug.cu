// debug.cu -- test-only entry points that certify kernel building blocks on
// the device (declared in include/int8mp_debug.h).
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/int8mp_debug.h"
#include "divide.cuh"

// code mismatches, pairs, fast-path pairs, quotients differing from IEEE
static __device__ unsigned long long g_div_counts[4];
static __device__ unsigned int g_div_first[2];  // first code mismatch: absmax bits, x bits

namespace {

// nearest-even code of a quotient: clamp(rint(v)), +0 for zero
__device__ __forceinline__ float rne_code_of(float v) {
  return __fadd_rn(fminf(fmaxf(rintf(v), -127.0f), 127.0f), 0.0f);
}

// What fixes the stochastic code for every draw u = k 2^-24: floor(v) and
// the number of draws below v - floor(v).
__device__ __forceinline__ void sr_signature(float v, float& f, float& below) {
  f = floorf(v);
  below = ceilf(__fmul_rn(__fsub_rn(v, f), 0x1p24f));
}

// One block per positive finite bf16 absmax (bit patterns 0x0001..0x7F7F);
// its threads sweep every bf16 x with |x| <= absmax (magnitude bits <= the
// absmax bits, both signs) and compare the codes from the fast division with
// the codes from IEEE division; a pair also counts as a mismatch if the
// packed two-lane form (row quantizers) and the scalar form (column
// quantizers) give different quotients.
__global__ void __launch_bounds__(256) check_division_kernel() {
  const uint32_t a = blockIdx.x + 1u;
  const float amax = __uint_as_float(a << 16);
  const float s = __fdiv_rn(amax, 127.0f);
  const int8mp::ScaleDiv d = int8mp::make_scale_div(s);
  unsigned long long bad = 0, pairs = 0, qdiff = 0;
  for (uint32_t m = threadIdx.x; m <= a; m += blockDim.x) {
    const float xp = __uint_as_float(m << 16), xn = __uint_as_float((0x8000u | m) << 16);
    const float2 fast = int8mp::div2_fast(make_float2(xp, xn), make_float2(d.s, d.s),
                                          make_float2(d.r, d.r));
    for (uint32_t sign = 0; sign < 2; ++sign) {
      const uint32_t xb = (sign << 15) | m;
      const float x = sign ? xn : xp;
      // both fast forms: the packed lane must equal the scalar result
      const float lane = sign ? fast.y : fast.x;
      const float got = d.fast ? int8mp::div_fast(x, d.s, d.r) : __fdiv_rn(x, d.s);
      const bool forms_agree = !d.fast || __float_as_uint(lane) == __float_as_uint(got);
      const float ref = __fdiv_rn(x, s);
      ++pairs;
      if (!(got == ref)) ++qdiff;
      float fg, bg, fr, br;
      sr_signature(got, fg, bg);
      sr_signature(ref, fr, br);
      const bool same = forms_agree &&
                        __float_as_uint(rne_code_of(got)) == __float_as_uint(rne_code_of(ref)) &&
                        fg == fr && bg == br;
      if (!same) {
        ++bad;
        if (atomicCAS(&g_div_first[0], 0u, a) == 0u) g_div_first[1] = xb;
      }
    }
  }
  if (bad) atomicAdd(&g_div_counts[0], bad);
  atomicAdd(&g_div_counts[1], pairs);
  if (d.fast) atomicAdd(&g_div_counts[2], pairs);
  if (qdiff) atomicAdd(&g_div_counts[3], qdiff);
}

}  // namespace

extern "C" int8mp_status int8mp_debug_check_division(uint64_t* results, uint32_t* first_bad) {
  if (!results || !first_bad) return INT8MP_ERR_INVALID_ARG;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return INT8MP_ERR_CUDA;
  if (major != 10 || minor != 3) return INT8MP_ERR_UNSUPPORTED_DEVICE;
  const unsigned long long zero4[4] = {0, 0, 0, 0};
  const unsigned int zero2[2] = {0, 0};
  if (cudaMemcpyToSymbol(g_div_counts, zero4, sizeof zero4) != cudaSuccess ||
      cudaMemcpyToSymbol(g_div_first, zero2, sizeof zero2) != cudaSuccess)
    return INT8MP_ERR_CUDA;
  check_division_kernel<<<0x7F7F, 256>>>();
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return INT8MP_ERR_CUDA;
  unsigned long long counts[4];
  unsigned int first[2];
  if (cudaMemcpyFromSymbol(counts, g_div_counts, sizeof counts) != cudaSuccess ||
      cudaMemcpyFromSymbol(first, g_div_first, sizeof first) != cudaSuccess)
    return INT8MP_ERR_CUDA;
  for (int i = 0; i < 4; ++i) results[i] = counts[i];
  first_bad[0] = first[0];
  first_bad[1] = first[1];
  return INT8MP_OK;
}
