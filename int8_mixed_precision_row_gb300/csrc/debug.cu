// debug.cu -- test-only entry points that certify kernel building blocks on
// the device (declared in include/int8mp_debug.h).
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/int8mp_debug.h"
#include "divide.cuh"

static __device__ unsigned long long g_div_counts[3];  // mismatches, pairs, fast-path pairs
static __device__ unsigned int g_div_first[3];  // a mismatch (absmax bits, x bits); largest |x| bits

namespace {

// One block per positive finite bf16 absmax (bit patterns 0x0001..0x7F7F);
// its threads sweep every bf16 x with |x| <= absmax (magnitude bits <= the
// absmax bits, both signs) and compare div_scale with IEEE division.
__global__ void __launch_bounds__(256) check_division_kernel() {
  const uint32_t a = blockIdx.x + 1u;
  const float amax = __uint_as_float(a << 16);
  const float s = __fdiv_rn(amax, 127.0f);
  const int8mp::ScaleDiv d = int8mp::make_scale_div(s);
  unsigned long long bad = 0, pairs = 0;
  for (uint32_t m = threadIdx.x; m <= a; m += blockDim.x) {
    for (uint32_t sign = 0; sign < 2; ++sign) {
      const uint32_t xb = (sign << 15) | m;
      const float x = __uint_as_float(xb << 16);
      const float got = int8mp::div_scale(x, d);
      const float ref = __fdiv_rn(x, s);
      ++pairs;
      if (!(got == ref)) {  // float equality: +0 == -0, which give the same code
        ++bad;
        if (atomicCAS(&g_div_first[0], 0u, a) == 0u) g_div_first[1] = xb;
        atomicMax(&g_div_first[2], m);
      }
    }
  }
  if (bad) atomicAdd(&g_div_counts[0], bad);
  atomicAdd(&g_div_counts[1], pairs);
  if (d.fast) atomicAdd(&g_div_counts[2], pairs);
}

}  // namespace

extern "C" int8mp_status int8mp_debug_check_division(uint64_t* mismatches, uint64_t* pairs,
                                                     uint64_t* fast_pairs, uint32_t* first_bad) {
  if (!mismatches || !pairs || !fast_pairs || !first_bad) return INT8MP_ERR_INVALID_ARG;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return INT8MP_ERR_CUDA;
  if (major != 10 || minor != 3) return INT8MP_ERR_UNSUPPORTED_DEVICE;
  const unsigned long long zero3[3] = {0, 0, 0};
  const unsigned int zero2[3] = {0, 0, 0};
  if (cudaMemcpyToSymbol(g_div_counts, zero3, sizeof zero3) != cudaSuccess ||
      cudaMemcpyToSymbol(g_div_first, zero2, sizeof zero2) != cudaSuccess)
    return INT8MP_ERR_CUDA;
  check_division_kernel<<<0x7F7F, 256>>>();
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return INT8MP_ERR_CUDA;
  unsigned long long counts[3];
  unsigned int first[3];
  if (cudaMemcpyFromSymbol(counts, g_div_counts, sizeof counts) != cudaSuccess ||
      cudaMemcpyFromSymbol(first, g_div_first, sizeof first) != cudaSuccess)
    return INT8MP_ERR_CUDA;
  *mismatches = counts[0];
  *pairs = counts[1];
  *fast_pairs = counts[2];
  first_bad[0] = first[0];
  first_bad[1] = first[1];
  first_bad[2] = first[2];
  return INT8MP_OK;
}
