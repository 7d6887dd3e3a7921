// noalloc.cu -- int8mp_linear_fwd_noalloc: the INT8 linear forward pass for
// callers that must not allocate device memory themselves.
//
// Who needs it: code embedded in a host program that owns every byte of
// device memory through its own pool (or has reserved the whole memory budget
// up front) and forbids direct cudaMalloc; and latency-critical callers that
// may not call cudaMalloc / cudaFree at run time because those calls can
// synchronize the device and take unbounded time.  Such callers cannot
// provide the workspace int8mp_linear_fwd asks for.
//
// How: the workspace (f16 codes and fp32 scales of X and W) lives in the
// file-scope array below, which every device that loads this library holds
// until the process exits.  Host code cannot use the array's name as a
// device address (on the host it is only a stand-in), so the first call on
// each device looks the address up with cudaGetSymbolAddress while that
// device is current, and every call passes that address on as the workspace
// of the ordinary forward pass.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/int8mp.h"

// One shared scratch area per device.  Every call uses all of it; a call
// leaves its codes and scales behind, and the next call overwrites them.
static __device__ __align__(256) unsigned char g_noalloc_scratch[INT8MP_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

struct ScratchSlot {
  std::mutex mu;
  void* ptr = nullptr;  // set once a lookup has succeeded
};
ScratchSlot g_slots[kMaxDevices];

// Device address of the scratch array on the current device, looked up with
// that device current.  Only a successful lookup is kept: a first call made
// in a state where the lookup fails (inside a stream capture, or with an
// error pending from earlier work) returns INT8MP_ERR_CUDA, and the next
// call tries again.
int8mp_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return INT8MP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return INT8MP_ERR_UNSUPPORTED_DEVICE;
  ScratchSlot& slot = g_slots[dev];
  std::lock_guard<std::mutex> lock(slot.mu);
  if (slot.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return INT8MP_ERR_CUDA;
    slot.ptr = p;
  }
  *out = slot.ptr;
  return INT8MP_OK;
}

inline uint64_t round256(uint64_t v) { return (v + 255u) / 256u * 256u; }

}  // namespace

extern "C" int8mp_status int8mp_linear_fwd_noalloc(const void* X, const void* W, void* Y,
                                                   int64_t T, int64_t N, int64_t K,
                                                   const int8mp_linear_cfg* cfg, void* stream) {
  if (!cfg || T < 0 || N < 0 || K < 0 || T > INT8MP_MAX_K || N > INT8MP_MAX_K || K > INT8MP_MAX_K)
    return INT8MP_ERR_INVALID_ARG;
  // the forward pass's workspace: codes (2 bytes each) and scales of X and W
  const uint64_t need = round256(2ull * T * K) + round256(4ull * T) + round256(2ull * N * K) +
                        round256(4ull * N);
  if (need > INT8MP_NOALLOC_SCRATCH_BYTES) return INT8MP_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int8mp_status st = scratch_on_current_device(&scratch);
  if (st != INT8MP_OK) return st;
  // Exactly the codes and scales: with no room past them the matmul runs
  // whole tiles only (no split last wave, whose counters it would read
  // before writing), so every byte a call reads it has written first.
  return int8mp_linear_fwd(X, W, Y, T, N, K, cfg, scratch, static_cast<size_t>(need), stream);
}
