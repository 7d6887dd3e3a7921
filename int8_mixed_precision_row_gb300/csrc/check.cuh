// check.cuh -- bounds checks of a checked build.
//
// Built with -DINT8MP_CHECK, the kernels check every global-memory index
// they compute (and the shared-memory slots they index) against the extent of
// the buffer it falls in before the access; a failed check skips the access
// and sets bit 1 of the device status word, which int8mp_poll_device_status
// reports as INT8MP_ERR_BOUNDS.  Nothing traps.  In the ordinary build the
// checks compile to nothing.
#pragma once

namespace int8mp {

#ifdef INT8MP_CHECK
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

constexpr unsigned int kStatusBounds = 2u;

// true if the access may go ahead: always in the ordinary build; in a
// checked build only when `ok`, else the failure is recorded.
__device__ __forceinline__ bool in_bounds(bool ok, unsigned int* status) {
  if (kChecked && !ok) {
    atomicOr(status, kStatusBounds);
    return false;
  }
  return true;
}

}  // namespace int8mp
