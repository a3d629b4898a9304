// checks.cuh - index checks of the checked build.
//
// Built with FA_DEBUG_CHECKS (libfa_checked.so), every plain global load and
// store of the kernels is first checked against the extent its buffer has by
// the call's arguments.  A failing access is skipped (a load yields 0) and
// FA_DEV_BAD_INDEX is set in the status word; nothing traps.  The release
// build compiles every check to `true`.  TMA copies need no check: their
// tensor maps bound them in hardware.
#pragma once

#include <cstddef>

#include "ptx.cuh"

namespace fa {

#ifdef FA_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// Elements [idx, idx + count) lie inside a buffer of n elements.
__device__ __forceinline__ bool in_bounds(size_t idx, size_t count, size_t n,
                                          unsigned int *status) {
  if constexpr (kDebugChecks) {
    if (idx + count > n) {
      raise_status(status, FA_DEV_BAD_INDEX);
      return false;
    }
  }
  return true;
}

// Load of element idx of a buffer of n elements (0 when outside).
template <typename T>
__device__ __forceinline__ T checked_load(const T *base, size_t idx, size_t n,
                                          unsigned int *status) {
  return in_bounds(idx, 1, n, status) ? base[idx] : T{};
}

}  // namespace fa
