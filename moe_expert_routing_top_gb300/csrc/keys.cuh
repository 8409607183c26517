// keys.cuh -- order-preserving integer keys of doubles, and a warp minimum over
// (key, index) pairs, for the assignment kernels' scans and reductions.
#pragma once

#include "common.cuh"

namespace moer {

// Order-preserving 64-bit key of a double that is not NaN: unsigned order of
// the keys is the numeric order of the values (-0.0 sorts just below +0.0;
// neither the costs, sums of squares, nor their differences produce -0.0).
// GB300 issues fp64 compares at a small fraction of the integer rate, so the
// assignment kernels' scans and reductions compare keys.
__device__ __forceinline__ unsigned long long okey(double x) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(x);
  return (b >> 63) ? ~b : b | 0x8000000000000000ull;
}
__device__ __forceinline__ double okey_value(unsigned long long k) {
  return __longlong_as_double((long long)((k >> 63) ? k & 0x7FFFFFFFFFFFFFFFull : ~k));
}

// Warp-wide lexicographic minimum of (key, idx) over the lanes; every lane
// gets the result.  Keys compare as two 32-bit halves with redux.sync.
__device__ __forceinline__ void warp_min_key(unsigned long long& key, int& idx) {
  const unsigned hi = (unsigned)(key >> 32), lo = (unsigned)key;
  const unsigned mhi = __reduce_min_sync(FULL, hi);
  const unsigned mlo = __reduce_min_sync(FULL, hi == mhi ? lo : 0xFFFFFFFFu);
  const bool at = hi == mhi && lo == mlo;
  idx = (int)__reduce_min_sync(FULL, at ? (unsigned)idx : 0xFFFFFFFFu);
  key = ((unsigned long long)mhi << 32) | mlo;
}

}  // namespace moer
