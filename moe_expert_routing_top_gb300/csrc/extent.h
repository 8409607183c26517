// extent.h -- host-only checks that a caller's buffers can hold what a call
// will touch, for the library's optional checked mode.
//
// The library receives raw device pointers and sizes, so a buffer that is
// too small would only show up as a memory fault inside a kernel.  In checked
// mode every entry point first asks the driver for the allocation that holds
// each buffer (its base and size) and refuses the call when
// [p, p + bytes) does not lie inside it.  The check sees allocation ends
// only: a buffer carved out of a larger allocation (a framework's memory
// pool) can still overrun into its neighbour.  Plain C++: the unit tests
// compile it with g++ and drive it with a made-up range query.
#pragma once

#include <cstddef>
#include <cstdint>
#include <initializer_list>

namespace moer {

// True when [p, p + bytes) lies inside [base, base + size).  Written so that
// no sum can wrap.
inline bool extent_within(uintptr_t p, size_t bytes, uintptr_t base, size_t size) {
  if (p < base) return false;
  const uintptr_t off = p - base;
  if (off > size) return false;
  return bytes <= size - off;
}

// One buffer argument of a call: its pointer and the bytes the call may touch
// from it.  A NULL pointer or zero bytes has nothing to check (optional
// arguments are NULL when unused; required ones are tested for NULL before).
struct Extent {
  const void* p;
  size_t bytes;
};

// Checks every extent with `range(p, &base, &size)`, which returns false when
// p is not in any device allocation.  Returns the index of the first extent
// that fails, or -1 when all hold.
template <typename RangeQuery>
int first_bad_extent(std::initializer_list<Extent> list, RangeQuery&& range) {
  int i = 0;
  for (const Extent& e : list) {
    if (e.p != nullptr && e.bytes != 0) {
      uintptr_t base = 0;
      size_t size = 0;
      const uintptr_t a = reinterpret_cast<uintptr_t>(e.p);
      if (!range(a, &base, &size) || !extent_within(a, e.bytes, base, size)) return i;
    }
    ++i;
  }
  return -1;
}

}  // namespace moer
