// ctx_cache.h -- host-only cache of one device address per CUDA context.
//
// A __device__ variable has one address per context that loads the module.
// Keying the cache on the context's unique ID (cuCtxGetId: IDs are never
// reused within a process) rather than on the device ordinal means that a
// context destroyed and created again (cudaDeviceReset, a primary context
// released and retained again) gets a fresh look-up instead of an address
// from the dead context.  Plain C++: the unit tests compile it with g++ and
// drive it with made-up IDs.
#pragma once

#include <mutex>

namespace moer {

template <int N>
class CtxAddressCache {
 public:
  // The address cached for context `ctx_id`.  On a miss, `lookup(void**)`
  // (returning true on success) supplies it; a failed look-up caches nothing
  // and returns nullptr.  When all N entries are taken, the oldest is
  // replaced.
  template <typename Lookup>
  void* get(unsigned long long ctx_id, Lookup&& lookup) {
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < used_; ++i)
      if (ids_[i] == ctx_id) return addr_[i];
    void* p = nullptr;
    if (!lookup(&p) || p == nullptr) return nullptr;
    const int slot = used_ < N ? used_++ : (next_++ % N);
    ids_[slot] = ctx_id;
    addr_[slot] = p;
    return p;
  }

  int size() {
    std::lock_guard<std::mutex> lock(mu_);
    return used_;
  }

 private:
  std::mutex mu_;
  unsigned long long ids_[N] = {};
  void* addr_[N] = {};
  int used_ = 0;
  int next_ = 0;
};

}  // namespace moer
