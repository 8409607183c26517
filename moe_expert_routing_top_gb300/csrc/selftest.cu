// selftest.cu -- moer_wait_selftest: the expiry path of the library's bounded
// device waits, exercised on purpose.
//
// The kernel's mbarrier is set up for one arrival that never comes, so the
// wait used by every pipelined kernel (mbar_wait) gives up after the given
// limit, records MOER_ETIMEOUT in the workspace status word and returns; the
// kernel then ends normally and the context stays usable.  Nothing faults,
// traps or spins without a bound.
#include "common.cuh"

namespace moer {

__global__ void wait_selftest_kernel(uint32_t* status, uint32_t* gave_up, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) gave_up[0] = mbar_wait(&bar, 0u, status, limit_ns) ? 0u : 1u;
}

moer_status wait_selftest_launch(void* ws, uint32_t limit_us, cudaStream_t st) {
  uint32_t* status = static_cast<uint32_t*>(ws);
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, status + 2, (unsigned long long)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
