// pdl.cuh -- programmatic dependent launch along the small kernels of a step
// (block counts, co-activation from ids, stitch, loads, routing).
//
// A kernel launched with launch_pdl may be scheduled before the kernel ahead
// of it in the stream has finished.  It calls pdl_wait() before anything
// else: that returns once the kernel ahead has completed and its writes are
// visible (at once when there is no such dependency).  Each of these kernels
// calls pdl_release() as its last statement, so the kernel behind it is
// launched while its last CTAs finish and lands on SMs that are by then free.
// (Released at the start instead, the successor's CTAs were placed on the
// few SMs free at that moment; a persistent grid that expects an even spread
// ran unbalanced, and the gate path's step took 8.35 instead of 8.24 ms.)
// Stream order is kept; what overlaps is one kernel's launch with the tail of
// the one before.
//
// The block counts and the co-activation from ids are persistent grids that
// split their work statically; they are launched normally (their CTAs then
// find every SM free) and release their successor at their end.  Launched
// early, the co-activation's CTAs crowded the SMs that freed first, and the
// gate path's step took 8.32-8.40 instead of 8.22 ms.
//
// The logits pass and the gate GEMM are launched normally and release
// nothing: the logits pass holds every SM's registers, so a successor
// launched early could only wait beside it, and the gate GEMM leaves room on
// each SM for a waiting block-count CTA (with an early release there the gate
// path's step took 8.36 instead of 8.23 ms).
#pragma once

#include <cuda_runtime.h>

namespace moer {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c = {};
  c.gridDim = grid;
  c.blockDim = block;
  c.dynamicSmemBytes = smem;
  c.stream = st;
  c.attrs = attr;
  c.numAttrs = 1;
  return cudaLaunchKernelEx(&c, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moer
