// noalloc.cu -- moer_topk_signature_noalloc: the same call as
// moer_topk_signature for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs inside another
// framework's allocator arena or memory pool, plugins that must not change
// the process's device-memory footprint after start-up, and code paths that
// have to stay free of allocation calls for latency or determinism.  For
// them the scratch that moer_topk_signature takes as a caller workspace lives
// here, in one fixed-size array in device memory that every GPU loading this
// library holds until the process exits.
#include <cuda.h>

#include "common.cuh"
#include "ctx_cache.h"

namespace moer {

moer_status topk_signature_check(const moer_dims* d, const float* logits, int64_t T,
                                 const int32_t* blk_tab, int32_t nblk, const uint8_t* topk,
                                 const uint8_t* blk_cnt, const int32_t* affinity);
moer_status topk_signature_noalloc_extents(const moer_dims* d, const float* logits, int64_t T,
                                           const int32_t* blk_tab, int32_t nblk, const uint8_t* topk,
                                           const uint8_t* blk_cnt, const int32_t* affinity);
moer_status topk_signature_launch(const moer_dims* d, const float* logits, int64_t T,
                                  const int32_t* blk_tab, int32_t nblk, uint8_t* topk,
                                  uint8_t* blk_cnt, int32_t* affinity, void* ws, cudaStream_t st);

// Status header (256 bytes) followed by room for the mask layers' top-k ids,
// which are staged here only when the caller passes topk == NULL.
static __device__ __align__(256) uint8_t noalloc_scratch[WS_HEADER + MOER_NOALLOC_IDS_BYTES];

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's cuCtxGetCurrent and cuCtxGetId, resolved through the runtime
// (the library does not link libcuda directly).
struct CtxApi {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const CtxApi& ctx_api() {
  static const CtxApi api = []() {
    CtxApi a;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      a.get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      a.get_id = reinterpret_cast<CtxGetIdFn>(f);
    return a;
  }();
  return api;
}

// ID of the context current on this thread; false when there is none yet.
bool current_context_id(unsigned long long* id) {
  const CtxApi& a = ctx_api();
  if (a.get_current == nullptr || a.get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (a.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return a.get_id(ctx, id) == CUDA_SUCCESS;
}

CtxAddressCache<64> g_scratch_addr;

bool lookup_scratch(void** p) { return cudaGetSymbolAddress(p, noalloc_scratch) == cudaSuccess; }

// Device address of the scratch array in the current context (the host-side
// symbol is not a device address), looked up once per context.
void* scratch_in_current_context() {
  unsigned long long id = 0;
  if (!current_context_id(&id)) {
    // No context is current on this thread yet: the runtime's look-up makes
    // the current device's primary context current, then it has an ID.
    void* p = nullptr;
    if (!lookup_scratch(&p) || !current_context_id(&id)) return nullptr;
  }
  return g_scratch_addr.get(id, lookup_scratch);
}

}  // namespace
}  // namespace moer

using namespace moer;

extern "C" MOER_API moer_status moer_topk_signature_noalloc(const moer_dims* d, const float* logits,
                                                           int64_t T, const int32_t* blk_tab,
                                                           int32_t nblk, uint8_t* topk, uint8_t* blk_cnt,
                                                           int32_t* affinity, moer_stream_t stream) {
  moer_status s = topk_signature_check(d, logits, T, blk_tab, nblk, topk, blk_cnt, affinity);
  if (s != MOER_OK || T == 0) return s;
  if (topk == nullptr && blk_cnt != nullptr && d->m > 0 &&
      (uint64_t)d->m * (uint64_t)T * (uint64_t)d->k > (uint64_t)MOER_NOALLOC_IDS_BYTES)
    return MOER_ENOMEM;
  s = topk_signature_noalloc_extents(d, logits, T, blk_tab, nblk, topk, blk_cnt, affinity);
  if (s != MOER_OK) return s;
  void* ws = scratch_in_current_context();
  if (ws == nullptr) return MOER_ECUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the status word must start at zero; earlier calls left their contents
  if (cudaMemsetAsync(ws, 0, WS_HEADER, st) != cudaSuccess) return MOER_ECUDA;
  return topk_signature_launch(d, logits, T, blk_tab, nblk, topk, blk_cnt, affinity, ws, st);
}
