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
#include <mutex>

#include "common.cuh"

namespace moer {

moer_status topk_signature_check(const moer_dims* d, const float* logits, int64_t T,
                                 const int32_t* blk_tab, int32_t nblk, const uint8_t* topk,
                                 const uint8_t* blk_cnt, const int32_t* affinity);
moer_status topk_signature_launch(const moer_dims* d, const float* logits, int64_t T,
                                  const int32_t* blk_tab, int32_t nblk, uint8_t* topk,
                                  uint8_t* blk_cnt, int32_t* affinity, void* ws, cudaStream_t st);

// Status header (256 bytes) followed by room for the mask layers' top-k ids,
// which are staged here only when the caller passes topk == NULL.
static __device__ __align__(256) uint8_t noalloc_scratch[WS_HEADER + MOER_NOALLOC_IDS_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (the host-side symbol is not a device address).
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, noalloc_scratch) != cudaSuccess) return nullptr;
    g_ptr[dev] = p;
  }
  return g_ptr[dev];
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
  void* ws = scratch_on_current_device();
  if (ws == nullptr) return MOER_ECUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the status word must start at zero; earlier calls left their contents
  if (cudaMemsetAsync(ws, 0, WS_HEADER, st) != cudaSuccess) return MOER_ECUDA;
  return topk_signature_launch(d, logits, T, blk_tab, nblk, topk, blk_cnt, affinity, ws, st);
}
