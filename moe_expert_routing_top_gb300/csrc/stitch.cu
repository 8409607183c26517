// stitch.cu -- prefix-cache stitching of per-KV-block counts.
//
// ELDR, table of what existing decode routing misses (signature cache row),
// component table (signature cache) and section "Practical interpretation":
// a signature cache co-indexed with the KV cache stores each KV block's
// expert footprint, so that a prefix-cache hit still yields the full-prompt
// signature.  Full computed blocks are inserted first; then each request's
// counts are the sum over its cached prefix blocks and its computed blocks.
//
// Both kernels move 32-bit words of packed 8-bit counts (four experts per
// word); a request's record of m*E counts is handled by one CTA whose threads
// own consecutive words, so every load and store is coalesced.
#include "common.cuh"

namespace moer {

__global__ void stitch_insert(const uint32_t* __restrict__ blk_w, const int32_t* __restrict__ blk_tab,
                              int nblk, int B, const int32_t* __restrict__ insert_slot,
                              uint32_t* __restrict__ cache_w, int nslots, int rec_words,
                              uint32_t* status) {
  const int64_t total = (int64_t)nblk * rec_words;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(i / rec_words);
    const int w = (int)(i - (int64_t)b * rec_words);
    const int slot = insert_slot[b];
    if (slot < 0 || blk_tab[2 * b + 1] != B) continue;
    if (slot >= nslots) {
      if (status != nullptr && w == 0) atomicOr(status, WS_BIT_EDATA);
      continue;
    }
    cache_w[(size_t)slot * rec_words + w] = blk_w[(size_t)b * rec_words + w];
  }
}

__global__ void stitch_sum(const uint32_t* __restrict__ blk_w, int nblk,
                           const int32_t* __restrict__ req_blk_off,
                           const int32_t* __restrict__ cache_idx,
                           const int32_t* __restrict__ req_cache_off,
                           const uint32_t* __restrict__ cache_w, int nslots, int rec_words,
                           int32_t* __restrict__ req_cnt, uint32_t* status) {
  const int r = blockIdx.x;
  const int b0 = req_blk_off[r], b1 = req_blk_off[r + 1];
  const int c0 = cache_w ? req_cache_off[r] : 0, c1 = cache_w ? req_cache_off[r + 1] : 0;
  const bool bad_blocks = b0 < 0 || b1 < b0 || b1 > nblk;
  if (bad_blocks && threadIdx.x == 0 && status != nullptr) atomicOr(status, WS_BIT_EDATA);
  for (int w = threadIdx.x; w < rec_words; w += blockDim.x) {
    uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
    for (int c = c0; c < c1; ++c) {
      const int slot = cache_idx[c];
      if (slot < 0 || slot >= nslots) {
        if (status != nullptr && w == 0) atomicOr(status, WS_BIT_EDATA);
        continue;
      }
      const uint32_t v = cache_w[(size_t)slot * rec_words + w];
      a0 += v & 0xFFu;
      a1 += (v >> 8) & 0xFFu;
      a2 += (v >> 16) & 0xFFu;
      a3 += v >> 24;
    }
    if (!bad_blocks)
      for (int b = b0; b < b1; ++b) {
        const uint32_t v = blk_w[(size_t)b * rec_words + w];
        a0 += v & 0xFFu;
        a1 += (v >> 8) & 0xFFu;
        a2 += (v >> 16) & 0xFFu;
        a3 += v >> 24;
      }
    int32_t* dst = req_cnt + (size_t)r * rec_words * 4 + (size_t)w * 4;
    dst[0] = (int32_t)a0;
    dst[1] = (int32_t)a1;
    dst[2] = (int32_t)a2;
    dst[3] = (int32_t)a3;
  }
}

moer_status block_stitch_launch(const moer_dims* d, const uint8_t* blk_cnt, const int32_t* blk_tab,
                                int32_t nblk, const int32_t* req_blk_off, int32_t R,
                                const int32_t* cache_idx, const int32_t* req_cache_off,
                                uint8_t* cache, int32_t nslots, const int32_t* insert_slot,
                                int32_t* req_cnt, uint32_t* status, cudaStream_t st) {
  const int rec_words = d->m * d->E / 4;
  if (cache != nullptr && insert_slot != nullptr && nblk > 0) {
    const int64_t total = (int64_t)nblk * rec_words;
    const int blocks = (int)min64((total + 255) / 256, 8192);
    stitch_insert<<<blocks, 256, 0, st>>>(reinterpret_cast<const uint32_t*>(blk_cnt), blk_tab, nblk,
                                          d->block, insert_slot, reinterpret_cast<uint32_t*>(cache),
                                          nslots, rec_words, status);
    if (cudaGetLastError() != cudaSuccess) return MOER_ECUDA;
  }
  const int threads = rec_words >= 256 ? 256 : ((rec_words + 31) / 32) * 32;
  stitch_sum<<<R, threads, 0, st>>>(reinterpret_cast<const uint32_t*>(blk_cnt), nblk, req_blk_off,
                                    cache_idx, req_cache_off,
                                    reinterpret_cast<const uint32_t*>(cache), nslots, rec_words,
                                    req_cnt, status);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
