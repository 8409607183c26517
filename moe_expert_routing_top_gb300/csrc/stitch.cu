// stitch.cu -- prefix-cache stitching of per-KV-block counts.
//
// ELDR, table of what existing decode routing misses (signature cache row),
// component table (signature cache) and section "Practical interpretation":
// a signature cache co-indexed with the KV cache stores each KV block's
// expert footprint, so that a prefix-cache hit still yields the full-prompt
// signature.  Full computed blocks are inserted first; then each request's
// counts are the sum over its cached prefix blocks and its computed blocks.
//
// Both kernels move 16-byte words of packed 8-bit counts (sixteen experts per
// word; 4-byte words when a record or buffer is not 16-byte aligned): the
// insert copies one block record per warp, and a request's record of m*E
// counts is summed by one CTA whose threads own consecutive words, so every
// load and store is coalesced.
#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "pdl.cuh"

namespace moer {

// One warp per KV block: the slot is checked once, the record is copied with
// 16-byte (V = uint4) or 4-byte (V = uint32_t) words.
template <typename V>
__global__ void stitch_insert(const V* __restrict__ blk_w, const int32_t* __restrict__ blk_tab, int nblk, int B,
                              const int32_t* __restrict__ insert_slot, V* __restrict__ cache_w, int nslots,
                              int rec_v, uint32_t* status) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nblk; b += stride) {
    const int slot = insert_slot[b];
    if (slot < 0 || blk_tab[2 * b + 1] != B) continue;
    if (slot >= nslots) {
      if (status != nullptr && lane == 0) atomicOr(status, WS_BIT_EDATA);
      continue;
    }
    const V* src = blk_w + (size_t)b * rec_v;
    V* dst = cache_w + (size_t)slot * rec_v;
    for (int w = lane; w < rec_v; w += 32) dst[w] = src[w];
  }
  pdl_release();
}

// block loads in flight per thread: 8 words of 4 bytes or 4 of 16 bytes (the
// sixteen 32-bit sums of a 16-byte word leave no registers for more)
template <typename V>
__host__ __device__ constexpr int stitch_su() { return sizeof(V) == 16 ? 4 : 8; }

__device__ __forceinline__ void acc4(uint32_t (&a)[4], uint32_t v) {
  a[0] += v & 0xFFu;
  a[1] += (v >> 8) & 0xFFu;
  a[2] += (v >> 16) & 0xFFu;
  a[3] += v >> 24;
}
__device__ __forceinline__ void accv(uint32_t (&a)[4], uint32_t v) { acc4(a, v); }
__device__ __forceinline__ void accv(uint32_t (&a)[16], uint4 v) {
  uint32_t* q = a;
  acc4(*reinterpret_cast<uint32_t(*)[4]>(q), v.x);
  acc4(*reinterpret_cast<uint32_t(*)[4]>(q + 4), v.y);
  acc4(*reinterpret_cast<uint32_t(*)[4]>(q + 8), v.z);
  acc4(*reinterpret_cast<uint32_t(*)[4]>(q + 12), v.w);
}

// One CTA per request, S groups of TW threads: thread (s, w) sums word w of
// the record (16 or 4 bytes of packed 8-bit counts) over the request's cached
// blocks s, s + S, ... and computed blocks s, s + S, ..., SU block loads in
// flight; group 0 adds the S partial sums (through shared memory, laid out
// [S][NB][TW] so every access is conflict-free) and writes the request's row.
// The kernel's length is set by its longest requests (a few hundred blocks):
// S groups with SU loads each keep S * SU of their blocks in flight at once.
template <typename V, int NB, int S>
__global__ void __launch_bounds__(1024) stitch_sum(const V* __restrict__ blk_w, int nblk, const int32_t* __restrict__ req_blk_off,
                           const int32_t* __restrict__ cache_idx, int ncached,
                           const int32_t* __restrict__ req_cache_off, const V* __restrict__ cache_w, int nslots,
                           int rec_v, int32_t* __restrict__ req_cnt, uint32_t* status) {
  extern __shared__ uint32_t part[];  // [S][NB][TW] partial sums
  pdl_wait();
  constexpr int SU = stitch_su<V>();
  const int TW = blockDim.x / S;
  const int grp = threadIdx.x / TW, wl = threadIdx.x - grp * TW;
  const int r = blockIdx.x;
  const int b0 = req_blk_off[r], b1 = req_blk_off[r + 1];
  int c0 = cache_w ? req_cache_off[r] : 0, c1 = cache_w ? req_cache_off[r + 1] : 0;
  const bool bad_blocks = b0 < 0 || b1 < b0 || b1 > nblk;
  // a cached-prefix range outside [0, ncached) is skipped whole, like a bad block range
  const bool bad_cache = c0 < 0 || c1 < c0 || c1 > ncached;
  if ((bad_blocks || bad_cache) && threadIdx.x == 0 && status != nullptr) atomicOr(status, WS_BIT_EDATA);
  if (bad_cache) c0 = c1 = 0;
  for (int w0 = 0; w0 < rec_v; w0 += TW) {
    const int w = w0 + wl;
    uint32_t a[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) a[i] = 0u;
    if (w < rec_v) {
      // cached prefix blocks: SU slot numbers, then their SU records, in flight together
      for (int c = c0 + grp; c < c1; c += SU * S) {
        int slot[SU];
#pragma unroll
        for (int u = 0; u < SU; ++u) slot[u] = c + u * S < c1 ? cache_idx[c + u * S] : -2;
        V v[SU];
#pragma unroll
        for (int u = 0; u < SU; ++u)
          if (slot[u] >= 0 && slot[u] < nslots) v[u] = cache_w[(size_t)slot[u] * rec_v + w];
#pragma unroll
        for (int u = 0; u < SU; ++u) {
          if (slot[u] >= 0 && slot[u] < nslots) {
            accv(a, v[u]);
          } else if (slot[u] != -2 && status != nullptr) {
            atomicOr(status, WS_BIT_EDATA);
          }
        }
      }
      if (!bad_blocks) {
        int b = b0 + grp;
        for (; b + (SU - 1) * S < b1; b += SU * S) {
          V v[SU];
#pragma unroll
          for (int u = 0; u < SU; ++u) v[u] = blk_w[(size_t)(b + u * S) * rec_v + w];
#pragma unroll
          for (int u = 0; u < SU; ++u) accv(a, v[u]);
        }
        for (; b < b1; b += S) accv(a, blk_w[(size_t)b * rec_v + w]);
      }
    }
    if constexpr (S > 1) {
#pragma unroll
      for (int i = 0; i < NB; ++i) part[((size_t)grp * NB + i) * TW + wl] = a[i];
      __syncthreads();
      if (grp == 0) {
        for (int q = 1; q < S; ++q)
#pragma unroll
          for (int i = 0; i < NB; ++i) a[i] += part[((size_t)q * NB + i) * TW + wl];
      }
      __syncthreads();  // the next word range reuses the partial sums
    }
    if (grp == 0 && w < rec_v) {
      int32_t* dst = req_cnt + (size_t)r * rec_v * NB + (size_t)w * NB;
      if constexpr (NB == 16) {
        int4* d4 = reinterpret_cast<int4*>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          d4[i] = make_int4((int)a[4 * i], (int)a[4 * i + 1], (int)a[4 * i + 2], (int)a[4 * i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < NB; ++i) dst[i] = (int32_t)a[i];
      }
    }
  }
  pdl_release();
}

moer_status block_stitch_launch(const moer_dims* d, const uint8_t* blk_cnt, const int32_t* blk_tab,
                                int32_t nblk, const int32_t* req_blk_off, int32_t R,
                                const int32_t* cache_idx, int32_t ncached, const int32_t* req_cache_off,
                                uint8_t* cache, int32_t nslots, const int32_t* insert_slot,
                                int32_t* req_cnt, uint32_t* status, cudaStream_t st) {
  const int rec_bytes = d->m * d->E;
  auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  // 16-byte words when every record, cache slot and request row stays 16-byte aligned
  const bool v16 = rec_bytes % 16 == 0 && a16(blk_cnt) && (cache == nullptr || a16(cache)) && a16(req_cnt);
  const int sms = device_sm_count();
  if (sms <= 0) return MOER_ECUDA;
  if (cache != nullptr && insert_slot != nullptr && nblk > 0) {
    const int grid = (int)min64(((int64_t)nblk + 7) / 8, (int64_t)sms * 8);
    const cudaError_t e =
        v16 ? launch_pdl(stitch_insert<uint4>, dim3(grid), dim3(256), 0, st, reinterpret_cast<const uint4*>(blk_cnt),
                         blk_tab, nblk, d->block, insert_slot, reinterpret_cast<uint4*>(cache), nslots, rec_bytes / 16,
                         status)
            : launch_pdl(stitch_insert<uint32_t>, dim3(grid), dim3(256), 0, st,
                         reinterpret_cast<const uint32_t*>(blk_cnt), blk_tab, nblk, d->block, insert_slot,
                         reinterpret_cast<uint32_t*>(cache), nslots, rec_bytes / 4, status);
    if (e != cudaSuccess) return MOER_ECUDA;
  }
  // TW threads per group cover the record's words, four groups (at most 1,024 threads,
  // partial sums within 64 KB of shared memory).  Eight groups of up to 96 threads were
  // slower on the Qwen3-shaped batch (0.096 against 0.088 ms for the stitch call): fewer
  // requests resident per SM.
  auto launch_sum = [&](auto vtag, auto nbtag) -> cudaError_t {
    using V = decltype(vtag);
    constexpr int NB = decltype(nbtag)::value;
    const int rec_v = rec_bytes / (int)sizeof(V);
    const int tw = rec_v >= 256 ? 256 : ((rec_v + 31) / 32) * 32;
    const size_t part1 = (size_t)NB * tw * sizeof(uint32_t);
    auto go = [&](auto stag) -> cudaError_t {
      constexpr int S = decltype(stag)::value;
      // the attribute is a ceiling kept for the process: set it once to the most any call
      // of this instance may ask for (64 KB), never to one call's size
      static std::atomic<unsigned long long> opted{0};
      cudaError_t e = smem_optin(stitch_sum<V, NB, S>, 64 * 1024, opted);
      if (e != cudaSuccess) return e;
      return launch_pdl(stitch_sum<V, NB, S>, dim3(R), dim3(S * tw), S * part1, st,
                        reinterpret_cast<const V*>(blk_cnt), nblk, req_blk_off, cache_idx, ncached, req_cache_off,
                        reinterpret_cast<const V*>(cache), nslots, rec_v, req_cnt, status);
    };
    return go(std::integral_constant<int, 4>{});  // tw <= 256 and part1 <= 16 KB always fit
  };
  const cudaError_t e = v16 ? launch_sum(uint4{}, std::integral_constant<int, 16>{})
                            : launch_sum(uint32_t{}, std::integral_constant<int, 4>{});
  return e == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
