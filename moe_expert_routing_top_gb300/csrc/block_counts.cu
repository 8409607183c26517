// block_counts.cu -- per-KV-block expert counts over the signature layers.
//
// ELDR, section "Key idea / structure / operation": the prefill hook records
// the request's expert signature at KV-block granularity -- for each block
// and each layer of the selected mask, how many of the block's tokens picked
// each expert in their top-k.
//
// A segmented histogram over the block table: one warp per (KV block, mask
// layer) pair reads the block's top-k ids (contiguous uint8, len * k bytes),
// counts them into a private shared-memory row of packed 8-bit counters (four
// experts per 32-bit word; a count never exceeds B <= 255) and writes the row
// out with coalesced 32-bit stores.  No global atomics, no pre-zeroing.  The
// block table is validated on the fly: a block whose length is outside
// [1, B], that runs past T or that does not start where the previous block
// ends is skipped and recorded as MOER_EDATA.
#include "common.cuh"

namespace moer {

constexpr int BC_WARPS = 8;

struct BcParams {
  const uint8_t* ids;     // top-k ids
  int64_t layer_stride;   // T * k
  int64_t T;
  int k, E, B, m, nblk;
  const int32_t* blk_tab;
  uint8_t* blk_cnt;
  uint32_t* status;
  int16_t layer_row[256];  // ids row-block of mask layer i
};

__global__ void __launch_bounds__(BC_WARPS * 32) block_counts_kernel(const __grid_constant__ BcParams p) {
  extern __shared__ uint32_t bc_smem[];  // [BC_WARPS][E / 4]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpb = p.E / 4;
  uint32_t* cnt = bc_smem + warp * wpb;
  const int64_t pair = (int64_t)blockIdx.x * BC_WARPS + warp;
  if (pair >= (int64_t)p.nblk * p.m) return;
  const int b = (int)(pair / p.m), i = (int)(pair - (int64_t)b * p.m);
  const int t0 = p.blk_tab[2 * b], ln = p.blk_tab[2 * b + 1];
  bool ok = ln >= 1 && ln <= p.B && t0 >= 0 && (int64_t)t0 + ln <= p.T;
  if (b == 0) {
    ok = ok && t0 == 0;
  } else {
    const int pt0 = p.blk_tab[2 * (b - 1)], pln = p.blk_tab[2 * (b - 1) + 1];
    ok = ok && (int64_t)pt0 + pln == (int64_t)t0;
  }
  if (b == p.nblk - 1) ok = ok && (int64_t)t0 + ln == p.T;
  if (!ok) {
    if (lane == 0 && i == 0) atomicOr(p.status, WS_BIT_EDATA);
    return;
  }
  for (int w = lane; w < wpb; w += 32) cnt[w] = 0u;
  __syncwarp();
  const uint8_t* src = p.ids + (int64_t)p.layer_row[i] * p.layer_stride + (int64_t)t0 * p.k;
  const int n = ln * p.k;
  for (int j = lane; j < n; j += 32) {
    const int e = src[j];
    atomicAdd(&cnt[e >> 2], 1u << ((e & 3) * 8));
  }
  __syncwarp();
  uint32_t* dst = reinterpret_cast<uint32_t*>(p.blk_cnt + ((size_t)b * p.m + i) * p.E);
  for (int w = lane; w < wpb; w += 32) dst[w] = cnt[w];
}

// ids: either the caller's [L][T][k] top-k (mask_only = false: row block of
// mask layer i is mask[i]) or a mask-only [m][T][k] buffer (row block i).
moer_status block_counts_launch(const moer_dims* d, const uint8_t* ids, bool mask_only, int64_t T,
                                const int32_t* blk_tab, int nblk, uint8_t* blk_cnt, uint32_t* status,
                                cudaStream_t st) {
  BcParams p;
  p.ids = ids;
  p.layer_stride = T * d->k;
  p.T = T;
  p.k = d->k;
  p.E = d->E;
  p.B = d->block;
  p.m = d->m;
  p.nblk = nblk;
  p.blk_tab = blk_tab;
  p.blk_cnt = blk_cnt;
  p.status = status;
  for (int i = 0; i < 256; ++i) p.layer_row[i] = 0;
  for (int i = 0; i < d->m; ++i) p.layer_row[i] = (int16_t)(mask_only ? i : d->mask[i]);
  const int64_t pairs = (int64_t)nblk * d->m;
  const int64_t grid = (pairs + BC_WARPS - 1) / BC_WARPS;
  if (grid <= 0) return MOER_OK;
  block_counts_kernel<<<(unsigned)grid, BC_WARPS * 32, BC_WARPS * (d->E / 4) * sizeof(uint32_t), st>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer

namespace moer {

// Per-layer co-activation counts from top-k ids (the gate path, where the ids
// come out of the GEMM epilogue rather than from a logits pass).  GRACE-MoE,
// section 3 and section 4 / Figure 2(a): A_l[a][b] += #tokens whose top-k
// at layer l holds both a and b.  Persistent grid over (layer, 512-token
// chunk) items in layer-major order; each CTA accumulates into a shared
// E x (E+1) tile and flushes it (atomic adds) when its layer changes.
constexpr int AI_CHUNK = 512;
constexpr int AI_THREADS = 256;

__global__ void __launch_bounds__(AI_THREADS) affinity_ids_kernel(const uint8_t* __restrict__ ids, int64_t T,
                                                                  int k, int E, int L, int nchunks,
                                                                  int32_t* __restrict__ affinity) {
  extern __shared__ int ai_tile[];  // [E][E+1]
  const int stride = E + 1;
  const int64_t nitems = (int64_t)L * nchunks;
  const int64_t i0 = (int64_t)blockIdx.x * nitems / gridDim.x;
  const int64_t i1 = ((int64_t)blockIdx.x + 1) * nitems / gridDim.x;
  for (int c = threadIdx.x; c < E * stride; c += AI_THREADS) ai_tile[c] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane >> 3, j = lane & 7;  // four rows per warp step, eight id lanes per row
  int cur = (int)(i0 / nchunks);
  for (int64_t it = i0; it < i1; ++it) {
    const int l = (int)(it / nchunks);
    if (l != cur) {
      __syncthreads();
      for (int c = threadIdx.x; c < E * E; c += AI_THREADS) {
        const int a = c / E, b = c - a * E;
        const int v = ai_tile[a * stride + b];
        if (v != 0) {
          atomicAdd(&affinity[(size_t)cur * E * E + c], v);
          ai_tile[a * stride + b] = 0;
        }
      }
      __syncthreads();
      cur = l;
    }
    const int64_t tb = (it - (int64_t)l * nchunks) * AI_CHUNK;
    for (int r = warp * 4; r < AI_CHUNK; r += (AI_THREADS / 32) * 4) {
      const int64_t t = tb + r + sub;
      const bool ok = t < T && j < k;
      const int e = ok ? ids[((size_t)l * T + t) * k + j] : 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int eb = __shfl_sync(FULL, e, (lane & ~7) | b);
        if (ok && b < k) atomicAdd(&ai_tile[e * stride + eb], 1);
      }
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < E * E; c += AI_THREADS) {
    const int a = c / E, b = c - a * E;
    const int v = ai_tile[a * stride + b];
    if (v != 0) atomicAdd(&affinity[(size_t)cur * E * E + c], v);
  }
}

moer_status affinity_ids_launch(const moer_dims* d, const uint8_t* ids, int64_t T, int32_t* affinity,
                                cudaStream_t st) {
  const int nchunks = (int)((T + AI_CHUNK - 1) / AI_CHUNK);
  const int64_t nitems = (int64_t)d->L * nchunks;
  const int sms = device_sm_count();
  if (sms <= 0) return MOER_ECUDA;
  const size_t smem = (size_t)d->E * (d->E + 1) * sizeof(int);
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(affinity_ids_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(129 * 128 * 4)) !=
        cudaSuccess)
      return MOER_ECUDA;
    configured = true;
  }
  const int grid = (int)min64(nitems, (int64_t)sms * 2);
  affinity_ids_kernel<<<grid, AI_THREADS, smem, st>>>(ids, T, d->k, d->E, d->L, nchunks, affinity);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
