// block_counts.cu -- per-KV-block expert counts over the signature layers.
//
// ELDR, section "Key idea / structure / operation": the prefill hook records
// the request's expert signature at KV-block granularity -- for each block
// and each layer of the selected mask, how many of the block's tokens picked
// each expert in their top-k.
//
// A segmented histogram over the block table: a persistent grid of warps walks
// the KV blocks; per block the warp reads the block's top-k ids of up to sixteen
// mask layers at once (contiguous uint8, len * k bytes per layer, as 4-byte
// words when k is a multiple of 4), counts them into private shared-memory
// rows of packed 8-bit counters (four
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

constexpr int BC_MC = 16;  // mask layers counted together (their loads in flight at once)

// CHECK: the ids come from the caller (moer_ids_signature); an id >= E is
// skipped and recorded as MOER_EDATA instead of being counted.
template <bool CHECK>
__global__ void __launch_bounds__(BC_WARPS * 32) block_counts_kernel(const __grid_constant__ BcParams p) {
  extern __shared__ uint32_t bc_smem[];  // [BC_WARPS][BC_MC][E / 4]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpb = p.E / 4;
  uint32_t* cnt = bc_smem + warp * BC_MC * wpb;
  const int64_t stride = (int64_t)gridDim.x * BC_WARPS;
  // 4-byte loads when every block's id row starts on a 4-byte boundary
  const bool vec = (p.k % 4) == 0;
  // persistent warps, one KV block at a time, all mask layers of the block
  for (int64_t bb = (int64_t)blockIdx.x * BC_WARPS + warp; bb < p.nblk; bb += stride) {
    const int b = (int)bb;
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
      if (lane == 0) atomicOr(p.status, WS_BIT_EDATA);
      continue;
    }
    const int n = ln * p.k;
    for (int i0 = 0; i0 < p.m; i0 += BC_MC) {
      const int nl = min(BC_MC, p.m - i0);
      for (int w = lane; w < nl * wpb; w += 32) cnt[w] = 0u;
      __syncwarp();
      if (vec) {
        const int nw = n >> 2;
        for (int q0 = 0; q0 < nw; q0 += 32) {
          const int q = q0 + lane;
          uint32_t v[BC_MC];
#pragma unroll
          for (int ii = 0; ii < BC_MC; ++ii) {
            v[ii] = 0u;
            if (ii < nl && q < nw) {
              const uint8_t* src = p.ids + (int64_t)p.layer_row[i0 + ii] * p.layer_stride + (int64_t)t0 * p.k;
              v[ii] = reinterpret_cast<const uint32_t*>(src)[q];
            }
          }
#pragma unroll
          for (int ii = 0; ii < BC_MC; ++ii) {
            if (ii < nl && q < nw) {
              uint32_t* c = cnt + ii * wpb;
#pragma unroll
              for (int by = 0; by < 4; ++by) {
                const int e = (v[ii] >> (8 * by)) & 0xFF;
                if (CHECK && e >= p.E) {
                  atomicOr(p.status, WS_BIT_EDATA);
                  continue;
                }
                atomicAdd(&c[e >> 2], 1u << ((e & 3) * 8));
              }
            }
          }
        }
      } else {
        for (int ii = 0; ii < nl; ++ii) {
          const uint8_t* src = p.ids + (int64_t)p.layer_row[i0 + ii] * p.layer_stride + (int64_t)t0 * p.k;
          uint32_t* c = cnt + ii * wpb;
          for (int j = lane; j < n; j += 32) {
            const int e = src[j];
            if (CHECK && e >= p.E) {
              atomicOr(p.status, WS_BIT_EDATA);
              continue;
            }
            atomicAdd(&c[e >> 2], 1u << ((e & 3) * 8));
          }
        }
      }
      __syncwarp();
      for (int ii = 0; ii < nl; ++ii) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.blk_cnt + ((size_t)b * p.m + i0 + ii) * p.E);
        for (int w = lane; w < wpb; w += 32) dst[w] = cnt[ii * wpb + w];
      }
      __syncwarp();
    }
  }
}

// ids: either the caller's [L][T][k] top-k (mask_only = false: row block of
// mask layer i is mask[i]) or a mask-only [m][T][k] buffer (row block i).
// check: ids from outside the library, bounded by E as they are read.
moer_status block_counts_launch(const moer_dims* d, const uint8_t* ids, bool mask_only, int64_t T,
                                const int32_t* blk_tab, int nblk, uint8_t* blk_cnt, uint32_t* status,
                                cudaStream_t st, bool check) {
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
  if (nblk <= 0 || d->m <= 0) return MOER_OK;
  const int sms = device_sm_count();
  if (sms <= 0) return MOER_ECUDA;
  const int64_t grid = min64(((int64_t)nblk + BC_WARPS - 1) / BC_WARPS, (int64_t)sms * 8);
  const size_t smem = BC_WARPS * BC_MC * (d->E / 4) * sizeof(uint32_t);
  if (check)
    block_counts_kernel<true><<<(unsigned)grid, BC_WARPS * 32, smem, st>>>(p);
  else
    block_counts_kernel<false><<<(unsigned)grid, BC_WARPS * 32, smem, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer

namespace moer {

// Per-layer co-activation counts from top-k ids (the gate path, where the ids
// come out of the GEMM epilogue rather than from a logits pass).  GRACE-MoE,
// section 3 and section 4 / Figure 2(a): A_l[a][b] += #tokens whose top-k
// at layer l holds both a and b.
//
// Persistent grid over (layer, 2048-token chunk) items in layer-major order,
// four token rows per thread with their id loads issued together.  A row's k
// distinct ids, in rank order, add its k(k-1)/2 rank-ordered pairs to a
// shared tile of directed counts D[a][b] (= # rows where a ranks above b).  When the CTA's layer changes
// the tile is folded into the symmetric co-activation -- A[a][b] = D[a][b] +
// D[b][a] off the diagonal, and A[a][a] = (sum over b != a of A[a][b]) /
// (k - 1), since each row holding a holds k - 1 other experts -- and added to
// global memory.  Needs k >= 2.
constexpr int AI_THREADS = 512;
constexpr int AI_U = 4;                      // tokens per thread per item, loads in flight together
constexpr int AI_CHUNK = AI_THREADS * AI_U;  // tokens per work item

// The tile's rows are E + 1 words apart, so the bank of D[a][b] depends on a
// as well as b.
__device__ void affinity_ids_flush(int* tile, int* rsum, int E, int k, int32_t* dst) {
  const int rs = E + 1;
  for (int c = threadIdx.x; c < E * E; c += AI_THREADS) {
    const int a = c / E, b = c - a * E;
    if (a < b) {
      const int v = tile[a * rs + b] + tile[b * rs + a];
      if (v != 0) {
        atomicAdd(&dst[a * E + b], v);
        atomicAdd(&dst[b * E + a], v);
        atomicAdd(&rsum[a], v);
        atomicAdd(&rsum[b], v);
      }
    }
  }
  __syncthreads();
  for (int a = threadIdx.x; a < E; a += AI_THREADS) {
    const int v = rsum[a];
    if (v != 0) {
      atomicAdd(&dst[a * E + a], v / (k - 1));
      rsum[a] = 0;
    }
  }
  for (int c = threadIdx.x; c < E * rs; c += AI_THREADS) tile[c] = 0;
  __syncthreads();
}

// CHECK: the ids come from the caller (moer_ids_signature); a row holding an
// id >= E or a repeated id is left out (the diagonal needs k distinct ids)
// and recorded as MOER_EDATA.
template <int K, bool CHECK>
__global__ void __launch_bounds__(AI_THREADS) affinity_ids_kernel(const uint8_t* __restrict__ ids, int64_t T,
                                                                  int E, int L, int nchunks,
                                                                  int32_t* __restrict__ affinity,
                                                                  uint32_t* status) {
  extern __shared__ int ai_tile[];  // [E][E + 1] directed counts, then [E] row sums
  const int rs = E + 1;
  int* rsum = ai_tile + E * rs;
  const uint32_t tile_base = smem_u32(ai_tile);
  const uint32_t row_bytes = (uint32_t)rs * 4u;
  const int64_t nitems = (int64_t)L * nchunks;
  const int64_t i0 = (int64_t)blockIdx.x * nitems / gridDim.x;
  const int64_t i1 = ((int64_t)blockIdx.x + 1) * nitems / gridDim.x;
  for (int c = threadIdx.x; c < E * rs + E; c += AI_THREADS) ai_tile[c] = 0;
  __syncthreads();
  int cur = (int)(i0 / nchunks);
  for (int64_t it = i0; it < i1; ++it) {
    const int l = (int)(it / nchunks);
    if (l != cur) {
      __syncthreads();
      affinity_ids_flush(ai_tile, rsum, E, K, affinity + (size_t)cur * E * E);
      cur = l;
    }
    const int64_t tb = (it - (int64_t)l * nchunks) * AI_CHUNK + threadIdx.x;
    const uint8_t* lay = ids + (size_t)l * T * K;
    uint32_t w[AI_U][(K + 3) / 4];
#pragma unroll
    for (int u = 0; u < AI_U; ++u) {
      const int64_t t = tb + (int64_t)u * AI_THREADS;
      if (t < T) {
        if constexpr (K == 8) {
          const uint2 v = *reinterpret_cast<const uint2*>(lay + (size_t)t * 8);
          w[u][0] = v.x;
          w[u][1] = v.y;
        } else {
          const uint8_t* src = lay + (size_t)t * K;
#pragma unroll
          for (int j = 0; j < K; j += 2) {
            const uint32_t h = *reinterpret_cast<const uint16_t*>(src + j);
            if (j % 4 == 0)
              w[u][j / 4] = h;
            else
              w[u][j / 4] |= h << 16;
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < AI_U; ++u) {
      if (tb + (int64_t)u * AI_THREADS < T) {
        int e[K];
#pragma unroll
        for (int j = 0; j < K; ++j) e[j] = (w[u][j / 4] >> (8 * (j % 4))) & 0xFF;
        if constexpr (CHECK) {
          // K distinct ids below E: their bits in a 256-bit set number exactly K
          unsigned long long m0 = 0, m1 = 0, m2 = 0, m3 = 0;
          bool inrange = true;
#pragma unroll
          for (int j = 0; j < K; ++j) {
            inrange = inrange && e[j] < E;
            const unsigned long long bit = 1ull << (e[j] & 63);
            const int q = e[j] >> 6;
            m0 |= q == 0 ? bit : 0ull;
            m1 |= q == 1 ? bit : 0ull;
            m2 |= q == 2 ? bit : 0ull;
            m3 |= q == 3 ? bit : 0ull;
          }
          if (!inrange || __popcll(m0) + __popcll(m1) + __popcll(m2) + __popcll(m3) != K) {
            atomicOr(status, WS_BIT_EDATA);
            continue;
          }
        }
        // shared address of D[a][b] = tile + 4 b + a * row pitch: one
        // multiply-add per pair (FMA pipe) rather than integer-ALU adds
        uint32_t colb[K];
#pragma unroll
        for (int j = 1; j < K; ++j) colb[j] = tile_base + 4u * (uint32_t)e[j];
#pragma unroll
        for (int i = 0; i < K - 1; ++i) {
#pragma unroll
          for (int j = i + 1; j < K; ++j) {
            uint32_t addr;
            asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(addr) : "r"((uint32_t)e[i]), "r"(row_bytes), "r"(colb[j]));
            asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(addr) : "memory");
          }
        }
      }
    }
  }
  __syncthreads();
  affinity_ids_flush(ai_tile, rsum, E, K, affinity + (size_t)cur * E * E);
}

// ids [L][T][k] (k = 6 or 8, 8-byte aligned rows for k = 8) -> affinity
// [L][E][E] accumulated.
moer_status affinity_ids_launch(const moer_dims* d, const uint8_t* ids, int64_t T, int32_t* affinity,
                                cudaStream_t st, uint32_t* status, bool check) {
  if (d->k != 8 && d->k != 6) return MOER_ERANGE;
  if (d->E > 128) return MOER_ERANGE;
  const int nchunks = (int)((T + AI_CHUNK - 1) / AI_CHUNK);
  const int64_t nitems = (int64_t)d->L * nchunks;
  const int sms = device_sm_count();
  if (sms <= 0) return MOER_ECUDA;
  const size_t smem = ((size_t)d->E * (d->E + 1) + d->E) * sizeof(int);
  static std::atomic<unsigned long long> set8{0}, set6{0}, set8c{0}, set6c{0};
  const int most = (int)((128 * 129 + 128) * sizeof(int));
  if (smem_optin(affinity_ids_kernel<8, false>, most, set8) != cudaSuccess ||
      smem_optin(affinity_ids_kernel<6, false>, most, set6) != cudaSuccess ||
      smem_optin(affinity_ids_kernel<8, true>, most, set8c) != cudaSuccess ||
      smem_optin(affinity_ids_kernel<6, true>, most, set6c) != cudaSuccess)
    return MOER_ECUDA;
  const int grid = (int)min64(nitems, (int64_t)sms * 2);
  if (d->k == 8 && !check)
    affinity_ids_kernel<8, false><<<grid, AI_THREADS, smem, st>>>(ids, T, d->E, d->L, nchunks, affinity, status);
  else if (d->k == 8)
    affinity_ids_kernel<8, true><<<grid, AI_THREADS, smem, st>>>(ids, T, d->E, d->L, nchunks, affinity, status);
  else if (!check)
    affinity_ids_kernel<6, false><<<grid, AI_THREADS, smem, st>>>(ids, T, d->E, d->L, nchunks, affinity, status);
  else
    affinity_ids_kernel<6, true><<<grid, AI_THREADS, smem, st>>>(ids, T, d->E, d->L, nchunks, affinity, status);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
