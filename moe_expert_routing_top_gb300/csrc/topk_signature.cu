// topk_signature.cu -- fused top-k gating, per-KV-block signature counts and
// per-layer expert co-activation, one pass over the router logits.
//
// What it computes:
//   ELDR (Expert-Locality-Aware Decode Routing), section "What it tries to
//   solve": every MoE token selects its own top-k experts; section "Key idea /
//   structure / operation": the standard top-k gate is left unchanged and the
//   prefill hook records discrete top-k counts per KV block over the selected
//   layer mask.  GRACE-MoE, section 3 "Key observations" and section 4
//   "Method" / Figure 2(a): expert selections are profiled layer by layer
//   into a co-activation (affinity) matrix whose diagonal is the expert load.
//
// Design (GB300):
//   * Persistent grid, one 544-thread CTA per SM.  Work items are
//     (layer, token tile) pairs in layer-major order; each CTA takes a
//     contiguous range, so its affinity tile spans at most a few layers.
//   * One producer warp streams each tile of logit rows (TT rows x E fp32,
//     contiguous in HBM) into shared memory with a single cp.async.bulk copy
//     completing on an mbarrier; 3-4 stages keep 64-96 KB per SM in flight.
//     It also builds the tile's token -> local KV block map and, when
//     consumers release a stage, writes that tile's block counts out.
//   * Sixteen consumer warps take one row each per step (warp per row).
//     Fast path (E = 64 or 128, k = 6 or 8): each lane forms 32-bit keys
//     from its logits (upper 24 bits of the float, lower 8 bits = 255 - e)
//     so every key is unique and carries its expert id; a lane pre-sorts its
//     top 3 keys and k rounds of redux.sync.max pop one winner each.  The
//     result is checked for exactness (all k+1 leading keys distinct in their
//     upper bits, all positive and finite); otherwise the row is redone by an
//     exact path on order-preserving 32-bit keys with ballot tie-breaking to
//     the lower expert id (also used for every other E and k).
//   * Co-activation pairs go to a shared-memory E x (E+1) int32 tile with
//     shared atomics, flushed to global memory (atomic adds) when the CTA's
//     layer changes.  Block counts use packed 8-bit counters in shared memory
//     (four experts per 32-bit word; counts never exceed B <= 255).
//   * Tiles are fixed TT-token ranges; KV blocks that straddle two tiles are
//     zeroed by the tile-index pre-pass and accumulated with atomic adds,
//     blocks inside one tile are written with plain stores.
#include <climits>

#include "common.cuh"
#include "k1_params.cuh"

namespace moer {

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <int EPL>
struct K1Geo {
  static constexpr int EMAX = 32 * EPL;
  static constexpr int TT = (EPL <= 2) ? 128 : (EPL == 4 ? 64 : 32);
  static constexpr int STAGES = (EPL == 4) ? 3 : 4;
  static constexpr bool SMEM_AFF = EPL <= 4;
  static constexpr int CWARPS = 16;
  static constexpr int NR = 4;  // rows a consumer warp works on at once
  static constexpr int CTHREADS = CWARPS * 32;
  static constexpr int THREADS = CTHREADS + 32;
  static constexpr size_t STAGE_BYTES = (size_t)TT * EMAX * 4;
  static constexpr size_t CNT_WORDS = (size_t)TT * EMAX / 4;
  static constexpr size_t OFF_ROWS = 0;
  static constexpr size_t OFF_CNT = OFF_ROWS + STAGES * STAGE_BYTES;
  static constexpr size_t OFF_MAP = OFF_CNT + STAGES * CNT_WORDS * 4;
  static constexpr size_t OFF_AFF = align_up(OFF_MAP + (size_t)STAGES * TT, 16);
  static constexpr size_t AFF_WORDS = SMEM_AFF ? (size_t)EMAX * (EMAX + 1) : 0;
  static constexpr size_t OFF_WSCR = align_up(OFF_AFF + AFF_WORDS * 4, 16);
  static constexpr size_t OFF_META = OFF_WSCR + (size_t)CWARPS * NR * 16 * 4;
  static constexpr size_t OFF_BAR = align_up(OFF_META + (size_t)STAGES * 8 * 4, 16);
  static constexpr size_t SMEM = OFF_BAR + 2 * STAGES * 8;
};

struct K1Params {
  const float* logits;
  int64_t T;
  int E, k, L, m, B;
  const int32_t* blk_tab;
  int nblk;
  uint8_t* topk;
  uint8_t* blk_cnt;
  int32_t* affinity;
  const int32_t* tile_blk0;
  int ntiles;
  int64_t nitems;
  uint32_t* status;     // sticky status word
  uint32_t* call_flag;  // validation result of this call's pre-pass
  int16_t slot_of_layer[256];
};

int k1_tile_tokens(int E) {
  if (E <= 64) return K1Geo<2>::TT;
  if (E <= 128) return K1Geo<4>::TT;
  return K1Geo<8>::TT;
}

// Workspace after the header: a per-tile table sized for the smallest tile
// (32 tokens), then one block id per token.
size_t k1_scratch_bytes(int64_t T) {
  const size_t tiles = (size_t)((T + 31) / 32) * sizeof(int32_t);
  return (tiles + 255) / 256 * 256 + ((size_t)T * sizeof(int32_t) + 255) / 256 * 256;
}



// ---------------------------------------------------------------- pre-pass
// Validates the block table, records each tile's first block (warp-per-row
// kernel) or each token's block (thread-per-row kernel), and zeroes the count
// rows of blocks that straddle a tile boundary.
__global__ void k1_tile_index(const int32_t* __restrict__ blk_tab, int nblk, int64_t T, int B,
                              int TT, int32_t* __restrict__ tile_blk0, int32_t* __restrict__ tok_blk,
                              uint32_t* status, uint32_t* call_flag, uint8_t* __restrict__ blk_cnt,
                              int m, int E) {
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += gridDim.x * blockDim.x) {
    const int t0 = blk_tab[2 * b], ln = blk_tab[2 * b + 1];
    bool ok = ln >= 1 && ln <= B && t0 >= 0 && (int64_t)t0 + ln <= T;
    if (b == 0) {
      ok = ok && t0 == 0;
    } else {
      const int pt0 = blk_tab[2 * (b - 1)], pln = blk_tab[2 * (b - 1) + 1];
      ok = ok && (int64_t)pt0 + pln == (int64_t)t0;
    }
    if (b == nblk - 1) ok = ok && (int64_t)t0 + ln == T;
    if (!ok) {
      atomicOr(status, WS_BIT_EDATA);
      atomicOr(call_flag, 1u);
      continue;
    }
    if (tile_blk0 != nullptr)
      for (int64_t j = ((int64_t)t0 + TT - 1) / TT; j * TT < (int64_t)t0 + ln; ++j) tile_blk0[j] = b;
    if (tok_blk != nullptr)
      for (int t = t0; t < t0 + ln; ++t) tok_blk[t] = b;
    if (blk_cnt != nullptr && m > 0 && (t0 / TT) != ((t0 + ln - 1) / TT)) {
      uint32_t* row = reinterpret_cast<uint32_t*>(blk_cnt + (size_t)b * m * E);
      for (int w = 0; w < m * E / 4; ++w) row[w] = 0u;
    }
  }
}

// ----------------------------------------------------------- row selection
// Order-preserving 32-bit key of the ranking: NaN lowest (above only the
// "removed" key 0), -0.0 equal to +0.0, otherwise by value.
__device__ __forceinline__ uint32_t rank_key(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 1u;
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exact top-k of one row held in shared memory, any E <= 32*EPL, k <= 32.
// Lane owns experts [lane*EPL, lane*EPL+EPL).  Returns, in lane r < k, the
// id ranked r-th; -1 in other lanes.
template <int EPL>
__device__ int topk_exact(const float* row, int E, int k, int lane) {
  uint32_t key[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane * EPL + j;
    key[j] = e < E ? rank_key(row[e]) : 0u;
  }
  int myidx = -1;
  for (int r = 0; r < k; ++r) {
    uint32_t best = 0u;
    int bj = 0;
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (key[j] > best) {
        best = key[j];
        bj = j;
      }
    const uint32_t M = __reduce_max_sync(FULL, best);
    const unsigned bal = __ballot_sync(FULL, best == M);
    const int w = __ffs(bal) - 1;
    const int e = __shfl_sync(FULL, lane * EPL + bj, w);
    if (lane == w) {
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (j == bj) key[j] = 0u;
    }
    if (lane == r) myidx = e;
  }
  return myidx;
}

// Fast top-K of NR rows at once (E == 32*EPL, EPL 2 or 4, K <= 8).  The NR
// rows are independent, so their redux chains interleave and hide each
// other's latency.  Keys: upper 24 bits of the float's bit pattern (as a
// signed int: exact order among positive floats), lower 8 bits 255 - e, so
// keys are unique and carry the expert id.  Row q's result is certified when
// its k+1 leading keys are positive, finite and pairwise distinct in their
// upper 24 bits; otherwise bit q of the returned mask is set and the caller
// redoes that row exactly.  Every lane writes the same winners to scr, so
// each lane reads back values it wrote itself (no warp barrier needed).
template <int EPL, int K, int NR>
__device__ __forceinline__ unsigned topk_fast_rows(const float* const (&rowp)[NR], int lane, int* scr,
                                                   int (&myidx)[NR]) {
  static_assert(EPL == 2 || EPL == 4, "fast path needs 2 or 4 experts per lane");
  static_assert(K >= 1 && K <= 8, "fast path needs k <= 8");
  int h[NR], s1[NR], s2[NR];
#pragma unroll
  for (int q = 0; q < NR; ++q) {
    int key[EPL];
    if constexpr (EPL == 4) {
      const float4 v = reinterpret_cast<const float4*>(rowp[q])[lane];
      key[0] = __float_as_int(v.x);
      key[1] = __float_as_int(v.y);
      key[2] = __float_as_int(v.z);
      key[3] = __float_as_int(v.w);
    } else {
      const float2 v = reinterpret_cast<const float2*>(rowp[q])[lane];
      key[0] = __float_as_int(v.x);
      key[1] = __float_as_int(v.y);
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j) key[j] = (key[j] & (int)0xFFFFFF00) | (255 - (lane * EPL + j));
    if constexpr (EPL == 4) {
      const int a = max(key[0], key[1]), b = min(key[0], key[1]);
      const int c = max(key[2], key[3]), d = min(key[2], key[3]);
      h[q] = max(a, c);
      const int x = min(a, c), y = max(b, d);
      s1[q] = max(x, y);
      s2[q] = max(min(x, y), min(b, d));
    } else {
      h[q] = max(key[0], key[1]);
      s1[q] = min(key[0], key[1]);
      s2[q] = INT_MIN;
    }
  }
#pragma unroll
  for (int r = 0; r < K; ++r) {
#pragma unroll
    for (int q = 0; q < NR; ++q) {
      const int M = __reduce_max_sync(FULL, h[q]);
      const bool p = (h[q] == M);
      h[q] = p ? s1[q] : h[q];
      s1[q] = p ? INT_MIN : s1[q];
      scr[q * 16 + r] = M;
    }
  }
#pragma unroll
  for (int q = 0; q < NR; ++q) scr[q * 16 + K] = __reduce_max_sync(FULL, max(h[q], s2[q]));
  unsigned badmask = 0u;
#pragma unroll
  for (int q = 0; q < NR; ++q) {
    const int Mr = scr[q * 16 + min(lane, K)];
    const int Mn = scr[q * 16 + min(lane + 1, K)];
    bool bad = (lane < K) && ((Mn >= (Mr & (int)0xFFFFFF00)) || (Mr < 256));
    bad = bad || (lane == 0 && Mr >= 0x7F800000);
    if (__any_sync(FULL, bad)) badmask |= 1u << q;
    myidx[q] = (lane < K) ? (255 - (Mr & 0xFF)) : -1;
  }
  return badmask;
}

// ------------------------------------------------------- co-activation adds
template <int KK>
__device__ __forceinline__ void aff_pairs_fixed(int* aff, int stride, int myidx, int lane) {
  constexpr int P = KK * KK;
#pragma unroll
  for (int base = 0; base < P; base += 32) {
    const int q = base + lane;
    const int a = q < P ? q / KK : 0;
    const int b = q < P ? q % KK : 0;
    const int ia = __shfl_sync(FULL, myidx, a);
    const int ib = __shfl_sync(FULL, myidx, b);
    if (q < P) atomicAdd(&aff[ia * stride + ib], 1);
  }
}

__device__ __forceinline__ void aff_pairs_any(int* aff, int stride, int myidx, int k, int lane) {
  const int P = k * k;
  for (int base = 0; base < P; base += 32) {
    const int q = base + lane;
    const int a = q < P ? q / k : 0;
    const int b = q < P ? q - (q / k) * k : 0;
    const int ia = __shfl_sync(FULL, myidx, a);
    const int ib = __shfl_sync(FULL, myidx, b);
    if (q < P) atomicAdd(&aff[ia * stride + ib], 1);
  }
}

// ---------------------------------------------------------------- producer
template <int EPL>
__device__ void k1_flush_counts(const K1Params& p, const int* meta, uint32_t* cnt, int lane) {
  using G = K1Geo<EPL>;
  const int slot = meta[3], nb = meta[5];
  if (slot < 0 || p.blk_cnt == nullptr || nb == 0) return;
  const int tile = meta[1], ntok = meta[2], blk0 = meta[4];
  const int64_t tok0 = (int64_t)tile * G::TT;
  const int wpb = p.E / 4;
  for (int j = 0; j < nb; ++j) {
    const int b = blk0 + j;
    const int t0 = p.blk_tab[2 * b], ln = p.blk_tab[2 * b + 1];
    const bool inside = t0 >= tok0 && (int64_t)t0 + ln <= tok0 + ntok;
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.blk_cnt + ((size_t)b * p.m + slot) * p.E);
    uint32_t* src = cnt + (size_t)j * wpb;
    for (int w = lane; w < wpb; w += 32) {
      const uint32_t v = src[w];
      if (inside)
        dst[w] = v;
      else if (v != 0u)
        atomicAdd(&dst[w], v);
      src[w] = 0u;
    }
  }
}

template <int EPL>
__device__ void k1_producer(const K1Params& p, char* smem, int64_t i0, int64_t i1) {
  using G = K1Geo<EPL>;
  const int lane = threadIdx.x & 31;
  float* rows = reinterpret_cast<float*>(smem + G::OFF_ROWS);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + G::OFF_CNT);
  uint8_t* map = reinterpret_cast<uint8_t*>(smem + G::OFF_MAP);
  int* meta = reinterpret_cast<int*>(smem + G::OFF_META);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  uint64_t* empty = full + G::STAGES;
  const bool hist = p.blk_cnt != nullptr && p.m > 0;
  int64_t issued = 0;
  bool ok = true;
  for (int64_t it = i0; it < i1; ++it) {
    const int64_t n = it - i0;
    const int s = (int)(n % G::STAGES);
    if (n >= G::STAGES) {
      if (!mbar_wait(&empty[s], (uint32_t)((n / G::STAGES - 1) & 1), p.status)) {
        ok = false;
        break;
      }
      k1_flush_counts<EPL>(p, meta + s * 8, cnt + (size_t)s * G::CNT_WORDS, lane);
      __syncwarp();
    }
    const int l = (int)(it / p.ntiles);
    const int tile = (int)(it - (int64_t)l * p.ntiles);
    const int64_t tok0 = (int64_t)tile * G::TT;
    const int ntok = (int)min64(G::TT, p.T - tok0);
    const int slot = p.slot_of_layer[l];
    int blk0 = 0, nb = 0;
    if (slot >= 0 && hist) {
      blk0 = p.tile_blk0[tile];
      for (int base = 0; base < G::TT; base += 32) {
        const int j = base + lane;
        const int b = blk0 + j;
        bool in = false;
        int t0 = 0, ln = 0;
        if (j < G::TT && b < p.nblk) {
          t0 = p.blk_tab[2 * b];
          ln = p.blk_tab[2 * b + 1];
          in = (int64_t)t0 < tok0 + ntok;
        }
        if (in) {
          const int64_t a = max64((int64_t)t0, tok0);
          const int64_t e = min64((int64_t)t0 + ln, tok0 + ntok);
          for (int64_t t = a; t < e; ++t) map[s * G::TT + (int)(t - tok0)] = (uint8_t)j;
        }
        const unsigned bal = __ballot_sync(FULL, in);
        nb += __popc(bal);
        if (bal != FULL) break;
      }
    }
    if (lane == 0) {
      int* mt = meta + s * 8;
      mt[0] = l;
      mt[1] = tile;
      mt[2] = ntok;
      mt[3] = hist ? slot : -1;
      mt[4] = blk0;
      mt[5] = nb;
    }
    __syncwarp();
    if (lane == 0) {
      const uint32_t bytes = (uint32_t)ntok * (uint32_t)p.E * 4u;
      mbar_arrive_expect_tx(&full[s], bytes);
      bulk_g2s(rows + (size_t)s * G::TT * G::EMAX, p.logits + ((size_t)l * p.T + tok0) * p.E, bytes,
               &full[s]);
    } else {
      mbar_arrive(&full[s]);
    }
    ++issued;
  }
  const int64_t first = issued > G::STAGES ? issued - G::STAGES : 0;
  for (int64_t n = first; n < issued; ++n) {
    const int s = (int)(n % G::STAGES);
    if (ok) {
      if (!mbar_wait(&empty[s], (uint32_t)((n / G::STAGES) & 1), p.status)) {
        ok = false;
      } else {
        k1_flush_counts<EPL>(p, meta + s * 8, cnt + (size_t)s * G::CNT_WORDS, lane);
        __syncwarp();
        continue;
      }
    }
    // error path: make sure no bulk copy into this CTA's shared memory is in flight
    mbar_wait(&full[s], (uint32_t)((n / G::STAGES) & 1), p.status);
  }
}

// --------------------------------------------------------------- consumers
template <int EPL>
__device__ void k1_flush_aff(const K1Params& p, int* aff, int layer, int ctid) {
  const int E = p.E, stride = E + 1;
  int32_t* dst = p.affinity + (size_t)layer * E * E;
  for (int c = ctid; c < E * E; c += K1Geo<EPL>::CTHREADS) {
    const int a = c / E, b = c - a * E;
    const int v = aff[a * stride + b];
    if (v != 0) {
      atomicAdd(&dst[c], v);
      aff[a * stride + b] = 0;
    }
  }
}

template <int EPL, int FASTK>
__device__ void k1_consumer(const K1Params& p, char* smem, int64_t i0, int64_t i1) {
  using G = K1Geo<EPL>;
  constexpr int NR = G::NR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* rows = reinterpret_cast<const float*>(smem + G::OFF_ROWS);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + G::OFF_CNT);
  const uint8_t* map = reinterpret_cast<const uint8_t*>(smem + G::OFF_MAP);
  int* aff = reinterpret_cast<int*>(smem + G::OFF_AFF);
  int* wscr = reinterpret_cast<int*>(smem + G::OFF_WSCR) + warp * 16 * G::NR;
  const int* meta = reinterpret_cast<const int*>(smem + G::OFF_META);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  uint64_t* empty = full + G::STAGES;
  const bool aff_on = p.affinity != nullptr;
  const int kk = FASTK > 0 ? FASTK : p.k;
  const int wpb = p.E / 4;
  const int stride = p.E + 1;
  bool dead = false;
  int cur = -1;
  for (int64_t it = i0; it < i1; ++it) {
    const int64_t n = it - i0;
    const int s = (int)(n % G::STAGES);
    const int l = (int)(it / p.ntiles);
    if (G::SMEM_AFF && aff_on && l != cur) {
      if (cur >= 0) {
        named_bar(1, G::CTHREADS);
        if (!dead) k1_flush_aff<EPL>(p, aff, cur, threadIdx.x);
        named_bar(1, G::CTHREADS);
      }
    }
    cur = l;
    if (dead) continue;
    if (!mbar_wait(&full[s], (uint32_t)((n / G::STAGES) & 1), p.status)) {
      dead = true;
      continue;
    }
    const int* mt = meta + s * 8;
    const int tile = mt[1], ntok = mt[2], slot = mt[3];
    const int64_t tok0 = (int64_t)tile * G::TT;
    const float* stage = rows + (size_t)s * G::TT * G::EMAX;
    uint32_t* scnt = cnt + (size_t)s * G::CNT_WORDS;
    for (int r0 = warp * NR; r0 < ntok; r0 += G::CWARPS * NR) {
      const float* rowp[NR];
      int myidx[NR];
#pragma unroll
      for (int q = 0; q < NR; ++q) rowp[q] = stage + (size_t)min(r0 + q, ntok - 1) * p.E;
      unsigned redo = (1u << NR) - 1u;
      if constexpr (FASTK > 0) redo = topk_fast_rows<EPL, FASTK, NR>(rowp, lane, wscr, myidx);
#pragma unroll
      for (int q = 0; q < NR; ++q)
        if ((redo >> q) & 1u) myidx[q] = topk_exact<EPL>(rowp[q], p.E, p.k, lane);
#pragma unroll
      for (int q = 0; q < NR; ++q) {
        const int r = r0 + q;
        if (r >= ntok) break;
        if (p.topk != nullptr && lane < kk)
          p.topk[((size_t)l * p.T + tok0 + r) * kk + lane] = (uint8_t)myidx[q];
        if (aff_on) {
          if constexpr (G::SMEM_AFF) {
            if constexpr (FASTK > 0)
              aff_pairs_fixed<FASTK>(aff, stride, myidx[q], lane);
            else
              aff_pairs_any(aff, stride, myidx[q], kk, lane);
          } else {
            aff_pairs_any(p.affinity + (size_t)l * p.E * p.E, p.E, myidx[q], kk, lane);
          }
        }
        if (slot >= 0 && lane < kk) {
          const int lb = map[s * G::TT + r];
          atomicAdd(&scnt[lb * wpb + (myidx[q] >> 2)], 1u << ((myidx[q] & 3) * 8));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (G::SMEM_AFF && aff_on && cur >= 0) {
    named_bar(1, G::CTHREADS);
    if (!dead) k1_flush_aff<EPL>(p, aff, cur, threadIdx.x);
  }
}

template <int EPL, int FASTK>
__global__ void __launch_bounds__(K1Geo<EPL>::THREADS, 1) k1_kernel(const __grid_constant__ K1Params p) {
  using G = K1Geo<EPL>;
  extern __shared__ __align__(128) char smem[];
  if (*reinterpret_cast<volatile uint32_t*>(p.call_flag) != 0u) return;
  const int64_t i0 = (int64_t)blockIdx.x * p.nitems / gridDim.x;
  const int64_t i1 = ((int64_t)blockIdx.x + 1) * p.nitems / gridDim.x;
  uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + G::OFF_CNT);
  for (size_t w = threadIdx.x; w < G::STAGES * G::CNT_WORDS; w += G::THREADS) cnt[w] = 0u;
  if constexpr (G::SMEM_AFF) {
    int* aff = reinterpret_cast<int*>(smem + G::OFF_AFF);
    if (p.affinity != nullptr)
      for (size_t w = threadIdx.x; w < G::AFF_WORDS; w += G::THREADS) aff[w] = 0;
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(&full[s], 32);
      mbar_init(&full[G::STAGES + s], G::CWARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x >= G::CTHREADS)
    k1_producer<EPL>(p, smem, i0, i1);
  else
    k1_consumer<EPL, FASTK>(p, smem, i0, i1);
}

// ------------------------------------------------------------------ launch
template <int EPL, int FASTK>
cudaError_t k1_launch(const K1Params& p, int grid, cudaStream_t st) {
  using G = K1Geo<EPL>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k1_kernel<EPL, FASTK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  k1_kernel<EPL, FASTK><<<grid, G::THREADS, G::SMEM, st>>>(p);
  return cudaGetLastError();
}

// Host side of moer_topk_signature after argument validation.
moer_status topk_signature_launch(const moer_dims* d, const float* logits, int64_t T,
                                  const int32_t* blk_tab, int32_t nblk, uint8_t* topk,
                                  uint8_t* blk_cnt, int32_t* affinity, void* ws,
                                  cudaStream_t st) {
  const int E = d->E, k = d->k;
  const bool tpr = tpr_supported(E, k);
  const int TT = tpr ? 32 : k1_tile_tokens(E);
  const int ntiles = (int)((T + TT - 1) / TT);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint32_t* call_flag = status + 1;
  int32_t* tile_blk0 = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + WS_HEADER);
  int32_t* tok_blk = reinterpret_cast<int32_t*>(
      static_cast<char*>(ws) + WS_HEADER + ((size_t)((T + 31) / 32) * sizeof(int32_t) + 255) / 256 * 256);
  if (cudaMemsetAsync(call_flag, 0, sizeof(uint32_t), st) != cudaSuccess) return MOER_ECUDA;
  const bool hist = blk_cnt != nullptr && d->m > 0;
  if (hist) {
    const int blocks = (int)min64((nblk + 255) / 256, 4096);
    k1_tile_index<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(blk_tab, nblk, T, d->block, TT,
                                                            tpr ? nullptr : tile_blk0,
                                                            tpr ? tok_blk : nullptr, status, call_flag,
                                                            blk_cnt, d->m, E);
    if (cudaGetLastError() != cudaSuccess) return MOER_ECUDA;
  }
  int sms = device_sm_count();
  if (sms <= 0) return MOER_ECUDA;
  if (tpr) {
    TprParams q;
    q.logits = logits;
    q.T = T;
    q.k = k;
    q.L = d->L;
    q.m = d->m;
    q.topk = topk;
    q.blk_cnt = hist ? blk_cnt : nullptr;
    q.affinity = affinity;
    q.tok_blk = tok_blk;
    q.ntiles = ntiles;
    q.nitems = (int64_t)d->L * ntiles;
    q.status = status;
    q.call_flag = call_flag;
    for (int l = 0; l < 256; ++l) q.slot_of_layer[l] = -1;
    for (int i = 0; i < d->m; ++i) q.slot_of_layer[d->mask[i]] = (int16_t)i;
    const int grid = (int)min64(q.nitems, sms);
    return tpr_run(E, k, q, grid, st) == cudaSuccess ? MOER_OK : MOER_ECUDA;
  }
  K1Params p;
  p.logits = logits;
  p.T = T;
  p.E = E;
  p.k = k;
  p.L = d->L;
  p.m = d->m;
  p.B = d->block;
  p.blk_tab = blk_tab;
  p.nblk = nblk;
  p.topk = topk;
  p.blk_cnt = hist ? blk_cnt : nullptr;
  p.affinity = affinity;
  p.tile_blk0 = tile_blk0;
  p.ntiles = ntiles;
  p.nitems = (int64_t)d->L * ntiles;
  p.status = status;
  p.call_flag = call_flag;
  for (int l = 0; l < 256; ++l) p.slot_of_layer[l] = -1;
  for (int i = 0; i < d->m; ++i) p.slot_of_layer[d->mask[i]] = (int16_t)i;
  const int grid = (int)min64(p.nitems, sms);
  cudaError_t e;
  if (E <= 32)
    e = k1_launch<1, 0>(p, grid, st);
  else if (E <= 64)
    e = k1_launch<2, 0>(p, grid, st);
  else if (E <= 128)
    e = k1_launch<4, 0>(p, grid, st);
  else
    e = k1_launch<8, 0>(p, grid, st);
  return e == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
