// topk_signature_tpr.cu -- thread-per-row logits pass of moer_topk_signature
// (top-k ids and expert co-activation) for the model shapes the path is
// built around (E = 64 or 128 experts, k = 6 or 8).
//
// What it computes is identical to the warp-per-row kernel (see
// topk_signature.cu): ELDR, sections "What it tries to solve" and "Key idea /
// structure / operation" (standard top-k gating; discrete top-k counts per
// KV block over the layer mask); GRACE-MoE, section 3 and section 4 /
// Figure 2(a) (per-layer expert co-activation).
//
// Design (GB300):
//   * Persistent grid, one CTA per SM: one producer warp and twelve consumer
//     warps.  Work items are (layer, 32-token tile); tile n of the CTA goes to
//     consumer warp n % 12 and to that warp's own ring stage (one
//     cp.async.bulk copy of 32 contiguous logit rows, completing on an
//     mbarrier).  Stages are never shared between consumer warps, so each
//     warp meets its stages' barrier phases strictly in order.
//   * One consumer lane per token row (two lanes per row is a build option:
//     the halves are then merged across the lane pair with shuffles).  A lane
//     reads its row from shared memory in 16-byte units whose order is
//     XOR-rotated by (lane & 7), which makes every LDS.128 conflict-free, and
//     folds it 8 values at a time into a sorted top-8 held in registers: an
//     optimal 19-comparator sorting network per chunk, then a bitonic
//     split/merge with the running top-8 (the split's losers, folded with
//     3-input maxima, give the 9th-ranked key).  Keys are the float's upper
//     24 bits (signed-int order equals value order for positive floats) with
//     the value's position in the lane's read order in the low 8 bits, so
//     keys are unique and min/max networks apply.
//   * A row's result is certified when its k leading keys are positive and
//     finite and the k+1 leading keys are pairwise distinct in their upper
//     24 bits (then truncation cannot have changed membership or order).
//     Rows that fail (ties, NaN, +-inf, zeros, negatives in the top k) are
//     redone exactly by the whole warp with the ballot tie-breaking path.
//   * Co-activation: each lane adds its row's k(k-1)/2 rank-ordered pairs to
//     a shared-memory tile of directed counts with shared atomics (28 adds per
//     row at k = 8 instead of the 64 of the full k x k block), 16 bits per
//     count so the tile takes 32 KB and the ring 192 KB; the consumer warps
//     fold the tile into the symmetric co-activation, diagonal included, and
//     add it to global memory at each layer change and at least every 2047
//     tiles (65504 rows), before any count could overflow.
//   * The top-k ids go out as 8 (or 6) bytes per row; the per-KV-block
//     counts are computed from them by block_counts.cu.
#include <climits>

#include "common.cuh"
#include "k1_params.cuh"

namespace moer {

// Geometry (compile-time tunables with the measured defaults).
#ifndef MOER_TPR_LPR
#define MOER_TPR_LPR 1
#endif
#ifndef MOER_TPR_CW
#define MOER_TPR_CW 12
#endif
#ifndef MOER_TPR_STAGE_KB
#define MOER_TPR_STAGE_KB 192
#endif
#ifndef MOER_TPR_FOLD_ROWS
#define MOER_TPR_FOLD_ROWS 65535  // rows between folds of the 16-bit co-activation tile
#endif

template <int E>
struct TprGeo {
  static constexpr int LPR = MOER_TPR_LPR;  // lanes per row: each folds E / LPR values
  static constexpr int TT = 32 / LPR;       // rows per tile (one tile per consumer warp)
  static constexpr int CW = MOER_TPR_CW;    // consumer warps
  static constexpr int STAGES = MOER_TPR_STAGE_KB * 1024 / (TT * E * 4);
  // Each stage belongs to one consumer warp (STAGES / CW stages per warp), so
  // a warp always waits on its stages' phases in order and can never pass a
  // barrier one phase early.
  static_assert(STAGES % CW == 0, "stages must divide evenly among consumer warps");
  static constexpr int SPW = STAGES / CW;
  // Ring stage of the CTA's n-th tile: warp n % CW, that warp's (n / CW)-th use.
  __device__ static int stage_of(int64_t n) { return (int)(n % CW) + CW * (int)((n / CW) % SPW); }
  // Phase (use count) of that stage: n / STAGES.
  static constexpr int CTHREADS = CW * 32;
  static constexpr int THREADS = CTHREADS + 32;
  static constexpr size_t STAGE_BYTES = (size_t)TT * E * 4;
  static constexpr size_t OFF_ROWS = 0;
  static constexpr size_t OFF_AFF = OFF_ROWS + STAGES * STAGE_BYTES;
  // directed pair counts, 16 bits each, two per word (D[a][b] is half (b & 1)
  // of word (a E + b) / 2); the tile is folded into global memory at least
  // every FT tiles, so no count passes 65535 (a count grows once per row at most)
  static constexpr size_t AFF_WORDS = (size_t)E * E / 2;
  static constexpr int FT = MOER_TPR_FOLD_ROWS / TT;
  static_assert(MOER_TPR_FOLD_ROWS <= 65535, "16-bit counts: at most 65535 rows between folds");
  static constexpr size_t OFF_RSUM = OFF_AFF + AFF_WORDS * 4;  // E row sums used by the flush
  static constexpr size_t OFF_BAR = OFF_RSUM + (size_t)E * 4;
  static constexpr size_t SMEM = OFF_BAR + 2 * STAGES * 8;
};


// ------------------------------------------------------ comparator networks
__device__ __forceinline__ void cas(int& a, int& b) {  // a <- max, b <- min
  const int hi = max(a, b), lo = min(a, b);
  a = hi;
  b = lo;
}

// Sorts 8 keys in descending order (19 comparators, depth 6).
__device__ __forceinline__ void sort8_desc(int (&c)[8]) {
  cas(c[0], c[2]); cas(c[1], c[3]); cas(c[4], c[6]); cas(c[5], c[7]);
  cas(c[0], c[4]); cas(c[1], c[5]); cas(c[2], c[6]); cas(c[3], c[7]);
  cas(c[0], c[1]); cas(c[2], c[3]); cas(c[4], c[5]); cas(c[6], c[7]);
  cas(c[2], c[4]); cas(c[3], c[5]);
  cas(c[1], c[4]); cas(c[3], c[6]);
  cas(c[1], c[2]); cas(c[3], c[4]); cas(c[5], c[6]);
}

// Sorts a bitonic sequence of 8 keys in descending order (half-cleaners).
__device__ __forceinline__ void clean8_desc(int (&m)[8]) {
  cas(m[0], m[4]); cas(m[1], m[5]); cas(m[2], m[6]); cas(m[3], m[7]);
  cas(m[0], m[2]); cas(m[1], m[3]); cas(m[4], m[6]); cas(m[5], m[7]);
  cas(m[0], m[1]); cas(m[2], m[3]); cas(m[4], m[5]); cas(m[6], m[7]);
}

// Folds the losers of a half-cleaner step (mins of T[i] and U[7 - i]) into
// the running 9th key with 3-input maxima (one ALU op each).
__device__ __forceinline__ int fold_losers(int L9, const int (&lo)[8]) {
  const int a = __vimax3_s32(lo[0], lo[1], lo[2]);
  const int b = __vimax3_s32(lo[3], lo[4], lo[5]);
  const int c = __vimax3_s32(lo[6], lo[7], L9);
  return __vimax3_s32(a, b, c);
}

// T <- top-8 of T and U (both sorted descending), sorted descending; with
// WANT9, L9 <- max(L9, 9th key of T and U).
template <bool WANT9>
__device__ __forceinline__ void merge8(int (&T)[8], const int (&U)[8], int& L9) {
  int mrg[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mrg[i] = max(T[i], U[7 - i]);
  if constexpr (WANT9) {
    int lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) lo[i] = min(T[i], U[7 - i]);
    L9 = fold_losers(L9, lo);
  }
  clean8_desc(mrg);
#pragma unroll
  for (int i = 0; i < 8; ++i) T[i] = mrg[i];
}

// Top-8 keys (descending) of this lane's part of a row and, if WANT9, the
// 9th key.  The part holds NV values starting at expert PART * NV; it is read
// in 16-byte units whose order is XOR-rotated by (lane & 7).  The value at
// read position p of part h gets the low key byte 255 - (h * NV + p); its
// expert id is h * NV + (p ^ (4 * rot)) with rot the reading lane's rotation.
// The key keeps the float's upper 24 bits: (bits >> 8) * 256 + byte, computed
// as a multiply-high and a multiply-add by the run-time constants hi_mul =
// 2^24 and lo_mul = 2^8.
template <int NV, bool WANT9>
__device__ __forceinline__ void part_top8(const float* part, int h, int rot, uint32_t hi_mul, uint32_t lo_mul,
                                          int (&T)[8], int& L9) {
  const char* base = reinterpret_cast<const char*>(part);
  const int r16 = rot * 16;
  const int hb = h * NV;
  L9 = INT_MIN;
#pragma unroll
  for (int g = 0; g < NV / 8; ++g) {
    const float4 a = *reinterpret_cast<const float4*>(base + (((2 * g) * 16) ^ r16));
    const float4 b = *reinterpret_cast<const float4*>(base + (((2 * g + 1) * 16) ^ r16));
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    int c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      c[j] = (int)(__umulhi(__float_as_uint(v[j]), hi_mul) * lo_mul + (uint32_t)(255 - hb - (8 * g + j)));
    sort8_desc(c);
    if (g == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) T[i] = c[i];
    } else {
      merge8<WANT9>(T, c, L9);
    }
  }
}

// Merges the sorted top-8 of the lanes that share a row (xor butterfly over
// LPR lanes); afterwards every lane of the row holds the row's top-8 and 9th.
template <int LPR, bool WANT9>
__device__ __forceinline__ void merge_lanes(int (&T)[8], int& L9) {
#pragma unroll
  for (int sh = 1; sh < LPR; sh <<= 1) {
    int P[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) P[i] = __shfl_xor_sync(FULL, T[i], sh);
    if constexpr (WANT9) L9 = max(L9, __shfl_xor_sync(FULL, L9, sh));
    merge8<WANT9>(T, P, L9);
  }
}

// Exact warp-cooperative top-k of one row (ties to the lower expert id, NaN
// lowest, -0.0 == +0.0); lane r < k receives the id ranked r-th.
__device__ __forceinline__ uint32_t exact_key(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 1u;
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <int E>
__device__ int row_topk_exact(const float* row, int k, int lane) {
  constexpr int EPL = E / 32;
  uint32_t key[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) key[j] = exact_key(row[lane * EPL + j]);
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

// --------------------------------------------------------------- producer
template <int E>
__device__ void tpr_producer(const K1Params& p, char* smem, int64_t i0, int64_t i1) {
  using G = TprGeo<E>;
  if ((threadIdx.x & 31) != 0) return;
  float* rows = reinterpret_cast<float*>(smem + G::OFF_ROWS);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  uint64_t* empty = full + G::STAGES;
  const int64_t N = i1 - i0;
  // (layer, tile) of the next copy, advanced incrementally (no division per item)
  int cl = (int)(i0 / p.ntiles), ct = (int)(i0 % p.ntiles);
  int64_t n = 0;
  for (; n < N; ++n) {
    const int s = G::stage_of(n);
    if (n >= G::STAGES && !mbar_wait(&empty[s], (uint32_t)((n / G::STAGES - 1) & 1), p.status)) break;
    const int64_t tok0 = (int64_t)ct * G::TT;
    const uint32_t bytes = (uint32_t)min64(G::TT, p.T - tok0) * E * 4u;
    mbar_arrive_expect_tx(&full[s], bytes);
    bulk_g2s(rows + (size_t)s * G::TT * E, p.logits + ((size_t)cl * p.T + tok0) * E, bytes, &full[s]);
    if (++ct == p.ntiles) {
      ct = 0;
      ++cl;
    }
  }
  if (n < N) {
    // a consumer stopped answering: wait (bounded) for the copies still in
    // flight into this CTA's shared memory before leaving
    for (int64_t q = (n > G::STAGES ? n - G::STAGES : 0); q < n; ++q)
      mbar_wait(&full[G::stage_of(q)], (uint32_t)((q / G::STAGES) & 1), nullptr);
  }
}

// -------------------------------------------------------------- consumers
// Directed pair count D[a][b]: 16-bit half (b & 1) of word (a E + b) / 2.
__device__ __forceinline__ uint32_t aff_get(const uint32_t* aff, int c) { return (aff[c >> 1] >> ((c & 1) << 4)) & 0xFFFFu; }

// The shared tile holds directed pair counts D[a][b] = # rows of this CTA's
// current layer (since the last fold) in which expert a ranks above expert b.
// Co-activation is symmetric: A[a][b] = D[a][b] + D[b][a] for a != b, and,
// every row holding k distinct experts, the diagonal (the expert's load) is
// its off-diagonal row sum divided by k - 1.  Adds the tile to layer `layer`
// of the global co-activation and clears it.  All consumer threads call this
// (it holds a barrier); `skip` leaves the tile alone (a consumer warp timed out).
template <int E, int K>
__device__ void tpr_flush_aff(const K1Params& p, uint32_t* aff, int* rsum, int layer, bool skip) {
  using G = TprGeo<E>;
  int32_t* dst = p.affinity + (size_t)layer * E * E;
  if (!skip) {
    for (int c = threadIdx.x; c < E * E; c += G::CTHREADS) {
      const int a = c / E, b = c % E;
      if (a < b) {
        const int v = (int)(aff_get(aff, a * E + b) + aff_get(aff, b * E + a));
        if (v != 0) {
          atomicAdd(&dst[a * E + b], v);
          atomicAdd(&dst[b * E + a], v);
          atomicAdd(&rsum[a], v);
          atomicAdd(&rsum[b], v);
        }
      }
    }
  }
  named_bar(1, G::CTHREADS);
  if (!skip) {
    for (int a = threadIdx.x; a < E; a += G::CTHREADS) {
      const int v = rsum[a];
      if (v != 0) {
        atomicAdd(&dst[a * E + a], v / (K - 1));
        rsum[a] = 0;
      }
    }
    for (int c = threadIdx.x; c < (int)G::AFF_WORDS; c += G::CTHREADS) aff[c] = 0u;
  }
}

template <int E, int K>
__device__ void tpr_consumer(const K1Params& p, char* smem, int64_t i0, int64_t i1) {
  using G = TprGeo<E>;
  constexpr int LPR = G::LPR;
  constexpr int NV = E / LPR;              // values folded by one lane
  static_assert(LPR == 1 || LPR == 2, "rank split assumes one or two lanes per row");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rrow = lane / LPR, h = lane % LPR, rot = lane & 7;
  const float* rows = reinterpret_cast<const float*>(smem + G::OFF_ROWS);
  uint32_t* aff = reinterpret_cast<uint32_t*>(smem + G::OFF_AFF);
  int* rsum = reinterpret_cast<int*>(smem + G::OFF_RSUM);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  uint64_t* empty = full + G::STAGES;
  const bool aff_on = p.affinity != nullptr;
  const int64_t N = i1 - i0;
  // fold epochs: (layer, tile / FT), numbered l * epl + tile / FT, monotone in the item
  const int epl = (p.ntiles + G::FT - 1) / G::FT;
  auto epoch_of = [&](int64_t item) {
    const int li = (int)(item / p.ntiles);
    return (int64_t)li * epl + (item - (int64_t)li * p.ntiles) / G::FT;
  };
  const int64_t ep_last = epoch_of(i1 - 1);
  int64_t cur = epoch_of(i0);
  bool dead = false;
  int l = (int)((i0 + warp) / p.ntiles);
  int tile = (int)((i0 + warp) - (int64_t)l * p.ntiles);
  for (int64_t n = warp; n < N; n += G::CW) {
    if (n > warp) {
      tile += G::CW;
      while (tile >= p.ntiles) {
        tile -= p.ntiles;
        ++l;
      }
    }
    const int64_t ep = (int64_t)l * epl + tile / G::FT;
    while (aff_on && cur < ep) {
      named_bar(1, G::CTHREADS);
      tpr_flush_aff<E, K>(p, aff, rsum, (int)(cur / epl), dead);
      named_bar(1, G::CTHREADS);
      ++cur;
    }
    cur = ep;
    if (dead) continue;
    const int s = G::stage_of(n);
    if (!mbar_wait(&full[s], (uint32_t)((n / G::STAGES) & 1), p.status)) {
      dead = true;
      continue;
    }
    const int64_t tok0 = (int64_t)tile * G::TT;
    const int ntok = (int)min64(G::TT, p.T - tok0);
    const int slot = p.slot_of_layer[l];
    uint8_t* out = nullptr;
    if (p.ids != nullptr && (!p.ids_mask_only || slot >= 0))
      out = p.ids + ((size_t)(p.ids_mask_only ? slot : l) * p.T + tok0) * K;
    const float* stage = rows + (size_t)s * G::TT * E;
    int Tk[8], L9;
    part_top8<NV, (K == 8)>(stage + (size_t)rrow * E + h * NV, h, rot, p.key_hi_mul, p.key_lo_mul, Tk, L9);
    merge_lanes<LPR, (K == 8)>(Tk, L9);
    // certification of the truncated-key result
    const int nxt = (K == 8) ? L9 : Tk[K < 8 ? K : 7];
    bool bad = (Tk[K - 1] < 256) || (Tk[0] >= 0x7F800000);
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const int a = Tk[i];
      const int b = (i + 1 < K) ? Tk[i + 1] : nxt;
      bad = bad || (b >= (a & (int)0xFFFFFF00));
    }
    const bool live = rrow < ntok;
    const unsigned redo = __ballot_sync(FULL, bad && live && h == 0);
    // expert ids: position pos = 255 - low byte lies in part hp = pos / NV,
    // read by lane (row lanes) | hp with rotation orot = that lane's & 7, so
    // id = hp * NV + ((pos % NV) ^ 4 orot).  4 orot < NV leaves bit log2(NV)
    // alone, hence id = pos ^ 4 orot = pos ^ xrow ^ 4 hp with the row's
    // constant xrow = 4 ((lane & ~(LPR-1)) & 7) and 4 hp = (pos >> (log2(NV) - 2)) & 4.
    static_assert(4 * 7 < NV && (NV & (NV - 1)) == 0, "id recovery assumes NV a power of two >= 32");
    constexpr int HSH = (NV == 64) ? 4 : 3;
    const int xrow = 4 * ((lane & ~(LPR - 1)) & 7);
    int idx[K];
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const int pos = (~Tk[i]) & 0xFF;
      idx[i] = (LPR == 2) ? (pos ^ xrow ^ ((pos >> HSH) & 4)) : (pos ^ xrow);
    }
    if (live && !bad) {
      if (out != nullptr && h == 0) {
        if constexpr (K == 8) {
          const uint32_t lo = (uint32_t)idx[0] | ((uint32_t)idx[1] << 8) | ((uint32_t)idx[2] << 16) |
                              ((uint32_t)idx[3] << 24);
          const uint32_t hi = (uint32_t)idx[4] | ((uint32_t)idx[5] << 8) | ((uint32_t)idx[6] << 16) |
                              ((uint32_t)idx[7] << 24);
          *reinterpret_cast<uint2*>(out + (size_t)rrow * 8) = make_uint2(lo, hi);
        } else {
          uint8_t* o = out + (size_t)rrow * K;
#pragma unroll
          for (int i = 0; i < K; i += 2)
            *reinterpret_cast<uint16_t*>(o + i) = (uint16_t)(idx[i] | (idx[i + 1] << 8));
        }
      }
      if (aff_on) {
        // directed pairs (rank i above rank j): k(k-1)/2 adds per row into the
        // packed 16-bit counts; with two lanes per row, lane h takes the ranks
        // i with i % 2 == h
        int wj[K];
        uint32_t sj[K];
#pragma unroll
        for (int j = 1; j < K; ++j) {
          wj[j] = idx[j] >> 1;
          sj[j] = 1u << ((idx[j] & 1) << 4);
        }
#pragma unroll
        for (int i = 0; i < K - 1; ++i) {
          if (i % LPR == h) {
            uint32_t* ra = aff + idx[i] * (E / 2);
#pragma unroll
            for (int j = i + 1; j < K; ++j) atomicAdd(ra + wj[j], sj[j]);
          }
        }
      }
    }
    // rows the fast path could not certify: the whole warp redoes each exactly
    unsigned todo = redo;
    while (todo) {
      const int f = (__ffs(todo) - 1) / LPR;
      todo &= todo - 1;
      const int e = row_topk_exact<E>(stage + (size_t)f * E, K, lane);
      if (out != nullptr && lane < K) out[(size_t)f * K + lane] = (uint8_t)e;
      if (aff_on) {
#pragma unroll
        for (int base = 0; base < K * K; base += 32) {
          const int q = base + lane;
          const int ia = __shfl_sync(FULL, e, q < K * K ? q / K : 0);
          const int ib = __shfl_sync(FULL, e, q < K * K ? q % K : 0);
          if (q < K * K && q / K < q % K) {
            const int c = ia * E + ib;
            atomicAdd(&aff[c >> 1], 1u << ((c & 1) << 4));
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (aff_on) {
    while (cur < ep_last) {
      named_bar(1, G::CTHREADS);
      tpr_flush_aff<E, K>(p, aff, rsum, (int)(cur / epl), dead);
      named_bar(1, G::CTHREADS);
      ++cur;
    }
    named_bar(1, G::CTHREADS);
    tpr_flush_aff<E, K>(p, aff, rsum, (int)(cur / epl), dead);
  }
}

template <int E, int K>
__global__ void __launch_bounds__(TprGeo<E>::THREADS, 1) k1_tpr_kernel(const __grid_constant__ K1Params p) {
  using G = TprGeo<E>;
  extern __shared__ __align__(1024) char smem[];
  const int64_t i0 = (int64_t)blockIdx.x * p.nitems / gridDim.x;
  const int64_t i1 = ((int64_t)blockIdx.x + 1) * p.nitems / gridDim.x;
  if (i1 <= i0) return;
  if (p.affinity != nullptr) {
    uint32_t* aff = reinterpret_cast<uint32_t*>(smem + G::OFF_AFF);
    for (size_t w = threadIdx.x; w < G::AFF_WORDS + E; w += G::THREADS) aff[w] = 0u;  // tile and row sums
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&full[G::STAGES + s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x >= G::CTHREADS)
    tpr_producer<E>(p, smem, i0, i1);
  else
    tpr_consumer<E, K>(p, smem, i0, i1);
}

template <int E, int K>
cudaError_t tpr_launch(const K1Params& p, int grid, cudaStream_t st) {
  using G = TprGeo<E>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k1_tpr_kernel<E, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)G::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  k1_tpr_kernel<E, K><<<grid, G::THREADS, G::SMEM, st>>>(p);
  return cudaGetLastError();
}

bool tpr_supported(int E, int k) { return (E == 128 || E == 64) && (k == 8 || k == 6); }

int tpr_tile_tokens(int E) { return E == 128 ? TprGeo<128>::TT : TprGeo<64>::TT; }

cudaError_t tpr_run(int E, int k, const K1Params& p, int grid, cudaStream_t st) {
  if (E == 128 && k == 8) return tpr_launch<128, 8>(p, grid, st);
  if (E == 128 && k == 6) return tpr_launch<128, 6>(p, grid, st);
  if (E == 64 && k == 8) return tpr_launch<64, 8>(p, grid, st);
  return tpr_launch<64, 6>(p, grid, st);
}

}  // namespace moer
