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
//   * Persistent grid, one CTA per SM, twenty warps, no producer warp.  Work
//     items are (layer, 32-token tile); tile n of the CTA goes to warp n % 20.
//     A tile is fetched in column slices (32 rows x 32 experts, 4 KB) by 3-D
//     TMA tensor copies ([L][T][E] logits, rows past T zero-filled) into two
//     slice buffers that the warp owns: as soon as the warp has folded a
//     slice, its lane 0 issues the copy of the slice two ahead into the same
//     buffer, so each copy lands while the other buffer is being folded.
//     With one whole-tile stage per warp instead, a warp sat idle a quarter of
//     its time waiting for its own refill.
//   * One lane per token row.  A lane reads its row's slice from shared memory
//     in 16-byte units whose order is XOR-rotated by (lane & 7), which makes
//     every LDS.128 conflict-free, and folds it 8 values at a time into a
//     sorted top-8 held in registers: an optimal 19-comparator sorting network
//     per chunk, then a merge with the running top-8 that also yields the
//     9th-ranked key (Batcher's odd-even merge pruned to its nine leading
//     outputs, rank.cuh).
//     Keys are the float's upper 24 bits (signed-int order equals value order
//     for positive floats) with the value's position in the lane's read order
//     in the low 8 bits, so keys are unique and min/max networks apply.
//   * A row's result is certified when its k leading keys are positive and
//     finite and the k+1 leading keys are pairwise distinct in their upper
//     24 bits (then truncation cannot have changed membership or order).
//     Rows that fail (ties, NaN, +-inf, zeros, negatives in the top k) are
//     redone exactly by the whole warp, from global memory, with the ballot
//     tie-breaking path.
//   * Co-activation: each lane adds its row's k(k-1)/2 rank-ordered pairs to
//     a shared-memory tile of directed counts with shared atomics (28 adds per
//     row at k = 8 instead of the 64 of the full k x k block), 32 bits per
//     count (66 KB with the bank padding; a 16-bit tile of half the size,
//     folded every 65,535 rows, is a build option and costs more per add);
//     the warps fold the tile into the symmetric co-activation, diagonal
//     included, and add it to global memory at each layer change.
//   * The top-k ids go out as 8 (or 6) bytes per row; the per-KV-block
//     counts are computed from them by block_counts.cu.
#include <climits>

#include "common.cuh"
#include "k1_params.cuh"
#include "rank.cuh"

namespace moer {

// Geometry (compile-time tunables with the measured defaults).
#ifndef MOER_TPR_CW
#define MOER_TPR_CW 20  // warps per CTA (the most whose slice buffers fit beside the 32-bit tile)
#endif
#ifndef MOER_TPR_RING
#define MOER_TPR_RING 2  // slice buffers per warp
#endif
#ifndef MOER_TPR_AFF32
#define MOER_TPR_AFF32 1  // 32-bit co-activation counts (else 16-bit, two per word)
#endif
#ifndef MOER_TPR_FOLD_ROWS
#define MOER_TPR_FOLD_ROWS 65535  // rows between folds of the 16-bit co-activation tile
#endif

template <int E>
struct TprGeo {
  static constexpr int TT = 32;             // rows per tile: one per lane
  static constexpr int SW = 32;             // experts per slice: 128-byte slice rows
  static constexpr int Q = E / SW;          // slices per tile
  static constexpr int R = MOER_TPR_RING;   // slice buffers per warp
  static constexpr int CW = MOER_TPR_CW;
  static constexpr int THREADS = CW * 32;
  static_assert(E % SW == 0 && Q >= 1, "whole slices per row");
  static_assert(R >= 2, "a warp needs a second slice buffer to overlap copy and compute");
  // every tile starts in buffer 0, so a slice's buffer and the refill that
  // follows it are fixed by its place q in the tile
  static_assert(R <= Q && Q % R == 0, "whole rounds of the slice buffers per tile");
  static constexpr uint32_t SLICE_BYTES = (uint32_t)TT * SW * 4;
  static constexpr size_t OFF_ROWS = 0;
  static constexpr size_t OFF_AFF = OFF_ROWS + (size_t)CW * R * SLICE_BYTES;
  // Directed pair counts D[a][b].  16-bit counts: half (b & 1) of word
  // a RS + b / 2, folded into global memory at least every FT tiles so that no
  // count passes 65535 (a count grows once per row at most).  32-bit counts:
  // word a RS + b, folded at layer changes only.  A tile row has one word of
  // padding, so the bank of a counter moves with its row as well as its
  // column (without it the column alone picks the bank).
  static constexpr bool W32 = MOER_TPR_AFF32 != 0;
  static constexpr int RS = W32 ? E + 1 : E / 2 + 1;
  static constexpr size_t AFF_WORDS = (size_t)E * RS;
  static constexpr int FT = W32 ? (1 << 30) / TT : MOER_TPR_FOLD_ROWS / TT;
  static_assert(MOER_TPR_FOLD_ROWS <= 65535, "16-bit counts: at most 65535 rows between folds");
  static constexpr size_t OFF_RSUM = OFF_AFF + AFF_WORDS * 4;  // E row sums used by the flush
  static constexpr size_t OFF_BAR = (OFF_RSUM + (size_t)E * 4 + 7) / 8 * 8;
  static constexpr size_t SMEM = OFF_BAR + (size_t)CW * R * 8;
  static_assert(SMEM <= 232448, "fits the 227 KB of shared memory a CTA may use");
};


// Folds one slice of this lane's row (SW values, experts col0 .. col0 + SW - 1)
// into the running top-8 keys T (descending) and, if WANT9, the 9th key L9.
// The slice row is read in 16-byte units whose order is XOR-rotated by
// rot = (lane & 7).  The value at read position p of the row gets the low key
// byte 255 - p; its expert id is p ^ (4 rot) (the rotation permutes the units
// of each 128-byte slice row, and col0 is a multiple of 32).  The key keeps
// the float's upper 24 bits: (bits >> 8) * 256 + byte, the value of
// trunc_key(bits, byte), computed as a multiply-high and a multiply-add by
// the run-time constants hi_mul = 2^24 and lo_mul = 2^8.  FIRST starts a
// row: the first chunk becomes T.
template <int SW, bool WANT9, bool FIRST>
__device__ __forceinline__ void slice_top8(const float* srow, int rot, int col0, uint32_t hi_mul,
                                           uint32_t lo_mul, int (&T)[8], int& L9) {
  const char* base = reinterpret_cast<const char*>(srow);
  const int r16 = rot * 16;
  if constexpr (FIRST) L9 = INT_MIN;
#pragma unroll
  for (int g = 0; g < SW / 8; ++g) {
    const float4 a = *reinterpret_cast<const float4*>(base + (((2 * g) * 16) ^ r16));
    const float4 b = *reinterpret_cast<const float4*>(base + (((2 * g + 1) * 16) ^ r16));
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    int c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      c[j] = (int)(__umulhi(__float_as_uint(v[j]), hi_mul) * lo_mul + (uint32_t)(255 - col0 - (8 * g + j)));
    sort8_desc(c);
    if (FIRST && g == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) T[i] = c[i];
    } else {
      merge8<WANT9>(T, c, L9);
    }
  }
}

// ------------------------------------------------------------- slice copy
// One tiled TMA copy of the 3-D logits map (x = expert, y = token, z = layer)
// into shared memory, completing on `bar` as transaction bytes; rows past T
// are zero-filled and counted.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// -------------------------------------------------------------- consumers
// Directed pair count D[a][b] in the shared tile.
template <int E>
__device__ __forceinline__ uint32_t aff_get(const uint32_t* aff, int a, int b) {
  using G = TprGeo<E>;
  if constexpr (G::W32) return aff[a * G::RS + b];
  return (aff[a * G::RS + (b >> 1)] >> ((b & 1) << 4)) & 0xFFFFu;
}

// Adds one to D[a][b].
template <int E>
__device__ __forceinline__ void aff_add(uint32_t* aff, int a, int b) {
  using G = TprGeo<E>;
  if constexpr (G::W32)
    atomicAdd(&aff[a * G::RS + b], 1u);
  else
    atomicAdd(&aff[a * G::RS + (b >> 1)], 1u << ((b & 1) << 4));
}

// The shared tile holds directed pair counts D[a][b] = # rows of this CTA's
// current layer (since the last fold) in which expert a ranks above expert b.
// Co-activation is symmetric: A[a][b] = D[a][b] + D[b][a] for a != b, and,
// every row holding k distinct experts, the diagonal (the expert's load) is
// its off-diagonal row sum divided by k - 1.  Adds the tile to layer `layer`
// of the global co-activation and clears it; the sums are formed by warp
// reductions, with no shared atomics (a row's lanes would all hit one
// counter).  All consumer threads call this (it holds a barrier); `skip`
// leaves the tile alone (a warp timed out).
template <int E, int K>
__device__ void tpr_flush_aff(const K1Params& p, uint32_t* aff, int* rsum, int layer, bool skip) {
  using G = TprGeo<E>;
  (void)rsum;
  int32_t* dst = p.affinity + (size_t)layer * E * E;
  if (!skip) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (p.aff_pairs64) {
      // a warp per row a: first the diagonal, the sum of the row and column of D
      // over all b (D[a][a] is 0: a row's k experts are distinct) over k - 1; then
      // the whole row A[a][b] = D[a][b] + D[b][a], two neighbouring counts per
      // 64-bit red
      for (int a = warp; a < E; a += G::CW) {
        uint32_t sum = 0u;
        for (int b = lane; b < E; b += 32) sum += aff_get<E>(aff, a, b) + aff_get<E>(aff, b, a);
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
        const uint32_t diag = sum / (uint32_t)(K - 1);
        for (int b = 2 * lane; b < E; b += 64) {
          const uint32_t v0 = b == a ? diag : aff_get<E>(aff, a, b) + aff_get<E>(aff, b, a);
          const uint32_t v1 = b + 1 == a ? diag : aff_get<E>(aff, a, b + 1) + aff_get<E>(aff, b + 1, a);
          if ((v0 | v1) != 0u) {
            const unsigned long long v = ((unsigned long long)v1 << 32) | v0;
            asm volatile("red.global.add.u64 [%0], %1;" ::"l"(dst + (size_t)a * E + b), "l"(v) : "memory");
          }
        }
      }
    } else {
      // the pairs a < b, a warp per row a and its lanes along b: A[a][b] = A[b][a] =
      // D[a][b] + D[b][a]
      for (int a = warp; a < E - 1; a += G::CW)
        for (int b = a + 1 + lane; b < E; b += 32) {
          const int v = (int)(aff_get<E>(aff, a, b) + aff_get<E>(aff, b, a));
          if (v != 0) {
            atomicAdd(&dst[a * E + b], v);
            atomicAdd(&dst[b * E + a], v);
          }
        }
      // the diagonal, a warp per expert a: the sum of its row and column of D over
      // all b (D[a][a] is 0: a row's k experts are distinct), divided by k - 1
      for (int a = warp; a < E; a += G::CW) {
        uint32_t sum = 0u;
        for (int b = lane; b < E; b += 32) sum += aff_get<E>(aff, a, b) + aff_get<E>(aff, b, a);
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
        if (lane == 0 && sum != 0u) atomicAdd(&dst[a * E + a], (int)(sum / (uint32_t)(K - 1)));
      }
    }
  }
  named_bar(1, G::THREADS);  // every read of the tile is done before it is cleared
  if (!skip)
    for (int c = threadIdx.x; c < (int)G::AFF_WORDS; c += G::THREADS) aff[c] = 0u;
}

template <int E, int K>
__device__ void tpr_consumer(const K1Params& p, char* smem, int64_t i0, int64_t i1) {
  using G = TprGeo<E>;
  constexpr int Q = G::Q, R = G::R, SW = G::SW;
  constexpr int SLICE_FLOATS = G::TT * SW;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rot = lane & 7;
  float* ring = reinterpret_cast<float*>(smem + G::OFF_ROWS) + (size_t)warp * R * SLICE_FLOATS;
  uint32_t* aff = reinterpret_cast<uint32_t*>(smem + G::OFF_AFF);
  const uint32_t aff_base = smem_u32(aff);
  int* rsum = reinterpret_cast<int*>(smem + G::OFF_RSUM);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR) + warp * R;
  const bool aff_on = p.affinity != nullptr;
  const int N = (int)(i1 - i0);  // this CTA's items (the host keeps them below 2^31)
  // fold epochs: (layer, tile / FT), numbered l * epl + tile / FT, monotone in
  // the item (below 2^24: fewer than 256 layers, epl <= 2^26 / FT)
  const int epl = (p.ntiles + G::FT - 1) / G::FT;
  auto epoch_of = [&](int64_t item) {
    const int li = (int)(item / p.ntiles);
    return li * epl + (int)(item - (int64_t)li * p.ntiles) / G::FT;
  };
  const int ep_last = epoch_of(i1 - 1);
  int cur = epoch_of(i0);
  const int l0 = (int)((i0 + warp) / p.ntiles);
  const int t0 = (int)((i0 + warp) - (int64_t)l0 * p.ntiles);
  // Slice q of the warp's tile i (its tile n = warp + i CW) is its slice
  // j = i Q + q: buffer j % R = q % R, use j / R of that buffer.  Lane 0
  // copies the first R slices of the first tile, then, each time a slice is
  // folded, refills its buffer with the slice R ahead -- slice q + R of the
  // same tile, or slice q + R - Q of the warp's next tile.
  const int ntw = N > warp ? (N - warp + G::CW - 1) / G::CW : 0;  // tiles of this warp
  auto copy = [&](int buf, int q, int tl, int ly) {
    mbar_arrive_expect_tx(&full[buf], G::SLICE_BYTES);
    tma_load_3d(ring + (size_t)buf * SLICE_FLOATS, &p.tm_logits, q * SW, tl * G::TT, ly, &full[buf]);
  };
  if (lane == 0 && ntw > 0)
#pragma unroll
    for (int r = 0; r < R; ++r) copy(r, r, t0, l0);
  bool dead = false;
  int dead_j = 0;  // the slice whose wait expired
  int l = l0, tile = t0, nl = l0, ntile = t0;
  int ti = 0;  // tiles of this warp begun
  for (int n = warp; n < N; n += G::CW, ++ti) {
    l = nl;
    tile = ntile;
    // the warp's next tile
    ntile = tile + G::CW;
    while (ntile >= p.ntiles) {
      ntile -= p.ntiles;
      ++nl;
    }
    const bool has_next = n + G::CW < N;
    const int ep = l * epl + tile / G::FT;
    while (aff_on && cur < ep) {
      named_bar(1, G::THREADS);
      tpr_flush_aff<E, K>(p, aff, rsum, (int)(cur / epl), dead);
      named_bar(1, G::THREADS);
      ++cur;
    }
    cur = ep;
    if (dead) continue;
    const int64_t tok0 = (int64_t)tile * G::TT;
    const int ntok = tile == p.ntiles - 1 ? p.tail_rows : G::TT;
    const int slot = p.slot_of_layer[l];
    uint8_t* out = nullptr;
    if (p.ids != nullptr && (!p.ids_mask_only || slot >= 0))
      out = p.ids + ((size_t)(p.ids_mask_only ? slot : l) * p.T + tok0) * K;
    // parity of the tile's first use of each buffer: (i Q / R) & 1
    const uint32_t par0 = ((Q / R) & 1) ? (uint32_t)(ti & 1) : 0u;
    int Tk[8], L9;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int buf = q % R;
      if (!__all_sync(FULL, mbar_wait(&full[buf], par0 ^ (uint32_t)((q / R) & 1), p.status))) {
        dead = true;
        dead_j = ti * Q + q;
        break;
      }
      const float* srow = ring + (size_t)buf * SLICE_FLOATS + lane * SW;
      if (q == 0)
        slice_top8<SW, (K == 8), true>(srow, rot, 0, p.key_hi_mul, p.key_lo_mul, Tk, L9);
      else
        slice_top8<SW, (K == 8), false>(srow, rot, q * SW, p.key_hi_mul, p.key_lo_mul, Tk, L9);
      // every lane has read the buffer: refill it with the slice R ahead
      __syncwarp();
      if (lane == 0) {
        if (q + R < Q)
          copy(buf, q + R, tile, l);
        else if (has_next)
          copy(buf, q + R - Q, ntile, nl);
      }
    }
    if (dead) continue;
    // certification of the truncated-key result
    const bool bad = trunc_top8_uncertain<K>(Tk, L9);
    const bool live = lane < ntok;
    const unsigned redo = __ballot_sync(FULL, bad && live);
    // expert ids: read position pos = 255 - low byte, id = pos ^ 4 (lane & 7)
    const int xrow = 4 * rot;
    int idx[K];
#pragma unroll
    for (int i = 0; i < K; ++i) idx[i] = ((~Tk[i]) & 0xFF) ^ xrow;
    if (live && !bad) {
      if (out != nullptr) {
        if constexpr (K == 8) {
          const uint32_t lo = (uint32_t)idx[0] | ((uint32_t)idx[1] << 8) | ((uint32_t)idx[2] << 16) |
                              ((uint32_t)idx[3] << 24);
          const uint32_t hi = (uint32_t)idx[4] | ((uint32_t)idx[5] << 8) | ((uint32_t)idx[6] << 16) |
                              ((uint32_t)idx[7] << 24);
          *reinterpret_cast<uint2*>(out + (size_t)lane * 8) = make_uint2(lo, hi);
        } else {
          uint8_t* o = out + (size_t)lane * K;
#pragma unroll
          for (int i = 0; i < K; i += 2)
            *reinterpret_cast<uint16_t*>(o + i) = (uint16_t)(idx[i] | (idx[i + 1] << 8));
        }
      }
      if (aff_on) {
        // directed pairs (rank i above rank j): k(k-1)/2 adds per row
        if constexpr (G::W32) {
          // shared address of D[a][b] = tile + 4 b + a * row pitch: one
          // multiply-add per pair (FMA pipe), the pitch known only at run time
          // so that it is not folded into integer-ALU shifts and adds
          uint32_t colb[K];
#pragma unroll
          for (int j = 1; j < K; ++j) colb[j] = aff_base + 4u * (uint32_t)idx[j];
#pragma unroll
          for (int i = 0; i < K - 1; ++i) {
#pragma unroll
            for (int j = i + 1; j < K; ++j) {
              uint32_t addr;
              asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(addr) : "r"((uint32_t)idx[i]), "r"(p.aff_row_bytes), "r"(colb[j]));
              asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(addr) : "memory");
            }
          }
        } else {
          int wj[K];
          uint32_t sj[K];
#pragma unroll
          for (int j = 1; j < K; ++j) {
            wj[j] = idx[j] >> 1;
            sj[j] = 1u << ((idx[j] & 1) << 4);
          }
#pragma unroll
          for (int i = 0; i < K - 1; ++i) {
            uint32_t* ra = aff + idx[i] * G::RS;
#pragma unroll
            for (int j = i + 1; j < K; ++j) atomicAdd(ra + wj[j], sj[j]);
          }
        }
      }
    }
    // rows the fast path could not certify: the whole warp redoes each exactly,
    // reading the row again from global memory (its slices are being refilled)
    unsigned todo = redo;
    while (todo) {
      const int f = __ffs(todo) - 1;
      todo &= todo - 1;
      const int e = warp_topk_exact<E / 32>(p.logits + ((size_t)l * p.T + tok0 + f) * E, E, K, lane);
      if (out != nullptr && lane < K) out[(size_t)f * K + lane] = (uint8_t)e;
      if (aff_on) {
#pragma unroll
        for (int base = 0; base < K * K; base += 32) {
          const int q = base + lane;
          const int ia = __shfl_sync(FULL, e, q < K * K ? q / K : 0);
          const int ib = __shfl_sync(FULL, e, q < K * K ? q % K : 0);
          if (q < K * K && q / K < q % K) aff_add<E>(aff, ia, ib);
        }
      }
    }
  }
  if (dead && lane == 0) {
    // a copy stopped answering: wait (bounded) for this warp's copies still in
    // flight into shared memory before leaving -- slices dead_j .. (issued: R
    // ahead of the slice that expired, within the warp's slices)
    const int js = min(dead_j + R, ntw * Q);
    for (int j = dead_j; j < js; ++j) mbar_wait(&full[j % R], (uint32_t)((j / R) & 1), nullptr);
  }
  if (aff_on) {
    while (cur < ep_last) {
      named_bar(1, G::THREADS);
      tpr_flush_aff<E, K>(p, aff, rsum, (int)(cur / epl), dead);
      named_bar(1, G::THREADS);
      ++cur;
    }
    named_bar(1, G::THREADS);
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
    for (int s = 0; s < G::CW * G::R; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  tpr_consumer<E, K>(p, smem, i0, i1);
}

template <int E, int K>
cudaError_t tpr_launch(const K1Params& p, int grid, cudaStream_t st) {
  using G = TprGeo<E>;
  static std::atomic<unsigned long long> set{0};
  const cudaError_t e = smem_optin(k1_tpr_kernel<E, K>, (int)G::SMEM, set);
  if (e != cudaSuccess) return e;
  k1_tpr_kernel<E, K><<<grid, G::THREADS, G::SMEM, st>>>(p);
  return cudaGetLastError();
}

bool tpr_supported(int E, int k) { return (E == 128 || E == 64) && (k == 8 || k == 6); }

int tpr_tile_tokens(int E) { return E == 128 ? TprGeo<128>::TT : TprGeo<64>::TT; }

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tiled_encoder() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// The logits [L][T][E] fp32 as a 3-D tensor map (x = expert, y = token,
// z = layer) with boxes of one slice: SW experts x TT tokens x 1 layer.
template <int E>
bool logits_map(CUtensorMap* m, const float* logits, int64_t T, int L) {
  using G = TprGeo<E>;
  EncodeTiledFn enc = tiled_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)E, (cuuint64_t)T, (cuuint64_t)L};
  const cuuint64_t strides[2] = {(cuuint64_t)E * 4, (cuuint64_t)T * E * 4};
  const cuuint32_t box[3] = {(cuuint32_t)G::SW, (cuuint32_t)G::TT, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(logits), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int E, int K>
cudaError_t tpr_launch_mapped(const K1Params& p0, int grid, cudaStream_t st) {
  K1Params p = p0;
  if (!logits_map<E>(&p.tm_logits, p.logits, p.T, p.L)) return cudaErrorInvalidValue;
  return tpr_launch<E, K>(p, grid, st);
}
}  // namespace

cudaError_t tpr_run(int E, int k, const K1Params& p, int grid, cudaStream_t st) {
  if (E == 128 && k == 8) return tpr_launch_mapped<128, 8>(p, grid, st);
  if (E == 128 && k == 6) return tpr_launch_mapped<128, 6>(p, grid, st);
  if (E == 64 && k == 8) return tpr_launch_mapped<64, 8>(p, grid, st);
  return tpr_launch_mapped<64, 6>(p, grid, st);
}

}  // namespace moer
