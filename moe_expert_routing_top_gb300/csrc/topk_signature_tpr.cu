// topk_signature_tpr.cu -- thread-per-row variant of the fused top-k /
// per-KV-block count / co-activation pass, for the model shapes the path is
// built around (E = 64 or 128 experts, k = 6 or 8).
//
// What it computes is identical to the warp-per-row kernel (see
// topk_signature.cu): ELDR, sections "What it tries to solve" and "Key idea /
// structure / operation" (standard top-k gating; discrete top-k counts per
// KV block over the layer mask); GRACE-MoE, section 3 and section 4 /
// Figure 2(a) (per-layer expert co-activation).
//
// Design (GB300):
//   * Persistent grid, one CTA per SM: one producer warp and four consumer
//     warps.  Work items are (layer, 32-token tile); tile n of the CTA goes to
//     ring stage n % STAGES (one cp.async.bulk copy of 32 contiguous logit
//     rows, completing on an mbarrier) and to consumer warp n % 4.
//   * Each consumer lane owns one token row.  It reads the row from shared
//     memory in 16-byte units whose order is XOR-rotated by (lane & 7), which
//     makes every LDS.128 conflict-free, and folds the row 8 values at a
//     time into a sorted top-8 held in registers: an optimal 19-comparator
//     sorting network per chunk, then a bitonic split/merge with the running
//     top-8 (the split's losers give the 9th-ranked key).  Keys are the
//     float's upper 24 bits (signed-int order equals value order for positive
//     floats) with the value's position in the lane's read order in the low
//     8 bits, so keys are unique and min/max networks apply.
//   * A row's result is certified when its k leading keys are positive and
//     finite and the k+1 leading keys are pairwise distinct in their upper
//     24 bits (then truncation cannot have changed membership or order).
//     Rows that fail (ties, NaN, +-inf, zeros, negatives in the top k) are
//     redone exactly by the whole warp with the ballot tie-breaking path.
//   * Co-activation: each lane adds its row's k*k ordered pairs to a
//     shared-memory E x E int32 tile with shared atomics; the four consumer
//     warps flush it to global memory (atomic adds) at each layer change.
//   * KV-block counts: each consumer warp accumulates its tile's counts in a
//     private packed-byte buffer (four experts per 32-bit word) indexed by
//     the token's block relative to the tile's first block (from the
//     per-token block ids the pre-pass writes), then writes the tile's blocks
//     out itself: plain stores for blocks inside the tile, atomic adds for
//     the two edge blocks that straddle tiles (zeroed by the pre-pass).
#include <climits>

#include "common.cuh"
#include "k1_params.cuh"

namespace moer {

template <int E>
struct TprGeo {
  static constexpr int NU = E / 4;  // 16-byte units per row
  static constexpr int TT = 32;     // rows per tile: one per consumer lane
  static constexpr int CW = 4;      // consumer warps
  static constexpr int STAGES = (E == 128) ? 8 : 16;
  static constexpr int CTHREADS = CW * 32;
  static constexpr int THREADS = CTHREADS + 32;
  static constexpr size_t STAGE_BYTES = (size_t)TT * E * 4;
  static constexpr size_t CNT_WORDS = (size_t)TT * E / 4;  // per consumer warp
  static constexpr size_t OFF_ROWS = 0;
  static constexpr size_t OFF_CNT = OFF_ROWS + STAGES * STAGE_BYTES;
  static constexpr size_t OFF_AFF = OFF_CNT + CW * CNT_WORDS * 4;
  static constexpr size_t AFF_WORDS = (size_t)E * E;
  static constexpr size_t OFF_BAR = OFF_AFF + AFF_WORDS * 4;
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

// Top-8 keys (descending) of the lane's row and, if WANT9, the 9th key.
// Position p (0..E-1) of a value in the lane's read order goes into the key's
// low byte as 255 - p; the expert id of position p is p ^ (4 * (lane & 7)).
template <int E, bool WANT9>
__device__ __forceinline__ void row_top8(const float* row, int lane, int (&T)[8], int& L9) {
  const char* base = reinterpret_cast<const char*>(row);
  const int rot = (lane & 7) * 16;
  L9 = INT_MIN;
#pragma unroll
  for (int g = 0; g < E / 8; ++g) {
    const float4 a = *reinterpret_cast<const float4*>(base + (((2 * g) * 16) ^ rot));
    const float4 b = *reinterpret_cast<const float4*>(base + (((2 * g + 1) * 16) ^ rot));
    int c[8];
    c[0] = (__float_as_int(a.x) & (int)0xFFFFFF00) | (255 - (8 * g + 0));
    c[1] = (__float_as_int(a.y) & (int)0xFFFFFF00) | (255 - (8 * g + 1));
    c[2] = (__float_as_int(a.z) & (int)0xFFFFFF00) | (255 - (8 * g + 2));
    c[3] = (__float_as_int(a.w) & (int)0xFFFFFF00) | (255 - (8 * g + 3));
    c[4] = (__float_as_int(b.x) & (int)0xFFFFFF00) | (255 - (8 * g + 4));
    c[5] = (__float_as_int(b.y) & (int)0xFFFFFF00) | (255 - (8 * g + 5));
    c[6] = (__float_as_int(b.z) & (int)0xFFFFFF00) | (255 - (8 * g + 6));
    c[7] = (__float_as_int(b.w) & (int)0xFFFFFF00) | (255 - (8 * g + 7));
    sort8_desc(c);
    if (g == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) T[i] = c[i];
    } else {
      int mrg[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mrg[i] = max(T[i], c[7 - i]);
        if constexpr (WANT9) L9 = max(L9, min(T[i], c[7 - i]));
      }
      clean8_desc(mrg);
#pragma unroll
      for (int i = 0; i < 8; ++i) T[i] = mrg[i];
    }
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
__device__ void tpr_producer(const TprParams& p, char* smem, int64_t i0, int64_t i1) {
  using G = TprGeo<E>;
  if ((threadIdx.x & 31) != 0) return;
  float* rows = reinterpret_cast<float*>(smem + G::OFF_ROWS);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  uint64_t* empty = full + G::STAGES;
  const int64_t N = i1 - i0;
  int64_t n = 0;
  for (; n < N; ++n) {
    const int s = (int)(n % G::STAGES);
    if (n >= G::STAGES && !mbar_wait(&empty[s], (uint32_t)((n / G::STAGES - 1) & 1), p.status)) break;
    const int64_t it = i0 + n;
    const int l = (int)(it / p.ntiles);
    const int64_t tok0 = (it - (int64_t)l * p.ntiles) * G::TT;
    const int ntok = (int)min64(G::TT, p.T - tok0);
    const uint32_t bytes = (uint32_t)ntok * E * 4u;
    mbar_arrive_expect_tx(&full[s], bytes);
    bulk_g2s(rows + (size_t)s * G::TT * E, p.logits + ((size_t)l * p.T + tok0) * E, bytes, &full[s]);
  }
  if (n < N) {
    // a consumer stopped answering: wait (bounded) for the copies still in
    // flight into this CTA's shared memory before leaving
    for (int64_t q = (n > G::STAGES ? n - G::STAGES : 0); q < n; ++q)
      mbar_wait(&full[q % G::STAGES], (uint32_t)((q / G::STAGES) & 1), nullptr);
  }
}

// -------------------------------------------------------------- consumers
template <int E>
__device__ void tpr_flush_aff(const TprParams& p, int* aff, int layer) {
  using G = TprGeo<E>;
  int32_t* dst = p.affinity + (size_t)layer * E * E;
  for (int c = threadIdx.x; c < E * E; c += G::CTHREADS) {
    const int v = aff[c];
    if (v != 0) {
      atomicAdd(&dst[c], v);
      aff[c] = 0;
    }
  }
}

template <int E, int K>
__device__ void tpr_consumer(const TprParams& p, char* smem, int64_t i0, int64_t i1) {
  using G = TprGeo<E>;
  constexpr int WPB = E / 4;  // packed count words per block
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* rows = reinterpret_cast<const float*>(smem + G::OFF_ROWS);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + G::OFF_CNT) + (size_t)warp * G::CNT_WORDS;
  int* aff = reinterpret_cast<int*>(smem + G::OFF_AFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  uint64_t* empty = full + G::STAGES;
  const bool aff_on = p.affinity != nullptr;
  const int64_t N = i1 - i0;
  const int l_first = (int)(i0 / p.ntiles), l_last = (int)((i1 - 1) / p.ntiles);
  const int x4 = 4 * (lane & 7);
  int cur = l_first;
  bool dead = false;
  for (int64_t n = warp; n < N; n += G::CW) {
    const int64_t it = i0 + n;
    const int l = (int)(it / p.ntiles);
    while (aff_on && cur < l) {
      named_bar(1, G::CTHREADS);
      if (!dead) tpr_flush_aff<E>(p, aff, cur);
      named_bar(1, G::CTHREADS);
      ++cur;
    }
    cur = l;
    if (dead) continue;
    const int s = (int)(n % G::STAGES);
    const int64_t tok0 = (it - (int64_t)l * p.ntiles) * G::TT;
    const int ntok = (int)min64(G::TT, p.T - tok0);
    const int slot = p.slot_of_layer[l];
    const bool hist = slot >= 0 && p.blk_cnt != nullptr;
    int tb = 0, nbr = -1;
    if (hist) {
      tb = lane < ntok ? p.tok_blk[tok0 + lane] : 0;
      if (lane == 0 && tok0 > 0) nbr = p.tok_blk[tok0 - 1];
      if (lane == 1 && tok0 + ntok < p.T) nbr = p.tok_blk[tok0 + ntok];
    }
    if (!mbar_wait(&full[s], (uint32_t)((n / G::STAGES) & 1), p.status)) {
      dead = true;
      continue;
    }
    const float* stage = rows + (size_t)s * G::TT * E;
    const float* row = stage + (size_t)lane * E;
    int Tk[8], L9;
    row_top8<E, (K == 8)>(row, lane, Tk, L9);
    // certification of the truncated-key result
    const int nxt = (K == 8) ? L9 : Tk[K < 8 ? K : 7];
    bool bad = (Tk[K - 1] < 256) || (Tk[0] >= 0x7F800000);
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const int a = Tk[i];
      const int b = (i + 1 < K) ? Tk[i + 1] : nxt;
      bad = bad || (b >= (a & (int)0xFFFFFF00));
    }
    const bool live = lane < ntok;
    const unsigned redo = __ballot_sync(FULL, bad && live);
    const bool mine = live && !bad;
    const int blk0 = __shfl_sync(FULL, tb, 0);
    const int lb = tb - blk0;
    int idx[K];
#pragma unroll
    for (int i = 0; i < K; ++i) idx[i] = ((~Tk[i]) & 0xFF) ^ x4;
    const size_t orow = (size_t)l * p.T + tok0;
    if (mine) {
      if (p.topk != nullptr) {
        if constexpr (K == 8) {
          const uint32_t lo = (uint32_t)idx[0] | ((uint32_t)idx[1] << 8) | ((uint32_t)idx[2] << 16) |
                              ((uint32_t)idx[3] << 24);
          const uint32_t hi = (uint32_t)idx[4] | ((uint32_t)idx[5] << 8) | ((uint32_t)idx[6] << 16) |
                              ((uint32_t)idx[7] << 24);
          *reinterpret_cast<uint2*>(p.topk + (orow + lane) * 8) = make_uint2(lo, hi);
        } else {
          uint8_t* o = p.topk + (orow + lane) * K;
#pragma unroll
          for (int i = 0; i < K; i += 2)
            *reinterpret_cast<uint16_t*>(o + i) = (uint16_t)(idx[i] | (idx[i + 1] << 8));
        }
      }
      if (aff_on) {
#pragma unroll
        for (int a = 0; a < K; ++a) {
          int* ra = aff + idx[a] * E;
#pragma unroll
          for (int b = 0; b < K; ++b) atomicAdd(ra + idx[b], 1);
        }
      }
      if (hist) {
#pragma unroll
        for (int i = 0; i < K; ++i) atomicAdd(&cnt[lb * WPB + (idx[i] >> 2)], 1u << ((idx[i] & 3) * 8));
      }
    }
    // rows the fast path could not certify: the whole warp redoes each exactly
    unsigned todo = redo;
    while (todo) {
      const int f = __ffs(todo) - 1;
      todo &= todo - 1;
      const int e = row_topk_exact<E>(stage + (size_t)f * E, K, lane);
      if (p.topk != nullptr && lane < K) p.topk[(orow + f) * K + lane] = (uint8_t)e;
      if (aff_on) {
#pragma unroll
        for (int base = 0; base < K * K; base += 32) {
          const int q = base + lane;
          const int ia = __shfl_sync(FULL, e, q < K * K ? q / K : 0);
          const int ib = __shfl_sync(FULL, e, q < K * K ? q % K : 0);
          if (q < K * K) atomicAdd(&aff[ia * E + ib], 1);
        }
      }
      const int lbf = __shfl_sync(FULL, lb, f);
      if (hist && lane < K) atomicAdd(&cnt[lbf * WPB + (e >> 2)], 1u << ((e & 3) * 8));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (hist) {
      // write this tile's block counts (edge blocks may be shared with the
      // neighbouring tiles: those were zeroed by the pre-pass and take atomics)
      __syncwarp();
      const int blkN = __shfl_sync(FULL, tb, ntok - 1);
      const int before = __shfl_sync(FULL, nbr, 0);
      const int after = __shfl_sync(FULL, nbr, 1);
      const int nb = blkN - blk0 + 1;
      for (int j = 0; j < nb; ++j) {
        const bool partial = (j == 0 && before == blk0) || (j == nb - 1 && after == blkN);
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.blk_cnt + ((size_t)(blk0 + j) * p.m + slot) * E);
        uint32_t* src = cnt + j * WPB;
#pragma unroll
        for (int w = lane; w < WPB; w += 32) {
          const uint32_t v = src[w];
          if (!partial)
            dst[w] = v;
          else if (v != 0u)
            atomicAdd(&dst[w], v);
          src[w] = 0u;
        }
      }
      __syncwarp();
    }
  }
  if (aff_on) {
    while (cur < l_last) {
      named_bar(1, G::CTHREADS);
      if (!dead) tpr_flush_aff<E>(p, aff, cur);
      named_bar(1, G::CTHREADS);
      ++cur;
    }
    named_bar(1, G::CTHREADS);
    if (!dead) tpr_flush_aff<E>(p, aff, cur);
  }
}

template <int E, int K>
__global__ void __launch_bounds__(TprGeo<E>::THREADS, 1) k1_tpr_kernel(const __grid_constant__ TprParams p) {
  using G = TprGeo<E>;
  extern __shared__ __align__(1024) char smem[];
  if (*reinterpret_cast<volatile uint32_t*>(p.call_flag) != 0u) return;
  const int64_t i0 = (int64_t)blockIdx.x * p.nitems / gridDim.x;
  const int64_t i1 = ((int64_t)blockIdx.x + 1) * p.nitems / gridDim.x;
  if (i1 <= i0) return;
  uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + G::OFF_CNT);
  for (size_t w = threadIdx.x; w < G::CW * G::CNT_WORDS; w += G::THREADS) cnt[w] = 0u;
  if (p.affinity != nullptr) {
    int* aff = reinterpret_cast<int*>(smem + G::OFF_AFF);
    for (size_t w = threadIdx.x; w < G::AFF_WORDS; w += G::THREADS) aff[w] = 0;
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
cudaError_t tpr_launch(const TprParams& p, int grid, cudaStream_t st) {
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

cudaError_t tpr_run(int E, int k, const TprParams& p, int grid, cudaStream_t st) {
  if (E == 128 && k == 8) return tpr_launch<128, 8>(p, grid, st);
  if (E == 128 && k == 6) return tpr_launch<128, 6>(p, grid, st);
  if (E == 64 && k == 8) return tpr_launch<64, 8>(p, grid, st);
  return tpr_launch<64, 6>(p, grid, st);
}

}  // namespace moer
