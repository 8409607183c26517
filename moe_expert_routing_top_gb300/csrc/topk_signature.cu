// topk_signature.cu -- moer_topk_signature: top-k gating, per-layer expert
// co-activation and per-KV-block signature counts from the router logits.
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
// The call runs two kernels on the caller's stream:
//   1. one pass over the logits that selects every row's top-k and adds the
//      row's k*k ordered expert pairs to the co-activation counts
//      (thread-per-row kernel in topk_signature_tpr.cu for E = 64 / 128 with
//      k = 6 / 8; the general kernel below for every other shape), writing
//      the top-k ids;
//   2. the segmented block histogram of block_counts.cu over those ids.
//
// General kernel (any E <= 256 with E % 4 == 0, any k <= 32):
//   * Persistent grid, one 544-thread CTA per SM.  Work items are
//     (layer, token tile) pairs in layer-major order; each CTA takes a
//     contiguous range, so its co-activation tile spans few layers.
//   * A producer warp streams each tile of logit rows (TT rows x E fp32,
//     contiguous in HBM) into shared memory with one cp.async.bulk copy
//     completing on an mbarrier.  All sixteen consumer warps share every
//     stage (rows split among them), so each warp meets every stage's
//     barrier phases in order.
//   * Warp per row: lanes hold E/32 order-preserving 32-bit keys and k
//     rounds of redux.sync.max with ballot tie-breaking pick the experts,
//     ties to the lower id.
//   * Co-activation pairs go to a shared-memory E x (E+1) int32 tile with
//     shared atomics (global atomics when E > 128), flushed when the CTA's
//     layer changes.
#include <climits>

#include "common.cuh"
#include "k1_params.cuh"
#include "rank.cuh"

namespace moer {

moer_status block_counts_launch(const moer_dims* d, const uint8_t* ids, bool mask_only, int64_t T,
                                const int32_t* blk_tab, int nblk, uint8_t* blk_cnt, uint32_t* status,
                                cudaStream_t st, bool check);

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <int EPL>
struct K1Geo {
  static constexpr int EMAX = 32 * EPL;
  static constexpr int TT = (EPL <= 2) ? 128 : (EPL == 4 ? 64 : 32);
  static constexpr int STAGES = 4;
  static constexpr bool SMEM_AFF = EPL <= 4;
  static constexpr int CWARPS = 16;
  static constexpr int CTHREADS = CWARPS * 32;
  static constexpr int THREADS = CTHREADS + 32;
  static constexpr size_t STAGE_BYTES = (size_t)TT * EMAX * 4;
  static constexpr size_t OFF_ROWS = 0;
  static constexpr size_t OFF_AFF = OFF_ROWS + STAGES * STAGE_BYTES;
  static constexpr size_t AFF_WORDS = SMEM_AFF ? (size_t)EMAX * (EMAX + 1) : 0;
  static constexpr size_t OFF_BAR = align_up(OFF_AFF + AFF_WORDS * 4, 16);
  static constexpr size_t SMEM = OFF_BAR + 2 * STAGES * 8;
};

int k1_tile_tokens(int E) {
  if (E <= 64) return K1Geo<2>::TT;
  if (E <= 128) return K1Geo<4>::TT;
  return K1Geo<8>::TT;
}

// Workspace after the header: the top-k ids of the mask layers, [m][T][k],
// used when the caller does not ask for the ids itself.
size_t k1_scratch_bytes(const moer_dims* d, int64_t T) {
  return ((size_t)d->m * (size_t)T * (size_t)d->k + 255) / 256 * 256;
}

// ----------------------------------------------------------- row selection
// Adds the k*k ordered pairs of one row (ids in lanes r < k) to a counter
// matrix with row stride `stride`.
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
__device__ void k1_producer(const K1Params& p, char* smem, int64_t i0, int64_t i1) {
  using G = K1Geo<EPL>;
  if ((threadIdx.x & 31) != 0) return;
  float* rows = reinterpret_cast<float*>(smem + G::OFF_ROWS);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  uint64_t* empty = full + G::STAGES;
  const int64_t N = i1 - i0;
  int cl = (int)(i0 / p.ntiles), ct = (int)(i0 % p.ntiles);
  int64_t n = 0;
  for (; n < N; ++n) {
    const int s = (int)(n % G::STAGES);
    if (n >= G::STAGES && !mbar_wait(&empty[s], (uint32_t)((n / G::STAGES - 1) & 1), p.status)) break;
    const int64_t tok0 = (int64_t)ct * G::TT;
    const uint32_t bytes = (uint32_t)min64(G::TT, p.T - tok0) * (uint32_t)p.E * 4u;
    mbar_arrive_expect_tx(&full[s], bytes);
    bulk_g2s(rows + (size_t)s * G::TT * G::EMAX, p.logits + ((size_t)cl * p.T + tok0) * p.E, bytes,
             &full[s]);
    if (++ct == p.ntiles) {
      ct = 0;
      ++cl;
    }
  }
  if (n < N) {
    // a consumer stopped answering: wait (bounded) for the copies still in
    // flight into this CTA's shared memory before leaving
    for (int64_t q = (n > G::STAGES ? n - G::STAGES : 0); q < n; ++q)
      mbar_wait(&full[q % G::STAGES], (uint32_t)((q / G::STAGES) & 1), nullptr);
  }
}

// --------------------------------------------------------------- consumers
template <int EPL>
__device__ void k1_flush_aff(const K1Params& p, int* aff, int layer) {
  const int E = p.E, stride = E + 1;
  int32_t* dst = p.affinity + (size_t)layer * E * E;
  for (int c = threadIdx.x; c < E * E; c += K1Geo<EPL>::CTHREADS) {
    const int a = c / E, b = c - a * E;
    const int v = aff[a * stride + b];
    if (v != 0) {
      atomicAdd(&dst[c], v);
      aff[a * stride + b] = 0;
    }
  }
}

template <int EPL>
__device__ void k1_consumer(const K1Params& p, char* smem, int64_t i0, int64_t i1) {
  using G = K1Geo<EPL>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* rows = reinterpret_cast<const float*>(smem + G::OFF_ROWS);
  int* aff = reinterpret_cast<int*>(smem + G::OFF_AFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  uint64_t* empty = full + G::STAGES;
  const bool aff_on = p.affinity != nullptr;
  const int k = p.k;
  const int stride = p.E + 1;
  bool dead = false;
  int l = (int)(i0 / p.ntiles), tile = (int)(i0 % p.ntiles);
  int cur = l;
  for (int64_t it = i0; it < i1; ++it) {
    if (it > i0 && ++tile == p.ntiles) {
      tile = 0;
      ++l;
    }
    const int64_t n = it - i0;
    const int s = (int)(n % G::STAGES);
    if (G::SMEM_AFF && aff_on && l != cur) {
      named_bar(1, G::CTHREADS);
      if (!dead) k1_flush_aff<EPL>(p, aff, cur);
      named_bar(1, G::CTHREADS);
    }
    cur = l;
    if (dead) continue;
    if (!mbar_wait(&full[s], (uint32_t)((n / G::STAGES) & 1), p.status)) {
      dead = true;
      continue;
    }
    const int64_t tok0 = (int64_t)tile * G::TT;
    const int ntok = (int)min64(G::TT, p.T - tok0);
    const float* stage = rows + (size_t)s * G::TT * G::EMAX;
    const int slot = p.slot_of_layer[l];
    uint8_t* out = nullptr;
    if (p.ids != nullptr && (!p.ids_mask_only || slot >= 0))
      out = p.ids + ((size_t)(p.ids_mask_only ? slot : l) * p.T + tok0) * k;
    for (int r = warp; r < ntok; r += G::CWARPS) {
      const int myidx = warp_topk_exact<EPL>(stage + (size_t)r * p.E, p.E, k, lane);
      if (out != nullptr && lane < k) out[(size_t)r * k + lane] = (uint8_t)myidx;
      if (aff_on) {
        if constexpr (G::SMEM_AFF)
          aff_pairs_any(aff, stride, myidx, k, lane);
        else
          aff_pairs_any(p.affinity + (size_t)l * p.E * p.E, p.E, myidx, k, lane);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (G::SMEM_AFF && aff_on) {
    named_bar(1, G::CTHREADS);
    if (!dead) k1_flush_aff<EPL>(p, aff, cur);
  }
}

template <int EPL>
__global__ void __launch_bounds__(K1Geo<EPL>::THREADS, 1) k1_kernel(const __grid_constant__ K1Params p) {
  using G = K1Geo<EPL>;
  extern __shared__ __align__(128) char smem[];
  const int64_t i0 = (int64_t)blockIdx.x * p.nitems / gridDim.x;
  const int64_t i1 = ((int64_t)blockIdx.x + 1) * p.nitems / gridDim.x;
  if (i1 <= i0) return;
  if constexpr (G::SMEM_AFF) {
    int* aff = reinterpret_cast<int*>(smem + G::OFF_AFF);
    if (p.affinity != nullptr)
      for (size_t w = threadIdx.x; w < G::AFF_WORDS; w += G::THREADS) aff[w] = 0;
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::OFF_BAR);
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&full[G::STAGES + s], G::CWARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x >= G::CTHREADS)
    k1_producer<EPL>(p, smem, i0, i1);
  else
    k1_consumer<EPL>(p, smem, i0, i1);
}

// ------------------------------------------------------------------ launch
template <int EPL>
cudaError_t k1_launch(const K1Params& p, int grid, cudaStream_t st) {
  using G = K1Geo<EPL>;
  static std::atomic<unsigned long long> set{0};
  const cudaError_t e = smem_optin(k1_kernel<EPL>, (int)G::SMEM, set);
  if (e != cudaSuccess) return e;
  k1_kernel<EPL><<<grid, G::THREADS, G::SMEM, st>>>(p);
  return cudaGetLastError();
}

// Host side of moer_topk_signature after argument validation.
moer_status topk_signature_launch(const moer_dims* d, const float* logits, int64_t T,
                                  const int32_t* blk_tab, int32_t nblk, uint8_t* topk,
                                  uint8_t* blk_cnt, int32_t* affinity, void* ws, cudaStream_t st) {
  const int E = d->E, k = d->k;
  const bool tpr = tpr_supported(E, k);
  const int TT = tpr ? tpr_tile_tokens(E) : k1_tile_tokens(E);
  const int ntiles = (int)((T + TT - 1) / TT);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  const bool hist = blk_cnt != nullptr && d->m > 0;
  // ids for the block histogram: the caller's top-k, else mask layers in ws
  uint8_t* ids = topk;
  bool mask_only = false;
  if (ids == nullptr && hist) {
    ids = static_cast<uint8_t*>(ws) + WS_HEADER;
    mask_only = true;
  }
  const int sms = device_sm_count();
  if (sms <= 0) return MOER_ECUDA;
  K1Params p;
  p.logits = logits;
  p.T = T;
  p.E = E;
  p.k = k;
  p.L = d->L;
  p.ids = ids;
  p.ids_mask_only = mask_only ? 1 : 0;
  p.affinity = affinity;
  p.ntiles = ntiles;
  p.tail_rows = (int)(T - (int64_t)(ntiles - 1) * TT);
  p.nitems = (int64_t)d->L * ntiles;
  p.status = status;
  p.key_hi_mul = 1u << 24;
  p.key_lo_mul = 1u << 8;
  p.aff_row_bytes = (uint32_t)(d->E + 1) * 4u;  // the 32-bit tile's row pitch (E + 1 words)
  p.aff_pairs64 = (reinterpret_cast<uintptr_t>(affinity) & 7u) == 0 ? 1 : 0;
  for (int l = 0; l < 256; ++l) p.slot_of_layer[l] = -1;
  for (int i = 0; i < d->m; ++i) p.slot_of_layer[d->mask[i]] = (int16_t)i;
  const int grid = (int)min64(p.nitems, sms);
  // a CTA counts its work items in 32 bits
  if (grid > 0 && (p.nitems + grid - 1) / grid >= (int64_t(1) << 31)) return MOER_ERANGE;
  cudaError_t e;
  if (tpr)
    e = tpr_run(E, k, p, grid, st);
  else if (E <= 32)
    e = k1_launch<1>(p, grid, st);
  else if (E <= 64)
    e = k1_launch<2>(p, grid, st);
  else if (E <= 128)
    e = k1_launch<4>(p, grid, st);
  else
    e = k1_launch<8>(p, grid, st);
  if (e != cudaSuccess) return MOER_ECUDA;
  if (!hist) return MOER_OK;
  return block_counts_launch(d, ids, mask_only, T, blk_tab, nblk, blk_cnt, status, st, false);
}

}  // namespace moer
