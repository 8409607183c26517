// api.cu -- the extern "C" entry points of libmoeroute: argument validation,
// workspace accounting and dispatch to the kernels.  Nothing here computes
// routing statistics; every step runs on the GPU.
#include <cuda.h>

#include <atomic>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "extent.h"

namespace moer {
size_t spectral_workspace_bytes(int L, int E, int G);
moer_status spectral_launch(const moer_dims* d, const int32_t* affinity, int32_t G, int32_t* group_of,
                            int32_t* knee, double* u_curve, double* s_curve, void* ws, cudaStream_t st);
size_t mask_select_workspace_bytes(int32_t L, int32_t R);
moer_status mask_select_launch(const moer_dims* d, const uint8_t* topk, int64_t T, const int32_t* req_off, int32_t R,
                               const float* idf, int32_t m, int32_t* mask_out, double* quality_out, void* ws,
                               cudaStream_t st);
moer_status replication_plan_launch(const moer_dims* d, const int64_t* W, const int32_t* group_of, int32_t G,
                                    int32_t* n_rep, int32_t* src, uint8_t* hot, int32_t* dst, double* w_pred,
                                    uint32_t* status, cudaStream_t st);
size_t kmeans_workspace_bytes(int32_t N, int32_t dim, int32_t D);
moer_status kmeans_launch(const float* sig, int32_t N, int32_t dim, int32_t D, const float* init, int32_t max_iter,
                          float* centroids, int32_t* assign, int32_t* info, double* objective, void* ws,
                          cudaStream_t st);
size_t k1_scratch_bytes(const moer_dims* d, int64_t T);
moer_status wait_selftest_launch(void* ws, uint32_t limit_us, cudaStream_t st);
moer_status topk_signature_launch(const moer_dims* d, const float* logits, int64_t T,
                                  const int32_t* blk_tab, int32_t nblk, uint8_t* topk,
                                  uint8_t* blk_cnt, int32_t* affinity, void* ws, cudaStream_t st);
moer_status block_stitch_launch(const moer_dims* d, const uint8_t* blk_cnt, const int32_t* blk_tab,
                                int32_t nblk, const int32_t* req_blk_off, int32_t R,
                                const int32_t* cache_idx, int32_t ncached, const int32_t* req_cache_off,
                                uint8_t* cache, int32_t nslots, const int32_t* insert_slot,
                                int32_t* req_cnt, uint32_t* status, cudaStream_t st);
moer_status affinity_load_launch(const moer_dims* d, const int32_t* affinity, const int32_t* group_of,
                                 int32_t G, int64_t* W_expert, int64_t* W_group, double* rho_group,
                                 double* rho_expert, cudaStream_t st);
size_t route_scratch_bytes(int32_t R);
moer_status route_launch(const moer_dims* d, const int32_t* req_cnt, int32_t R, const float* idf,
                         const float* centroids, int32_t D, float tau, int32_t* loads, int32_t live,
                         float* sig, float* dist, int32_t* choice, void* ws, cudaStream_t st);
moer_status idf_fit_launch(const moer_dims* d, const int32_t* req_cnt, int32_t R, float* idf,
                           cudaStream_t st);
size_t gate_scratch_bytes(const moer_dims* d, int32_t H);
moer_status gate_topk_launch(const moer_dims* d, const uint16_t* hidden, int64_t T, int32_t H,
                             const uint16_t* w_gate, float* logits, uint8_t* topk, void* ws, cudaStream_t st);
moer_status affinity_ids_launch(const moer_dims* d, const uint8_t* ids, int64_t T, int32_t* affinity,
                                cudaStream_t st, uint32_t* status, bool check);
moer_status block_counts_launch(const moer_dims* d, const uint8_t* ids, bool mask_only, int64_t T,
                                const int32_t* blk_tab, int nblk, uint8_t* blk_cnt, uint32_t* status,
                                cudaStream_t st, bool check);

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------- checked mode
// Off by default; on with moer_set_extent_checks(1) or MOER_CHECK_EXTENTS=1 in
// the environment (read at the first call).  -1: not read yet.
std::atomic<int> g_extent_checks{-1};

bool extent_checks_on() {
  int v = g_extent_checks.load(std::memory_order_acquire);
  if (v < 0) {
    const char* e = std::getenv("MOER_CHECK_EXTENTS");
    const int want = (e != nullptr && e[0] != '\0' && e[0] != '0') ? 1 : 0;
    int expected = -1;
    g_extent_checks.compare_exchange_strong(expected, want, std::memory_order_acq_rel);
    v = g_extent_checks.load(std::memory_order_acquire);
  }
  return v == 1;
}

using AddrRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);

// The driver's cuMemGetAddressRange, resolved through the runtime (the library
// does not link libcuda directly).
AddrRangeFn addr_range_fn() {
  static const AddrRangeFn fn = []() -> AddrRangeFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<AddrRangeFn>(f);
  }();
  return fn;
}

bool device_range(uintptr_t p, uintptr_t* base, size_t* size) {
  const AddrRangeFn fn = addr_range_fn();
  if (fn == nullptr) return false;
  CUdeviceptr b = 0;
  size_t n = 0;
  if (fn(&b, &n, static_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) return false;
  *base = static_cast<uintptr_t>(b);
  *size = n;
  return true;
}

// MOER_EEXTENT when checked mode is on and a buffer's allocation cannot hold
// its extent, else MOER_OK.  Sizes are computed by the caller in size_t.
moer_status check_extents(std::initializer_list<Extent> list) {
  if (!extent_checks_on()) return MOER_OK;
  return first_bad_extent(list, device_range) < 0 ? MOER_OK : MOER_EEXTENT;
}

size_t sz(int64_t a) { return a > 0 ? static_cast<size_t>(a) : 0; }


moer_status check_dims(const moer_dims* d, bool need_mask) {
  if (d == nullptr) return MOER_EINVAL;
  if (d->E < 4 || d->E > 256 || d->E % 4 != 0) return MOER_ERANGE;
  if (d->k < 1 || d->k > 32 || d->k > d->E) return MOER_ERANGE;
  if (d->L < 1 || d->L > 256) return MOER_ERANGE;
  if (d->m < 0 || d->m > d->L) return MOER_ERANGE;
  if (d->block < 1 || d->block > 255) return MOER_ERANGE;
  if (d->m > 0 || need_mask) {
    if (d->m > 0 && d->mask == nullptr) return MOER_EINVAL;
    for (int i = 0; i < d->m; ++i) {
      if (d->mask[i] < 0 || d->mask[i] >= d->L) return MOER_ERANGE;
      if (i > 0 && d->mask[i] <= d->mask[i - 1]) return MOER_EINVAL;
    }
  }
  return MOER_OK;
}

// Extents of the logits-pass buffers (moer_topk_signature and its no-alloc form).
moer_status topk_signature_extents(const moer_dims* d, const float* logits, int64_t T, const int32_t* blk_tab,
                                   int32_t nblk, const uint8_t* topk, const uint8_t* blk_cnt,
                                   const int32_t* affinity, const void* ws, size_t ws_bytes, bool hist) {
  const size_t L = sz(d->L), E = sz(d->E), k = sz(d->k), m = sz(d->m), t = sz(T), nb = sz(nblk);
  return check_extents({{logits, L * t * E * 4},
                        {hist ? blk_tab : nullptr, nb * 2 * 4},
                        {topk, L * t * k},
                        {hist ? blk_cnt : nullptr, nb * m * E},
                        {affinity, L * E * E * 4},
                        {ws, ws_bytes}});
}

}  // namespace

// Host-side argument check of moer_topk_signature_noalloc: the same checks as
// moer_topk_signature except the workspace, which that entry point does not take.
moer_status topk_signature_check(const moer_dims* d, const float* logits, int64_t T,
                                 const int32_t* blk_tab, int32_t nblk, const uint8_t* topk,
                                 const uint8_t* blk_cnt, const int32_t* affinity) {
  moer_status s = check_dims(d, false);
  if (s != MOER_OK) return s;
  if (T < 0 || nblk < 0) return MOER_ERANGE;
  if (T >= (int64_t(1) << 31)) return MOER_ERANGE;
  if (T == 0) return MOER_OK;
  if (logits == nullptr || !aligned(logits, 16)) return MOER_EINVAL;
  if (affinity != nullptr && !aligned(affinity, 4)) return MOER_EINVAL;
  if (topk != nullptr && !aligned(topk, 8)) return MOER_EINVAL;
  if (blk_cnt != nullptr && d->m > 0) {
    if (blk_tab == nullptr || !aligned(blk_tab, 4) || !aligned(blk_cnt, 4)) return MOER_EINVAL;
    if (nblk < 1 || nblk > T) return MOER_ESHAPE;
  }
  return MOER_OK;
}

// Checked mode's extents for moer_topk_signature_noalloc (after its own
// argument and staging-size checks, as in the workspace form).
moer_status topk_signature_noalloc_extents(const moer_dims* d, const float* logits, int64_t T,
                                           const int32_t* blk_tab, int32_t nblk, const uint8_t* topk,
                                           const uint8_t* blk_cnt, const int32_t* affinity) {
  const bool hist = blk_cnt != nullptr && d->m > 0;
  return topk_signature_extents(d, logits, T, blk_tab, nblk, topk, blk_cnt, affinity, nullptr, 0, hist);
}
}  // namespace moer

using namespace moer;

extern "C" {

size_t moer_workspace_bytes(const moer_dims* d, int64_t T, int32_t nblk, int32_t R, int32_t D) {
  (void)nblk;
  size_t scratch = 0;
  if (d != nullptr && T > 0 && d->m > 0 && d->m <= 256 && d->k > 0) scratch = k1_scratch_bytes(d, T);
  if (R > 0 && D > 0) {
    const size_t route = route_scratch_bytes(R);
    scratch = route > scratch ? route : scratch;
  }
  return WS_HEADER + scratch;
}

moer_status moer_topk_signature(const moer_dims* d, const float* logits, int64_t T,
                                const int32_t* blk_tab, int32_t nblk, uint8_t* topk,
                                uint8_t* blk_cnt, int32_t* affinity, void* ws, size_t ws_bytes,
                                moer_stream_t stream) {
  moer_status s = check_dims(d, false);
  if (s != MOER_OK) return s;
  if (T < 0 || nblk < 0) return MOER_ERANGE;
  if (T >= (int64_t(1) << 31)) return MOER_ERANGE;
  if (T == 0) return MOER_OK;
  if (logits == nullptr || !aligned(logits, 16)) return MOER_EINVAL;
  if (affinity != nullptr && !aligned(affinity, 4)) return MOER_EINVAL;
  if (topk != nullptr && !aligned(topk, 8)) return MOER_EINVAL;
  const bool hist = blk_cnt != nullptr && d->m > 0;
  if (hist) {
    if (blk_tab == nullptr || !aligned(blk_tab, 4) || !aligned(blk_cnt, 4)) return MOER_EINVAL;
    if (nblk < 1 || nblk > T) return MOER_ESHAPE;
  }
  if (ws == nullptr || !aligned(ws, 16)) return MOER_EINVAL;
  if (ws_bytes < moer_workspace_bytes(d, T, nblk, 0, 0)) return MOER_ENOMEM;
  s = topk_signature_extents(d, logits, T, blk_tab, nblk, topk, blk_cnt, affinity, ws, ws_bytes, hist);
  if (s != MOER_OK) return s;
  return topk_signature_launch(d, logits, T, blk_tab, nblk, topk, blk_cnt, affinity, ws,
                               reinterpret_cast<cudaStream_t>(stream));
}

moer_status moer_block_stitch(const moer_dims* d, const uint8_t* blk_cnt, const int32_t* blk_tab,
                              int32_t nblk, const int32_t* req_blk_off, int32_t R,
                              const int32_t* cache_idx, int32_t ncached, const int32_t* req_cache_off,
                              uint8_t* cache, int32_t nslots, const int32_t* insert_slot,
                              int32_t* req_cnt, void* ws, size_t ws_bytes, moer_stream_t stream) {
  moer_status s = check_dims(d, true);
  if (s != MOER_OK) return s;
  if (d->m < 1) return MOER_ERANGE;
  if (R < 0 || nblk < 0 || nslots < 0 || ncached < 0) return MOER_ERANGE;
  if (R == 0) return MOER_OK;
  if (req_blk_off == nullptr || req_cnt == nullptr) return MOER_EINVAL;
  if (nblk > 0 && (blk_cnt == nullptr || !aligned(blk_cnt, 4))) return MOER_EINVAL;
  const bool has_cache = cache != nullptr;
  if (has_cache) {
    if (!aligned(cache, 4) || req_cache_off == nullptr) return MOER_EINVAL;
    if (ncached > 0 && cache_idx == nullptr) return MOER_EINVAL;
    if (insert_slot != nullptr && blk_tab == nullptr) return MOER_EINVAL;
  } else if (cache_idx != nullptr || req_cache_off != nullptr || insert_slot != nullptr || ncached != 0) {
    return MOER_EINVAL;
  }
  if (ws != nullptr && (!aligned(ws, 16) || ws_bytes < WS_HEADER)) return MOER_ENOMEM;
  {
    const size_t rec = sz(d->m) * sz(d->E), nb = sz(nblk), r1 = sz(R) + 1;
    s = check_extents({{blk_cnt, nb * rec},
                       {(has_cache && insert_slot != nullptr) ? blk_tab : nullptr, nb * 2 * 4},
                       {req_blk_off, r1 * 4},
                       {cache_idx, sz(ncached) * 4},
                       {req_cache_off, r1 * 4},
                       {cache, sz(nslots) * rec},
                       {insert_slot, nb * 4},
                       {req_cnt, sz(R) * rec * 4},
                       {ws, ws_bytes}});
    if (s != MOER_OK) return s;
  }
  return block_stitch_launch(d, blk_cnt, blk_tab, nblk, req_blk_off, R, cache_idx, ncached, req_cache_off,
                             cache, nslots, insert_slot, req_cnt,
                             ws ? reinterpret_cast<uint32_t*>(ws) : nullptr,
                             reinterpret_cast<cudaStream_t>(stream));
}

moer_status moer_affinity_load(const moer_dims* d, const int32_t* affinity, const int32_t* group_of,
                               int32_t G, int64_t* W_expert, int64_t* W_group, double* rho_group,
                               double* rho_expert, moer_stream_t stream) {
  moer_status s = check_dims(d, false);
  if (s != MOER_OK) return s;
  if (affinity == nullptr) return MOER_EINVAL;
  if ((W_group != nullptr || rho_group != nullptr)) {
    if (group_of == nullptr) return MOER_EINVAL;
    if (G < 1 || G > 4096) return MOER_ERANGE;
  }
  if (G < 1) G = 1;
  {
    const size_t L = sz(d->L), E = sz(d->E), g = sz(G);
    const bool groups = W_group != nullptr || rho_group != nullptr;
    s = check_extents({{affinity, L * E * E * 4},
                       {groups ? group_of : nullptr, L * E * 4},
                       {W_expert, L * E * 8},
                       {W_group, L * g * 8},
                       {rho_group, L * 8},
                       {rho_expert, L * 8}});
    if (s != MOER_OK) return s;
  }
  return affinity_load_launch(d, affinity, group_of, G, W_expert, W_group, rho_group, rho_expert,
                              reinterpret_cast<cudaStream_t>(stream));
}

moer_status moer_route(const moer_dims* d, const int32_t* req_cnt, int32_t R, const float* idf,
                       const float* centroids, int32_t D, float tau, int32_t* loads, int32_t live,
                       float* sig, float* dist, int32_t* choice, void* ws, size_t ws_bytes,
                       moer_stream_t stream) {
  moer_status s = check_dims(d, true);
  if (s != MOER_OK) return s;
  if (d->m < 1) return MOER_ERANGE;
  if (R < 0 || D < 1 || D > 64) return MOER_ERANGE;
  if (live != 0 && live != 1) return MOER_EINVAL;
  if (!(tau >= 0.f)) return MOER_ERANGE;
  if (R == 0) return MOER_OK;
  if (req_cnt == nullptr || idf == nullptr || centroids == nullptr || loads == nullptr ||
      choice == nullptr)
    return MOER_EINVAL;
  if (live) {  // the band masks of live routing live in the workspace
    if (ws == nullptr || !aligned(ws, 16)) return MOER_EINVAL;
    if (ws_bytes < moer_workspace_bytes(d, 0, 0, R, D)) return MOER_ENOMEM;
  }
  {
    const size_t dim = sz(d->m) * sz(d->E), r = sz(R), nd = sz(D);
    s = check_extents({{req_cnt, r * dim * 4},
                       {idf, dim * 4},
                       {centroids, nd * dim * 4},
                       {loads, nd * 4},
                       {sig, r * dim * 4},
                       {dist, r * nd * 4},
                       {choice, r * 4},
                       {live ? ws : nullptr, ws_bytes}});
    if (s != MOER_OK) return s;
  }
  return route_launch(d, req_cnt, R, idf, centroids, D, tau, loads, live, sig, dist, choice, ws,
                      reinterpret_cast<cudaStream_t>(stream));
}

moer_status moer_idf_fit(const moer_dims* d, const int32_t* req_cnt, int32_t R, float* idf,
                         moer_stream_t stream) {
  moer_status s = check_dims(d, true);
  if (s != MOER_OK) return s;
  if (d->m < 1) return MOER_ERANGE;
  if (R < 1) return MOER_ERANGE;
  if (req_cnt == nullptr || idf == nullptr) return MOER_EINVAL;
  s = check_extents({{req_cnt, sz(R) * sz(d->m) * sz(d->E) * 4}, {idf, sz(d->m) * sz(d->E) * 4}});
  if (s != MOER_OK) return s;
  return idf_fit_launch(d, req_cnt, R, idf, reinterpret_cast<cudaStream_t>(stream));
}

size_t moer_gate_workspace_bytes(const moer_dims* d, int32_t H) {
  if (d == nullptr || d->L < 1 || H < 1) return WS_HEADER;
  return WS_HEADER + gate_scratch_bytes(d, H);
}

moer_status moer_gate_topk(const moer_dims* d, const uint16_t* hidden, int64_t T, int32_t H,
                           const uint16_t* w_gate, const int32_t* blk_tab, int32_t nblk, float* logits,
                           uint8_t* topk, uint8_t* blk_cnt, int32_t* affinity, void* ws, size_t ws_bytes,
                           moer_stream_t stream) {
  moer_status s = check_dims(d, false);
  if (s != MOER_OK) return s;
  if (d->E != 128 || (d->k != 8 && d->k != 6)) return MOER_ERANGE;
  if (H < 64 || H % 64 != 0 || H > 65536) return MOER_ERANGE;
  if (T < 0 || T >= (int64_t(1) << 31) || nblk < 0) return MOER_ERANGE;
  if (T == 0) return MOER_OK;
  if (hidden == nullptr || w_gate == nullptr || topk == nullptr) return MOER_EINVAL;
  if (!aligned(hidden, 16) || !aligned(w_gate, 16) || !aligned(topk, 8)) return MOER_EINVAL;
  if (logits != nullptr && !aligned(logits, 16)) return MOER_EINVAL;
  if (affinity != nullptr && !aligned(affinity, 4)) return MOER_EINVAL;
  const bool hist = blk_cnt != nullptr && d->m > 0;
  if (hist) {
    if (blk_tab == nullptr || !aligned(blk_tab, 4) || !aligned(blk_cnt, 4)) return MOER_EINVAL;
    if (nblk < 1 || nblk > T) return MOER_ESHAPE;
  }
  if (ws == nullptr || !aligned(ws, 256)) return MOER_EINVAL;
  if (ws_bytes < moer_gate_workspace_bytes(d, H)) return MOER_ENOMEM;
  {
    const size_t L = sz(d->L), E = sz(d->E), k = sz(d->k), m = sz(d->m), t = sz(T), h = sz(H), nb = sz(nblk);
    s = check_extents({{hidden, t * h * 2},
                       {w_gate, L * h * E * 2},
                       {hist ? blk_tab : nullptr, nb * 2 * 4},
                       {logits, L * t * E * 4},
                       {topk, L * t * k},
                       {hist ? blk_cnt : nullptr, nb * m * E},
                       {affinity, L * E * E * 4},
                       {ws, ws_bytes}});
    if (s != MOER_OK) return s;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  s = gate_topk_launch(d, hidden, T, H, w_gate, logits, topk, ws, st);
  if (s != MOER_OK) return s;
  if (affinity != nullptr) {
    s = affinity_ids_launch(d, topk, T, affinity, st, reinterpret_cast<uint32_t*>(ws), false);
    if (s != MOER_OK) return s;
  }
  if (hist)
    s = block_counts_launch(d, topk, false, T, blk_tab, nblk, blk_cnt, reinterpret_cast<uint32_t*>(ws), st, false);
  return s;
}

moer_status moer_ids_signature(const moer_dims* d, const uint8_t* topk, int64_t T, const int32_t* blk_tab,
                               int32_t nblk, uint8_t* blk_cnt, int32_t* affinity, void* ws, size_t ws_bytes,
                               moer_stream_t stream) {
  moer_status s = check_dims(d, false);
  if (s != MOER_OK) return s;
  if (T < 0 || T >= (int64_t(1) << 31) || nblk < 0) return MOER_ERANGE;
  if (T == 0) return MOER_OK;
  if (topk == nullptr || !aligned(topk, 8)) return MOER_EINVAL;
  const bool hist = blk_cnt != nullptr && d->m > 0;
  if (hist) {
    if (blk_tab == nullptr || !aligned(blk_tab, 4) || !aligned(blk_cnt, 4)) return MOER_EINVAL;
    if (nblk < 1 || nblk > T) return MOER_ESHAPE;
  }
  if (affinity != nullptr) {
    if (!aligned(affinity, 4)) return MOER_EINVAL;
    if (d->E > 128 || (d->k != 8 && d->k != 6)) return MOER_ERANGE;
  }
  if (ws == nullptr || !aligned(ws, 16)) return MOER_EINVAL;
  if (ws_bytes < WS_HEADER) return MOER_ENOMEM;
  {
    const size_t L = sz(d->L), E = sz(d->E), k = sz(d->k), m = sz(d->m), t = sz(T), nb = sz(nblk);
    s = check_extents({{topk, L * t * k},
                       {hist ? blk_tab : nullptr, nb * 2 * 4},
                       {hist ? blk_cnt : nullptr, nb * m * E},
                       {affinity, L * E * E * 4},
                       {ws, ws_bytes}});
    if (s != MOER_OK) return s;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  if (affinity != nullptr) {
    s = affinity_ids_launch(d, topk, T, affinity, st, status, true);
    if (s != MOER_OK) return s;
  }
  if (hist) s = block_counts_launch(d, topk, false, T, blk_tab, nblk, blk_cnt, status, st, true);
  return s;
}

moer_status moer_replication_plan(const moer_dims* d, const int64_t* W, const int32_t* group_of, int32_t G,
                                  int32_t* n_rep, int32_t* src, uint8_t* hot, int32_t* dst, double* w_pred,
                                  void* ws, size_t ws_bytes, moer_stream_t stream) {
  moer_status s = check_dims(d, false);
  if (s != MOER_OK) return s;
  if (G < 1 || G > 64) return MOER_ERANGE;
  if (W == nullptr || group_of == nullptr || n_rep == nullptr || src == nullptr || hot == nullptr ||
      dst == nullptr || w_pred == nullptr)
    return MOER_EINVAL;
  if (!aligned(W, 8) || !aligned(w_pred, 8) || !aligned(group_of, 4) || !aligned(n_rep, 4) || !aligned(src, 4) ||
      !aligned(dst, 4))
    return MOER_EINVAL;
  if (ws == nullptr || !aligned(ws, 256)) return MOER_EINVAL;
  if (ws_bytes < WS_HEADER) return MOER_ENOMEM;
  {
    const size_t L = sz(d->L), E = sz(d->E), g = sz(G);
    s = check_extents({{W, L * E * 8}, {group_of, L * E * 4}, {n_rep, L * 4}, {src, L * 4}, {hot, L * E},
                       {dst, L * g * 4}, {w_pred, L * g * 8}, {ws, ws_bytes}});
    if (s != MOER_OK) return s;
  }
  return moer::replication_plan_launch(d, W, group_of, G, n_rep, src, hot, dst, w_pred,
                                       reinterpret_cast<uint32_t*>(ws), reinterpret_cast<cudaStream_t>(stream));
}

size_t moer_mask_select_workspace_bytes(const moer_dims* d, int32_t R) {
  if (d == nullptr || d->L < 1 || R < 1) return WS_HEADER;
  return moer::mask_select_workspace_bytes(d->L, R);
}

moer_status moer_mask_select(const moer_dims* d, const uint8_t* topk, int64_t T, const int32_t* req_off, int32_t R,
                             const float* idf, int32_t m, int32_t* mask_out, double* quality_out, void* ws,
                             size_t ws_bytes, moer_stream_t stream) {
  moer_status s = check_dims(d, false);
  if (s != MOER_OK) return s;
  if (R < 1 || T < 1 || m < 1 || m > d->L) return MOER_ERANGE;
  if (topk == nullptr || req_off == nullptr || mask_out == nullptr) return MOER_EINVAL;
  if (!aligned(req_off, 4) || !aligned(mask_out, 4) || (idf != nullptr && !aligned(idf, 4)) ||
      (quality_out != nullptr && !aligned(quality_out, 8)))
    return MOER_EINVAL;
  if (ws == nullptr || !aligned(ws, 256)) return MOER_EINVAL;
  if (ws_bytes < moer_mask_select_workspace_bytes(d, R)) return MOER_ENOMEM;
  {
    const size_t L = sz(d->L), E = sz(d->E), k = sz(d->k), t = sz(T), mm = sz(m);
    s = check_extents({{topk, L * t * k}, {req_off, (sz(R) + 1) * 4}, {idf, L * E * 4}, {mask_out, mm * 4},
                       {quality_out, mm * 8}, {ws, ws_bytes}});
    if (s != MOER_OK) return s;
  }
  return moer::mask_select_launch(d, topk, T, req_off, R, idf, m, mask_out, quality_out, ws,
                                  reinterpret_cast<cudaStream_t>(stream));
}

size_t moer_spectral_workspace_bytes(const moer_dims* d, int32_t G) {
  if (d == nullptr || d->L < 1 || d->E < 1 || G < 1) return WS_HEADER;
  return moer::spectral_workspace_bytes(d->L, d->E, G);
}

moer_status moer_spectral_groups(const moer_dims* d, const int32_t* affinity, int32_t G, int32_t* group_of,
                                 int32_t* knee, double* u_curve, double* s_curve, void* ws, size_t ws_bytes,
                                 moer_stream_t stream) {
  moer_status s = check_dims(d, false);
  if (s != MOER_OK) return s;
  if (d->E > 128 || G < 2 || G > 31 || G > d->E) return MOER_ERANGE;
  if (affinity == nullptr || group_of == nullptr || knee == nullptr || u_curve == nullptr || s_curve == nullptr)
    return MOER_EINVAL;
  if (!aligned(affinity, 4) || !aligned(group_of, 4) || !aligned(knee, 4) || !aligned(u_curve, 8) ||
      !aligned(s_curve, 8))
    return MOER_EINVAL;
  if (ws == nullptr || !aligned(ws, 256)) return MOER_EINVAL;
  if (ws_bytes < moer_spectral_workspace_bytes(d, G)) return MOER_ENOMEM;
  {
    const size_t L = sz(d->L), E = sz(d->E);
    s = check_extents({{affinity, L * E * E * 4}, {group_of, L * E * 4}, {knee, L * 4}, {u_curve, L * 17 * 8},
                       {s_curve, L * 17 * 8}, {ws, ws_bytes}});
    if (s != MOER_OK) return s;
  }
  return moer::spectral_launch(d, affinity, G, group_of, knee, u_curve, s_curve, ws,
                               reinterpret_cast<cudaStream_t>(stream));
}

size_t moer_kmeans_workspace_bytes(int32_t N, int32_t dim, int32_t D) {
  if (N < 1 || dim < 1 || D < 1) return WS_HEADER;
  return moer::kmeans_workspace_bytes(N, dim, D);
}

moer_status moer_kmeans_balanced(const float* sig, int32_t N, int32_t dim, int32_t D, const float* init_centroids,
                                 int32_t max_iter, float* centroids, int32_t* assign, int32_t* info,
                                 double* objective, void* ws, size_t ws_bytes, moer_stream_t stream) {
  if (D < 1 || D > 32 || N < D || N > (1 << 20) || dim < 1 || dim > 65536) return MOER_ERANGE;
  if (max_iter < 1 || max_iter > 1000) return MOER_ERANGE;
  if (sig == nullptr || init_centroids == nullptr || centroids == nullptr || assign == nullptr)
    return MOER_EINVAL;
  if (!aligned(sig, 4) || !aligned(init_centroids, 4) || !aligned(centroids, 4) || !aligned(assign, 4))
    return MOER_EINVAL;
  if ((info != nullptr && !aligned(info, 4)) || (objective != nullptr && !aligned(objective, 8)))
    return MOER_EINVAL;
  if (ws == nullptr || !aligned(ws, 256)) return MOER_EINVAL;
  if (ws_bytes < moer_kmeans_workspace_bytes(N, dim, D)) return MOER_ENOMEM;
  {
    const size_t n = sz(N), dm = sz(dim), nd = sz(D);
    const moer_status s = check_extents({{sig, n * dm * 4}, {init_centroids, nd * dm * 4}, {centroids, nd * dm * 4},
                                         {assign, n * 4}, {info, 3 * 4}, {objective, 8}, {ws, ws_bytes}});
    if (s != MOER_OK) return s;
  }
  return moer::kmeans_launch(sig, N, dim, D, init_centroids, max_iter, centroids, assign, info, objective, ws,
                       reinterpret_cast<cudaStream_t>(stream));
}

moer_status moer_wait_selftest(void* ws, size_t ws_bytes, uint32_t limit_us, moer_stream_t stream) {
  if (ws == nullptr || !aligned(ws, 16)) return MOER_EINVAL;
  if (ws_bytes < WS_HEADER) return MOER_ENOMEM;
  if (limit_us < 1 || limit_us > 1000000) return MOER_ERANGE;
  {
    const moer_status s = check_extents({{ws, ws_bytes}});
    if (s != MOER_OK) return s;
  }
  return moer::wait_selftest_launch(ws, limit_us, reinterpret_cast<cudaStream_t>(stream));
}

moer_status moer_ws_status(void* ws, moer_stream_t stream) {
  if (ws == nullptr) return MOER_EINVAL;
  {
    const moer_status s = check_extents({{ws, 8}});
    if (s != MOER_OK) return s;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t h[2] = {0u, 0u};
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOER_ECUDA;
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOER_ECUDA;
  if (cudaMemset(ws, 0, sizeof(h)) != cudaSuccess) return MOER_ECUDA;
  if (h[0] & WS_BIT_ETIMEOUT) return MOER_ETIMEOUT;
  if (h[0] & WS_BIT_EDATA) return MOER_EDATA;
  return MOER_OK;
}

const char* moer_status_str(moer_status s) {
  switch (s) {
    case MOER_OK: return "ok";
    case MOER_EINVAL: return "invalid argument (null or misaligned pointer, bad flag)";
    case MOER_ESHAPE: return "inconsistent sizes";
    case MOER_ERANGE: return "size or parameter outside the library limits";
    case MOER_ECUDA: return "CUDA call or kernel launch failed";
    case MOER_ENOMEM: return "workspace too small";
    case MOER_EDATA: return "device-side validation rejected input data";
    case MOER_ETIMEOUT: return "bounded device wait expired";
    case MOER_EEXTENT: return "checked mode: a buffer's allocation cannot hold what the call would touch";
  }
  return "unknown status";
}

int32_t moer_version(void) { return 100; }

void moer_set_extent_checks(int32_t on) { g_extent_checks.store(on ? 1 : 0, std::memory_order_release); }

int32_t moer_buffer_holds(const void* p, size_t bytes) {
  if (p == nullptr) return 0;
  return first_bad_extent({{p, bytes == 0 ? 1 : bytes}}, device_range) < 0 ? 1 : 0;
}

int32_t moer_extent_checks(void) { return extent_checks_on() ? 1 : 0; }

}  // extern "C"
