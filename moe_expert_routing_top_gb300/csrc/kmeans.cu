// kmeans.cu -- moer_kmeans_balanced: balanced K-means of calibration signatures
// into D decoder centroids.
//
// ELDR, section "Key idea / structure / operation": offline, the signatures of
// the calibration prompts are split into D clusters, one per decode worker, by
// K-means with a balance constraint (the Hungarian method), so that locality
// does not pile requests onto one decoder.  Cluster d holds floor(N/D) points,
// plus one for d < N mod D.  Each step assigns the points to clusters at the
// least total squared distance under those sizes, then moves every centroid to
// the mean of its points; the fit stops after a step that changes nothing, or
// after max_iter steps.
//
// Design (GB300):
//   * Squared distances in fp64 (one CTA per point, one warp per centroid:
//     the assignment decisions are taken in double precision).
//   * The balanced assignment is a transportation problem with N unit sources
//     and D sinks.  One CTA keeps a feasible assignment (the previous step's,
//     or a greedy one at the first step) and cancels negative cycles of the
//     residual graph collapsed onto the D cluster nodes: the edge u -> v costs
//     min over points p in u of cost[p][v] - cost[p][u] (moving p from u to v).
//     A cycle moves one point out of and one into every cluster on it, so the
//     sizes stay put; with no negative cycle left the assignment is optimal
//     (min-cost flow optimality).  Edge minima are scans of per-cluster member
//     lists (a few threads per edge, shuffle-reduced).  Each pass first applies
//     every disjoint negative 2-cycle (pairwise swap) it finds; only when none
//     is left does one warp run Bellman-Ford over the D <= 32 nodes and cancel
//     a longer cycle read off the predecessor graph.
//   * Means: one thread per (centroid, coordinate), points in index order.
//   * Every kernel of a step returns at once after convergence, so the host
//     launches max_iter steps without reading anything back.
#include <climits>

#include "common.cuh"

namespace moer {

constexpr int KM_MAXD = 32;
constexpr int KM_THREADS = 1024;
constexpr int KM_SORT_MAX = 2048;  // points put in regret order for the first step's start

struct KmState {
  int32_t steps;      // assignment steps done
  int32_t converged;  // set by the step that changed nothing
  int32_t cancelled;  // negative cycles cancelled, all steps
  int32_t capped;     // set if a step hit its cancellation bound
};

struct KmLayout {
  size_t state, cost, cent, prev, mem, pos, total;
};

static KmLayout km_layout(int32_t N, int32_t dim, int32_t D) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  KmLayout l;
  l.state = WS_HEADER;
  l.cost = l.state + 256;
  l.cent = l.cost + r256((size_t)N * D * sizeof(double));
  l.prev = l.cent + r256((size_t)D * dim * sizeof(double));
  l.mem = l.prev + r256((size_t)N * sizeof(int32_t));
  l.pos = l.mem + r256((size_t)N * sizeof(int32_t));
  l.total = l.pos + r256((size_t)N * sizeof(int32_t));
  return l;
}

__device__ __forceinline__ int km_cap(int d, int N, int D) { return N / D + (d < N % D ? 1 : 0); }

__global__ void km_init_kernel(const float* __restrict__ init, double* __restrict__ cent, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) cent[i] = (double)init[i];
}

// cost[i][d] = ||s_i - c_d||^2 in fp64; block i, warp w takes centroids w, w + 8, ...
__global__ void __launch_bounds__(256) km_cost_kernel(const float* __restrict__ sig, int32_t dim, int32_t D,
                                                      const double* __restrict__ cent, double* __restrict__ cost,
                                                      const KmState* state, int force) {
  if (!force && state->converged) return;
  const int i = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* s = sig + (size_t)i * dim;
  for (int d = warp; d < D; d += 8) {
    const double* c = cent + (size_t)d * dim;
    double acc = 0.0;
    for (int j = lane; j < dim; j += 32) {
      const double t = (double)s[j] - c[j];
      acc = fma(t, t, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL, acc, o);
    if (lane == 0) cost[(size_t)i * D + d] = acc;
  }
}

// Lexicographic (value, point) minimum, for edge minima that do not depend on
// the order in which the points are visited.
__device__ __forceinline__ void vmin(double& v, int& p, double v2, int p2) {
  if (v2 < v || (v2 == v && p2 < p)) {
    v = v2;
    p = p2;
  }
}

// One balanced assignment step (single CTA).  `a` holds the result; `prev` the
// previous step's assignment; `mem` / `pos` the per-cluster member lists
// (cluster u's members at mem[off_u .. off_u + cap_u), pos[p] = p's slot).
__global__ void __launch_bounds__(KM_THREADS, 1)
    km_assign_kernel(const double* __restrict__ cost, int32_t N, int32_t D, int32_t* __restrict__ a,
                     int32_t* __restrict__ prev, int32_t* __restrict__ mem, int32_t* __restrict__ pos,
                     KmState* state, int32_t max_pass, uint32_t* status) {
  __shared__ double wval[KM_MAXD * KM_MAXD];
  __shared__ int widx[KM_MAXD * KM_MAXD];
  __shared__ int off[KM_MAXD + 1], fill[KM_MAXD];
  __shared__ int mv_pt[KM_MAXD], mv_from[KM_MAXD], mv_to[KM_MAXD], freed[KM_MAXD];
  __shared__ int nmv;
  __shared__ int s_pred[KM_MAXD];
  __shared__ double red[KM_THREADS / 32];
  __shared__ int s_first;
  __shared__ double s_key[KM_SORT_MAX];
  __shared__ int s_ord[KM_SORT_MAX];
  if (state->converged) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    s_first = (state->steps == 0);
    off[0] = 0;
    for (int d = 0; d < D; ++d) {
      off[d + 1] = off[d] + km_cap(d, N, D);
      fill[d] = 0;
    }
  }
  __syncthreads();
  const bool first = s_first != 0;

  // 1. a feasible start: the previous assignment, or greedy nearest-with-room in
  //    regret order (the points whose nearest centroid beats their second nearest
  //    by most go first; index order when N > KM_SORT_MAX), which leaves fewer
  //    cycles to cancel than index order
  const bool sorted = first && N <= KM_SORT_MAX;
  if (sorted) {
    int P = 1;
    while (P < N) P <<= 1;
    for (int i = tid; i < P; i += KM_THREADS) {
      double rk = -1.0;  // padding sorts last
      if (i < N) {
        double b1 = INFINITY, b2 = INFINITY;
        for (int d = 0; d < D; ++d) {
          const double c = cost[(size_t)i * D + d];
          if (c < b1) {
            b2 = b1;
            b1 = c;
          } else if (c < b2) {
            b2 = c;
          }
        }
        rk = D > 1 ? b2 - b1 : 0.0;
      }
      s_key[i] = rk;
      s_ord[i] = i;
    }
    __syncthreads();
    // bitonic sort: larger regret first, then lower index
    for (int k = 2; k <= P; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < P; i += KM_THREADS) {
          const int m = i ^ j;
          if (m > i) {
            const double ki = s_key[i], km = s_key[m];
            const int oi = s_ord[i], om = s_ord[m];
            const bool i_first = ki > km || (ki == km && oi < om);
            if (((i & k) == 0) != i_first) {
              s_key[i] = km;
              s_key[m] = ki;
              s_ord[i] = om;
              s_ord[m] = oi;
            }
          }
        }
        __syncthreads();
      }
  }
  if (first) {
    if (tid == 0) {
      int cnt[KM_MAXD];
      for (int d = 0; d < D; ++d) cnt[d] = 0;
      for (int r = 0; r < N; ++r) {
        const int i = sorted ? s_ord[r] : r;
        int best = -1;
        double bc = 0.0;
        for (int d = 0; d < D; ++d) {
          if (cnt[d] >= off[d + 1] - off[d]) continue;
          const double c = cost[(size_t)i * D + d];
          if (best < 0 || c < bc) {
            best = d;
            bc = c;
          }
        }
        a[i] = best;
        cnt[best] += 1;
      }
    }
  } else {
    for (int i = tid; i < N; i += KM_THREADS) a[i] = prev[i];
  }
  __syncthreads();
  // member lists (slot order within a cluster does not matter)
  for (int i = tid; i < N; i += KM_THREADS) {
    const int u = a[i];
    const int slot = off[u] + atomicAdd(&fill[u], 1);
    mem[slot] = i;
    pos[i] = slot;
  }
  // 2. tolerance: a move must gain more than 1e-12 of the largest cost
  double mx = 0.0;
  for (int64_t q = tid; q < (int64_t)N * D; q += KM_THREADS) mx = fmax(mx, fabs(cost[q]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(FULL, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (warp == 0) {
    mx = lane < KM_THREADS / 32 ? red[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(FULL, mx, o));
    if (lane == 0) red[0] = mx;
  }
  __syncthreads();
  const double eps = 1e-12 * red[0] + 1e-300;

  // threads per edge (a power of two <= 32, so an edge's threads share a warp)
  const int npairs = D * D;
  int tpp = 32;
  while (tpp > 1 && tpp * npairs > KM_THREADS) tpp >>= 1;

  // 3. improve until no negative cycle is left
  int done = 0;
  for (int pass = 0; pass < max_pass; ++pass) {
    // edge minima: W[u][v] = min over members p of u of cost[p][v] - cost[p][u]
    {
      const int q = tid / tpp, sub = tid % tpp;
      const int u = q / D, v = q - (q / D) * D;
      double best = INFINITY;
      int bp = INT_MAX;
      if (q < npairs && u != v) {
        for (int k = off[u] + sub; k < off[u + 1]; k += tpp) {
          const int p = mem[k];
          vmin(best, bp, cost[(size_t)p * D + v] - cost[(size_t)p * D + u], p);
        }
      }
      for (int o = tpp >> 1; o > 0; o >>= 1) {
        const double ob = __shfl_xor_sync(FULL, best, o);
        const int op = __shfl_xor_sync(FULL, bp, o);
        vmin(best, bp, ob, op);
      }
      if (q < npairs && sub == 0) {
        wval[q] = best;
        widx[q] = bp;
      }
    }
    __syncthreads();
    // disjoint pairwise swaps first (negative 2-cycles), first fit in (u, v) order
    if (tid == 0) {
      unsigned used = 0u;
      int n = 0;
      for (int u = 0; u < D; ++u)
        for (int v = u + 1; v < D; ++v) {
          if ((used >> u) & 1u || (used >> v) & 1u) continue;
          if (wval[u * D + v] + wval[v * D + u] < -eps) {
            used |= (1u << u) | (1u << v);
            mv_pt[n] = widx[u * D + v], mv_from[n] = u, mv_to[n] = v, ++n;
            mv_pt[n] = widx[v * D + u], mv_from[n] = v, mv_to[n] = u, ++n;
          }
        }
      nmv = n;
    }
    __syncthreads();
    if (nmv == 0 && warp == 0) {
      // no swap left: Bellman-Ford from a virtual source (0-weight edges to
      // every node) for a longer negative cycle; lane v owns node v, rounds
      // are synchronous (old distances through shuffles all lanes execute)
      double dist = 0.0;
      int pred = -1;
      for (int round = 0; round < 2 * (D + 1); ++round) {
        double best = dist;
        int from = pred;
        for (int u = 0; u < D; ++u) {
          const double du = __shfl_sync(FULL, dist, u);
          if (lane < D && u != lane) {
            const double cand = du + wval[u * D + lane];
            if (cand < best) {
              best = cand;
              from = u;
            }
          }
        }
        const bool changed = best < dist;
        dist = best;
        pred = from;
        if (!__any_sync(FULL, changed)) break;
      }
      if (lane < D) s_pred[lane] = pred;
      __syncwarp();
      // A cycle of the predecessor graph has negative weight.  A walk of D
      // steps along predecessors that never reaches the source ends on one.
      int x = lane;
      bool alive = lane < D;
      for (int st = 0; st < D && alive; ++st) {
        const int nx = s_pred[x];
        if (nx < 0) alive = false;
        else x = nx;
      }
      const unsigned on = __ballot_sync(FULL, alive);
      const int start = __shfl_sync(FULL, x, on ? (__ffs(on) - 1) : 0);
      if (lane == 0 && on) {
        // walk the cycle backwards (edges pred[y] -> y)
        int y = start, n = 0;
        double w = 0.0;
        bool ok = true;
        do {
          const int py = s_pred[y];
          if (py < 0 || widx[py * D + y] >= N) {  // cannot happen on a cycle; checked anyway
            ok = false;
            break;
          }
          mv_pt[n] = widx[py * D + y], mv_from[n] = py, mv_to[n] = y, ++n;
          w += wval[py * D + y];
          y = py;
        } while (y != start && n < D);
        nmv = (ok && y == start && w < -eps) ? n : 0;
      }
    }
    __syncthreads();
    if (nmv == 0) {
      done = 1;
      break;
    }
    if (tid == 0) {
      // every cluster on the moves loses one point and gains one: the incoming
      // point takes the outgoing point's slot (points are distinct: each move
      // leaves a different cluster)
      for (int m = 0; m < nmv; ++m) freed[mv_from[m]] = pos[mv_pt[m]];
      for (int m = 0; m < nmv; ++m) {
        const int pt = mv_pt[m], slot = freed[mv_to[m]];
        a[pt] = mv_to[m];
        mem[slot] = pt;
        pos[pt] = slot;
      }
      state->cancelled += 1;
    }
    __syncthreads();
  }
  // 4. convergence and bookkeeping
  int changed = 0;
  if (!first)
    for (int i = tid; i < N; i += KM_THREADS) changed |= (a[i] != prev[i]);
  changed = __syncthreads_or(changed);
  for (int i = tid; i < N; i += KM_THREADS) prev[i] = a[i];
  if (tid == 0) {
    if (!first && !changed) state->converged = 1;
    if (!done) {
      state->capped = 1;
      atomicOr(status, WS_BIT_ETIMEOUT);
    }
    state->steps += 1;
  }
}

// cent[d][j] = mean of sig[p][j] over the points p of cluster d.
__global__ void __launch_bounds__(256) km_update_kernel(const float* __restrict__ sig, int32_t N, int32_t dim,
                                                        int32_t D, const int32_t* __restrict__ a,
                                                        double* __restrict__ cent, const KmState* state) {
  if (state->converged) return;
  const int d = blockIdx.y;
  const int j = blockIdx.x * 256 + threadIdx.x;
  double sum = 0.0;
  int n = 0;
  for (int p = 0; p < N; ++p) {
    if (a[p] != d) continue;  // uniform across the block
    if (j < dim) sum += (double)sig[(size_t)p * dim + j];
    ++n;
  }
  if (j < dim && n > 0) cent[(size_t)d * dim + j] = sum / n;
}

__global__ void __launch_bounds__(KM_THREADS) km_finalize_kernel(const double* __restrict__ cost,
                                                                  const double* __restrict__ cent,
                                                                  const int32_t* __restrict__ a, int32_t N,
                                                                  int32_t dim, int32_t D, float* __restrict__ out,
                                                                  int32_t* info, double* objective,
                                                                  const KmState* state) {
  __shared__ double red[KM_THREADS / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int64_t q = tid; q < (int64_t)D * dim; q += KM_THREADS) out[q] = (float)cent[q];
  double acc = 0.0;
  for (int i = tid; i < N; i += KM_THREADS) acc += cost[(size_t)i * D + a[i]];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL, acc, o);
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (warp == 0) {
    acc = lane < KM_THREADS / 32 ? red[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL, acc, o);
    if (lane == 0) {
      if (objective != nullptr) *objective = acc;
      if (info != nullptr) {
        info[0] = state->steps;
        info[1] = state->cancelled;
        info[2] = state->capped;
      }
    }
  }
}

size_t kmeans_workspace_bytes(int32_t N, int32_t dim, int32_t D) { return km_layout(N, dim, D).total; }

moer_status kmeans_launch(const float* sig, int32_t N, int32_t dim, int32_t D, const float* init, int32_t max_iter,
                          float* centroids, int32_t* assign, int32_t* info, double* objective, void* ws,
                          cudaStream_t st) {
  const KmLayout l = km_layout(N, dim, D);
  char* w = static_cast<char*>(ws);
  KmState* state = reinterpret_cast<KmState*>(w + l.state);
  double* cost = reinterpret_cast<double*>(w + l.cost);
  double* cent = reinterpret_cast<double*>(w + l.cent);
  int32_t* prev = reinterpret_cast<int32_t*>(w + l.prev);
  int32_t* mem = reinterpret_cast<int32_t*>(w + l.mem);
  int32_t* pos = reinterpret_cast<int32_t*>(w + l.pos);
  uint32_t* status = reinterpret_cast<uint32_t*>(w);
  if (cudaMemsetAsync(state, 0, sizeof(KmState), st) != cudaSuccess) return MOER_ECUDA;
  const int64_t nc = (int64_t)D * dim;
  km_init_kernel<<<(unsigned)((nc + 255) / 256), 256, 0, st>>>(init, cent, nc);
  const int32_t max_cancel = 16 * N + 1024;
  const dim3 ug((unsigned)((dim + 255) / 256), (unsigned)D);
  for (int it = 0; it < max_iter; ++it) {
    km_cost_kernel<<<(unsigned)N, 256, 0, st>>>(sig, dim, D, cent, cost, state, 0);
    km_assign_kernel<<<1, KM_THREADS, 0, st>>>(cost, N, D, assign, prev, mem, pos, state, max_cancel, status);
    km_update_kernel<<<ug, 256, 0, st>>>(sig, N, dim, D, assign, cent, state);
  }
  km_cost_kernel<<<(unsigned)N, 256, 0, st>>>(sig, dim, D, cent, cost, state, 1);
  km_finalize_kernel<<<1, KM_THREADS, 0, st>>>(cost, cent, assign, N, dim, D, centroids, info, objective, state);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
