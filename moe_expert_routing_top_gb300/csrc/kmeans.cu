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
//   * Squared distances in fp64 as ||s||^2 + ||c||^2 - 2 s.c (one CTA per
//     point, one warp per centroid: the assignment decisions are taken in
//     double precision).
//   * The balanced assignment is a transportation problem with N unit sources
//     and D sinks.  One CTA keeps a feasible assignment (the previous step's,
//     or a greedy one at the first step) and cancels negative cycles of the
//     residual graph collapsed onto the D cluster nodes: the edge u -> v costs
//     min over points p in u of cost[p][v] - cost[p][u] (moving p from u to v).
//     A cycle moves one point out of and one into every cluster on it, so the
//     sizes stay put; with no negative cycle left the assignment is optimal
//     (min-cost flow optimality).  Edge minima are scans of per-cluster member
//     lists (a few threads per edge, shuffle-reduced); the costs, assignment
//     and member lists are staged in shared memory when they fit.  Each pass first applies
//     every disjoint negative 2-cycle (pairwise swap) it finds; only when none
//     is left does one warp run Bellman-Ford over the D <= 32 nodes and cancel
//     a longer cycle read off the predecessor graph.
//   * Means: one thread per (centroid, coordinate), points in index order,
//     read from per-cluster member lists that the assignment step leaves in
//     index order.
//   * Every kernel of a step returns at once after convergence, so the host
//     launches max_iter steps without reading anything back.
#include <climits>

#include "common.cuh"
#include "keys.cuh"

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
  size_t state, cost, cent, cpart, prev, mem, pos, dkey, total;
};

static KmLayout km_layout(int32_t N, int32_t dim, int32_t D) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  KmLayout l;
  l.state = WS_HEADER;
  l.cost = l.state + 256;
  l.cent = l.cost + r256((size_t)N * D * sizeof(double));
  l.cpart = l.cent + r256((size_t)D * dim * sizeof(double));
  l.prev = l.cpart + r256((size_t)D * ((dim + 255) / 256) * sizeof(double));
  l.mem = l.prev + r256((size_t)N * sizeof(int32_t));
  l.pos = l.mem + r256((size_t)N * sizeof(int32_t));
  l.dkey = l.pos + r256((size_t)N * sizeof(int32_t));
  l.total = l.dkey + r256((size_t)N * (D + 1) * sizeof(unsigned long long));
  return l;
}

__device__ __forceinline__ int km_cap(int d, int N, int D) { return N / D + (d < N % D ? 1 : 0); }

// The kernels of a fit are chained by programmatic dependent launch: each
// waits for the grid before it in the stream (whose writes are then visible),
// then lets the next grid start launching, so that a launch's latency overlaps
// the work before it (after convergence the steps return at once, and their
// launches are the fit's cost).  A dependent grid is scheduled only after every
// CTA of the grid it waits for has started.
__device__ __forceinline__ void km_chain() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Sum of v over a block of 256 threads, in a fixed order; thread 0 gets it.
__device__ __forceinline__ double km_block_sum256(double v, double* red8) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  if (lane == 0) red8[warp] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < 8; ++w) t += red8[w];
  return t;
}

// cent = init widened to fp64; block (bx, d) also leaves the sum of squares of
// its 256 coordinates of centroid d in cpart[d][bx] (see km_cost_kernel).
__global__ void __launch_bounds__(256) km_init_kernel(const float* __restrict__ init, int32_t dim,
                                                      double* __restrict__ cent, double* __restrict__ cpart) {
  __shared__ double red8[8];
  const int d = blockIdx.y, j = blockIdx.x * 256 + threadIdx.x;
  double c = 0.0;
  if (j < dim) {
    c = (double)init[(size_t)d * dim + j];
    cent[(size_t)d * dim + j] = c;
  }
  const double t = km_block_sum256(c * c, red8);
  if (threadIdx.x == 0) cpart[(size_t)d * gridDim.x + blockIdx.x] = t;
}

// cost[i][d] = ||s_i - c_d||^2 in fp64, as ||s_i||^2 + ||c_d||^2 - 2 s_i.c_d:
// one fused multiply-add per element instead of a subtraction and one (fp64
// runs at about 16 cycles per warp instruction per SM on this part).  Block i,
// warp w takes centroids w, w + 8, ...; the signature row is widened to fp64
// once per block, a chunk at a time, into shared memory, and its squares are
// summed on the way.  ||c_d||^2 is the sum, in block order, of the partials
// cpart[d][0 .. nbk) left by the kernel that wrote the centroids.
constexpr int KM_COST_CHUNK = 2048;
__global__ void __launch_bounds__(256) km_cost_kernel(const float* __restrict__ sig, int32_t dim, int32_t D,
                                                      const double* __restrict__ cent,
                                                      const double* __restrict__ cpart, int32_t nbk,
                                                      double* __restrict__ cost, const KmState* state, int force) {
  __shared__ double s64[KM_COST_CHUNK];
  __shared__ double red8[8];
  __shared__ double s_ss;
  km_chain();
  if (!force && state->converged) return;
  const int i = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* s = sig + (size_t)i * dim;
  double acc[KM_MAXD / 8];
#pragma unroll
  for (int q = 0; q < KM_MAXD / 8; ++q) acc[q] = 0.0;
  double ssp = 0.0;
  for (int j0 = 0; j0 < dim; j0 += KM_COST_CHUNK) {
    const int n = min(KM_COST_CHUNK, dim - j0);
    for (int j = threadIdx.x; j < n; j += 256) {
      const double v = (double)s[j0 + j];
      s64[j] = v;
      ssp = fma(v, v, ssp);
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < KM_MAXD / 8; ++q) {
      const int d = warp + 8 * q;
      if (d < D) {
        const double* c = cent + (size_t)d * dim + j0;
        double t_acc = acc[q];
        for (int j = lane; j < n; j += 32) t_acc = fma(s64[j], c[j], t_acc);
        acc[q] = t_acc;
      }
    }
    __syncthreads();
  }
  const double sst = km_block_sum256(ssp, red8);
  if (threadIdx.x == 0) s_ss = sst;
  __syncthreads();
  const double ss = s_ss;
#pragma unroll
  for (int q = 0; q < KM_MAXD / 8; ++q) {
    const int d = warp + 8 * q;
    if (d < D) {
      double t_acc = acc[q];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t_acc += __shfl_xor_sync(FULL, t_acc, o);
      if (lane == 0) {
        double cc = 0.0;
        for (int b = 0; b < nbk; ++b) cc += cpart[(size_t)d * nbk + b];
        cost[(size_t)i * D + d] = fma(-2.0, t_acc, ss + cc);
      }
    }
  }
}

// One balanced assignment step (single CTA).  `a` holds the result; `prev` the
// previous step's assignment; `mem` / `pos` the per-cluster member lists
// (cluster u's members at mem[off_u .. off_u + cap_u), pos[p] = p's slot);
// `dkey` row p holds okey(cost[p][v] - cost[p][a(p)]) for every v (stride
// D + 1), the gain of moving p, rewritten only for the points that move.  With
// `staged`, the assignment, member lists and keys live in shared memory
// instead (the global arrays then only receive the result).
__global__ void __launch_bounds__(KM_THREADS, 1)
    km_assign_kernel(const double* __restrict__ cost, int32_t N, int32_t D, int32_t* __restrict__ a,
                     int32_t* __restrict__ prev, int32_t* __restrict__ mem, int32_t* __restrict__ pos,
                     unsigned long long* __restrict__ dkey, KmState* state, int32_t max_pass, int32_t staged,
                     uint32_t* status) {
  extern __shared__ __align__(16) unsigned char km_dyn[];
  __shared__ double wval[KM_MAXD * KM_MAXD];
  __shared__ int widx[KM_MAXD * KM_MAXD];
  __shared__ int off[KM_MAXD + 1], fill[KM_MAXD];
  __shared__ int mv_pt[KM_MAXD], mv_from[KM_MAXD], mv_to[KM_MAXD], freed[KM_MAXD];
  __shared__ int nmv;
  __shared__ int s_pred[KM_MAXD];
  __shared__ double bf_dist[2][KM_MAXD];
  __shared__ unsigned negmask[KM_MAXD];
  __shared__ unsigned long long red[KM_THREADS / 32];
  __shared__ int wcnt[KM_MAXD][KM_THREADS / 32];
  __shared__ int s_first;
  __shared__ unsigned long long s_key[KM_SORT_MAX];
  __shared__ int s_ord[KM_SORT_MAX];
  km_chain();
  if (state->converged) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int DS = D + 1;  // key row stride: consecutive rows start in different banks
  int32_t* as = a;
  int32_t* mm = mem;
  int32_t* ps = pos;
  unsigned long long* dk = dkey;
  if (staged) {
    dk = reinterpret_cast<unsigned long long*>(km_dyn);
    as = reinterpret_cast<int32_t*>(dk + (size_t)N * DS);
    mm = as + N;
    ps = as + 2 * (size_t)N;
  }
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
      unsigned long long rk = 0ull;  // padding sorts last
      if (i < N) {
        unsigned long long b1 = ~0ull, b2 = ~0ull;
        for (int d = 0; d < D; ++d) {
          const unsigned long long c = okey(cost[(size_t)i * D + d]);
          if (c < b1) {
            b2 = b1;
            b1 = c;
          } else if (c < b2) {
            b2 = c;
          }
        }
        rk = okey(D > 1 ? okey_value(b2) - okey_value(b1) : 0.0);
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
            const unsigned long long ki = s_key[i], km = s_key[m];
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
    if (warp == 0) {
      // greedy nearest-with-room, one point at a time; lane d owns cluster d's
      // fill, and a warp minimum over the lanes with room (ties: lower d) picks
      const int capd = lane < D ? off[lane + 1] - off[lane] : 0;
      int cnt = 0;
      int i = sorted ? s_ord[0] : 0;
      double c = lane < D ? cost[(size_t)i * D + lane] : 0.0;
      for (int r = 0; r < N; ++r) {
        const int inext = r + 1 < N ? (sorted ? s_ord[r + 1] : r + 1) : i;
        const double cnext = lane < D ? cost[(size_t)inext * D + lane] : 0.0;  // next row in flight
        unsigned long long key = lane < D && cnt < capd ? okey(c) : ~0ull;
        int d = lane;
        warp_min_key(key, d);
        if (lane == d) ++cnt;
        if (lane == 0) as[i] = d;
        i = inext;
        c = cnext;
      }
    }
  } else {
    for (int i = tid; i < N; i += KM_THREADS) as[i] = prev[i];
  }
  __syncthreads();
  // member lists (slot order within a cluster does not matter)
  for (int i = tid; i < N; i += KM_THREADS) {
    const int u = as[i];
    const int slot = off[u] + atomicAdd(&fill[u], 1);
    mm[slot] = i;
    ps[i] = slot;
  }
  // gain keys of every point, and the largest |cost| (bit patterns of
  // non-negative doubles order as integers)
  unsigned long long mx = 0ull;
  for (int64_t q = tid; q < (int64_t)N * D; q += KM_THREADS) {
    const int p = (int)(q / D), v = (int)(q - (int64_t)p * D);
    const double c = cost[q];
    dk[(size_t)p * DS + v] = okey(c - cost[(size_t)p * D + as[p]]);
    const unsigned long long ab = (unsigned long long)__double_as_longlong(c) & 0x7FFFFFFFFFFFFFFFull;
    mx = ab > mx ? ab : mx;
  }
  {
    unsigned long long cm = ~mx;  // the maximum is the complement of the complements' minimum
    int unused = 0;
    warp_min_key(cm, unused);
    mx = ~cm;
  }
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (warp == 0) {
    unsigned long long cm = lane < KM_THREADS / 32 ? ~red[lane] : ~0ull;
    int unused = 0;
    warp_min_key(cm, unused);
    if (lane == 0) red[0] = ~cm;
  }
  __syncthreads();
  // 2. tolerance: a move must gain more than 1e-12 of the largest cost
  const double eps = 1e-12 * __longlong_as_double((long long)red[0]) + 1e-300;

  // threads per edge (a power of two <= 32, so an edge's threads share a warp)
  const int npairs = D * D;
  int tpp = 32;
  while (tpp > 1 && tpp * npairs > KM_THREADS) tpp >>= 1;

  // 3. improve until no negative cycle is left
  int done = 0, ncancel = 0;
  for (int pass = 0; pass < max_pass; ++pass) {
    // edge minima: W[u][v] = min over members p of u of cost[p][v] - cost[p][u]
    // (ties: the lower point)
    {
      const int q = tid / tpp, sub = tid % tpp;
      const int u = q / D, v = q - (q / D) * D;
      unsigned long long best = ~0ull;
      int bp = INT_MAX;
      if (q < npairs && u != v) {
        for (int k = off[u] + sub; k < off[u + 1]; k += tpp) {
          const int p = mm[k];
          const unsigned long long kk = dk[(size_t)p * DS + v];
          if (kk < best || (kk == best && p < bp)) {
            best = kk;
            bp = p;
          }
        }
      }
      for (int o = tpp >> 1; o > 0; o >>= 1) {
        const unsigned long long ob = __shfl_xor_sync(FULL, best, o);
        const int op = __shfl_xor_sync(FULL, bp, o);
        if (ob < best || (ob == best && op < bp)) {
          best = ob;
          bp = op;
        }
      }
      if (q < npairs && sub == 0) {
        wval[q] = bp == INT_MAX ? INFINITY : okey_value(best);
        widx[q] = bp;
      }
      if (tid < D) negmask[tid] = 0u;
    }
    __syncthreads();
    // disjoint pairwise swaps first (negative 2-cycles), first fit in (u, v)
    // order: the negative pairs of each row u are marked (bit v, v > u), then
    // one thread takes, for u ascending, the lowest v that is still free
    if (tid < npairs) {
      const int u = tid / D, v = tid - (tid / D) * D;
      if (v > u && wval[u * D + v] + wval[v * D + u] < -eps) atomicOr(&negmask[u], 1u << v);
    }
    __syncthreads();
    if (tid == 0) {
      unsigned used = 0u;
      int n = 0;
      for (int u = 0; u < D; ++u) {
        if ((used >> u) & 1u) continue;
        const unsigned m = negmask[u] & ~used;
        if (m == 0u) continue;
        const int v = __ffs(m) - 1;
        used |= (1u << u) | (1u << v);
        mv_pt[n] = widx[u * D + v], mv_from[n] = u, mv_to[n] = v, ++n;
        mv_pt[n] = widx[v * D + u], mv_from[n] = v, mv_to[n] = u, ++n;
      }
      nmv = n;
      if (n == 0) {
        for (int x = 0; x < D; ++x) {
          bf_dist[0][x] = 0.0;
          s_pred[x] = -1;
        }
      }
    }
    __syncthreads();
    if (nmv == 0) {
      // no swap left: Bellman-Ford from a virtual source (0-weight edges to
      // every node) for a longer negative cycle.  Synchronous rounds; warp v
      // relaxes node v, lane u offering dist[u] + W[u][v]; a node takes the
      // smallest offer (ties: the lower u) only if it beats its distance.
      int cur = 0;
      for (int round = 0; round < 2 * (D + 1); ++round) {
        int changed = 0;
        if (warp < D) {
          const int v = warp;
          unsigned long long key = ~0ull;
          int from = lane;
          if (lane < D && lane != v) key = okey(bf_dist[cur][lane] + wval[lane * D + v]);
          warp_min_key(key, from);
          if (lane == 0) {
            const double dv = bf_dist[cur][v];
            if (key < okey(dv)) {
              bf_dist[cur ^ 1][v] = okey_value(key);
              s_pred[v] = from;
              changed = 1;
            } else {
              bf_dist[cur ^ 1][v] = dv;
            }
          }
        }
        cur ^= 1;
        changed = __syncthreads_or(changed);
        if (warp == 0) {
          // A cycle of the predecessor graph has negative weight (its sum is
          // checked anyway): stop at the first round that closes one.  A walk
          // of D steps along predecessors that never reaches the source ends
          // on a cycle.
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
        if (nmv != 0 || !changed) break;
      }
    }
    if (nmv == 0) {
      done = 1;
      break;
    }
    if (tid == 0) {
      // every cluster on the moves loses one point and gains one: the incoming
      // point takes the outgoing point's slot (points are distinct: each move
      // leaves a different cluster)
      for (int m = 0; m < nmv; ++m) freed[mv_from[m]] = ps[mv_pt[m]];
      for (int m = 0; m < nmv; ++m) {
        const int pt = mv_pt[m], slot = freed[mv_to[m]];
        as[pt] = mv_to[m];
        mm[slot] = pt;
        ps[pt] = slot;
      }
      ++ncancel;
    }
    __syncthreads();
    // the moved points' gain keys, against their new clusters
    for (int t = tid; t < nmv * D; t += KM_THREADS) {
      const int p = mv_pt[t / D], v = t - (t / D) * D;
      dk[(size_t)p * DS + v] = okey(cost[(size_t)p * D + v] - cost[(size_t)p * D + as[p]]);
    }
    __syncthreads();
  }
  // 4. convergence and bookkeeping
  int changed = 0;
  if (!first)
    for (int i = tid; i < N; i += KM_THREADS) changed |= (as[i] != prev[i]);
  changed = __syncthreads_or(changed);
  // 5. each cluster's members in index order, for the means: mem[off_u + r]
  //    is the r-th lowest point of cluster u (a stable counting sort: warp
  //    ballots per cluster, then a scan over the warps)
  if (tid < D) fill[tid] = 0;
  for (int base = 0; base < N; base += KM_THREADS) {
    const int i = base + tid;
    const int ai = i < N ? as[i] : -1;
    int rank = 0;
    for (int d = 0; d < D; ++d) {
      const unsigned b = __ballot_sync(FULL, ai == d);
      if (lane == 0) wcnt[d][warp] = __popc(b);
      if (ai == d) rank = __popc(b & ((1u << lane) - 1u));
    }
    __syncthreads();
    if (tid < D) {
      int run = fill[tid];
      for (int w = 0; w < KM_THREADS / 32; ++w) {
        const int c = wcnt[tid][w];
        wcnt[tid][w] = run;
        run += c;
      }
      fill[tid] = run;
    }
    __syncthreads();
    if (ai >= 0) mem[off[ai] + wcnt[ai][warp] + rank] = i;
    __syncthreads();
  }
  for (int i = tid; i < N; i += KM_THREADS) {
    prev[i] = as[i];
    if (staged) a[i] = as[i];
  }
  if (tid == 0) {
    state->cancelled += ncancel;
    if (!first && !changed) state->converged = 1;
    if (!done) {
      state->capped = 1;
      atomicOr(status, WS_BIT_ETIMEOUT);
    }
    state->steps += 1;
  }
}

// cent[d][j] = mean of sig[p][j] over the points p of cluster d, summed in
// index order: `ord` holds each cluster's members in index order at the
// cluster's offset (written by the assignment step), eight loads in flight.
__global__ void __launch_bounds__(256) km_update_kernel(const float* __restrict__ sig, int32_t N, int32_t dim,
                                                        int32_t D, const int32_t* __restrict__ ord,
                                                        double* __restrict__ cent, double* __restrict__ cpart,
                                                        const KmState* state) {
  __shared__ double red8[8];
  km_chain();
  if (state->converged) return;
  const int d = blockIdx.y;
  const int j = blockIdx.x * 256 + threadIdx.x;
  const int jj = j < dim ? j : dim - 1;  // threads past the end read a valid column, store nothing
  const int base = N / D, rem = N % D;
  const int o = d * base + min(d, rem), n = base + (d < rem ? 1 : 0);
  const int32_t* m = ord + o;
  double sum = 0.0;
  int k = 0;
  for (; k + 8 <= n; k += 8) {
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = sig[(size_t)m[k + q] * dim + jj];
#pragma unroll
    for (int q = 0; q < 8; ++q) sum += (double)v[q];
  }
  for (; k < n; ++k) sum += (double)sig[(size_t)m[k] * dim + jj];
  double c = 0.0;
  if (j < dim && n > 0) {
    c = sum / n;
    cent[(size_t)d * dim + j] = c;
  }
  const double t = km_block_sum256(c * c, red8);
  if (threadIdx.x == 0) cpart[(size_t)d * gridDim.x + blockIdx.x] = t;
}

__global__ void __launch_bounds__(KM_THREADS) km_finalize_kernel(const double* __restrict__ cost,
                                                                  const double* __restrict__ cent,
                                                                  const int32_t* __restrict__ a, int32_t N,
                                                                  int32_t dim, int32_t D, float* __restrict__ out,
                                                                  int32_t* info, double* objective,
                                                                  const KmState* state) {
  km_chain();
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
  double* cpart = reinterpret_cast<double*>(w + l.cpart);
  int32_t* prev = reinterpret_cast<int32_t*>(w + l.prev);
  int32_t* mem = reinterpret_cast<int32_t*>(w + l.mem);
  int32_t* pos = reinterpret_cast<int32_t*>(w + l.pos);
  unsigned long long* dkey = reinterpret_cast<unsigned long long*>(w + l.dkey);
  uint32_t* status = reinterpret_cast<uint32_t*>(w);
  if (cudaMemsetAsync(state, 0, sizeof(KmState), st) != cudaSuccess) return MOER_ECUDA;
  const int32_t nbk = (dim + 255) / 256;
  km_init_kernel<<<dim3((unsigned)nbk, (unsigned)D), 256, 0, st>>>(init, dim, cent, cpart);
  const int32_t max_cancel = 16 * N + 1024;
  const dim3 ug((unsigned)((dim + 255) / 256), (unsigned)D);
  // shared-memory staging of the assignment step when it fits beside the
  // kernel's static arrays (1,000 points x 16 clusters: 148 KB)
  static std::atomic<unsigned long long> assign_set{0};
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, km_assign_kernel) != cudaSuccess) return MOER_ECUDA;
  const int64_t dyn_max = 232448 - (int64_t)fa.sharedSizeBytes;
  const int64_t dyn = (int64_t)N * (D + 1) * (int64_t)sizeof(unsigned long long) +
                      3 * (int64_t)N * (int64_t)sizeof(int32_t);
  const bool staged = dyn <= dyn_max;
  if (staged && smem_optin(km_assign_kernel, (int)dyn_max, assign_set) != cudaSuccess) return MOER_ECUDA;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  auto cfg = [&](dim3 g, dim3 b, size_t smem) {
    cudaLaunchConfig_t c = {};
    c.gridDim = g;
    c.blockDim = b;
    c.dynamicSmemBytes = smem;
    c.stream = st;
    c.attrs = pdl;
    c.numAttrs = 1;
    return c;
  };
  const cudaLaunchConfig_t c_cost = cfg(dim3((unsigned)N), dim3(256), 0);
  const cudaLaunchConfig_t c_assign = cfg(dim3(1), dim3(KM_THREADS), staged ? (size_t)dyn : 0);
  const cudaLaunchConfig_t c_update = cfg(ug, dim3(256), 0);
  const cudaLaunchConfig_t c_final = cfg(dim3(1), dim3(KM_THREADS), 0);
  const int32_t stg = staged ? 1 : 0;
  for (int it = 0; it < max_iter; ++it) {
    if (cudaLaunchKernelEx(&c_cost, km_cost_kernel, sig, dim, D, (const double*)cent, (const double*)cpart, nbk,
                           cost, (const KmState*)state, 0) != cudaSuccess ||
        cudaLaunchKernelEx(&c_assign, km_assign_kernel, (const double*)cost, N, D, assign, prev, mem, pos, dkey,
                           state, max_cancel, stg, status) != cudaSuccess ||
        cudaLaunchKernelEx(&c_update, km_update_kernel, sig, N, dim, D, (const int32_t*)mem, cent, cpart,
                           (const KmState*)state) != cudaSuccess)
      return MOER_ECUDA;
  }
  if (cudaLaunchKernelEx(&c_cost, km_cost_kernel, sig, dim, D, (const double*)cent, (const double*)cpart, nbk,
                         cost, (const KmState*)state, 1) != cudaSuccess ||
      cudaLaunchKernelEx(&c_final, km_finalize_kernel, (const double*)cost, (const double*)cent,
                         (const int32_t*)assign, N, dim, D, centroids, info, objective,
                         (const KmState*)state) != cudaSuccess)
    return MOER_ECUDA;
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
