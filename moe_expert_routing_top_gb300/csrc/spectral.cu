// spectral.cu -- moer_spectral_groups: spectral grouping of experts per layer
// with a controlled size tolerance.
//
// GRACE-MoE, section 4.1 (expert grouping, communication first): spectral
// clustering of the affinity (co-activation) matrix puts experts that are
// selected together on the same GPU; fully non-uniform groups minimise
// communication but worsen load balance, so the group sizes are held within
// [E_bar - delta, E_bar + delta], delta = E_bar * r, and r is taken at the knee
// point of the affinity utilisation U(r) (with the size deviation S(r)).
// Per layer, for G groups (one node of G GPUs), in fp64:
//   * M = D^-1/2 A D^-1/2 with A the co-activation counts off the diagonal;
//     the embedding is the eigenvectors of M's G largest eigenvalues, each
//     expert's row scaled to unit length;
//   * for r = j/16, j = 0..16, sizes in [max(1, floor(E(16-j)/(16G))),
//     min(E, ceil(E(16+j)/(16G)))]: K-means on the embedding rows under those
//     bounds, seeded with the expert of largest degree and then the farthest
//     expert from the seeds so far; each step assigns at the least total
//     squared distance under the bounds and moves the centroids to the means;
//   * U(r) = affinity inside groups / all affinity off the diagonal; S(r) =
//     std of the group sizes / (E/G); the knee of U over r (scaled to [0, 1],
//     the point farthest above the chord from r = 0 to r = 1) picks the groups.
//
// Design (GB300):
//   * spec_embed_kernel, one CTA per layer: M lives in shared memory (fp64,
//     128 KB at E = 128); parallel cyclic Jacobi with the round-robin pairing,
//     E/2 disjoint rotations per round (rows, then columns with the pairs
//     fastest so a warp touches 32 different columns, and the eigenvector
//     matrix, kept transposed in global memory so its update is coalesced),
//     until a sweep finds every off-diagonal entry negligible against its
//     diagonal pair (|a_pq| <= 1e-15 sqrt|a_pp a_qq|: threshold Jacobi, which
//     stops at the rounding floor instead of chasing it); the G largest
//     diagonal entries pick the columns.  A full solve rather than an
//     iteration on the top-G subspace: the co-activation spectra of real
//     layers are nearly degenerate just below the leading eigenvalues, where
//     subspace iteration needs 10^4 - 10^5 steps, while Jacobi's accuracy
//     (backward stable) only needs the gap at the G-th eigenvalue.
//   * spec_group_kernel, one CTA per (grid point, layer): the size-bounded
//     assignment is a transportation problem with lower and upper bounds; one
//     warp keeps a feasible assignment and cancels negative cycles of the
//     residual graph collapsed onto the G groups plus one slack node t (t -> u
//     when u may shrink, u -> t when u may grow, a large negative u -> t while u
//     is below its lower bound), Bellman-Ford with a lane per node.
//   * spec_knee_kernel, one warp per layer: the knee and the chosen groups.
#include <climits>

#include "common.cuh"

namespace moer {

constexpr int SP_MAXE = 128;
constexpr int SP_MAXG = 31;
constexpr int SP_NGRID = 17;
constexpr int SP_EMBED_THREADS = 1024;
constexpr int SP_GROUP_THREADS = 256;
constexpr int SP_MAX_SWEEPS = 40;
constexpr int SP_MAX_STEPS = 100;

__device__ __forceinline__ int sp_seq(int j, int r, int E) { return j == 0 ? 0 : ((j - 1 + r) % (E - 1)) + 1; }

__global__ void __launch_bounds__(SP_EMBED_THREADS, 1)
    spec_embed_kernel(const int32_t* __restrict__ affinity, int E, int G, double* __restrict__ V,
                      double* __restrict__ Uo, double* __restrict__ deg_out) {
  extern __shared__ double sp_sm[];
  double* M = sp_sm;                 // [E][E]
  double* inv = M + E * E;           // [E]
  double* cs = inv + E;              // [E/2]
  double* sn = cs + E / 2;           // [E/2]
  double* red = sn + E / 2;          // [32]
  int* pp = reinterpret_cast<int*>(red + 32);
  int* qq = pp + E / 2;
  __shared__ int s_done;
  const int l = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const int32_t* A = affinity + (size_t)l * E * E;
  double* Vl = V + (size_t)l * E * E;
  for (int a = tid; a < E; a += nt) {
    long long d = 0;
    for (int b = 0; b < E; ++b)
      if (b != a) d += A[(size_t)a * E + b] > 0 ? A[(size_t)a * E + b] : 0;
    deg_out[(size_t)l * E + a] = (double)d;
    inv[a] = d > 0 ? 1.0 / sqrt((double)d) : 0.0;
  }
  __syncthreads();
  for (int q = tid; q < E * E; q += nt) {
    const int a = q / E, b = q - a * E;
    const int32_t x = A[q] > 0 ? A[q] : 0;
    M[q] = (a == b) ? 0.0 : inv[a] * (double)x * inv[b];
    Vl[q] = (a == b) ? 1.0 : 0.0;
  }
  __syncthreads();
  // threshold Jacobi: a rotation is skipped when |a_pq| <= 1e-15 sqrt(|a_pp a_qq|)
  // (negligible against the diagonal); the solve ends after a sweep that rotates nothing
  for (int sweep = 0; sweep < SP_MAX_SWEEPS; ++sweep) {
    if (tid == 0) s_done = 1;
    __syncthreads();
    for (int r = 0; r < E - 1; ++r) {
      if (tid < E / 2) {
        const int p = sp_seq(tid, r, E), q = sp_seq(E - 1 - tid, r, E);
        const double apq = M[p * E + q], app = M[p * E + p], aqq = M[q * E + q];
        double c = 1.0, s = 0.0;
        if (fabs(apq) > 1e-15 * sqrt(fabs(app * aqq)) && fabs(apq) > 1e-300) {
          const double th = (aqq - app) / (2.0 * apq);
          double t;
          if (fabs(th) > 1e150) t = 1.0 / (2.0 * th);
          else if (th == 0.0) t = 1.0;
          else t = (th > 0.0 ? 1.0 : -1.0) / (fabs(th) + sqrt(th * th + 1.0));
          c = 1.0 / sqrt(1.0 + t * t);
          s = t * c;
          s_done = 0;
        }
        pp[tid] = p;
        qq[tid] = q;
        cs[tid] = c;
        sn[tid] = s;
      }
      __syncthreads();
      for (int w = tid; w < (E / 2) * E; w += nt) {  // rows p, q of every pair
        const int i = w / E, j = w - i * E;
        const int p = pp[i], q = qq[i];
        const double c = cs[i], s = sn[i];
        const double mp = M[p * E + j], mq = M[q * E + j];
        M[p * E + j] = c * mp - s * mq;
        M[q * E + j] = s * mp + c * mq;
      }
      __syncthreads();
      for (int w = tid; w < (E / 2) * E; w += nt) {  // columns p, q: pairs fastest (distinct banks)
        const int i = w % (E / 2), j = w / (E / 2);
        const int p = pp[i], q = qq[i];
        const double c = cs[i], s = sn[i];
        const double mp = M[j * E + p], mq = M[j * E + q];
        M[j * E + p] = c * mp - s * mq;
        M[j * E + q] = s * mp + c * mq;
      }
      for (int w = tid; w < (E / 2) * E; w += nt) {  // eigenvectors, stored transposed: rows p, q
        const int i = w / E, j = w - i * E;
        const int p = pp[i], q = qq[i];
        const double c = cs[i], s = sn[i];
        const double vp = Vl[(size_t)p * E + j], vq = Vl[(size_t)q * E + j];
        Vl[(size_t)p * E + j] = c * vp - s * vq;
        Vl[(size_t)q * E + j] = s * vp + c * vq;
      }
      __syncthreads();
    }
    const bool stop = s_done != 0;  // read by every thread before thread 0 resets it
    __syncthreads();
    if (stop) break;
  }
  // the G largest eigenvalues (ties: lower index) pick the embedding's columns
  double* U = Uo + (size_t)l * E * G;
  for (int a = tid; a < E; a += nt) {
    const double la = M[a * E + a];
    int rank = 0;
    for (int b = 0; b < E; ++b) {
      const double lb = M[b * E + b];
      rank += (lb > la || (lb == la && b < a)) ? 1 : 0;
    }
    if (rank < G)  // eigenvector a is row a of the transposed matrix
      for (int e = 0; e < E; ++e) U[(size_t)e * G + rank] = Vl[(size_t)a * E + e];
  }
  __syncthreads();
  for (int e = tid; e < E; e += nt) {  // unit rows
    double n2 = 0.0;
    for (int g = 0; g < G; ++g) n2 += U[(size_t)e * G + g] * U[(size_t)e * G + g];
    const double n = sqrt(n2);
    for (int g = 0; g < G; ++g) U[(size_t)e * G + g] = n > 0.0 ? U[(size_t)e * G + g] / n : 0.0;
  }
}

size_t spec_embed_smem(int E);

// Size-bounded assignment by warp 0 (lanes 0..31): a = previous assignment or
// greedy nearest-with-room at the first step, then negative cycles of the
// residual graph on the G groups plus the slack node t = G are cancelled.
__device__ void sp_assign(const double* cost, int E, int G, int lo, int hi, int* a, const int* prev, bool first,
                          double* W, int* widx, int* sz, int* s_pred, int* mv_pt, int* mv_to, int* nmv,
                          uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int n = G + 1, t = G, ld = G + 1;
  if (first) {
    if (lane == 0) {
      for (int g = 0; g < G; ++g) sz[g] = 0;
      for (int e = 0; e < E; ++e) {
        int best = -1;
        for (int g = 0; g < G; ++g) {
          if (sz[g] >= hi) continue;
          if (best < 0 || cost[e * G + g] < cost[e * G + best]) best = g;
        }
        a[e] = best;
        sz[best] += 1;
      }
    }
  } else {
    for (int e = lane; e < E; e += 32) a[e] = prev[e];
  }
  double mx = 0.0;
  for (int q = lane; q < E * G; q += 32) mx = fmax(mx, fabs(cost[q]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(FULL, mx, o));
  const double eps = 1e-12 * mx + 1e-300;
  const double big = 1.0 + 4.0 * (mx + 1.0) * E;  // any lower-bound repair beats any cost change
  __syncwarp();
  const int max_pass = 16 * E + 1024;
  int done = 0;
  for (int pass = 0; pass < max_pass; ++pass) {
    if (lane == 0) {
      for (int g = 0; g < G; ++g) sz[g] = 0;
      for (int e = 0; e < E; ++e) sz[a[e]] += 1;
    }
    __syncwarp();
    for (int q = lane; q < G * G; q += 32) {  // edge u -> v: the cheapest member of u to move
      const int u = q / G, v = q - u * G;
      double best = INFINITY;
      int bp = INT_MAX;
      if (u != v)
        for (int p = 0; p < E; ++p) {
          if (a[p] != u) continue;
          const double val = cost[p * G + v] - cost[p * G + u];
          if (val < best) {
            best = val;
            bp = p;
          }
        }
      W[u * ld + v] = best;
      widx[q] = bp;
    }
    for (int u = lane; u < G; u += 32) {
      W[t * ld + u] = sz[u] > lo ? 0.0 : INFINITY;                        // u may shrink
      W[u * ld + t] = sz[u] < lo ? -big : (sz[u] < hi ? 0.0 : INFINITY);  // u may (must) grow
    }
    if (lane == 0) W[t * ld + t] = INFINITY;
    __syncwarp();
    double dist = 0.0;
    int pred = -1;
    for (int round = 0; round < 2 * (n + 1); ++round) {
      double best = dist;
      int from = pred;
      for (int u = 0; u < n; ++u) {
        const double du = __shfl_sync(FULL, dist, u);
        if (lane < n && u != lane) {
          const double w = W[u * ld + lane];
          if (w < INFINITY && du + w < best) {
            best = du + w;
            from = u;
          }
        }
      }
      const bool changed = best < dist;
      dist = best;
      pred = from;
      if (!__any_sync(FULL, changed)) break;
    }
    if (lane < n) s_pred[lane] = pred;
    __syncwarp();
    int x = lane;
    bool alive = lane < n;
    for (int st = 0; st < n && alive; ++st) {
      const int nx = s_pred[x];
      if (nx < 0) alive = false;
      else x = nx;
    }
    const unsigned on = __ballot_sync(FULL, alive);
    const int start = __shfl_sync(FULL, x, on ? (__ffs(on) - 1) : 0);
    if (lane == 0) {
      *nmv = 0;
      if (on) {
        int y = start, k = 0, m = 0;
        double w = 0.0;
        bool ok = true;
        do {
          const int py = s_pred[y];
          if (py < 0) {
            ok = false;
            break;
          }
          w += W[py * ld + y];
          if (py != t && y != t) {
            if (widx[py * G + y] >= E) {
              ok = false;
              break;
            }
            mv_pt[m] = widx[py * G + y];
            mv_to[m] = y;
            ++m;
          }
          y = py;
          ++k;
        } while (y != start && k <= n);
        if (ok && y == start && w < -eps) *nmv = m;
      }
    }
    __syncwarp();
    if (*nmv == 0) {
      done = 1;
      break;
    }
    if (lane == 0)
      for (int m = 0; m < *nmv; ++m) a[mv_pt[m]] = mv_to[m];
    __syncwarp();
  }
  if (lane == 0 && !done) atomicOr(status, WS_BIT_ETIMEOUT);
  __syncwarp();
}

__global__ void __launch_bounds__(SP_GROUP_THREADS, 1)
    spec_group_kernel(const int32_t* __restrict__ affinity, int E, int G, const double* __restrict__ Uo,
                      const double* __restrict__ deg, int32_t* __restrict__ groups, double* __restrict__ ucurve,
                      double* __restrict__ scurve, uint32_t* status) {
  extern __shared__ double gp_sm[];
  double* Us = gp_sm;                        // [E][G]
  double* C = Us + E * G;                    // [G][G]
  double* cost = C + G * G;                  // [E][G]
  double* mind = cost + E * G;               // [E]
  double* W = mind + E;                      // [G+1][G+1]
  int* a = reinterpret_cast<int*>(W + (G + 1) * (G + 1));  // [E]
  int* prev = a + E;                         // [E]
  int* widx = prev + E;                      // [G][G]
  int* sz = widx + G * G;                    // [G]
  int* s_pred = sz + G;                      // [32]
  int* mv_pt = s_pred + 32;                  // [32]
  int* mv_to = mv_pt + 32;                   // [32]
  __shared__ int s_seed, s_nmv;
  __shared__ long long red_same[SP_GROUP_THREADS / 32], red_tot[SP_GROUP_THREADS / 32];
  const int j = blockIdx.x, l = blockIdx.y, tid = threadIdx.x, nt = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int lo = max(1, (E * (16 - j)) / (16 * G));
  const int hi = min(E, (E * (16 + j) + 16 * G - 1) / (16 * G));
  const double* Ul = Uo + (size_t)l * E * G;
  for (int q = tid; q < E * G; q += nt) Us[q] = Ul[q];
  if (tid == 0) {
    int best = 0;
    for (int e = 1; e < E; ++e)
      if (deg[(size_t)l * E + e] > deg[(size_t)l * E + best]) best = e;
    s_seed = best;
  }
  __syncthreads();
  // seeds: the largest degree, then repeatedly the farthest row from the seeds so far
  for (int g = 0; g < G; ++g) {
    if (g > 0) {
      if (tid == 0) {
        int best = 0;
        for (int e = 1; e < E; ++e)
          if (mind[e] > mind[best]) best = e;
        s_seed = best;
      }
      __syncthreads();
    }
    const int sd = s_seed;
    for (int d = tid; d < G; d += nt) C[g * G + d] = Us[sd * G + d];
    for (int e = tid; e < E; e += nt) {
      double dd = 0.0;
      for (int d = 0; d < G; ++d) {
        const double x = Us[e * G + d] - Us[sd * G + d];
        dd += x * x;
      }
      mind[e] = g == 0 ? dd : fmin(mind[e], dd);
    }
    __syncthreads();
  }
  // size-bounded K-means
  bool first = true;
  for (int step = 0; step < SP_MAX_STEPS; ++step) {
    for (int q = tid; q < E * G; q += nt) {
      const int e = q / G, g = q - e * G;
      double dd = 0.0;
      for (int d = 0; d < G; ++d) {
        const double x = Us[e * G + d] - C[g * G + d];
        dd += x * x;
      }
      cost[q] = dd;
    }
    __syncthreads();
    if (warp == 0) sp_assign(cost, E, G, lo, hi, a, prev, first, W, widx, sz, s_pred, mv_pt, mv_to, &s_nmv, status);
    __syncthreads();
    int changed = 0;
    if (!first)
      for (int e = tid; e < E; e += nt) changed |= (a[e] != prev[e]);
    changed = __syncthreads_or(changed);
    if (!first && !changed) break;
    first = false;
    for (int e = tid; e < E; e += nt) prev[e] = a[e];
    for (int q = tid; q < G * G; q += nt) {  // centroid g, coordinate d: mean over its rows
      const int g = q / G, d = q - g * G;
      double sum = 0.0;
      int cnt = 0;
      for (int e = 0; e < E; ++e)
        if (a[e] == g) {
          sum += Us[e * G + d];
          ++cnt;
        }
      C[q] = cnt > 0 ? sum / cnt : 0.0;
    }
    __syncthreads();
  }
  // outputs for this grid point: groups, utilisation, size deviation
  int32_t* gout = groups + ((size_t)l * SP_NGRID + j) * E;
  for (int e = tid; e < E; e += nt) gout[e] = a[e];
  const int32_t* A = affinity + (size_t)l * E * E;
  long long same = 0, tot = 0;
  for (int q = tid; q < E * E; q += nt) {
    const int x = q / E, y = q - x * E;
    if (x == y) continue;
    const long long v = A[q] > 0 ? A[q] : 0;
    tot += v;
    if (a[x] == a[y]) same += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    same += __shfl_xor_sync(FULL, same, o);
    tot += __shfl_xor_sync(FULL, tot, o);
  }
  if (lane == 0) {
    red_same[warp] = same;
    red_tot[warp] = tot;
  }
  __syncthreads();
  if (tid == 0) {
    long long S_ = 0, T_ = 0;
    for (int w = 0; w < nt / 32; ++w) {
      S_ += red_same[w];
      T_ += red_tot[w];
    }
    ucurve[(size_t)l * SP_NGRID + j] = T_ > 0 ? (double)S_ / (double)T_ : 0.0;
    for (int g = 0; g < G; ++g) sz[g] = 0;
    for (int e = 0; e < E; ++e) sz[a[e]] += 1;
    const double mean = (double)E / (double)G;
    double acc = 0.0;
    for (int g = 0; g < G; ++g) {
      const double dlt = (double)sz[g] - mean;
      acc = __dadd_rn(acc, __dmul_rn(dlt, dlt));
    }
    scurve[(size_t)l * SP_NGRID + j] = sqrt(acc / (double)G) / mean;
  }
}

// Knee of U over r and the chosen groups, one warp per layer.
__global__ void __launch_bounds__(32) spec_knee_kernel(const int32_t* __restrict__ groups,
                                                       const double* __restrict__ ucurve, int E,
                                                       int32_t* __restrict__ group_of, int32_t* __restrict__ knee) {
  __shared__ int s_k;
  const int l = blockIdx.x, lane = threadIdx.x;
  if (lane == 0) {
    const double* Uc = ucurve + (size_t)l * SP_NGRID;
    double mn = Uc[0], mx = Uc[0];
    for (int j = 1; j < SP_NGRID; ++j) {
      mn = fmin(mn, Uc[j]);
      mx = fmax(mx, Uc[j]);
    }
    const double rng = __dsub_rn(mx, mn);
    double y[SP_NGRID];
    for (int j = 0; j < SP_NGRID; ++j) y[j] = rng > 0.0 ? __ddiv_rn(__dsub_rn(Uc[j], mn), rng) : 0.0;
    const double x0 = 0.0, dx = 1.0, dy = __dsub_rn(y[SP_NGRID - 1], y[0]);
    int best = 0;
    double bc = 0.0;
    for (int j = 0; j < SP_NGRID; ++j) {
      const double xj = __ddiv_rn((double)j, (double)(SP_NGRID - 1));
      const double c = __dsub_rn(__dmul_rn(dx, __dsub_rn(y[j], y[0])), __dmul_rn(dy, __dsub_rn(xj, x0)));
      if (c > bc) {
        best = j;
        bc = c;
      }
    }
    s_k = best;
    knee[l] = best;
  }
  __syncwarp();
  const int k = s_k;
  for (int e = lane; e < E; e += 32) group_of[(size_t)l * E + e] = groups[((size_t)l * SP_NGRID + k) * E + e];
}

size_t spec_group_smem(int E, int G) {
  return ((size_t)E * G * 2 + (size_t)G * G + E + (size_t)(G + 1) * (G + 1)) * sizeof(double) +
         ((size_t)E * 2 + (size_t)G * G + G + 96) * sizeof(int);
}

struct SpLayout {
  size_t V, U, deg, groups, total;
};

static SpLayout sp_layout(int L, int E, int G) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  SpLayout o;
  o.V = WS_HEADER;
  o.U = o.V + r256((size_t)L * E * E * sizeof(double));
  o.deg = o.U + r256((size_t)L * E * G * sizeof(double));
  o.groups = o.deg + r256((size_t)L * E * sizeof(double));
  o.total = o.groups + r256((size_t)L * SP_NGRID * E * sizeof(int32_t));
  return o;
}

size_t spectral_workspace_bytes(int L, int E, int G) { return sp_layout(L, E, G).total; }

moer_status spectral_launch(const moer_dims* d, const int32_t* affinity, int32_t G, int32_t* group_of,
                            int32_t* knee, double* u_curve, double* s_curve, void* ws, cudaStream_t st) {
  const int L = d->L, E = d->E;
  const SpLayout o = sp_layout(L, E, G);
  char* w = static_cast<char*>(ws);
  double* V = reinterpret_cast<double*>(w + o.V);
  double* U = reinterpret_cast<double*>(w + o.U);
  double* deg = reinterpret_cast<double*>(w + o.deg);
  int32_t* groups = reinterpret_cast<int32_t*>(w + o.groups);
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(spec_embed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)spec_embed_smem(SP_MAXE)) != cudaSuccess ||
        cudaFuncSetAttribute(spec_group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)spec_group_smem(SP_MAXE, SP_MAXG)) != cudaSuccess)
      return MOER_ECUDA;
    configured = true;
  }
  spec_embed_kernel<<<L, SP_EMBED_THREADS, spec_embed_smem(E), st>>>(affinity, E, G, V, U, deg);
  spec_group_kernel<<<dim3(SP_NGRID, L), SP_GROUP_THREADS, spec_group_smem(E, G), st>>>(
      affinity, E, G, U, deg, groups, u_curve, s_curve, reinterpret_cast<uint32_t*>(ws));
  spec_knee_kernel<<<L, 32, 0, st>>>(groups, u_curve, E, group_of, knee);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

size_t spec_embed_smem(int E) { return ((size_t)E * E + E + E + 32) * sizeof(double) + (size_t)E * sizeof(int); }

}  // namespace moer
