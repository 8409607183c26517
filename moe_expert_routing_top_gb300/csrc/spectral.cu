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
//     std of the group sizes / (E/G), evaluated as sqrt(G sum size^2 - E^2) / E
//     from an exact integer; the knee of U over r (scaled to [0, 1],
//     the point farthest above the chord from r = 0 to r = 1) picks the groups.
//
// Design (GB300):
//   * spec_embed_kernel, one CTA per layer: M lives in shared memory (fp64,
//     128 KB at E = 128).  Householder reduction to tridiagonal form (the
//     matrix-vector product eight threads per row, the rank-2 update over the
//     whole trailing block), the G largest eigenvalues by Sturm-count
//     multisection (a warp per eigenvalue, a lane per trial point), their
//     eigenvectors by inverse iteration on the tridiagonal form, taken back
//     through the reflections.  A full solve of the spectrum is not needed:
//     only G eigenpairs are formed.  Subspace iteration on the top-G space is
//     not an option either: the co-activation spectra of real layers are
//     nearly degenerate just below the leading eigenvalues, where it needs
//     10^4 - 10^5 steps.
//   * spec_group_kernel, one CTA per (grid point, layer), six per SM: the
//     size-bounded assignment is a transportation problem with lower and upper
//     bounds; the CTA keeps a feasible assignment and cancels negative cycles of
//     the residual graph collapsed onto the G groups plus one slack node t
//     (t -> u when u may shrink, u -> t when u may grow, a large negative u -> t
//     while u is below its lower bound).  Scans and minima compare integer keys
//     of the fp64 gains; Bellman-Ford relaxes the nodes a warp each.
//   * spec_knee_kernel, one warp per layer: the knee and the chosen groups.
#include <climits>

#include "common.cuh"
#include "keys.cuh"

namespace moer {

constexpr int SP_MAXE = 128;
constexpr int SP_MAXG = 31;
constexpr int SP_NGRID = 17;
constexpr int SP_EMBED_THREADS = 1024;
constexpr int SP_GROUP_THREADS = 256;
constexpr int SP_MAX_STEPS = 100;
constexpr int SP_LU_SLOTS = 8;  // eigenvectors whose inverse iterations run at once (a warp each)
constexpr int SP_MS_POINTS = 16;  // multisection trial points per eigenvalue (a lane each)


__device__ __forceinline__ double sp_warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

// Number of eigenvalues of the tridiagonal form below x: the sign changes in
// the leading principal minors of T - x I (p_0 = 1, p_1 = d_0 - x,
// p_{i+1} = (d_i - x) p_i - e_i^2 p_{i-1}, e_i^2 = e2[i]).  This is the ratio
// form's count (pivot q_i = p_{i+1} / p_i < 0) without its division: fp64
// divisions are a long instruction sequence on this part, and a Sturm count
// is the multisection's whole cost.  A minor below 2^-52 of the one before it
// is replaced by -2^-52 times that one (the ratio form's pivot floored to a
// tiny negative), and both carried minors are rescaled by an exact power of
// two when the newer leaves [2^-256, 2^256]; both tests read the exponent
// field.
__device__ __forceinline__ int sp_sturm(const double* dg, const double* e2, int n, double x) {
  auto expo = [](double v) { return (int)(((unsigned long long)__double_as_longlong(v) >> 52) & 0x7FF); };
  auto sgn = [](double v) { return (unsigned)((unsigned long long)__double_as_longlong(v) >> 63); };
  double pm = 1.0, p = dg[0] - x;
  if (expo(p) + 52 < 1023) p = -0x1p-52;
  int c = (int)sgn(p);
  for (int i = 1; i < n; ++i) {
    const double pn = fma(dg[i] - x, p, -(e2[i] * pm));
    pm = p;
    p = pn;
    const int ep = expo(p);
    if (ep + 52 < expo(pm)) {
      p = -0x1p-52 * pm;
    } else if (ep > 1023 + 256 || ep < 1023 - 256) {
      const double sc = __longlong_as_double((long long)(2046 - ep) << 52);  // 2^(1023 - ep)
      p *= sc;
      pm *= sc;
    }
    c += (int)(sgn(p) ^ sgn(pm));
  }
  return c;
}

// Spectral embedding of one layer (CTA l), all in fp64:
//   * M = D^-1/2 A D^-1/2 (A the co-activation without its diagonal, D its
//     row sums) in shared memory, reduced to tridiagonal form T by E - 2
//     Householder reflections H_k (x = column k below the diagonal,
//     v = x - alpha e_1 with alpha = -sign(x_0) |x|, beta = 2 / v.v; the
//     trailing block becomes A - v w^T - w v^T with p = beta A v,
//     w = p - (beta v.p / 2) v).  v is kept in row k right of the diagonal.
//   * The G largest eigenvalues of T by multisection: a group of sixteen lanes
//     brackets the (j+1)-th largest between Gershgorin bounds and narrows the
//     bracket 17-fold per step with Sturm counts at sixteen points (one per
//     lane), two eigenvalues per warp.
//   * Their eigenvectors by inverse iteration on T (LU with partial pivoting,
//     three solves from a fixed start vector; after each solve, in eigenvalue
//     order, re-orthogonalised against the earlier vectors whose eigenvalues
//     lie within 1e-3 |T|), eight vectors at once, a warp each; then taken
//     back through the reflections: x = H_0 ... H_{E-3} y.
//   Rows of the embedding are the G eigenvectors' components, scaled to unit
//   length.  Only the G vectors are formed: fp64 divisions and square roots
//   are slow on this part, and a full QL solve spent ~37 M clock cycles per
//   layer in its sequential recurrence.
__global__ void __launch_bounds__(SP_EMBED_THREADS, 1)
    spec_embed_kernel(const int32_t* __restrict__ affinity, int E, int G, double* __restrict__ Uo,
                      double* __restrict__ deg_out) {
  extern __shared__ double sp_sm[];
  const int n = E;
  double* M = sp_sm;         // [E][E + 1] (padded rows)
  double* inv = M + E * (E + 1);  // [E] D^-1/2
  double* vv = inv + E;      // [E] Householder vector
  double* pw = vv + E;       // [E] p, then w; later e2[i] = sd[i-1]^2
  double* dg = pw + E;       // [E] diagonal of T
  double* sd = dg + E;       // [E] subdiagonal: sd[i] couples i and i + 1
  double* bet = sd + E;      // [E] beta of reflection k (0: none needed)
  double* lam = bet + E;     // [32] eigenvalues, largest first
  double* red = lam + 32;    // [32]
  double* Y = red + 32;      // [G][E] eigenvectors
  // LU of T - lambda I for up to SP_LU_SLOTS eigenvectors at once, slot s at
  // s * E: reciprocal pivots, first and second superdiagonal, multipliers,
  // row swaps
  double* lu0 = Y + (size_t)G * E;
  double* lu1 = lu0 + SP_LU_SLOTS * E;
  double* lu2 = lu1 + SP_LU_SLOTS * E;
  double* lmul = lu2 + SP_LU_SLOTS * E;
  int* lsw = reinterpret_cast<int*>(lmul + SP_LU_SLOTS * E);
  const int l = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int S = E + 1;  // row stride of M: consecutive rows start two banks apart
  const int32_t* A = affinity + (size_t)l * E * E;
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
    M[a * S + b] = (a == b) ? 0.0 : inv[a] * (double)x * inv[b];
  }
  __syncthreads();
  // ---- Householder reduction to tridiagonal form
  for (int k = 0; k + 2 < n; ++k) {
    const int m = n - k - 1;  // length of x = M[k+1 ..][k]
    if (warp == 0) {
      double s2 = 0.0;
      for (int j = 1 + lane; j < m; j += 32) {
        const double x = M[(k + 1 + j) * S + k];
        s2 = fma(x, x, s2);
      }
      s2 = sp_warp_sum(s2);
      if (lane == 0) {
        const double x0 = M[(k + 1) * S + k];
        if (s2 == 0.0) {  // already reduced
          sd[k] = x0;
          bet[k] = 0.0;
        } else {
          const double sig = fma(x0, x0, s2);
          const double alpha = x0 > 0.0 ? -sqrt(sig) : sqrt(sig);
          sd[k] = alpha;
          bet[k] = 1.0 / (sig - alpha * x0);
          red[0] = x0 - alpha;
        }
        dg[k] = M[k * S + k];
      }
    }
    __syncthreads();
    const double beta = bet[k];
    if (beta == 0.0) continue;
    for (int j = tid; j < m; j += nt) vv[j] = j == 0 ? red[0] : M[(k + 1 + j) * S + k];
    __syncthreads();
    {  // p = beta A22 v, eight threads per row (nt / 8 >= m rows); only the
       // lower triangle of A22 is kept, so A22[i][j] for j > i is read as A22[j][i]
      const int i = tid >> 3;
      double acc = 0.0;
      if (i < m) {
        const double* a22 = M + (k + 1) * S + (k + 1);
        for (int j = tid & 7; j < m; j += 8) acc = fma(j <= i ? a22[i * S + j] : a22[j * S + i], vv[j], acc);
      }
      acc += __shfl_xor_sync(FULL, acc, 1);
      acc += __shfl_xor_sync(FULL, acc, 2);
      acc += __shfl_xor_sync(FULL, acc, 4);
      if (i < m && (tid & 7) == 0) pw[i] = beta * acc;
    }
    __syncthreads();
    if (warp == 0) {
      double t = 0.0;
      for (int j = lane; j < m; j += 32) t = fma(vv[j], pw[j], t);
      t = sp_warp_sum(t);
      if (lane == 0) red[1] = 0.5 * beta * t;
    }
    __syncthreads();
    const double kc = red[1];
    for (int j = tid; j < m; j += nt) pw[j] = fma(-kc, vv[j], pw[j]);
    __syncthreads();
    {  // A22 -= v w^T + w v^T on the lower triangle: warp u takes rows u and
       // m-1-u (together m+1 elements), then u + 32 and m-1-(u+32), ...
      double* a22 = M + (k + 1) * S + (k + 1);
      const int nw = nt >> 5;
      for (int pr = warp; pr < (m + 1) / 2; pr += nw) {
        const int ra = pr, rb = m - 1 - pr;
        const int len = (ra + 1) + (rb != ra ? rb + 1 : 0);
        for (int t = lane; t < len; t += 32) {
          const int i = t <= ra ? ra : rb, j = t <= ra ? t : t - (ra + 1);
          double* e = a22 + i * S + j;
          *e = *e - vv[i] * pw[j] - pw[i] * vv[j];
        }
      }
    }
    for (int j = tid; j < m; j += nt) M[k * S + (k + 1 + j)] = vv[j];  // v, for the eigenvectors
    __syncthreads();
  }
  if (tid == 0) {
    dg[n - 2] = M[(n - 2) * S + (n - 2)];
    sd[n - 2] = M[(n - 1) * S + (n - 2)];
    dg[n - 1] = M[(n - 1) * S + (n - 1)];
    sd[n - 1] = 0.0;
    double tn = 0.0;  // Gershgorin bound of T
    for (int i = 0; i < n; ++i) tn = fmax(tn, fabs(dg[i]) + fabs(sd[i]) + (i > 0 ? fabs(sd[i - 1]) : 0.0));
    red[2] = tn;
  }
  __syncthreads();
  for (int i = tid; i < n; i += nt) pw[i] = i > 0 ? sd[i - 1] * sd[i - 1] : 0.0;
  __syncthreads();
  const double eps = 2.220446049250313e-16;
  const double tn = red[2];
  const double pivmin = eps * tn + 1e-300;
  // ---- the G largest eigenvalues by multisection: lanes in groups of
  //      SP_MS_POINTS, group e (warp e / groups-per-warp) for the (e+1)-th
  //      largest, a trial point per lane.  Two eigenvalues share a warp: half
  //      the warps of one per warp (32 points), for 4.1 rather than 5 bits a
  //      step; the counts of fewer warps contend less for the fp64 pipe.
  {
    constexpr int P = SP_MS_POINTS, GPW = 32 / SP_MS_POINTS;
    const int ev = warp * GPW + lane / P, sub = lane % P, base = lane - sub;
    if (warp * GPW < G) {
      const bool act = ev < G;
      const int j = n - 1 - ev;  // eigenvalues below the (ev+1)-th largest
      double lo = -tn - pivmin, hi = tn + pivmin;
      bool done = !act;
      for (int it = 0; it < 256; ++it) {
        const double x = lo + (hi - lo) * ((double)(sub + 1) / (double)(P + 1));
        const int cnt = act ? sp_sturm(dg, pw, n, x) : 0;
        const unsigned gb = (__ballot_sync(FULL, act && cnt > j) >> base) & ((1u << P) - 1u);
        const int f = gb ? __ffs(gb) - 1 : 0;
        const double xl = __shfl_sync(FULL, x, base + P - 1);
        const double xf = __shfl_sync(FULL, x, base + f);
        const double xp = __shfl_sync(FULL, x, base + (f > 0 ? f - 1 : 0));
        if (!done) {
          if (gb == 0u) {
            lo = xl;
          } else {
            hi = xf;
            if (f > 0) lo = xp;
          }
          done = hi - lo <= 2.0 * eps * fmax(fabs(lo), fabs(hi)) + pivmin;
        }
        if (__all_sync(FULL, done)) break;
      }
      if (act && sub == 0) lam[ev] = 0.5 * (lo + hi);
    }
  }
  __syncthreads();
  // ---- inverse iteration, up to SP_LU_SLOTS eigenvectors at once: warp w
  //      factors and solves for vector w0 + w (lane 0 runs the recurrences);
  //      between iterations warp 0 re-orthogonalises the batch in order against
  //      the earlier vectors with eigenvalues within 1e-3 |T| and normalises
  for (int w0 = 0; w0 < G; w0 += SP_LU_SLOTS) {
    const int nb = min(SP_LU_SLOTS, G - w0);
    const int w = warp;
    double* y = Y + (size_t)(w0 + w) * n;
    double* f0 = lu0 + (size_t)w * n;
    double* f1 = lu1 + (size_t)w * n;
    double* f2 = lu2 + (size_t)w * n;
    double* fm = lmul + (size_t)w * n;
    int* fs = lsw + (size_t)w * n;
    if (w < nb) {
      const double lambda = lam[w0 + w];
      if (lane == 0) {
        double ca = dg[0] - lambda, cb = sd[0];
        for (int i = 0; i + 1 < n; ++i) {
          const double nc = sd[i], na = dg[i + 1] - lambda, nb2 = i + 2 < n ? sd[i + 1] : 0.0;
          if (fabs(ca) >= fabs(nc) || fabs(nc) <= pivmin) {  // no swap; a pivot below pivmin is floored
            const double piv = fabs(ca) > pivmin ? ca : (ca >= 0.0 ? pivmin : -pivmin);
            const double r = 1.0 / piv;
            f0[i] = r;
            f1[i] = cb;
            f2[i] = 0.0;
            fm[i] = nc * r;
            fs[i] = 0;
            ca = na - fm[i] * cb;
            cb = nb2;
          } else {
            const double r = 1.0 / nc;
            f0[i] = r;
            f1[i] = na;
            f2[i] = nb2;
            fm[i] = ca * r;
            fs[i] = 1;
            ca = cb - fm[i] * na;
            cb = -fm[i] * nb2;
          }
        }
        f0[n - 1] = 1.0 / (fabs(ca) > pivmin ? ca : (ca >= 0.0 ? pivmin : -pivmin));
      }
      for (int i = lane; i < n; i += 32) y[i] = (double)(((unsigned)i * 2654435761u) % 1000u) / 1000.0 - 0.499;
      __syncwarp();
    }
    for (int it = 0; it < 3; ++it) {
      if (w < nb && lane == 0) {  // solve (T - lambda I) y' = y
        for (int i = 0; i + 1 < n; ++i) {
          if (fs[i]) {
            const double t = y[i];
            y[i] = y[i + 1];
            y[i + 1] = t;
          }
          y[i + 1] -= fm[i] * y[i];
        }
        y[n - 1] *= f0[n - 1];
        y[n - 2] = (y[n - 2] - f1[n - 2] * y[n - 1]) * f0[n - 2];
        for (int i = n - 3; i >= 0; --i) y[i] = (y[i] - f1[i] * y[i + 1] - f2[i] * y[i + 2]) * f0[i];
      }
      __syncthreads();
      if (warp == 0) {
        for (int v = w0; v < w0 + nb; ++v) {
          double* yv = Y + (size_t)v * n;
          for (int u = 0; u < v; ++u) {
            if (fabs(lam[u] - lam[v]) > 1e-3 * tn) continue;
            const double* z = Y + (size_t)u * n;
            double t = 0.0;
            for (int i = lane; i < n; i += 32) t = fma(z[i], yv[i], t);
            t = sp_warp_sum(t);
            for (int i = lane; i < n; i += 32) yv[i] = fma(-t, z[i], yv[i]);
            __syncwarp();
          }
          double s2 = 0.0;
          for (int i = lane; i < n; i += 32) s2 = fma(yv[i], yv[i], s2);
          s2 = sp_warp_sum(s2);
          const double sc = s2 > 0.0 ? 1.0 / sqrt(s2) : 0.0;
          for (int i = lane; i < n; i += 32) yv[i] *= sc;
          __syncwarp();
        }
      }
      __syncthreads();
    }
  }
  // ---- back through the reflections: y <- H_k y for k = E-3 .. 0, warp j for vector j
  if (warp < G) {
    double* y = Y + (size_t)warp * n;
    for (int k = n - 3; k >= 0; --k) {
      if (bet[k] == 0.0) continue;
      const int m = n - k - 1;
      const double* v = M + k * S + (k + 1);
      double t = 0.0;
      for (int j = lane; j < m; j += 32) t = fma(v[j], y[k + 1 + j], t);
      const double f = bet[k] * sp_warp_sum(t);
      for (int j = lane; j < m; j += 32) y[k + 1 + j] = fma(-f, v[j], y[k + 1 + j]);
      __syncwarp();
    }
  }
  __syncthreads();
  double* U = Uo + (size_t)l * E * G;
  for (int e = tid; e < E; e += nt) {  // unit rows
    double n2 = 0.0;
    for (int g = 0; g < G; ++g) n2 = fma(Y[(size_t)g * n + e], Y[(size_t)g * n + e], n2);
    const double sc = n2 > 0.0 ? 1.0 / sqrt(n2) : 0.0;
    for (int g = 0; g < G; ++g) U[(size_t)e * G + g] = Y[(size_t)g * n + e] * sc;
  }
}

size_t spec_embed_smem(int E, int G);

// Size-bounded assignment by the whole CTA: a = previous assignment or, at the
// first step, greedy nearest-with-room in regret order, then negative cycles of the residual
// graph on the G groups plus the slack node t = G are cancelled.  Each expert
// keeps a row of its gains cost[p][v] - cost[p][a(p)] as order-preserving
// integer keys (rewritten only for the experts that move), so the edge minima
// (the cheapest member of u to move to v, ties to the lower point), taken by
// all threads a few per edge, compare integers.  Disjoint negative 2-cycles
// between groups (swaps) go first, several per pass; when none is left,
// Bellman-Ford runs with a warp per node in synchronous rounds and stops at the
// first round whose predecessor graph closes a negative cycle (through the
// slack node when sizes must change).  Thread 0 moves the points.
__device__ void sp_assign(const double* cost, int E, int G, int lo, int hi, int* a, const int* prev, bool first,
                          double* W, int* widx, int* sz, int* s_pred, int* mv_pt, int* mv_to, int* nmv,
                          unsigned long long* dk, uint32_t* status) {
  __shared__ unsigned long long sp_red[SP_GROUP_THREADS / 32];
  __shared__ unsigned long long s_key[SP_MAXE];
  __shared__ int s_ord[SP_MAXE];
  __shared__ double bf_dist[2][32];
  __shared__ unsigned negmask[32];
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int n = G + 1, t = G, ld = G + 1, DS = G + 1;
  if (first) {
    // greedy nearest-with-room in regret order: the experts whose nearest centroid
    // beats their second nearest by most go first (larger regret, then lower id)
    int P = 1;
    while (P < E) P <<= 1;
    for (int i = tid; i < P; i += nt) {
      unsigned long long rk = 0ull;  // padding sorts last
      if (i < E) {
        unsigned long long b1 = ~0ull, b2 = ~0ull;
        for (int g = 0; g < G; ++g) {
          const unsigned long long c = okey(cost[i * G + g]);
          if (c < b1) {
            b2 = b1;
            b1 = c;
          } else if (c < b2) {
            b2 = c;
          }
        }
        rk = okey(okey_value(b2) - okey_value(b1));
      }
      s_key[i] = rk;
      s_ord[i] = i;
    }
    __syncthreads();
    for (int k = 2; k <= P; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = tid; i < P; i += nt) {
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
    if (warp == 0) {
      // lane g owns group g's size; a keyed warp minimum over the lanes with
      // room picks the nearest (ties: the lower group)
      int cnt = 0;
      for (int r = 0; r < E; ++r) {
        const int e = s_ord[r];
        unsigned long long key = lane < G && cnt < hi ? okey(cost[e * G + lane]) : ~0ull;
        int g = lane;
        warp_min_key(key, g);
        if (lane == g) ++cnt;
        if (lane == 0) a[e] = g;
      }
    }
  } else {
    for (int e = tid; e < E; e += nt) a[e] = prev[e];
  }
  __syncthreads();
  // gain keys of every expert, and the largest |cost| (bit patterns of
  // non-negative doubles order as integers)
  unsigned long long mx = 0ull;
  for (int q = tid; q < E * G; q += nt) {
    const int p = q / G, v = q - p * G;
    const double c = cost[q];
    dk[p * DS + v] = okey(c - cost[p * G + a[p]]);
    const unsigned long long ab = (unsigned long long)__double_as_longlong(c) & 0x7FFFFFFFFFFFFFFFull;
    mx = ab > mx ? ab : mx;
  }
  {
    unsigned long long cm = ~mx;  // the maximum is the complement of the complements' minimum
    int unused = 0;
    warp_min_key(cm, unused);
    mx = ~cm;
  }
  if (lane == 0) sp_red[warp] = mx;
  __syncthreads();
  mx = 0ull;
  for (int w = 0; w < nt / 32; ++w) mx = sp_red[w] > mx ? sp_red[w] : mx;
  const double mxd = __longlong_as_double((long long)mx);
  const double eps = 1e-12 * mxd + 1e-300;
  const double big = 1.0 + 4.0 * (mxd + 1.0) * E;  // any lower-bound repair beats any cost change
  int tpe = 32;  // threads per edge: a power of two, so an edge's threads share a warp
  while (tpe > 1 && tpe * G * G > nt) tpe >>= 1;
  const int max_pass = 16 * E + 1024;
  int done = 0;
  for (int pass = 0; pass < max_pass; ++pass) {
    for (int g = tid; g < G; g += nt) {
      sz[g] = 0;
      negmask[g] = 0u;
    }
    __syncthreads();
    for (int e = tid; e < E; e += nt) atomicAdd(&sz[a[e]], 1);
    for (int q0 = 0; q0 < G * G; q0 += nt / tpe) {  // edge u -> v: the cheapest member of u to move
      const int q = q0 + tid / tpe, sub = tid % tpe;
      const int u = q / G, v = q - u * G;
      unsigned long long best = ~0ull;
      int bp = INT_MAX;
      if (q < G * G && u != v)
        for (int p = sub; p < E; p += tpe) {
          if (a[p] != u) continue;
          const unsigned long long kk = dk[p * DS + v];
          if (kk < best || (kk == best && p < bp)) {
            best = kk;
            bp = p;
          }
        }
      for (int o = tpe >> 1; o > 0; o >>= 1) {
        const unsigned long long ob = __shfl_xor_sync(FULL, best, o);
        const int op = __shfl_xor_sync(FULL, bp, o);
        if (ob < best || (ob == best && op < bp)) {
          best = ob;
          bp = op;
        }
      }
      if (q < G * G && sub == 0) {
        W[u * ld + v] = bp == INT_MAX ? INFINITY : okey_value(best);
        widx[q] = bp;
      }
    }
    __syncthreads();
    for (int u = tid; u < G; u += nt) {
      W[t * ld + u] = sz[u] > lo ? 0.0 : INFINITY;                        // u may shrink
      W[u * ld + t] = sz[u] < lo ? -big : (sz[u] < hi ? 0.0 : INFINITY);  // u may (must) grow
    }
    if (tid == 0) W[t * ld + t] = INFINITY;
    // disjoint negative 2-cycles between groups first, first fit in (u, v)
    // order: each swaps two points and leaves the sizes as they are; the
    // negative pairs of each row u are marked (bit v, v > u), then one thread
    // takes, for u ascending, the lowest v that is still free
    for (int q = tid; q < G * G; q += nt) {
      const int u = q / G, v = q - u * G;
      if (v > u && W[u * ld + v] + W[v * ld + u] < -eps) atomicOr(&negmask[u], 1u << v);
    }
    __syncthreads();
    if (tid == 0) {
      unsigned used = 0u;
      int m = 0;
      for (int u = 0; u < G; ++u) {
        if ((used >> u) & 1u) continue;
        const unsigned msk = negmask[u] & ~used;
        if (msk == 0u) continue;
        const int v = __ffs(msk) - 1;
        used |= (1u << u) | (1u << v);
        mv_pt[m] = widx[u * G + v], mv_to[m] = v, ++m;
        mv_pt[m] = widx[v * G + u], mv_to[m] = u, ++m;
      }
      *nmv = m;
      if (m == 0)
        for (int x = 0; x < n; ++x) {
          bf_dist[0][x] = 0.0;
          s_pred[x] = -1;
        }
    }
    __syncthreads();
    if (*nmv == 0) {
      // Bellman-Ford from a virtual source (0-weight edges to every node):
      // warp w relaxes nodes w, w + 8, ..., lane u offering dist[u] + W[u][v];
      // a node takes the smallest offer (ties: the lower u) only if it beats
      // its distance.  After each round warp 0 walks the predecessor graph: a
      // cycle there has negative weight (its sum is checked anyway).
      int cur = 0;
      for (int round = 0; round < 2 * (n + 1); ++round) {
        int changed = 0;
        for (int v = warp; v < n; v += nt / 32) {
          unsigned long long key = ~0ull;
          int from = lane;
          if (lane < n && lane != v) key = okey(bf_dist[cur][lane] + W[lane * ld + v]);
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
          // a walk of n steps along predecessors that never reaches the source
          // ends on a cycle
          int x = lane;
          bool alive = lane < n;
          for (int st = 0; st < n && alive; ++st) {
            const int nx = s_pred[x];
            if (nx < 0) alive = false;
            else x = nx;
          }
          const unsigned on = __ballot_sync(FULL, alive);
          const int start = __shfl_sync(FULL, x, on ? (__ffs(on) - 1) : 0);
          if (lane == 0 && on) {
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
        __syncthreads();
        if (*nmv != 0 || !changed) break;
      }
    }
    if (*nmv == 0) {
      done = 1;
      break;
    }
    if (tid == 0)
      for (int m = 0; m < *nmv; ++m) a[mv_pt[m]] = mv_to[m];
    __syncthreads();
    // the moved experts' gain keys, against their new groups
    for (int q = tid; q < *nmv * G; q += nt) {
      const int p = mv_pt[q / G], v = q - (q / G) * G;
      dk[p * DS + v] = okey(cost[p * G + v] - cost[p * G + a[p]]);
    }
  }
  if (tid == 0 && !done) atomicOr(status, WS_BIT_ETIMEOUT);
  __syncthreads();
}

__global__ void __launch_bounds__(SP_GROUP_THREADS, 6)
    spec_group_kernel(const int32_t* __restrict__ affinity, int E, int G, const double* __restrict__ Uo,
                      const double* __restrict__ deg, int32_t* __restrict__ groups, double* __restrict__ ucurve,
                      double* __restrict__ scurve, uint32_t* status) {
  extern __shared__ double gp_sm[];
  double* Us = gp_sm;                        // [E][G]
  double* C = Us + E * G;                    // [G][G]
  double* cost = C + G * G;                  // [E][G]
  double* mind = cost + E * G;               // [E]
  double* W = mind + E;                      // [G+1][G+1]
  unsigned long long* dk = reinterpret_cast<unsigned long long*>(W + (G + 1) * (G + 1));  // [E][G+1]
  int* a = reinterpret_cast<int*>(dk + E * (G + 1));  // [E]
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
    sp_assign(cost, E, G, lo, hi, a, prev, first, W, widx, sz, s_pred, mv_pt, mv_to, &s_nmv, dk, status);
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
    // S = sqrt(mean_g (size_g - E/G)^2) / (E/G) = sqrt(G sum_g size_g^2 - E^2) / E
    // (the sizes sum to E): an exact integer under the root
    long long s2 = 0;
    for (int g = 0; g < G; ++g) s2 += (long long)sz[g] * sz[g];
    const long long num = (long long)G * s2 - (long long)E * E;
    scurve[(size_t)l * SP_NGRID + j] = __dsqrt_rn((double)num) / (double)E;
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
  return ((size_t)E * G * 2 + (size_t)G * G + E + (size_t)(G + 1) * (G + 1) + (size_t)E * (G + 1)) *
             sizeof(double) +
         ((size_t)E * 2 + (size_t)G * G + G + 96) * sizeof(int);
}

struct SpLayout {
  size_t U, deg, groups, total;
};

static SpLayout sp_layout(int L, int E, int G) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  SpLayout o;
  o.U = WS_HEADER;
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
  double* U = reinterpret_cast<double*>(w + o.U);
  double* deg = reinterpret_cast<double*>(w + o.deg);
  int32_t* groups = reinterpret_cast<int32_t*>(w + o.groups);
  static std::atomic<unsigned long long> embed_set{0}, group_set{0};
  if (smem_optin(spec_embed_kernel, (int)spec_embed_smem(SP_MAXE, SP_MAXG), embed_set) != cudaSuccess ||
      smem_optin(spec_group_kernel, (int)spec_group_smem(SP_MAXE, SP_MAXG), group_set) != cudaSuccess)
    return MOER_ECUDA;
  spec_embed_kernel<<<L, SP_EMBED_THREADS, spec_embed_smem(E, G), st>>>(affinity, E, G, U, deg);
  spec_group_kernel<<<dim3(SP_NGRID, L), SP_GROUP_THREADS, spec_group_smem(E, G), st>>>(
      affinity, E, G, U, deg, groups, u_curve, s_curve, reinterpret_cast<uint32_t*>(ws));
  spec_knee_kernel<<<L, 32, 0, st>>>(groups, u_curve, E, group_of, knee);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

size_t spec_embed_smem(int E, int G) {
  return ((size_t)E * (E + 1) + 6 * (size_t)E + 64 + (size_t)G * E + 4 * (size_t)SP_LU_SLOTS * E) * sizeof(double) +
         (size_t)SP_LU_SLOTS * E * sizeof(int);
}

}  // namespace moer
