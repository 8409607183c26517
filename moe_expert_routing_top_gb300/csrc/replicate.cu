// replicate.cu -- moer_replication_plan: GRACE expert replication per layer.
//
// GRACE-MoE, section 4.2 (expert replication, load balance first) and section
// 4.3 (predicted load after replication, equation 3: W' = W - W_r + W_p).
// Each expert group sits on one GPU (G GPUs).  Per layer:
//   * the source is the most loaded group (ties: lower index); the replica
//     count is n = min(max(1, floor(rho)), G - 1) with rho = W_max / mean_g W_g,
//     floor(rho) taken exactly as floor(W_max * G / sum_g W_g); a layer with no
//     load, or G = 1, plans nothing;
//   * hot experts: the source group's experts in descending load (ties: lower
//     id), the shortest prefix whose cumulative load exceeds W_max n / (1 + n)
//     (compared exactly: cumulative * (1 + n) > W_max * n);
//   * the replicas go to the n least-loaded other groups (ties: lower index);
//   * predicted loads: the hot load H is split evenly over the original and
//     its n copies -- the source keeps W_max - H n / (1 + n), every replica
//     group gains H / (1 + n) (fp64: one division and one add or subtract of
//     exactly converted integers).
// One warp per layer: the lanes sum the group loads and initialise the output
// rows; lane 0 takes the decisions, which are sequential and tiny (E <= 256).
#include "common.cuh"

namespace moer {

constexpr int RP_MAXG = 64;

__global__ void __launch_bounds__(32) replication_plan_kernel(const int64_t* __restrict__ W,
                                                              const int32_t* __restrict__ group_of, int E, int G,
                                                              int32_t* __restrict__ n_rep, int32_t* __restrict__ src,
                                                              uint8_t* __restrict__ hot, int32_t* __restrict__ dst,
                                                              double* __restrict__ w_pred, uint32_t* status) {
  __shared__ unsigned long long wg[RP_MAXG];
  __shared__ int bad;
  const int l = blockIdx.x, lane = threadIdx.x;
  const int64_t* We = W + (size_t)l * E;
  const int32_t* ge = group_of + (size_t)l * E;
  if (lane == 0) bad = 0;
  for (int g = lane; g < G; g += 32) wg[g] = 0ull;
  __syncwarp();
  for (int e = lane; e < E; e += 32) {
    const int g = ge[e];
    const int64_t w = We[e];
    if (g < 0 || g >= G || w < 0) {
      bad = 1;
      continue;
    }
    atomicAdd(&wg[g], (unsigned long long)w);
  }
  for (int e = lane; e < E; e += 32) hot[(size_t)l * E + e] = 0;
  for (int g = lane; g < G; g += 32) {
    dst[(size_t)l * G + g] = -1;
    w_pred[(size_t)l * G + g] = (double)wg[g];
  }
  __syncwarp();
  if (lane != 0) return;
  int32_t n = 0, s = 0;
  if (bad) {
    atomicOr(status, WS_BIT_EDATA);
  } else {
    unsigned long long total = 0ull;
    for (int g = 0; g < G; ++g) {
      total += wg[g];
      if (wg[g] > wg[s]) s = g;
    }
    const unsigned long long wmax = wg[s];
    if (G >= 2 && wmax > 0ull) {
      const unsigned long long fr = wmax * (unsigned long long)G / total;
      n = (int32_t)(fr < 1ull ? 1ull : fr);
      if (n > G - 1) n = G - 1;
      // hot prefix of the source group in descending load (ties: lower id),
      // picked by repeated maximum over the members not taken yet
      unsigned long long acc = 0ull;
      int prev_e = -1;
      unsigned long long prev_w = 0ull;
      for (;;) {
        int best = -1;
        unsigned long long bw = 0ull;
        for (int e = 0; e < E; ++e) {
          if (ge[e] != s) continue;
          const unsigned long long w = (unsigned long long)We[e];
          // strictly after (prev_w, prev_e) in (descending load, ascending id) order
          const bool after = prev_e < 0 || w < prev_w || (w == prev_w && e > prev_e);
          if (!after) continue;
          if (best < 0 || w > bw) {
            best = e;
            bw = w;
          }
        }
        if (best < 0) break;
        hot[(size_t)l * E + best] = 1;
        acc += bw;
        prev_e = best;
        prev_w = bw;
        if (acc * (unsigned long long)(1 + n) > wmax * (unsigned long long)n) break;
      }
      const unsigned long long H = acc;
      // the n least-loaded other groups (ties: lower index)
      unsigned long long taken = 1ull << s;
      const double share = (double)H / (double)(1 + n);
      for (int r = 0; r < n; ++r) {
        int bg = -1;
        for (int g = 0; g < G; ++g) {
          if ((taken >> g) & 1ull) continue;
          if (bg < 0 || wg[g] < wg[bg]) bg = g;
        }
        taken |= 1ull << bg;
        dst[(size_t)l * G + r] = bg;
        w_pred[(size_t)l * G + bg] = (double)wg[bg] + share;
      }
      w_pred[(size_t)l * G + s] = (double)wmax - (double)(H * (unsigned long long)n) / (double)(1 + n);
    }
  }
  n_rep[l] = n;
  src[l] = s;
}

moer_status replication_plan_launch(const moer_dims* d, const int64_t* W, const int32_t* group_of, int32_t G,
                                    int32_t* n_rep, int32_t* src, uint8_t* hot, int32_t* dst, double* w_pred,
                                    uint32_t* status, cudaStream_t st) {
  replication_plan_kernel<<<d->L, 32, 0, st>>>(W, group_of, d->E, G, n_rep, src, hot, dst, w_pred, status);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
