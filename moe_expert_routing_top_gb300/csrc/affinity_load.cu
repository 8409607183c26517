// affinity_load.cu -- expert loads, group loads and load skew per layer.
//
// GRACE-MoE, section 4 "Method" (profiling yields load statistics), section
// 4.2 "Expert replication" (load skew rho = W_max / W_mean decides the
// replica count) and section 7 glossary ("load skew").  The load of expert e
// at layer l is the diagonal of the co-activation matrix (tokens whose top-k
// holds e); a group's load sums its experts' loads; the mean is taken over
// all G groups (E experts for the per-expert skew).
#include "common.cuh"
#include "pdl.cuh"

namespace moer {

__global__ void affinity_load_kernel(const int32_t* __restrict__ affinity, int E,
                                     const int32_t* __restrict__ group_of, int G,
                                     int64_t* __restrict__ W_expert, int64_t* __restrict__ W_group,
                                     double* __restrict__ rho_group, double* __restrict__ rho_expert) {
  extern __shared__ unsigned long long gsum[];  // [G]
  __shared__ unsigned long long red_sum[8], red_max[8];
  pdl_wait();
  const int l = blockIdx.x;
  for (int g = threadIdx.x; g < G; g += blockDim.x) gsum[g] = 0ull;
  __syncthreads();
  unsigned long long s = 0ull, mx = 0ull;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int32_t a = affinity[((size_t)l * E + e) * E + e];
    const unsigned long long w = a > 0 ? (unsigned long long)a : 0ull;
    if (W_expert) W_expert[(size_t)l * E + e] = (int64_t)w;
    s += w;
    mx = w > mx ? w : mx;
    const int g = group_of ? group_of[(size_t)l * E + e] : 0;
    if (g >= 0 && g < G) atomicAdd(&gsum[g], w);
  }
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(FULL, s, o);
    const unsigned long long t = __shfl_xor_sync(FULL, mx, o);
    mx = t > mx ? t : mx;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red_sum[warp] = s;
    red_max[warp] = mx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long S = 0ull, MX = 0ull;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      S += red_sum[w];
      MX = red_max[w] > MX ? red_max[w] : MX;
    }
    if (rho_expert) rho_expert[l] = S > 0ull ? (double)MX / ((double)S / (double)E) : 0.0;
    unsigned long long GS = 0ull, GM = 0ull;
    for (int g = 0; g < G; ++g) {
      GS += gsum[g];
      GM = gsum[g] > GM ? gsum[g] : GM;
    }
    if (rho_group) rho_group[l] = GS > 0ull ? (double)GM / ((double)GS / (double)G) : 0.0;
  }
  if (W_group)
    for (int g = threadIdx.x; g < G; g += blockDim.x) W_group[(size_t)l * G + g] = (int64_t)gsum[g];
  pdl_release();
}

moer_status affinity_load_launch(const moer_dims* d, const int32_t* affinity, const int32_t* group_of,
                                 int32_t G, int64_t* W_expert, int64_t* W_group, double* rho_group,
                                 double* rho_expert, cudaStream_t st) {
  const cudaError_t e = launch_pdl(affinity_load_kernel, dim3(d->L), dim3(256), (size_t)G * sizeof(unsigned long long),
                                   st, affinity, d->E, group_of, G, W_expert, W_group, rho_group, rho_expert);
  return e == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
