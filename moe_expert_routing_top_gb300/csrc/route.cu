// route.cu -- request signatures, decoder-centroid distances and tau-band
// least-loaded decoder selection; smoothed idf calibration.
//
// ELDR, section "Key idea / structure / operation": the signature is the
// discrete top-k count reweighted by idf over the selected layers; after
// prefill the router compares it with the D decoder centroids and, rather
// than always taking the nearest, sends the request to the least-loaded
// decoder among those within the tau = 0.1 locality band.  Component table:
// "locality-band routing" trades expert reuse against live load balance.
//
// Kernels:
//   route_sig_dist  one CTA per request: w = cnt * idf, ||w||_2, s = w / ||w||,
//                   d_q = ||s - c_q||_2 for all decoders (centroids stay
//                   L2-resident across requests); in static mode the same CTA
//                   also picks the decoder.
//   route_live      one CTA for the whole batch: requests are decided in
//                   arrival order by warp 0 while the other warps stage the
//                   next chunk of band masks into shared memory; each
//                   decision adds one to the chosen decoder's load.  The band
//                   does not depend on the loads, so route_sig_dist computes
//                   each request's band as a decoder bit mask in parallel and
//                   the sequential part only picks the least-loaded member.
//   idf_fit         per (mask layer, expert): df over the calibration
//                   requests and ln((1 + N) / (1 + df)) + 1.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "pdl.cuh"

namespace moer {

constexpr int ROUTE_THREADS = 256;
constexpr int ROUTE_DMAX = 64;

__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x < 32) {
    t = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(FULL, t, o);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  return red[0];
}

// The band of D <= 64 distances as a bit mask: d_min, then bit q set when
// d_q <= d_min + tau.  NaN distances are outside the band and take no part in
// d_min (fminf skips them); with no non-NaN distance the mask is 0.
__device__ __forceinline__ unsigned long long band_mask(const float* dist, int D, float tau) {
  float dmin = dist[0];
  for (int q = 1; q < D; ++q) dmin = fminf(dmin, dist[q]);
  const float thr = __fadd_rn(dmin, tau);
  unsigned long long m = 0ull;
  for (int q = 0; q < D; ++q)
    if (dist[q] <= thr) m |= 1ull << q;
  return m;
}

// The band member with the smallest load, ties to the lowest index; -1 for
// an empty band.  Sequential form used by the static path (one thread).
__device__ __forceinline__ int band_pick(unsigned long long m, const int32_t* loads) {
  int best = -1;
  while (m) {
    const int q = __ffsll((long long)m) - 1;
    m &= m - 1;
    if (best < 0 || loads[q] < loads[best]) best = q;
  }
  return best;
}

// pick = 1 (static): the CTA chooses the decoder; pick = 0 (live): it leaves
// the band mask in band[r] for route_live.
template <int DM>
__global__ void __launch_bounds__(ROUTE_THREADS) route_sig_dist(
    const int32_t* __restrict__ req_cnt, int dim, const float* __restrict__ idf,
    const float* __restrict__ centroids, int D, float tau, const int32_t* __restrict__ loads,
    int pick, float* __restrict__ sig, float* __restrict__ dist, int32_t* __restrict__ choice,
    unsigned long long* __restrict__ band) {
  __shared__ float red[32];
  __shared__ float part[ROUTE_THREADS / 32][DM];
  __shared__ float dsh[DM];
  pdl_wait();
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* cnt = req_cnt + (size_t)r * dim;
  float ss = 0.f;
  for (int j = threadIdx.x; j < dim; j += blockDim.x) {
    const float w = __fmul_rn((float)cnt[j], idf[j]);
    ss = __fmaf_rn(w, w, ss);
  }
  const float nrm = sqrtf(block_sum(ss, red));
  float acc[DM];
#pragma unroll
  for (int q = 0; q < DM; ++q) acc[q] = 0.f;
  for (int j = threadIdx.x; j < dim; j += blockDim.x) {
    const float w = __fmul_rn((float)cnt[j], idf[j]);
    const float s = nrm > 0.f ? __fdiv_rn(w, nrm) : 0.f;
    if (sig) sig[(size_t)r * dim + j] = s;
#pragma unroll
    for (int q = 0; q < DM; ++q)
      if (q < D) {
        const float diff = __fsub_rn(s, centroids[(size_t)q * dim + j]);
        acc[q] = __fmaf_rn(diff, diff, acc[q]);
      }
  }
#pragma unroll
  for (int q = 0; q < DM; ++q) {
    float v = acc[q];
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    if (lane == 0) part[warp][q] = v;
  }
  __syncthreads();
  if (threadIdx.x < D) {
    float t = 0.f;
    for (int w = 0; w < ROUTE_THREADS / 32; ++w) t += part[w][threadIdx.x];
    dsh[threadIdx.x] = sqrtf(t);
  }
  __syncthreads();
  if (threadIdx.x < D && dist) dist[(size_t)r * D + threadIdx.x] = dsh[threadIdx.x];
  if (threadIdx.x == 0) {
    const unsigned long long m = band_mask(dsh, D, tau);
    if (pick)
      choice[r] = band_pick(m, loads);
    else
      band[r] = m;
  }
  pdl_release();
}

// Sequential live routing over the requests' band masks.  Lane q of warp 0
// owns decoders q and q + 32; per request one warp minimum of the in-band
// loads and a ballot for the lowest decoder holding it.
constexpr int LIVE_BUF = 2048;  // band masks per staging buffer

template <bool WIDE>  // WIDE: D > 32, lanes also own decoders 32 .. 63
__global__ void __launch_bounds__(ROUTE_THREADS) route_live(const unsigned long long* __restrict__ band, int R,
                                                            int D, int32_t* __restrict__ loads,
                                                            int32_t* __restrict__ choice) {
  __shared__ unsigned long long buf[2][LIVE_BUF];
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int ld0 = 0, ld1 = 0;
  if (warp == 0) {
    ld0 = lane < D ? loads[lane] : INT_MAX;
    ld1 = WIDE && lane + 32 < D ? loads[lane + 32] : INT_MAX;
  }
  const int nch = (R + LIVE_BUF - 1) / LIVE_BUF;
  for (int i = threadIdx.x; i < min(R, LIVE_BUF); i += blockDim.x) buf[0][i] = band[i];
  __syncthreads();
  for (int c = 0; c < nch; ++c) {
    const int r0 = c * LIVE_BUF;
    const int nr = min(LIVE_BUF, R - r0);
    if (warp == 0) {
      const unsigned long long* b = buf[c & 1];
      for (int i = 0; i < nr; ++i) {
        const unsigned long long m = b[i];
        // bits only for decoders below D; an empty mask (no non-NaN distance)
        // leaves every lane out, so the choice is -1 and no load changes
        const bool in0 = (m >> lane) & 1ull;
        const bool in1 = WIDE && ((m >> (lane + 32)) & 1ull);
        const int lm = __reduce_min_sync(FULL, min(in0 ? ld0 : INT_MAX, in1 ? ld1 : INT_MAX));
        const unsigned b0 = __ballot_sync(FULL, in0 && ld0 == lm);
        const unsigned b1 = WIDE ? __ballot_sync(FULL, in1 && ld1 == lm) : 0u;
        const int q = b0 ? __ffs(b0) - 1 : (b1 ? 32 + __ffs(b1) - 1 : -1);
        if (lane == 0) choice[r0 + i] = q;
        if (q >= 0 && lane == (q & 31)) {
          if (q < 32)
            ld0 += 1;
          else
            ld1 += 1;
        }
      }
    } else if (c + 1 < nch) {
      const int n1 = min(LIVE_BUF, R - (r0 + LIVE_BUF));
      const unsigned long long* src = band + (size_t)(r0 + LIVE_BUF);
      unsigned long long* dstb = buf[(c + 1) & 1];
      for (int i = threadIdx.x - 32; i < n1; i += blockDim.x - 32) dstb[i] = src[i];
    }
    __syncthreads();
  }
  if (warp == 0) {
    if (lane < D) loads[lane] = ld0;
    if (WIDE && lane + 32 < D) loads[lane + 32] = ld1;
  }
  pdl_release();
}

__global__ void idf_fit_kernel(const int32_t* __restrict__ req_cnt, int R, int dim, float* __restrict__ idf) {
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < dim; j += gridDim.x * blockDim.x) {
    int df = 0;
    for (int r = 0; r < R; ++r) df += req_cnt[(size_t)r * dim + j] > 0;
    idf[j] = (float)(log((1.0 + (double)R) / (1.0 + (double)df)) + 1.0);
  }
}

size_t route_scratch_bytes(int32_t R) { return ((size_t)R * sizeof(unsigned long long) + 255) / 256 * 256; }

moer_status route_launch(const moer_dims* d, const int32_t* req_cnt, int32_t R, const float* idf,
                         const float* centroids, int32_t D, float tau, int32_t* loads, int32_t live,
                         float* sig, float* dist, int32_t* choice, void* ws, cudaStream_t st) {
  const int dim = d->m * d->E;
  unsigned long long* band =
      live ? reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + WS_HEADER) : nullptr;
  const int pick = live ? 0 : 1;
  cudaError_t e = D <= 16 ? launch_pdl(route_sig_dist<16>, dim3(R), dim3(ROUTE_THREADS), 0, st, req_cnt, dim, idf,
                                       centroids, D, tau, loads, pick, sig, dist, choice, band)
                          : launch_pdl(route_sig_dist<ROUTE_DMAX>, dim3(R), dim3(ROUTE_THREADS), 0, st, req_cnt,
                                       dim, idf, centroids, D, tau, loads, pick, sig, dist, choice, band);
  if (e != cudaSuccess) return MOER_ECUDA;
  if (live) {
    e = D <= 32 ? launch_pdl(route_live<false>, dim3(1), dim3(ROUTE_THREADS), 0, st, (const unsigned long long*)band,
                             R, D, loads, choice)
                : launch_pdl(route_live<true>, dim3(1), dim3(ROUTE_THREADS), 0, st, (const unsigned long long*)band,
                             R, D, loads, choice);
    if (e != cudaSuccess) return MOER_ECUDA;
  }
  return MOER_OK;
}

moer_status idf_fit_launch(const moer_dims* d, const int32_t* req_cnt, int32_t R, float* idf,
                           cudaStream_t st) {
  const int dim = d->m * d->E;
  const int blocks = (dim + 255) / 256;
  idf_fit_kernel<<<blocks, 256, 0, st>>>(req_cnt, R, dim, idf);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
