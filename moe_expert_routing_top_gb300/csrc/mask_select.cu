// mask_select.cu -- moer_mask_select: greedy choice of the signature's layer mask.
//
// ELDR, section "Key idea / structure / operation": the signature keeps only
// the subset of MoE layers with the highest signature quality, chosen
// greedily on the calibration prompts.  The pages do not print the quality
// objective (the paper relates prefill signatures to decode-time expert reuse,
// which needs decode traces); the objective here is a labelled proxy: each
// calibration prompt is split into its first half (tokens [0, floor(len/2)))
// and its second half, and quality(M) is the mean over all requests of the
// cosine between the two halves' count.idf signatures restricted to the layers
// in M (0 when either is the zero vector).  Greedy: starting from the empty
// set, m times add the layer with the largest quality(M + {l}) (ties: the
// lower layer).
//
// Design: the cosine over a layer set only needs, per (request, layer), the
// three sums s11 = sum_e w1^2, s22 = sum_e w2^2, s12 = sum_e w1 w2 (w = count *
// idf): quality(M) = mean_r S12 / sqrt(S11 S22) with S = sum over l in M.
//   * mask_stats_kernel: one CTA per (request, layer); the two halves' ids go
//     into shared-memory histograms (at k = 8 one 8-byte load per token, four
//     in flight per thread), then the three sums in fp64.
//   * per greedy step, one mask_step_kernel: CTAs over (request slice,
//     candidate layer) evaluate the candidates (fp64 cosines of the running
//     sums plus the candidate's), and the last CTA to finish picks the layer
//     and adds its sums to the running sums.  The fp64 square roots and
//     divisions are spread over the SMs, a step is one launch, and the steps
//     are chained by programmatic dependent launch.
#include <algorithm>

#include "common.cuh"

namespace moer {

constexpr int MS_STATS_THREADS = 128;
constexpr int MS_UNROLL = 4;  // token loads in flight per thread
constexpr int MS_EVAL_THREADS = 256;
constexpr int MS_MAX_SLICES = 16;  // request slices per candidate layer in one greedy step

__global__ void __launch_bounds__(MS_STATS_THREADS) mask_stats_kernel(const uint8_t* __restrict__ topk, int64_t T,
                                                                      int k, int E, int L,
                                                                      const int32_t* __restrict__ req_off,
                                                                      const float* __restrict__ idf,
                                                                      double* __restrict__ stats, uint32_t* status) {
  __shared__ int c1[256], c2[256];
  const int r = blockIdx.x, l = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t t0 = req_off[r], t1 = req_off[r + 1];
  const int R = gridDim.x;
  double* out = stats + ((size_t)l * R + r) * 3;  // layer-major: the greedy's lanes read consecutive requests
  if (t0 < 0 || t1 < t0 || t1 > T) {
    if (tid == 0) {
      out[0] = out[1] = out[2] = 0.0;
      if (l == 0) atomicOr(status, WS_BIT_EDATA);
    }
    return;
  }
  for (int e = tid; e < E; e += MS_STATS_THREADS) c1[e] = c2[e] = 0;
  __syncthreads();
  const int64_t mid = t0 + (t1 - t0) / 2;
  const uint8_t* row = topk + (size_t)l * T * k;
  bool bad_id = false;
  if (k == 8 && (reinterpret_cast<uintptr_t>(row) & 7u) == 0) {
    // whole tokens: one 8-byte word of ids each, MS_UNROLL loads in flight per
    // thread; a lane starts its token's ranks at (lane & 7), so the lanes of
    // one add mostly hit different experts (ranks, not tokens, correlate)
    const uint2* tok_ids = reinterpret_cast<const uint2*>(row);
    const int rot = 8 * (lane & 3);
    const bool swap = (lane & 4) != 0;
    for (int64_t t = t0 + tid; t < t1; t += MS_STATS_THREADS * MS_UNROLL) {
      uint2 v[MS_UNROLL];
#pragma unroll
      for (int u = 0; u < MS_UNROLL; ++u) {
        const int64_t tu = t + (int64_t)u * MS_STATS_THREADS;
        v[u] = tu < t1 ? tok_ids[tu] : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < MS_UNROLL; ++u) {
        const int64_t tu = t + (int64_t)u * MS_STATS_THREADS;
        if (tu < t1) {
          int* c = tu < mid ? c1 : c2;
          const uint32_t a = swap ? v[u].y : v[u].x, b = swap ? v[u].x : v[u].y;
          const uint32_t lo = __funnelshift_r(a, b, rot), hi = __funnelshift_r(b, a, rot);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int e = (int)(((j < 4 ? lo : hi) >> (8 * (j & 3))) & 0xFFu);
            if (e < E)
              atomicAdd(&c[e], 1);
            else
              bad_id = true;
          }
        }
      }
    }
  } else {
    for (int64_t q = t0 * k + tid; q < t1 * k; q += MS_STATS_THREADS) {
      const int e = row[q];
      if (e < E)
        atomicAdd(q < mid * k ? &c1[e] : &c2[e], 1);
      else
        bad_id = true;
    }
  }
  if (bad_id) atomicOr(status, WS_BIT_EDATA);  // an id outside [0, E) is skipped and reported
  __syncthreads();
  // the three sums, by warp 0 alone: GB300 issues fp64 at about 16 cycles per
  // warp instruction per SM, and the grid has one CTA per (request, layer)
  if (warp != 0) return;
  if (idf == nullptr) {
    // unit weights: sums of integer products, exact in int64 (and in the
    // double they are converted to, being far below 2^53)
    long long a = 0, b = 0, c = 0;
    for (int e = lane; e < E; e += 32) {
      const long long x = c1[e], y = c2[e];
      a += x * x;
      b += y * y;
      c += x * y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(FULL, a, o);
      b += __shfl_xor_sync(FULL, b, o);
      c += __shfl_xor_sync(FULL, c, o);
    }
    if (lane == 0) {
      out[0] = (double)a;
      out[1] = (double)b;
      out[2] = (double)c;
    }
  } else {
    double a = 0.0, b = 0.0, c = 0.0;
    for (int e = lane; e < E; e += 32) {
      const double w = (double)idf[(size_t)l * E + e];
      const double w1 = c1[e] * w, w2 = c2[e] * w;
      a = fma(w1, w1, a);
      b = fma(w2, w2, b);
      c = fma(w1, w2, c);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(FULL, a, o);
      b += __shfl_xor_sync(FULL, b, o);
      c += __shfl_xor_sync(FULL, c, o);
    }
    if (lane == 0) {
      out[0] = a;
      out[1] = b;
      out[2] = c;
    }
  }
}

__device__ __forceinline__ double ms_cos(double s11, double s22, double s12) {
  return (s11 > 0.0 && s22 > 0.0) ? s12 / sqrt(s11 * s22) : 0.0;
}

// One greedy step.  CTA (s, l) evaluates candidate layer l over its slice of
// the requests: running sums of the chosen layers + the candidate's, fp64
// cosines, a block reduction to one partial sum.  The CTA that finishes last
// (a counter that every CTA bumps once, after publishing its partial: no CTA
// waits for another) sums each layer's partials in slice order, takes the best
// layer not chosen yet (ties: the lower layer; chosen layers read -inf),
// records it, adds its sums to every request's running sums and resets the
// counter for the next step.
__global__ void __launch_bounds__(MS_EVAL_THREADS) mask_step_kernel(const double* __restrict__ stats, int R, int L,
                                                                    double* run, unsigned char* taken,
                                                                    double* part, unsigned int* counter, int step,
                                                                    int32_t* __restrict__ mask_out,
                                                                    double* __restrict__ quality_out) {
  __shared__ double red[MS_EVAL_THREADS / 32];
  __shared__ int s_last;
  // the greedy steps are chained by programmatic dependent launch: wait for
  // the grid before this one (its pick and running sums are then visible),
  // then let the next step start launching
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int S = gridDim.x, s = blockIdx.x, l = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (R + S - 1) / S, r0 = s * per, r1 = min(R, r0 + per);
  double acc = 0.0;
  if (!taken[l]) {
    for (int r = r0 + tid; r < r1; r += MS_EVAL_THREADS) {
      const double* sv = stats + ((size_t)l * R + r) * 3;
      const double* u = run + (size_t)r * 3;
      acc += ms_cos(u[0] + sv[0], u[1] + sv[1], u[2] + sv[2]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL, acc, o);
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (tid == 0) {
    double sum = 0.0;
    for (int w = 0; w < MS_EVAL_THREADS / 32; ++w) sum += red[w];
    part[(size_t)l * S + s] = sum;
    __threadfence();
    s_last = atomicAdd(counter, 1u) == (unsigned)(S * L) - 1u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Each thread takes layers tid, tid + blockDim, ...; then an argmax over the
  // threads' (quality, layer) pairs, ties to the lower layer.
  __shared__ double s_q[MS_EVAL_THREADS / 32];
  __shared__ int s_c[MS_EVAL_THREADS / 32];
  __shared__ int s_best;
  double bq = -INFINITY;
  int bc = L;
  for (int c = tid; c < L; c += MS_EVAL_THREADS) {
    double q = -INFINITY;
    if (!taken[c]) {
      double sum = 0.0;
      for (int j = 0; j < S; ++j) sum += __ldcg(part + (size_t)c * S + j);
      q = sum / (double)R;
    }
    if (bc == L || q > bq) bq = q, bc = c;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double oq = __shfl_xor_sync(FULL, bq, o);
    const int oc = __shfl_xor_sync(FULL, bc, o);
    if (oc < L && (bc == L || oq > bq || (oq == bq && oc < bc))) bq = oq, bc = oc;
  }
  if (lane == 0) s_q[warp] = bq, s_c[warp] = bc;
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < MS_EVAL_THREADS / 32; ++w)
      if (s_c[w] < L && (bc == L || s_q[w] > bq || (s_q[w] == bq && s_c[w] < bc))) bq = s_q[w], bc = s_c[w];
    s_best = bc;
    taken[bc] = 1;
    mask_out[step] = bc;
    if (quality_out != nullptr) quality_out[step] = bq;
    *counter = 0u;
  }
  __syncthreads();
  const int best = s_best;
  for (int r = tid; r < R; r += MS_EVAL_THREADS) {
    const double* sv = stats + ((size_t)best * R + r) * 3;
    double* u = run + (size_t)r * 3;
    u[0] += sv[0];
    u[1] += sv[1];
    u[2] += sv[2];
  }
}

size_t mask_select_workspace_bytes(int32_t L, int32_t R) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  return WS_HEADER + r256((size_t)R * L * 3 * sizeof(double)) + r256((size_t)R * 3 * sizeof(double)) +
         r256((size_t)L * MS_MAX_SLICES * sizeof(double)) + r256((size_t)L) + 256;
}

moer_status mask_select_launch(const moer_dims* d, const uint8_t* topk, int64_t T, const int32_t* req_off, int32_t R,
                               const float* idf, int32_t m, int32_t* mask_out, double* quality_out, void* ws,
                               cudaStream_t st) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  char* w = static_cast<char*>(ws);
  double* stats = reinterpret_cast<double*>(w + WS_HEADER);
  double* run = reinterpret_cast<double*>(w + WS_HEADER + r256((size_t)R * d->L * 3 * sizeof(double)));
  double* part = reinterpret_cast<double*>(reinterpret_cast<char*>(run) + r256((size_t)R * 3 * sizeof(double)));
  unsigned char* taken = reinterpret_cast<unsigned char*>(part) + r256((size_t)d->L * MS_MAX_SLICES * sizeof(double));
  unsigned int* counter = reinterpret_cast<unsigned int*>(taken + r256((size_t)d->L));
  if (cudaMemsetAsync(run, 0, (size_t)R * 3 * sizeof(double), st) != cudaSuccess) return MOER_ECUDA;
  if (cudaMemsetAsync(taken, 0, r256((size_t)d->L) + sizeof(unsigned int), st) != cudaSuccess) return MOER_ECUDA;
  mask_stats_kernel<<<dim3((unsigned)R, (unsigned)d->L), MS_STATS_THREADS, 0, st>>>(
      topk, T, d->k, d->E, d->L, req_off, idf, stats, reinterpret_cast<uint32_t*>(ws));
  // Request slices per layer: about two CTAs per SM in all, at least one
  // request per thread.
  const int64_t want = std::max<int64_t>(1, 2 * (int64_t)device_sm_count() / d->L);
  const unsigned S = (unsigned)std::min<int64_t>(
      std::min<int64_t>(((int64_t)R + MS_EVAL_THREADS - 1) / MS_EVAL_THREADS, want), MS_MAX_SLICES);
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c_step = {};
  c_step.gridDim = dim3(std::max(1u, S), (unsigned)d->L);
  c_step.blockDim = dim3(MS_EVAL_THREADS);
  c_step.dynamicSmemBytes = 0;
  c_step.stream = st;
  c_step.attrs = pdl;
  c_step.numAttrs = 1;
  for (int step = 0; step < m; ++step)
    if (cudaLaunchKernelEx(&c_step, mask_step_kernel, (const double*)stats, R, d->L, run, taken, part, counter, step,
                           mask_out, quality_out) != cudaSuccess)
      return MOER_ECUDA;
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
