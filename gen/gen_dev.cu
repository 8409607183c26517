// gen_dev.cu -- device filler of the synthetic input generator (test and
// bench infrastructure, run outside every timed region).  Bit-identical to
// gen_host.c; the definitions live in ih12.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ih12.h"

namespace {

__global__ void logits_kernel(uint64_t ss, const int64_t* __restrict__ tok_key,
                              const int32_t* __restrict__ tok_dom, int64_t T,
                              int L, int E, const uint8_t* __restrict__ bias_mask,
                              int ndom, float bias, float* __restrict__ out) {
  const int64_t quads = (int64_t)L * T * (E / 4);
  const int eq = E / 4;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < quads;
       q += (int64_t)gridDim.x * blockDim.x) {
    int64_t row = q / eq;
    int e0 = (int)(q - row * eq) * 4;
    int l = (int)(row / T);
    int64_t t = row - (int64_t)l * T;
    int64_t key = tok_key[t];
    int dom = tok_dom ? tok_dom[t] : -1;
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = e0 + j;
      float x = gen_ih12(ss, gen_logit_ctr((uint64_t)key, (uint32_t)l, (uint32_t)e));
      if (bias_mask != nullptr && dom >= 0 && dom < ndom &&
          bias_mask[((size_t)dom * L + l) * E + e])
        x = __fadd_rn(x, bias);
      v[j] = x;
    }
    reinterpret_cast<float4*>(out)[q] = make_float4(v[0], v[1], v[2], v[3]);
  }
}

__global__ void hidden_kernel(uint64_t ss, int64_t T, int H, uint16_t* __restrict__ out) {
  const int64_t n = T * (int64_t)H;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = gen_bf16_rne(gen_ih12(ss, (uint64_t)i));
}

__global__ void wgate_kernel(uint64_t ss, int64_t n, float scale, uint16_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = gen_bf16_rne(__fmul_rn(gen_ih12(ss, (uint64_t)i), scale));
}

int grid_for(int64_t n) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t want = (n + 255) / 256;
  int64_t cap = (int64_t)sms * 16;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

extern "C" {

// Fills logits [L][T][E] (E a multiple of 4).  Returns a cudaError_t code.
int gen_dev_logits(uint64_t seed, const int64_t* tok_key, const int32_t* tok_dom,
                   int64_t T, int L, int E, const uint8_t* bias_mask, int ndom,
                   float bias, float* out, cudaStream_t stream) {
  if (E % 4 != 0 || T <= 0 || L <= 0) return (int)cudaErrorInvalidValue;
  int64_t quads = (int64_t)L * T * (E / 4);
  logits_kernel<<<grid_for(quads), 256, 0, stream>>>(
      gen_stream_seed(seed, GEN_STREAM_LOGITS), tok_key, tok_dom, T, L, E,
      bias_mask, ndom, bias, out);
  return (int)cudaGetLastError();
}

// Fills hidden states [T][H] as bf16 bits.
int gen_dev_hidden(uint64_t seed, int64_t T, int H, uint16_t* out, cudaStream_t stream) {
  int64_t n = T * (int64_t)H;
  hidden_kernel<<<grid_for(n), 256, 0, stream>>>(
      gen_stream_seed(seed, GEN_STREAM_HIDDEN), T, H, out);
  return (int)cudaGetLastError();
}

// Fills gate weights [L][H][E] as bf16 bits of scale * N(0,1).
int gen_dev_wgate(uint64_t seed, int L, int H, int E, float scale, uint16_t* out,
                  cudaStream_t stream) {
  int64_t n = (int64_t)L * H * E;
  wgate_kernel<<<grid_for(n), 256, 0, stream>>>(
      gen_stream_seed(seed, GEN_STREAM_WGATE), n, scale, out);
  return (int)cudaGetLastError();
}

}  // extern "C"
