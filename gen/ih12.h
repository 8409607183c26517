/*
 * ih12.h -- seeded, counter-based synthetic input generator (test and bench
 * infrastructure; holds none of the routing method's arithmetic).
 *
 * One definition, compiled twice: by gcc for the host twin (gen_host.c) and
 * by nvcc for the device filler (gen_dev.cu).  Every value is produced with
 * integer arithmetic followed by exactly-representable floating-point steps,
 * so the host and device outputs are bit-identical.
 *
 * Definitions
 *   mix64(z)     : the SplitMix64 output function (Steele, Lea & Flood,
 *                  "Fast splittable pseudorandom number generators",
 *                  OOPSLA 2014; constants as published by S. Vigna).
 *   draw(s, n)   : mix64(s + n * 0x9E3779B97F4A7C15), i.e. the n-th output of
 *                  a SplitMix64 stream seeded with s (counter-based access).
 *   ih12(s, c)   : "Irwin-Hall of 12": the twelve 16-bit fields of
 *                  draw(s,3c+1), draw(s,3c+2), draw(s,3c+3) are summed
 *                  (an integer in [0, 12*65535]); the result is
 *                  (sum - 6*65535) * 2^-16 as fp32.  Mean 0, variance
 *                  1 - 2^-32, support [-6, 6).  Both steps are exact in fp32
 *                  (|sum - 393210| < 2^19, scaling by a power of two).
 *   logit value  : ih12(seed, (key << 16) | (layer << 8) | e) + bias, where
 *                  the bias (0 or a constant such as 1.5) is added with one
 *                  round-to-nearest fp32 add.  key < 2^48, layer < 256,
 *                  e < 256.
 *   bf16_rne(x)  : fp32 -> bf16 round-to-nearest-even on the bit pattern
 *                  (inputs here are finite).
 */
#ifndef MOER_GEN_IH12_H
#define MOER_GEN_IH12_H

#include <stdint.h>

#if defined(__CUDACC__)
#define GEN_HD __host__ __device__ __forceinline__
#else
#define GEN_HD static inline
#endif

#define GEN_GOLDEN 0x9E3779B97F4A7C15ULL

/* Sub-stream tags: distinct tensors draw from distinct streams. */
#define GEN_STREAM_LOGITS 0x4C4F4749ULL /* "LOGI" */
#define GEN_STREAM_HIDDEN 0x48494444ULL /* "HIDD" */
#define GEN_STREAM_WGATE 0x57474154ULL  /* "WGAT" */

GEN_HD uint64_t gen_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

GEN_HD uint64_t gen_draw(uint64_t seed, uint64_t n) {
  return gen_mix64(seed + n * GEN_GOLDEN);
}

GEN_HD uint32_t gen_sum16x4(uint64_t w) {
  return (uint32_t)(w & 0xFFFFu) + (uint32_t)((w >> 16) & 0xFFFFu) +
         (uint32_t)((w >> 32) & 0xFFFFu) + (uint32_t)(w >> 48);
}

/* Stream seed for a tensor kind: mixes the user seed with the tag. */
GEN_HD uint64_t gen_stream_seed(uint64_t seed, uint64_t tag) {
  return gen_mix64(seed ^ (tag * GEN_GOLDEN));
}

GEN_HD float gen_ih12(uint64_t sseed, uint64_t ctr) {
  uint64_t n = ctr * 3ULL;
  uint32_t s = gen_sum16x4(gen_draw(sseed, n + 1)) +
               gen_sum16x4(gen_draw(sseed, n + 2)) +
               gen_sum16x4(gen_draw(sseed, n + 3));
  int32_t c = (int32_t)s - 393210; /* 6 * 65535 */
  return (float)c * (1.0f / 65536.0f);
}

GEN_HD uint64_t gen_logit_ctr(uint64_t key, uint32_t layer, uint32_t e) {
  return (key << 16) | ((uint64_t)layer << 8) | (uint64_t)e;
}

GEN_HD uint16_t gen_bf16_rne(float x) {
  union {
    float f;
    uint32_t u;
  } v;
  v.f = x;
  uint32_t lsb = (v.u >> 16) & 1u;
  return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

#endif /* MOER_GEN_IH12_H */
