/*
 * gen_host.c -- host twin of the synthetic input generator (test and bench
 * infrastructure).  Produces exactly the bits gen_dev.cu produces on the GPU.
 * The generator definitions live in ih12.h.
 */
#include <stddef.h>
#include <stdint.h>

#include "ih12.h"

static float logit_value(uint64_t sseed, int64_t key, int32_t dom, int layer,
                         int e, int L, int E, const uint8_t* bias_mask,
                         int ndom, float bias) {
  float v = gen_ih12(sseed, gen_logit_ctr((uint64_t)key, (uint32_t)layer,
                                           (uint32_t)e));
  if (bias_mask != NULL && dom >= 0 && dom < ndom &&
      bias_mask[((size_t)dom * (size_t)L + (size_t)layer) * (size_t)E + (size_t)e])
    v = v + bias;
  return v;
}

/* Full logits tensor, layout [L][T][E]. */
void gen_host_logits(uint64_t seed, const int64_t* tok_key,
                     const int32_t* tok_dom, int64_t T, int L, int E,
                     const uint8_t* bias_mask, int ndom, float bias,
                     float* out) {
  uint64_t ss = gen_stream_seed(seed, GEN_STREAM_LOGITS);
  for (int l = 0; l < L; ++l)
    for (int64_t t = 0; t < T; ++t)
      for (int e = 0; e < E; ++e)
        out[((size_t)l * (size_t)T + (size_t)t) * (size_t)E + (size_t)e] =
            logit_value(ss, tok_key[t], tok_dom ? tok_dom[t] : -1, l, e, L, E,
                        bias_mask, ndom, bias);
}

/* Selected rows: row n is (layers[n], toks[n]); out is [n][E]. */
void gen_host_logit_rows(uint64_t seed, const int64_t* tok_key,
                         const int32_t* tok_dom, const int32_t* layers,
                         const int64_t* toks, int64_t n, int L, int E,
                         const uint8_t* bias_mask, int ndom, float bias,
                         float* out) {
  uint64_t ss = gen_stream_seed(seed, GEN_STREAM_LOGITS);
  for (int64_t r = 0; r < n; ++r) {
    int64_t t = toks[r];
    for (int e = 0; e < E; ++e)
      out[(size_t)r * (size_t)E + (size_t)e] =
          logit_value(ss, tok_key[t], tok_dom ? tok_dom[t] : -1, layers[r], e,
                      L, E, bias_mask, ndom, bias);
  }
}

/* Logits of explicit (key, dom) tokens, out is [L][n][E]. */
void gen_host_logits_keys(uint64_t seed, const int64_t* keys,
                          const int32_t* doms, int64_t n, int L, int E,
                          const uint8_t* bias_mask, int ndom, float bias,
                          float* out) {
  gen_host_logits(seed, keys, doms, n, L, E, bias_mask, ndom, bias, out);
}

/* Hidden states, bf16 bits, rows [t0, t0 + nt) of a [T][H] tensor. */
void gen_host_hidden(uint64_t seed, int64_t t0, int64_t nt, int H,
                     uint16_t* out) {
  uint64_t ss = gen_stream_seed(seed, GEN_STREAM_HIDDEN);
  for (int64_t t = 0; t < nt; ++t)
    for (int h = 0; h < H; ++h)
      out[(size_t)t * (size_t)H + (size_t)h] = gen_bf16_rne(
          gen_ih12(ss, (uint64_t)(t0 + t) * (uint64_t)H + (uint64_t)h));
}

/* Gate weights, bf16 bits, layout [L][H][E]: bf16(scale * ih12). */
void gen_host_wgate(uint64_t seed, int L, int H, int E, float scale,
                    uint16_t* out) {
  uint64_t ss = gen_stream_seed(seed, GEN_STREAM_WGATE);
  size_t n = (size_t)L * (size_t)H * (size_t)E;
  for (size_t i = 0; i < n; ++i) {
    float v = gen_ih12(ss, (uint64_t)i) * scale;
    out[i] = gen_bf16_rne(v);
  }
}
