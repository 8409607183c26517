/*
 * oracle.c -- plain, slow CPU oracle (TEST INFRASTRUCTURE ONLY; see oracle.h).
 *
 * Each function writes out the plain definition of one quantity of the MoE
 * expert-routing statistics path, with no blocking, fusion or reordering.
 * Where the pages leave a step open, the reading taken is stated beside it.
 *
 * Mutation hooks: building with -DORACLE_MUTANT=n plants one deliberate
 * mistake (listed at each `#if ORACLE_MUTANT == n`).  The pin tests build
 * these mutants and check that the pins reject every one of them.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ------------------------------------------------------------------ O1 --
 * Top-k gating.  [ELDR] section "What it tries to solve": in an MoE layer
 * every token picks its own top-k experts; section "Key idea / structure /
 * operation": routing statistics observe the standard top-k gate, whose
 * output is left unchanged.  [GRACE] section 3 "Key observations": top-k
 * routing.
 * Reading (ties and special values): experts are ranked by logit, larger
 * first; equal logits (including -0.0 and +0.0) rank the lower expert index
 * first; NaN ranks below every number (NaNs among themselves by index).
 * The k experts ranked first are kept, in rank order.
 */
typedef struct {
  float v;
  int i;
} ranked;

static int rank_cmp(const void* pa, const void* pb) {
  const ranked* a = (const ranked*)pa;
  const ranked* b = (const ranked*)pb;
  int an = isnan(a->v) != 0, bn = isnan(b->v) != 0;
  if (an != bn) return an ? 1 : -1;
  if (!an) {
#if ORACLE_MUTANT == 1 /* mutant: smaller logits first */
    if (a->v < b->v) return -1;
    if (a->v > b->v) return 1;
#else
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
#endif
  }
#if ORACLE_MUTANT == 2 /* mutant: ties to the higher index */
  return (a->i > b->i) ? -1 : (a->i < b->i);
#else
  return (a->i < b->i) ? -1 : (a->i > b->i);
#endif
}

void orc_topk(const float* logits, int64_t rows, int E, int k, uint8_t* out) {
  ranked* buf = (ranked*)malloc(sizeof(ranked) * (size_t)E);
  for (int64_t r = 0; r < rows; ++r) {
    const float* x = logits + (size_t)r * (size_t)E;
    for (int e = 0; e < E; ++e) {
      buf[e].v = x[e];
      buf[e].i = e;
    }
    qsort(buf, (size_t)E, sizeof(ranked), rank_cmp);
    for (int j = 0; j < k; ++j) out[(size_t)r * (size_t)k + (size_t)j] = (uint8_t)buf[j].i;
  }
  free(buf);
}

/* ------------------------------------------------------------------ O2 --
 * Per-KV-block expert counts.  [ELDR] section "Key idea / structure /
 * operation": the prefill hook records the expert signature at KV-block
 * granularity; the signature is a discrete top-k count (how many prompt
 * tokens picked each expert), restricted to the selected layer mask.
 * Block j of request r covers its computed tokens [jB, min((j+1)B, n_r)),
 * relative to the request's first computed token.
 */
int64_t orc_num_blocks(const int32_t* req_off, int R, int B) {
  int64_t n = 0;
  for (int r = 0; r < R; ++r) {
    int64_t len = (int64_t)req_off[r + 1] - req_off[r];
    n += (len + B - 1) / B;
  }
  return n;
}

void orc_block_counts(const uint8_t* topk, int L, int64_t T, int k, int E,
                      const int32_t* req_off, int R, int B, const int32_t* mask,
                      int m, uint8_t* blk_cnt) {
  (void)L;
  int64_t b = 0;
  for (int r = 0; r < R; ++r) {
    int64_t start = req_off[r], end = req_off[r + 1];
    for (int64_t t0 = start; t0 < end; t0 += B, ++b) {
      int64_t t1 = t0 + B < end ? t0 + B : end;
      for (int i = 0; i < m; ++i) {
        uint8_t* c = blk_cnt + ((size_t)b * (size_t)m + (size_t)i) * (size_t)E;
        memset(c, 0, (size_t)E);
        int layer = mask[i];
#if ORACLE_MUTANT == 3 /* mutant: last token of the block dropped */
        int64_t tend = t1 - 1 > t0 ? t1 - 1 : t1;
#else
        int64_t tend = t1;
#endif
        for (int64_t t = t0; t < tend; ++t)
          for (int j = 0; j < k; ++j)
            c[topk[((size_t)layer * (size_t)T + (size_t)t) * (size_t)k + (size_t)j]] += 1;
      }
    }
  }
}

/* ------------------------------------------------------------------ O3 --
 * Prefix-cache stitching.  [ELDR] table "what existing decode routing
 * misses" (signature cache row), component table (signature cache) and
 * section "Practical interpretation": a signature cache co-indexed with the
 * KV cache stores each KV block's expert footprint, so that a prefix-cache
 * hit still yields the full-prompt signature.
 * Reading: the request count is the sum of the stored counts of its cached
 * prefix blocks and of its computed blocks; every full computed block is
 * stored in its cache slot (a partial last block is never stored, since only
 * full KV blocks are cacheable).  Requests are taken in order, so a request
 * may reuse blocks stored by an earlier one.
 */
void orc_stitch(const uint8_t* blk_cnt, const int32_t* req_off, int R, int B,
                int m, int E, const int32_t* cache_idx,
                const int32_t* req_cache_off, uint8_t* cache,
                const int32_t* insert_slot, int32_t* req_cnt) {
  const size_t rec = (size_t)m * (size_t)E;
  int64_t b = 0;
  for (int r = 0; r < R; ++r) {
    int32_t* acc = req_cnt + (size_t)r * rec;
    memset(acc, 0, rec * sizeof(int32_t));
    for (int32_t c = req_cache_off[r]; c < req_cache_off[r + 1]; ++c) {
      const uint8_t* src = cache + (size_t)cache_idx[c] * rec;
      for (size_t x = 0; x < rec; ++x) acc[x] += src[x];
    }
    int64_t start = req_off[r], end = req_off[r + 1];
    for (int64_t t0 = start; t0 < end; t0 += B, ++b) {
      const uint8_t* src = blk_cnt + (size_t)b * rec;
#if ORACLE_MUTANT == 4 /* mutant: computed blocks after the first are dropped */
      if (t0 == start)
#endif
        for (size_t x = 0; x < rec; ++x) acc[x] += src[x];
      int full = (end - t0) >= B;
      if (full && insert_slot != NULL && insert_slot[b] >= 0)
        memcpy(cache + (size_t)insert_slot[b] * rec, src, rec);
    }
  }
}

/* ------------------------------------------------------------------ O4 --
 * Expert signature.  [ELDR] section "Key idea / structure / operation": the
 * signature is the discrete top-k count reweighted by IDF ("count * idf"),
 * over the selected layers.  Reading: w[i*E+e] = cnt[i][e] * idf[i][e] over
 * the concatenated mask layers, then s = w / ||w||_2; a zero vector maps to
 * zero (the pages print no normalisation; the L2 reading is the one the
 * task statement gives).
 */
void orc_signature(const int32_t* cnt, const float* idf, int m, int E, double* s) {
  const int dim = m * E;
  double ss = 0.0;
  for (int j = 0; j < dim; ++j) {
    s[j] = (double)cnt[j] * (double)idf[j];
    ss += s[j] * s[j];
  }
  double nrm = sqrt(ss);
#if ORACLE_MUTANT == 5 /* mutant: no normalisation */
  nrm = 1.0;
#endif
  for (int j = 0; j < dim; ++j) s[j] = nrm > 0.0 ? s[j] / nrm : 0.0;
}

/* ------------------------------------------------------------------ O5 --
 * Centroid comparison.  [ELDR] section "Key idea / structure / operation":
 * after prefill the router compares the request signature with the decoder
 * centroids (fit by K-means).  Reading: Euclidean distance, the K-means
 * geometry; not squared.
 */
void orc_distances(const double* s, const float* centroids, int D, int dim, double* d) {
  for (int q = 0; q < D; ++q) {
    const float* c = centroids + (size_t)q * (size_t)dim;
    double acc = 0.0;
    for (int j = 0; j < dim; ++j) {
      double diff = s[j] - (double)c[j];
#if ORACLE_MUTANT == 6 /* mutant: sign error in the difference */
      diff = s[j] + (double)c[j];
#endif
      acc += diff * diff;
    }
    d[q] = sqrt(acc);
  }
}

void orc_sig_dist(const int32_t* req_cnt, int R, const float* idf, int m, int E,
                  const float* centroids, int D, double* sig, double* dist) {
  const int dim = m * E;
  for (int r = 0; r < R; ++r) {
    orc_signature(req_cnt + (size_t)r * (size_t)dim, idf, m, E, sig + (size_t)r * (size_t)dim);
    orc_distances(sig + (size_t)r * (size_t)dim, centroids, D, dim, dist + (size_t)r * (size_t)D);
  }
}

/* ------------------------------------------------------------------ O6 --
 * Locality-band routing.  [ELDR] section "Key idea / structure / operation"
 * and its component table ("locality-band routing"): rather than always the
 * nearest centroid, the router picks the least-loaded decoder among the
 * candidates inside the tau = 0.1 locality band.
 * Reading: d_min = min_d dist[d]; band = { d : dist[d] <= d_min + tau }
 * (additive band); choice = the band member with the smallest load, ties to
 * the lowest decoder index.  Live mode takes requests in arrival order and
 * adds one routed request to the chosen decoder's load after each decision.
 * The pages do not consider undefined distances; reading: a NaN distance is
 * outside the band and does not take part in d_min, and a request with no
 * finite distance gets no decoder (-1) and changes no load.
 */
void orc_route(const double* dist, int R, int D, double tau,
               const int32_t* loads_in, int live, int32_t* choice,
               int32_t* loads_out) {
  int32_t* load = (int32_t*)malloc(sizeof(int32_t) * (size_t)D);
  memcpy(load, loads_in, sizeof(int32_t) * (size_t)D);
  for (int r = 0; r < R; ++r) {
    const double* d = dist + (size_t)r * (size_t)D;
    /* NaN distances are outside the band and do not define d_min */
    double dmin = NAN;
    for (int q = 0; q < D; ++q)
      if (!isnan(d[q]) && (isnan(dmin) || d[q] < dmin)) dmin = d[q];
    int best = -1;
    for (int q = 0; q < D; ++q) {
#if ORACLE_MUTANT == 7 /* mutant: band test dropped (pure least-loaded) */
      int in_band = 1;
#else
      int in_band = d[q] <= dmin + tau;
#endif
      if (!in_band) continue;
      if (best < 0 || load[q] < load[best]) best = q;
    }
    choice[r] = best;
    /* no finite distance: the band is empty, no decoder is chosen */
    if (live && best >= 0) load[best] += 1;
  }
  if (loads_out) memcpy(loads_out, load, sizeof(int32_t) * (size_t)D);
  free(load);
}

/* ------------------------------------------------------------------ O7 --
 * Expert affinity.  [GRACE] section 3 "Key observations" (experts are
 * co-activated under top-k routing), section 4 "Method" and Figure 2(a)
 * (profiling expert selections per layer builds the affinity matrix) and
 * section 7 glossary ("expert affinity / co-activation").
 * Reading: A_l[a][b] = number of tokens whose top-k set at layer l contains
 * both a and b (a == b included, so the diagonal is the expert's load),
 * over the tokens routed in this call.
 */
void orc_affinity(const uint8_t* topk, int L, int64_t T, int k, int E, int64_t* A) {
  memset(A, 0, sizeof(int64_t) * (size_t)L * (size_t)E * (size_t)E);
  for (int l = 0; l < L; ++l)
    for (int64_t t = 0; t < T; ++t) {
      const uint8_t* s = topk + ((size_t)l * (size_t)T + (size_t)t) * (size_t)k;
      for (int a = 0; a < k; ++a)
        for (int b = 0; b < k; ++b) {
#if ORACLE_MUTANT == 8 /* mutant: transposed update below the diagonal only */
          if (s[a] < s[b]) continue;
#endif
          A[((size_t)l * (size_t)E + s[a]) * (size_t)E + s[b]] += 1;
        }
    }
}

/* ------------------------------------------------------------------ O8 --
 * Load statistics and skew.  [GRACE] section 4 "Method" (profiling yields
 * load statistics), section 4.2 "Expert replication" (load skew
 * rho = W_max / W_mean drives the replica count) and section 7 glossary
 * ("load skew (rho): maximum load / mean load").
 * Reading: the load unit is one (token, expert) selection; W_l[e] counts
 * tokens whose top-k set at layer l contains e; a group's load sums its
 * experts' loads; rho_l = max_g W_l,g / ((1/G) sum_g W_l,g), the mean taken
 * over all G groups including empty ones; rho = 0 for a layer with no load.
 * The per-expert skew applies the same formula over the E experts.
 */
void orc_loads(const uint8_t* topk, int L, int64_t T, int k, int E,
               const int32_t* group_of, int G, int64_t* W, int64_t* Wg,
               double* rho_group, double* rho_expert) {
  memset(W, 0, sizeof(int64_t) * (size_t)L * (size_t)E);
  memset(Wg, 0, sizeof(int64_t) * (size_t)L * (size_t)G);
  for (int l = 0; l < L; ++l)
    for (int64_t t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        W[(size_t)l * (size_t)E + topk[((size_t)l * (size_t)T + (size_t)t) * (size_t)k + (size_t)j]] += 1;
  for (int l = 0; l < L; ++l) {
    for (int e = 0; e < E; ++e) {
      /* W_{l,g} sums the experts whose group is g; an id outside [0, G) names no group */
      const int g = group_of[(size_t)l * (size_t)E + (size_t)e];
      if (g >= 0 && g < G) Wg[(size_t)l * (size_t)G + (size_t)g] += W[(size_t)l * (size_t)E + (size_t)e];
    }
    double sum = 0.0, mx = 0.0;
    for (int g = 0; g < G; ++g) {
      double w = (double)Wg[(size_t)l * (size_t)G + (size_t)g];
      sum += w;
      if (w > mx) mx = w;
    }
#if ORACLE_MUTANT == 9 /* mutant: mean over non-empty groups only */
    int ne = 0;
    for (int g = 0; g < G; ++g) ne += Wg[(size_t)l * (size_t)G + (size_t)g] > 0;
    rho_group[l] = sum > 0.0 ? mx / (sum / (double)ne) : 0.0;
#else
    rho_group[l] = sum > 0.0 ? mx / (sum / (double)G) : 0.0;
#endif
    sum = 0.0;
    mx = 0.0;
    for (int e = 0; e < E; ++e) {
      double w = (double)W[(size_t)l * (size_t)E + (size_t)e];
      sum += w;
      if (w > mx) mx = w;
    }
    rho_expert[l] = sum > 0.0 ? mx / (sum / (double)E) : 0.0;
  }
}

/* ------------------------------------------------------------------ O9 --
 * IDF weights.  [ELDR] section "Key idea / structure / operation": the
 * signature is reweighted by IDF, fit offline on 1,000 calibration prompts.
 * The formula is not printed.  Reading: each request is a document and each
 * (mask layer, expert) a term; df = number of calibration requests whose
 * count for the term is non-zero; smoothed idf = ln((1 + N) / (1 + df)) + 1.
 */
void orc_idf_fit(const int32_t* req_cnt, int R, int m, int E, double* idf) {
  const int dim = m * E;
  for (int j = 0; j < dim; ++j) {
    int64_t df = 0;
    for (int r = 0; r < R; ++r) df += req_cnt[(size_t)r * (size_t)dim + (size_t)j] > 0;
#if ORACLE_MUTANT == 10 /* mutant: smoothing term dropped from the numerator */
    idf[j] = log((double)R / (1.0 + (double)df)) + 1.0;
#else
    idf[j] = log((1.0 + (double)R) / (1.0 + (double)df)) + 1.0;
#endif
  }
}

/* ----------------------------------------------------------------- O10 --
 * Gate logits.  The router output of each MoE layer is the hidden state
 * times the layer's gate matrix ([ELDR] section "What it tries to solve":
 * the MoE gate scores every token; the gate itself is unchanged).
 * Definition: logit[l][t][e] = sum_h x[t][h] * W[l][h][e], bf16 operands,
 * summed in double and rounded once to fp32.
 */
static double bf16_to_double(uint16_t b) {
  union {
    uint32_t u;
    float f;
  } v;
  v.u = (uint32_t)b << 16;
  return (double)v.f;
}

void orc_gate_logits(const uint16_t* hidden, int64_t T, int H,
                     const uint16_t* wgate, int L, int E, float* out) {
  for (int l = 0; l < L; ++l)
    for (int64_t t = 0; t < T; ++t)
      for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h)
          acc += bf16_to_double(hidden[(size_t)t * (size_t)H + (size_t)h]) *
                 bf16_to_double(wgate[((size_t)l * (size_t)H + (size_t)h) * (size_t)E + (size_t)e]);
        out[((size_t)l * (size_t)T + (size_t)t) * (size_t)E + (size_t)e] = (float)acc;
      }
}
