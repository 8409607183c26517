/*
 * oracle.h -- plain, slow CPU oracle of the MoE expert-routing statistics
 * path.  TEST INFRASTRUCTURE ONLY: it is built and called by the tests, by
 * the package's smoke check and by the bench's CPU-baseline leg, never by the
 * library.  It shares no code, header or table with the CUDA path.
 *
 * Sources (cited per function in oracle.c):
 *   [ELDR]  "ELDR: Expert-Locality-Aware Decode Routing for PD-Disaggregated
 *           MoE Serving" (blog summary of arXiv 2607.00466).
 *   [GRACE] "GRACE-MoE: grouping, replication and locality-aware routing for
 *           distributed MoE inference" (research-notes summary, ICLR'26
 *           submission).
 *
 * Conventions: all pointers are host memory owned by the caller; floating
 * point results are computed in double precision; layouts are row-major:
 * logits [L][T][E], top-k ids [L][T][k], block counts [nblk][m][E],
 * request counts [R][m][E], affinity [L][E][E].
 *
 * Parity status: every function below is pinned by tests/test_oracle_pins.py
 * (brute force, closed forms, invariants, library special cases).
 */
#ifndef MOER_ORACLE_H
#define MOER_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* O1 top-k: out[row][0..k) = the k experts ranked first, in rank order. */
void orc_topk(const float* logits, int64_t rows, int E, int k, uint8_t* out);

/* Number of KV blocks of block size B over the CSR request offsets. */
int64_t orc_num_blocks(const int32_t* req_off, int R, int B);

/* O2 per-KV-block counts for the mask layers; blocks in (request, position) order. */
void orc_block_counts(const uint8_t* topk, int L, int64_t T, int k, int E,
                      const int32_t* req_off, int R, int B, const int32_t* mask,
                      int m, uint8_t* blk_cnt);

/* O3 stitch: request counts = cached prefix blocks + computed blocks; inserts
 * full computed blocks into the cache (cache is in/out, [nslots][m][E]). */
void orc_stitch(const uint8_t* blk_cnt, const int32_t* req_off, int R, int B,
                int m, int E, const int32_t* cache_idx,
                const int32_t* req_cache_off, uint8_t* cache,
                const int32_t* insert_slot, int32_t* req_cnt);

/* O4 signature of one request: s = w / ||w||_2, w = cnt * idf (dim m*E). */
void orc_signature(const int32_t* cnt, const float* idf, int m, int E, double* s);

/* O5 Euclidean distance of one signature to D centroids [D][dim]. */
void orc_distances(const double* s, const float* centroids, int D, int dim, double* d);

/* O4+O5 for R requests: sig [R][m*E], dist [R][D]. */
void orc_sig_dist(const int32_t* req_cnt, int R, const float* idf, int m, int E,
                  const float* centroids, int D, double* sig, double* dist);

/* O6 tau-band least-loaded routing; live != 0 applies load[choice] += 1
 * after each request.  loads_out may alias nothing; it receives the final loads. */
void orc_route(const double* dist, int R, int D, double tau,
               const int32_t* loads_in, int live, int32_t* choice,
               int32_t* loads_out);

/* O7 per-layer co-activation matrix A [L][E][E] (overwritten). */
void orc_affinity(const uint8_t* topk, int L, int64_t T, int k, int E, int64_t* A);

/* O8 loads W [L][E], group loads Wg [L][G], skew rho over groups and experts [L]. */
void orc_loads(const uint8_t* topk, int L, int64_t T, int k, int E,
               const int32_t* group_of, int G, int64_t* W, int64_t* Wg,
               double* rho_group, double* rho_expert);

/* O9 smoothed idf fit over R calibration requests: idf [m][E]. */
void orc_idf_fit(const int32_t* req_cnt, int R, int m, int E, double* idf);

/* O10 gate logits from bf16 bit patterns: out [L][T][E] = fp32(sum_h x*w)
 * with the sum in double; hidden [T][H], wgate [L][H][E]. */
void orc_gate_logits(const uint16_t* hidden, int64_t T, int H,
                     const uint16_t* wgate, int L, int E, float* out);

#ifdef __cplusplus
}
#endif

#endif /* MOER_ORACLE_H */
