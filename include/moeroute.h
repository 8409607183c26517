/*
 * moeroute.h -- C ABI of libmoeroute: MoE expert-routing statistics for
 * locality-aware serving, on one NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations:
 *   [ELDR]  "ELDR: Expert-Locality-Aware Decode Routing for PD-Disaggregated
 *           MoE Serving" (blog summary of arXiv 2607.00466).
 *   [GRACE] "GRACE-MoE: grouping, replication and locality-aware routing for
 *           distributed MoE inference" (research-notes summary).
 *
 * General conventions (every entry point):
 *   - All tensor pointers are DEVICE pointers to caller-owned memory unless a
 *     comment says "host".  The library allocates nothing and never frees.
 *   - Layouts are dense and row-major as stated per argument.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *     never synchronise the device, except moer_ws_status.
 *   - Argument errors detectable on the host return a non-zero status and
 *     launch nothing.  A failed launch returns MOER_ECUDA.
 *   - Malformed DEVICE data (a block table that does not tile the tokens, a
 *     cache slot out of range) is detected by the kernels, which then skip
 *     the offending work and record MOER_EDATA in the workspace's status
 *     word; moer_ws_status reports it.  No kernel traps.
 *   - Device waits are bounded; an expired wait records MOER_ETIMEOUT.
 *   - Checked mode (off by default; see moer_set_extent_checks): before
 *     launching, every entry point verifies that each buffer's device
 *     allocation can hold the bytes the call would touch, and returns
 *     MOER_EEXTENT otherwise.
 *   - Limits: 4 <= E <= 256 with E % 4 == 0; 1 <= k <= min(E, 32);
 *     1 <= L <= 256; 0 <= m <= L; 1 <= B <= 255; 1 <= D <= 64;
 *     T < 2^31 per call; every count fits in int32.
 */
#ifndef MOEROUTE_H
#define MOEROUTE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOER_API __attribute__((visibility("default")))
#else
#define MOER_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st* moer_stream_t;

typedef enum moer_status {
  MOER_OK = 0,
  MOER_EINVAL = 1,   /* NULL or misaligned pointer, bad enum/flag value      */
  MOER_ESHAPE = 2,   /* sizes inconsistent with each other                   */
  MOER_ERANGE = 3,   /* a size or parameter outside the library limits        */
  MOER_ECUDA = 4,    /* a CUDA runtime call or kernel launch failed           */
  MOER_ENOMEM = 5,   /* the workspace passed is smaller than required         */
  MOER_EDATA = 6,    /* device-side validation rejected input data            */
  MOER_ETIMEOUT = 7, /* a bounded device-side wait expired                    */
  MOER_EEXTENT = 8   /* checked mode: a buffer's allocation is too small      */
} moer_status;

/* Shape of the routing problem. */
typedef struct moer_dims {
  int32_t E;            /* experts per MoE layer                                    */
  int32_t k;            /* experts selected per token (top-k)                       */
  int32_t L;            /* MoE layers present in the logits tensor                  */
  int32_t m;            /* number of signature (mask) layers                        */
  const int32_t* mask;  /* HOST pointer: m strictly increasing layer ids in [0, L)  */
  int32_t block;        /* KV block size B in tokens                                */
} moer_dims;

/* Bytes of device workspace the calls below need for T computed tokens,
 * nblk KV blocks, R requests and D decoders (pass 0 for sizes a call does not
 * use).  One workspace may serve every call issued on one stream in order. */
MOER_API size_t moer_workspace_bytes(const moer_dims* d, int64_t T, int32_t nblk, int32_t R, int32_t D);

/* Top-k gating, per-KV-block signature counts and expert co-activation, in
 * one pass over the router logits.
 *   [ELDR] section "What it tries to solve" (each MoE token picks its own
 *   top-k experts) and section "Key idea / structure / operation" (the gate
 *   output is unchanged; the prefill hook records discrete top-k counts per
 *   KV block over the selected layer mask); [GRACE] section 3 "Key
 *   observations" and section 4 "Method", Figure 2(a) (per-layer expert
 *   co-activation profiling).
 *
 * logits    [L][T][E] fp32, 16-byte aligned.  Row (l, t) holds the router
 *           logits of computed token t at MoE layer l.
 * T         computed tokens in this call (0 is a no-op).
 * blk_tab   [nblk][2] int32 (tok0, len): the KV blocks of the computed
 *           tokens in order; they must tile [0, T) contiguously and have
 *           1 <= len <= B.  A block that breaks this (wrong length, gap or
 *           overlap with its predecessor, past T) is skipped -- its blk_cnt
 *           rows are left untouched -- and MOER_EDATA is recorded in ws; the
 *           top-k ids and co-activation counts are still produced.  May be
 *           NULL when blk_cnt is NULL.
 * topk      [L][T][k] uint8 or NULL, 8-byte aligned: expert ids in rank
 *           order.  Ranking: larger logit first; equal logits (-0.0 == +0.0)
 *           rank the lower expert id first; NaN ranks below every number.
 * blk_cnt   [nblk][m][E] uint8 or NULL: blk_cnt[b][i][e] = number of tokens
 *           of block b whose top-k at layer mask[i] contains e (<= B).
 * affinity  [L][E][E] int32 or NULL: ACCUMULATED (+=) co-activation counts,
 *           affinity[l][a][b] += #tokens whose top-k at layer l holds a and b
 *           (diagonal = expert load).  The caller zeroes it; streamed chunks
 *           sum.  4-byte aligned.
 * ws        device workspace of at least moer_workspace_bytes(d, T, nblk, 0, 0)
 *           bytes, 16-byte aligned (it holds the status word and, when topk
 *           is NULL, the mask layers' top-k ids).
 */
MOER_API moer_status moer_topk_signature(const moer_dims* d, const float* logits, int64_t T,
                                const int32_t* blk_tab, int32_t nblk, uint8_t* topk,
                                uint8_t* blk_cnt, int32_t* affinity, void* ws,
                                size_t ws_bytes, moer_stream_t stream);

/* moer_topk_signature for callers that cannot allocate device memory.
 *
 * No passage of the pages corresponds to this entry point; it exists for
 * the integration.  Some callers cannot call cudaMalloc: code running inside
 * another framework's memory pool or arena, plugins that must not grow the
 * process's device-memory footprint after start-up, and latency-critical
 * paths that must not allocate.  This call takes no workspace.  Its scratch
 * is one fixed array in device memory, compiled into the library: 256 bytes
 * of status plus MOER_NOALLOC_IDS_BYTES (32 MiB) for staging the mask
 * layers' top-k ids, so every GPU that loads the library holds about 32 MiB
 * until the process exits.
 *
 * Arguments and results are those of moer_topk_signature, without ws.
 * The caller still passes every input and output.
 *  - With topk == NULL and blk_cnt requested, m * T * k must not exceed
 *    MOER_NOALLOC_IDS_BYTES, else MOER_ENOMEM is returned and nothing is
 *    launched.  With a topk buffer the size limit does not apply.
 *  - The first call in a CUDA context looks up the array's device address
 *    (cudaGetSymbolAddress) with that context current, and keeps it for that
 *    context only; a context created later (after cudaDeviceReset, say)
 *    gets its own look-up.  Make the first call in each context before any
 *    stream capture.
 *  - Every call on a device shares the one array; each call clears the
 *    status part before use.  Calls whose kernels overlap on the GPU (for
 *    example on different streams without ordering) race on it.
 *  - The device-side statuses are not readable from the host: malformed
 *    block-table entries are skipped as in moer_topk_signature (MOER_EDATA
 *    there), and a bounded device wait that expires (MOER_ETIMEOUT there)
 *    leaves that part of the top-k ids, block counts or co-activation
 *    unwritten, both without a report.  Use moer_topk_signature with a
 *    workspace when those reports are needed.
 */
#define MOER_NOALLOC_IDS_BYTES (32u << 20)
MOER_API moer_status moer_topk_signature_noalloc(const moer_dims* d, const float* logits, int64_t T,
                                                 const int32_t* blk_tab, int32_t nblk, uint8_t* topk,
                                                 uint8_t* blk_cnt, int32_t* affinity,
                                                 moer_stream_t stream);

/* Prefix-cache stitching of per-block counts into per-request counts.
 *   [ELDR] table of what existing decode routing misses (signature cache),
 *   component table (signature cache) and section "Practical
 *   interpretation": a signature cache co-indexed with the KV cache keeps
 *   the full-prompt signature on prefix hits.
 * First every FULL computed block b (len == B) with insert_slot[b] >= 0 is
 * copied into cache[insert_slot[b]]; then
 *   req_cnt[r][i][e] = sum over c in [req_cache_off[r], req_cache_off[r+1])
 *                      of cache[cache_idx[c]][i][e]
 *                    + sum over b in [req_blk_off[r], req_blk_off[r+1])
 *                      of blk_cnt[b][i][e].
 * A request may therefore reuse blocks inserted in the same call by an
 * earlier request.  Partial blocks are never inserted.
 *
 * blk_cnt [nblk][m][E] uint8; blk_tab [nblk][2] (tok0, len) as above;
 * req_blk_off [R+1] int32; cache [nslots][m][E] uint8 (in/out) or NULL
 * together with cache_idx [ncached], req_cache_off [R+1] and
 * insert_slot [nblk] (all NULL, and ncached 0, when there is no cache;
 * cache_idx may be NULL when ncached is 0); req_cnt [R][m][E] int32
 * (overwritten).  Device data is checked as it is read: a request whose
 * block range is not within [0, nblk) or whose cached range
 * [req_cache_off[r], req_cache_off[r+1]) is not within [0, ncached) has
 * that part skipped, and a slot id outside [0, nslots) is skipped; each is
 * recorded as MOER_EDATA in ws (ws may be NULL: then they are skipped
 * silently).
 */
MOER_API moer_status moer_block_stitch(const moer_dims* d, const uint8_t* blk_cnt,
                              const int32_t* blk_tab, int32_t nblk,
                              const int32_t* req_blk_off, int32_t R,
                              const int32_t* cache_idx, int32_t ncached, const int32_t* req_cache_off,
                              uint8_t* cache, int32_t nslots, const int32_t* insert_slot,
                              int32_t* req_cnt, void* ws, size_t ws_bytes,
                              moer_stream_t stream);

/* Expert loads, group loads and load skew per MoE layer.
 *   [GRACE] section 4 "Method" (profiling yields the load statistics),
 *   section 4.2 "Expert replication" (the load skew rho = W_max / W_mean
 *   decides the replica count) and section 7 (glossary: load skew).  The
 *   load of expert e at layer l is the diagonal of the co-activation matrix
 *   (the tokens whose top-k holds e); a group's load sums its experts'
 *   loads; the mean runs over all G groups, empty ones included (over the E
 *   experts for the per-expert skew); a layer with no load has skew 0.
 * affinity  [L][E][E] int32, 4-byte aligned (moer_topk_signature's
 *           co-activation); only the diagonal is read.
 * group_of  [L][E] int32: the group of each expert, in [0, G); required
 *           when W_group or rho_group is asked for, else may be NULL.  An
 *           expert whose group id is outside [0, G) counts in no group.
 * G         1 <= G <= 4096 when group outputs are asked for.
 * W_expert  [L][E] int64 out or NULL: W[l][e] = affinity[l][e][e].
 * W_group   [L][G] int64 out or NULL: the sum of W over each group's experts.
 * rho_group [L] fp64 out or NULL: max_g W_group / mean_g W_group.
 * rho_expert [L] fp64 out or NULL: max_e W / mean_e W.
 * Caller-owned device buffers; nothing is accumulated (outputs are
 * overwritten).  Returns MOER_EINVAL for a NULL affinity (or a NULL
 * group_of when group outputs are asked for), MOER_ERANGE for G outside
 * its limits, MOER_ECUDA if the launch fails.
 */
MOER_API moer_status moer_affinity_load(const moer_dims* d, const int32_t* affinity,
                               const int32_t* group_of, int32_t G, int64_t* W_expert,
                               int64_t* W_group, double* rho_group, double* rho_expert,
                               moer_stream_t stream);

/* Signature, centroid distances and tau-band least-loaded decoder choice.
 *   [ELDR] section "Key idea / structure / operation": count * idf
 *   signature over the layer mask; comparison with D decoder centroids; the
 *   least-loaded decoder within the tau = 0.1 locality band of the nearest.
 * req_cnt [R][m][E] int32; idf [m][E] fp32; centroids [D][m*E] fp32.
 * sig   [R][m*E] fp32 or NULL: s = w / ||w||_2, w = req_cnt * idf (0 if w == 0).
 * dist  [R][D] fp32 or NULL: Euclidean ||s - c_d||_2.
 * choice [R] int32: d_min = min_d dist; band = {d : dist_d <= d_min + tau};
 *        the band member with the smallest load, ties to the lowest index.
 * loads [D] int32: live == 0: read only; live == 1: requests are routed in
 *        index order and each adds 1 to its decoder's load (updated in place).
 *        A request without any non-NaN distance gets choice -1 and changes no
 *        load.
 * ws    live == 1: at least moer_workspace_bytes(d, 0, 0, R, D) bytes, 16-byte
 *       aligned (each request's band as a decoder bit mask); live == 0: may
 *       be NULL.
 */
MOER_API moer_status moer_route(const moer_dims* d, const int32_t* req_cnt, int32_t R,
                       const float* idf, const float* centroids, int32_t D, float tau,
                       int32_t* loads, int32_t live, float* sig, float* dist,
                       int32_t* choice, void* ws, size_t ws_bytes, moer_stream_t stream);

/* Router (gate) GEMM with the top-k gate fused into its epilogue, on the
 * 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA operands).
 *   The router logits of every MoE layer, logit[l][t][e] = sum_h x[t][h] *
 *   W[l][h][e] with bf16 operands and fp32 accumulation, feed the standard
 *   top-k gate ([ELDR] section "What it tries to solve": each MoE token
 *   picks its own top-k experts; section "Key idea / structure / operation":
 *   the gate is unchanged), then the same per-KV-block counts and
 *   co-activation counts as moer_topk_signature.
 * Limits: E == 128, k in {6, 8}, H a multiple of 64 (64 .. 65536).
 * hidden  [T][H] bf16 bits (uint16), 16-byte aligned; one hidden state per
 *         computed token, shared by all L layers.
 * w_gate  [L][H][E] bf16 bits, 16-byte aligned.
 * logits  [L][T][E] fp32 or NULL: the fp32 logits (for inspection).
 * topk    [L][T][k] uint8, required, 8-byte aligned: ranking as in
 *         moer_topk_signature (on the fp32 accumulated logits).
 * blk_tab, blk_cnt, affinity: as in moer_topk_signature (blk_cnt and
 *         affinity may be NULL).
 * ws      at least moer_gate_workspace_bytes(d, H) bytes, 256-byte aligned
 *         (status word and the transposed gate weights).
 */
MOER_API size_t moer_gate_workspace_bytes(const moer_dims* d, int32_t H);
MOER_API moer_status moer_gate_topk(const moer_dims* d, const uint16_t* hidden, int64_t T, int32_t H,
                                    const uint16_t* w_gate, const int32_t* blk_tab, int32_t nblk,
                                    float* logits, uint8_t* topk, uint8_t* blk_cnt, int32_t* affinity,
                                    void* ws, size_t ws_bytes, moer_stream_t stream);

/* Per-KV-block signature counts and expert co-activation from top-k ids
 * computed elsewhere -- by the serving engine's own router, or by
 * moer_topk_signature / moer_gate_topk called without blk_cnt and affinity.
 *   [ELDR] section "Key idea / structure / operation": the gate is left
 *   unchanged and the prefill hook records, per KV block, the discrete
 *   top-k counts over the selected layer mask; [GRACE] section 3 and
 *   section 4, Figure 2(a): co-activation profiled from the selections.
 * topk      [L][T][k] uint8, 8-byte aligned: each row's k expert ids.
 * blk_tab, blk_cnt: as in moer_topk_signature (blk_cnt may be NULL).
 * affinity  [L][E][E] int32 or NULL, ACCUMULATED (+=) as in
 *           moer_topk_signature; requires E <= 128 and k in {6, 8}.
 * The ids are checked as they are read: an id >= E is not counted, and a
 * row holding an id >= E or a repeated id is left out of the
 * co-activation (its diagonal assumes k distinct ids); both are recorded
 * as MOER_EDATA in ws.  A repeated id below E is counted as given in
 * blk_cnt.
 * ws        at least 256 bytes, 16-byte aligned (the status word).
 */
MOER_API moer_status moer_ids_signature(const moer_dims* d, const uint8_t* topk, int64_t T,
                                        const int32_t* blk_tab, int32_t nblk, uint8_t* blk_cnt,
                                        int32_t* affinity, void* ws, size_t ws_bytes, moer_stream_t stream);

/* Expert grouping per MoE layer.  [GRACE-MoE] section 4.1: spectral
 * clustering of the co-activation matrix puts experts that are selected
 * together on the same GPU; the group sizes are held within
 * [E_bar - delta, E_bar + delta], delta = E_bar * r, with r at the knee of
 * the affinity utilisation U(r) (the size deviation S(r) beside it).  For G
 * groups, per layer, in fp64:
 *   M = D^-1/2 A D^-1/2 (A: co-activation off the diagonal, D: its row sums);
 *   embedding: eigenvectors of M's G largest eigenvalues, rows scaled to unit
 *   length; for r = j/16 (j = 0..16) group sizes in [max(1, floor(E(16-j)/16G)),
 *   min(E, ceil(E(16+j)/16G))]: K-means on the embedding under those bounds
 *   (seeds: largest degree, then farthest from the seeds so far; exact bounded
 *   assignment each step, centroids to the means, at most 100 steps);
 *   U(r) = affinity inside groups / affinity off the diagonal, S(r) = std of
 *   the sizes / (E/G); the knee of U over r (both scaled to [0, 1]: the point
 *   farthest above the chord from r = 0 to r = 1, ties to smaller r, r = 0
 *   when none is above) picks the groups.
 * affinity [L][E][E] int32 (moer_topk_signature's co-activation).
 * group_of [L][E] int32 out: the group of each expert (usable as the group
 *          map of moer_affinity_load and moer_replication_plan).
 * knee     [L] int32 out: j of the chosen r = j/16.
 * u_curve, s_curve [L][17] fp64 out: U and S at every grid point.
 * Limits: E <= 128, 2 <= G <= 31, G <= E.
 * ws       at least moer_spectral_workspace_bytes(d, G) bytes, 256-byte aligned
 *          (status word, eigenvectors, embedding, degrees, groups per grid
 *          point).  A bounded assignment that hits its pass bound records
 *          MOER_ETIMEOUT.
 */
MOER_API size_t moer_spectral_workspace_bytes(const moer_dims* d, int32_t G);
MOER_API moer_status moer_spectral_groups(const moer_dims* d, const int32_t* affinity, int32_t G,
                                          int32_t* group_of, int32_t* knee, double* u_curve, double* s_curve,
                                          void* ws, size_t ws_bytes, moer_stream_t stream);

/* Replication planning per MoE layer.  [GRACE-MoE] section 4.2 (expert
 * replication: only the hot experts of the most loaded group are copied, the
 * replica count follows the load skew) and section 4.3 (predicted load after
 * replication, W' = W - W_r + W_p).  Each of the G expert groups sits on one
 * GPU.  Per layer l:
 *   src[l]   the most loaded group (ties: lower index);
 *   n_rep[l] min(max(1, floor(W_max * G / sum_g W_g)), G - 1), or 0 when G = 1
 *            or the layer has no load;
 *   hot[l][e] 1 for the source group's experts, in descending load (ties:
 *            lower id), up to and including the one that takes the
 *            cumulative load past W_max * n / (1 + n) (exact integer test);
 *   dst[l][r] for r < n_rep: the n least-loaded other groups (ties: lower
 *            index), in that order; -1 beyond;
 *   w_pred[l][g] predicted load: the hot load H is split evenly over the
 *            original and its copies (source: W_max - H n / (1 + n), each
 *            replica group: W_g + H / (1 + n), fp64), other groups W_g.
 * W        [L][E] int64 expert loads (moer_affinity_load's W_expert), >= 0.
 * group_of [L][E] int32 group of each expert, in [0, G).
 * Limits: 1 <= G <= 64.  An entry out of range leaves its layer unplanned
 * (n_rep 0) and records MOER_EDATA in the workspace status word.
 * ws       at least 256 bytes, 256-byte aligned (the status word).
 */
MOER_API moer_status moer_replication_plan(const moer_dims* d, const int64_t* W, const int32_t* group_of,
                                           int32_t G, int32_t* n_rep, int32_t* src, uint8_t* hot,
                                           int32_t* dst, double* w_pred, void* ws, size_t ws_bytes,
                                           moer_stream_t stream);

/* Calibration (not on the per-request path): greedy choice of the signature's
 * layer mask.  [ELDR] section "Key idea / structure / operation": the
 * signature keeps only the MoE layers with the highest signature quality,
 * chosen greedily offline.  The pages do not print the quality objective; the
 * one here is a labelled proxy: each calibration request is split into its
 * first half (tokens [0, floor(len/2))) and its second half, and quality(M)
 * is the mean over the R requests of the cosine between the two halves'
 * count.idf signatures over the layers in M (0 if either is zero).  m times,
 * the layer outside M with the largest quality(M + {l}) is added (ties: the
 * lower layer).  Sums in fp64.
 * topk     [L][T][k] uint8 (moer_topk_signature's output over the calibration
 *          batch); d->E, d->k, d->L give its shape (d->mask is not used).
 * req_off  [R + 1] int32 token offsets of the requests (0 = req_off[0] <= ...
 *          <= req_off[R] = T); a malformed request or an id >= E is skipped
 *          and recorded as MOER_EDATA.
 * idf      [L][E] fp32 per-layer idf, or NULL for 1.
 * mask_out [m] int32: the layers in the order chosen (sort them for a mask).
 * quality_out [m] fp64 or NULL: quality after each addition.
 * Limits: 1 <= m <= L, R >= 1.
 * ws       at least moer_mask_select_workspace_bytes(d, R) bytes, 256-byte
 *          aligned (status word, per (request, layer) sums, running sums,
 *          per-step partial sums and a step counter, zeroed by the call).
 */
MOER_API size_t moer_mask_select_workspace_bytes(const moer_dims* d, int32_t R);
MOER_API moer_status moer_mask_select(const moer_dims* d, const uint8_t* topk, int64_t T, const int32_t* req_off,
                                      int32_t R, const float* idf, int32_t m, int32_t* mask_out,
                                      double* quality_out, void* ws, size_t ws_bytes, moer_stream_t stream);

/* Calibration (not on the per-request path): balanced K-means of N
 * calibration signatures into D decoder centroids.  [ELDR] section "Key idea
 * / structure / operation": offline, the calibration prompts' signatures are
 * split into D clusters, one per decode worker, by K-means with a balance
 * constraint solved by the Hungarian method, so that locality alone cannot
 * pile requests onto one decoder.
 *   Cluster d holds floor(N/D) points, plus one for d < N mod D.  Starting
 *   from init_centroids, each step assigns the points to clusters at the least
 *   total squared Euclidean distance under those sizes (exactly: a min-cost
 *   transportation problem, solved in fp64), then moves every centroid to the
 *   mean of its points (no renormalisation).  The fit stops after the first
 *   step whose assignment equals the previous one (no update follows it) or
 *   after max_iter steps.
 * Limits: 1 <= D <= 32, D <= N <= 2^20, 1 <= dim <= 65536, 1 <= max_iter <= 1000.
 * sig        [N][dim] fp32, device, finite (e.g. moer_route's signatures).
 * init_centroids [D][dim] fp32, device (the caller's seeding).
 * centroids  [D][dim] fp32 out (usable as moer_route's centroids).
 * assign     [N] int32 out: the cluster of each signature.
 * info       [3] int32 out or NULL: assignment steps run, negative cycles
 *            cancelled, 1 if a step stopped at its cancellation bound (then
 *            the status word also records MOER_ETIMEOUT).
 * objective  [1] fp64 out or NULL: sum of squared distances of the points to
 *            their returned centroids.
 * ws         at least moer_kmeans_workspace_bytes(N, dim, D) bytes, 256-byte
 *            aligned (status word, fp64 distances, centroids and their norm
 *            partials, previous assignment, member lists, gain keys).
 *            Launches 3 * max_iter + 3 kernels, chained by programmatic
 *            dependent launch on the caller's stream; steps after
 *            convergence return at once.
 */
MOER_API size_t moer_kmeans_workspace_bytes(int32_t N, int32_t dim, int32_t D);
MOER_API moer_status moer_kmeans_balanced(const float* sig, int32_t N, int32_t dim, int32_t D,
                                          const float* init_centroids, int32_t max_iter, float* centroids,
                                          int32_t* assign, int32_t* info, double* objective, void* ws,
                                          size_t ws_bytes, moer_stream_t stream);

/* Calibration helper (not on the per-request path): smoothed idf over R
 * calibration requests.  [ELDR] section "Key idea / structure / operation"
 * (idf reweighting fit offline on calibration prompts; formula not printed).
 * idf[i][e] = ln((1 + R) / (1 + df)) + 1, df = #{r : req_cnt[r][i][e] > 0},
 * evaluated in double and rounded to fp32.  req_cnt [R][m][E] int32.
 */
MOER_API moer_status moer_idf_fit(const moer_dims* d, const int32_t* req_cnt, int32_t R, float* idf,
                         moer_stream_t stream);

/* Waits for `stream`, then returns the status recorded in the workspace
 * (MOER_OK, MOER_EDATA or MOER_ETIMEOUT) and clears it.  `ws` is a device
 * workspace passed to earlier calls. */
MOER_API moer_status moer_ws_status(void* ws, moer_stream_t stream);

/* Diagnostic of the bounded device waits (no passage of the pages: it checks
 * the library's own failure reporting).  Launches one small kernel whose
 * mbarrier wait can never complete; the wait gives up after limit_us
 * microseconds, records MOER_ETIMEOUT in ws's status word (read it with
 * moer_ws_status) and writes 1 to ws's 32-bit word 2 (0 had the wait passed).
 * The kernel then ends normally; nothing faults.
 * ws        device workspace of at least 256 bytes, 16-byte aligned.
 * limit_us  1 .. 1,000,000.
 * Returns MOER_EINVAL / MOER_ENOMEM / MOER_ERANGE for bad arguments (nothing
 * launched), MOER_ECUDA if the launch fails, else MOER_OK. */
MOER_API moer_status moer_wait_selftest(void* ws, size_t ws_bytes, uint32_t limit_us, moer_stream_t stream);

/* Checked mode.  With `on` non-zero, every entry point first asks the CUDA
 * driver (cuMemGetAddressRange) for the allocation that holds each buffer it
 * is given and returns MOER_EEXTENT, launching nothing, when that allocation
 * does not contain [p, p + bytes) for the bytes the call would read or write
 * (the extents follow each argument's layout above; the workspace's extent is
 * ws_bytes), or when a pointer is not in any device allocation.  It turns a
 * buffer that is too small into an error instead of a memory fault.  The
 * check sees allocation ends only: a buffer carved from a larger allocation
 * (a framework's memory pool) can still overrun into its neighbour.  Cost:
 * one driver query per buffer per call.  Off by default; the environment
 * variable MOER_CHECK_EXTENTS=1 turns it on at the process's first call.
 * Process-wide; takes effect for calls made after it returns. */
MOER_API void moer_set_extent_checks(int32_t on);
/* 1 when checked mode is on, else 0. */
MOER_API int32_t moer_extent_checks(void);
/* The test checked mode applies, for one buffer: 1 when [p, p + bytes) lies
 * inside one device allocation (bytes 0 is taken as 1), else 0 (also for a
 * NULL or non-device pointer).  Host-side; launches nothing. */
MOER_API int32_t moer_buffer_holds(const void* p, size_t bytes);

/* Static description of a status code. */
MOER_API const char* moer_status_str(moer_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
MOER_API int32_t moer_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOEROUTE_H */
