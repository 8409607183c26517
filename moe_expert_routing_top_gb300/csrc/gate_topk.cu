// gate_topk.cu -- moer_gate_topk: the MoE gate (router) GEMM on the 5th-gen
// tensor cores, with the top-k selection fused into its epilogue.
//
// What it computes: the router logits of every MoE layer, logit[l][t][e] =
// sum_h x[t][h] * W[l][h][e] (bf16 operands, fp32 accumulation), followed by
// the standard top-k gate over each (token, layer) row -- the input of the
// routing statistics of ELDR (section "What it tries to solve": every MoE
// token picks its own top-k experts; section "Key idea / structure /
// operation": the gate itself is left unchanged).
//
// Design (GB300, sm_103a):
//   * The weights are transposed once per call into the workspace,
//     Wt[l*128 + e][h], so both operands are K-major.
//   * Clusters of two CTAs on the two SMs of a TPC, persistent over tiles of
//     256 tokens x 2 layers (UMMA M = 256, N = 256 experts) computed with
//     tcgen05.mma.cta_group::2, K = H in blocks of 64.  Each CTA loads its
//     own 128 tokens and one layer's 128 weight rows per K block (32 KB, six
//     stages, 128-byte swizzled TMA) and receives its 128 tokens x 256
//     columns in TMEM.  Tiles, token block major, are handed out in order
//     from a global counter, so the grid works on a few token blocks at a
//     time: each hidden-state panel is read from HBM once and shared through
//     L2; the 25 MB of weights stay in L2.
//   * Per CTA: warp 0 loads (in the leader, rank 0, it also takes the tile
//     ids and posts both CTAs' transaction bytes); warp 1 allocates two
//     256-column fp32 accumulators (both CTAs, collectively) and, in the
//     leader, one elected thread issues the MMAs and multicasts its commits
//     to both CTAs; warps 2-5 drain an accumulator with tcgen05.ld while the
//     next tile's MMAs run: each thread owns one token row (one TMEM lane)
//     and selects its top-k per layer with comparator networks on truncated
//     keys (rank.cuh), certified, else redone exactly.
//   * Every wait is bounded; on expiry the kernel records MOER_ETIMEOUT,
//     waits for its copies in flight and frees its TMEM before returning.
#include <cuda.h>
#include <climits>
#include <mutex>

#include "common.cuh"
#include "rank.cuh"

namespace moer {

struct GateParams {
  CUtensorMap tmx;  // hidden [T][H] bf16, box 64 x 128, 128B swizzle
  CUtensorMap tmw;  // Wt [L*128][H] bf16, box 64 x 128, 128B swizzle
  int64_t T;
  int H, L, k;
  int npairs;       // ceil(L / 2)
  int64_t ntiles;   // ceil(T / 256) * npairs
  float* logits;    // [L][T][128] or nullptr
  uint8_t* topk;    // [L][T][k]
  uint32_t* status;
  uint32_t* tile_ctr;  // next tile to hand out (zeroed before the launch)
};

// ------------------------------------------------------------ PTX helpers
// UMMA shared-memory descriptor: K-major operand tile with 128-byte swizzle
// (rows of 128 bytes, 8-row groups 1024 bytes apart), sm_100 descriptor version.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024u >> 4) << 32;         // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Truncated keys of the epilogue: E = 128 experts need 7 index bits.
constexpr int GK_IDX_BITS = 7;
constexpr int GK_IDX_MAX = (1 << GK_IDX_BITS) - 1;
constexpr int GK_VAL_MASK = (int)~((1u << GK_IDX_BITS) - 1u);

// Folds 32 logits (expert ids e0 .. e0+31) into the running top-8 keys T
// (and, if WANT9, the 9th key L9), with truncated keys (rank.cuh).
template <bool FIRST, bool WANT9>
__device__ __forceinline__ void fold32(const uint32_t (&r)[32], int e0, int (&T)[8], int& L9) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    int c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = trunc_key<GK_IDX_BITS>(r[8 * g + j], GK_IDX_MAX - (e0 + 8 * g + j));
    sort8_desc(c);
    if (FIRST && g == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) T[i] = c[i];
    } else {
      merge8<WANT9>(T, c, L9);
    }
  }
}

// Top-k ids of one row (K of them, rank order) into its output slot.
template <int K>
__device__ __forceinline__ void gate_store_ids(uint8_t* o, const int (&idx)[8]) {
  if constexpr (K == 8) {
    const uint32_t lo = (uint32_t)idx[0] | ((uint32_t)idx[1] << 8) | ((uint32_t)idx[2] << 16) | ((uint32_t)idx[3] << 24);
    const uint32_t hi = (uint32_t)idx[4] | ((uint32_t)idx[5] << 8) | ((uint32_t)idx[6] << 16) | ((uint32_t)idx[7] << 24);
    *reinterpret_cast<uint2*>(o) = make_uint2(lo, hi);
  } else {
#pragma unroll
    for (int i = 0; i < K; i += 2) *reinterpret_cast<uint16_t*>(o + i) = (uint16_t)(idx[i] | (idx[i + 1] << 8));
  }
}

__device__ __forceinline__ void store_logits32(float* lrow, const uint32_t (&r)[32]) {
#pragma unroll
  for (int c = 0; c < 32; c += 4)
    *reinterpret_cast<float4*>(lrow + c) =
        make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]), __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
}

// Exact top-8 of one layer's 128 logits (TMEM columns tbase ..), for rows the
// truncated keys could not certify: 40-bit keys inserted into a sorted list.
// Only lanes with `bad` take part and take its result.  With `thr` > 127
// (the row's k-th truncated key is a positive finite float) only values
// whose truncated key reaches thr can be in the exact top-k -- truncation is
// monotone on positive floats, so the k-th largest value truncates to
// exactly thr -- and only those few are inserted; with thr <= 127 (zeros,
// negatives, infinities or NaN near the top) every value is.  Warp-collective
// (tcgen05.ld).
__device__ __forceinline__ void gate_exact_row(uint32_t tbase, bool bad, int thr, int (&idx)[8]) {
  uint64_t X[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) X[i] = 0;
  const int lo = thr > GK_IDX_MAX ? thr : INT_MIN;
#pragma unroll 1
  for (int cb = 0; cb < 4; ++cb) {
    uint32_t r[32];
    tmem_ld32(tbase + (uint32_t)(cb * 32), r);
    tmem_ld_wait();
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      if (bad && trunc_key<GK_IDX_BITS>(r[jj], 0) >= lo) {
        uint64_t x = rank_key40(r[jj], cb * 32 + jj);
#pragma unroll
        for (int i = 0; i < 8; ++i) cas64(X[i], x);
      }
    }
  }
  if (bad) {
#pragma unroll
    for (int i = 0; i < 8; ++i) idx[i] = 255 - (int)(X[i] & 0xFF);
  }
}

// Drains one layer of an accumulator: this thread's token row `tok`, 128
// logits of layer `layer` in TMEM columns tbase .. tbase + 127 of the warp's
// lane quarter.  Stores the logits if asked, selects the row's top-k on
// truncated keys and redoes uncertified rows exactly.  Warp-collective
// (tcgen05.ld); a row past T or a layer past L is read but not written.
template <int K>
__device__ __forceinline__ void gate_drain_layer(const GateParams& p, uint32_t tbase, int64_t tok, int layer) {
  const bool valid = tok < p.T && layer < p.L;
  float* lrow = (p.logits != nullptr && valid) ? p.logits + ((size_t)layer * p.T + tok) * 128 : nullptr;
  int T[8], L9 = INT_MIN;
  {
    uint32_t r[32];
    tmem_ld32(tbase, r);
    tmem_ld_wait();
    if (lrow) store_logits32(lrow, r);
    fold32<true, (K == 8)>(r, 0, T, L9);
  }
#pragma unroll 1
  for (int cb = 1; cb < 4; ++cb) {
    uint32_t r[32];
    tmem_ld32(tbase + (uint32_t)(cb * 32), r);
    tmem_ld_wait();
    if (lrow) store_logits32(lrow + cb * 32, r);
    fold32<false, (K == 8)>(r, cb * 32, T, L9);
  }
  // certification of the truncated-key result
  const bool bad = trunc_top8_uncertain<K, GK_IDX_BITS>(T, L9) && valid;
  int idx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) idx[i] = GK_IDX_MAX - (T[i] & GK_IDX_MAX);
  if (__any_sync(FULL, bad)) {
    // the k-th truncated key, value bits only; the row qualifies for the
    // candidate filter when it and every key above it are positive finite
    const int thr = (T[0] < 0x7F800000) ? (T[K - 1] & GK_VAL_MASK) : INT_MIN;
    gate_exact_row(tbase, bad, thr, idx);
  }
  if (valid && p.topk != nullptr) gate_store_ids<K>(p.topk + ((size_t)layer * p.T + tok) * K, idx);
}

// Both layers of a tile's accumulator (TMEM columns tacc .. tacc + 255).
template <int K>
__device__ __forceinline__ void gate_drain_rows(const GateParams& p, uint32_t tacc, int64_t tok, int pair) {
#pragma unroll 1
  for (int hl = 0; hl < 2; ++hl) gate_drain_layer<K>(p, tacc + (uint32_t)(hl * 128), tok, 2 * pair + hl);
}

// ------------------------------------------------- CTA-pair (cta_group::2)
// One tile is 256 tokens x 2 layers, computed by the two CTAs of a cluster
// (two SMs of one TPC) with tcgen05.mma.cta_group::2 at M = 256, N = 256.
// CTA rank r loads A rows = tokens 256 mt + 128 r .. + 127 and B rows = the
// 128 experts of layer 2 pair + r; its TMEM receives its own 128 tokens x all
// 256 columns.  Rank 0 (the leader) takes tile ids, posts the stages'
// transaction counts and issues the MMAs; both CTAs load and drain.
constexpr int GP_BM = 128;   // tokens per CTA (UMMA M = 256 over the pair)
constexpr int GP_BN = 256;   // experts per tile: two layers (UMMA N)
constexpr int GP_BK = 64;
#ifndef MOER_GATE_PREFETCH_ID
#define MOER_GATE_PREFETCH_ID 1
#endif
#ifndef MOER_GATE_PAIR_STAGES
#define MOER_GATE_PAIR_STAGES 6
#endif
constexpr int GP_STAGES = MOER_GATE_PAIR_STAGES;
constexpr int GP_A_BYTES = GP_BM * GP_BK * 2;      // 16 KB
constexpr int GP_B_BYTES = (GP_BN / 2) * GP_BK * 2;  // 16 KB: this CTA's layer
constexpr int GP_STAGE_BYTES = GP_A_BYTES + GP_B_BYTES;
constexpr uint32_t GP_TX_BYTES = 2u * GP_STAGE_BYTES;  // both CTAs' halves land on the leader's barrier
// Epilogue warps per CTA: 4 (each drains both layers of its TMEM lane
// quarter) or 8 (warps 2-5 the first layer, 6-9 the second).
#ifndef MOER_GATE_EPI_WARPS
#define MOER_GATE_EPI_WARPS 4
#endif
constexpr int GP_EPI_WARPS = MOER_GATE_EPI_WARPS;
static_assert(GP_EPI_WARPS == 4 || GP_EPI_WARPS == 8, "4 or 8 epilogue warps");
constexpr int GP_THREADS = (2 + GP_EPI_WARPS) * 32;
constexpr int GP_TMEM_COLS = 512;
constexpr int GP_TRING = 16;
// The leader producer is at most GP_STAGES + 3 tiles ahead of the slowest
// reader of a ring slot (the peer's producer, the MMA thread, either CTA's
// epilogue), so a slot is never rewritten unread.
static_assert(GP_TRING >= GP_STAGES + 3, "tile-id ring shorter than the pipeline's lead");
constexpr size_t GP_OFF_BAR = (size_t)GP_STAGES * GP_STAGE_BYTES;
// barriers (full, empty, tfull, tempty, drain, tile ids), the TMEM address and
// the failure flag, the tile-id ring
constexpr size_t GP_BAR_BYTES = (2 * GP_STAGES + 2 + 2 + 1 + GP_TRING) * 8 + 16 + GP_TRING * 4;
static_assert(GP_BAR_BYTES <= 512, "barrier area");
constexpr size_t GP_SMEM = GP_OFF_BAR + 512 + 1024;
static_assert(GP_SMEM <= 232448, "fits the 227 KB of shared memory a CTA may use");

// Instruction descriptor: D fp32, A and B bf16, both K-major, M = 256, N = 256.
constexpr uint32_t GP_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(GP_BN >> 3) << 17) |
                              ((uint32_t)((2 * GP_BM) >> 4) << 24);

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_u32(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Every thread of both CTAs; release/acquire at cluster scope.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t caddr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(caddr), "r"(v) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

// (barrier given by its shared::cta address)
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for a phase whose arrivals may come from the other CTA.
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, uint32_t* status) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if ((it & 63u) == 63u && (globaltimer_ns() - t0 > WAIT_LIMIT_NS || it >= WAIT_LIMIT_ITERS)) {
      if (status) atomicOr(status, WS_BIT_ETIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, uint32_t* status) {
  return mbar_wait_cl(smem_u32(bar), parity, status);
}

// Tiled 2-D copy into this CTA's shared memory, completing on a barrier that
// may sit in either CTA of the pair (caddr: its shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* tm, int c0, int c1, uint32_t bar_caddr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(c0), "r"(c1), "r"(bar_caddr)
      : "memory");
}

// The operand descriptors come as 32-bit halves: the high half is the same for
// every stage, so the issuing thread only advances the low half (start
// address) with 32-bit adds.
__device__ __forceinline__ void umma_bf16_pair(uint32_t dt, uint32_t a_lo, uint32_t b_lo, uint32_t d_hi,
                                               uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %3};\n\tmov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, p;\n\t}" ::"r"(dt),
      "r"(a_lo), "r"(b_lo), "r"(d_hi), "r"(GP_IDESC), "r"(accum));
}

// Arrives on the barrier at this offset in both CTAs once every MMA issued so
// far by this thread has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) { umma_commit_pair(smem_u32(bar)); }

template <int K>
__global__ void __launch_bounds__(GP_THREADS, 1) gate_pair_kernel(const __grid_constant__ GateParams p) {
  extern __shared__ __align__(1024) char gsm_raw[];
  // 1024-byte alignment of the stage ring (128-byte swizzle atoms); the
  // offsets are the same in both CTAs, as the MMA's descriptors require
  char* gsm = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(gsm + GP_OFF_BAR);  // used in the leader
  uint64_t* empty = full + GP_STAGES;
  uint64_t* tfull = empty + GP_STAGES;
  uint64_t* tempty = tfull + 2;  // used in the leader: the epilogue warps of both CTAs
  uint64_t* drain = tempty + 2;
  uint64_t* tid_full = drain + 1;  // [GP_TRING]: slot j % GP_TRING holds tile j's id
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tid_full + GP_TRING);
  volatile int& failed = *reinterpret_cast<int*>(tmem_slot + 1);  // a wait in this CTA expired
  int* tile_ring = reinterpret_cast<int*>(tmem_slot + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int nkb = p.H / GP_BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < GP_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * GP_EPI_WARPS);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < GP_TRING; ++i) mbar_init(&tid_full[i], 1);
    failed = 0;
    fence_mbar_init();
  }
  // both CTAs running, barriers initialised and visible to the peer
  cluster_sync();
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(GP_TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producers
    if (lane == 0) {
      const uint32_t bar0 = mapa_u32(smem_u32(full), 0);  // the leader's full[0]
      int64_t g = 0;  // stages filled so far
      int s = 0;      // next stage (g mod STAGES) and its round (g / STAGES)
      int64_t round = 0;
      uint32_t ph = 0;  // parity of the release that round `round` >= 1 waits for: (round - 1) & 1
      bool ok = true;
      // the leader fetches each tile id one tile ahead, so the atomic's round
      // trip overlaps the previous tile's loads
      int t_next = (leader && MOER_GATE_PREFETCH_ID) ? (int)atomicAdd(p.tile_ctr, 1u) : -1;
      for (int64_t j = 0;; ++j) {
        const int slot = (int)(j % GP_TRING);
        int t;
        if (leader) {
          t = ok ? (MOER_GATE_PREFETCH_ID ? t_next : (int)atomicAdd(p.tile_ctr, 1u)) : -1;
          if (t >= p.ntiles) t = -1;
          if (MOER_GATE_PREFETCH_ID && t >= 0) t_next = (int)atomicAdd(p.tile_ctr, 1u);
          tile_ring[slot] = t;
          st_cluster_u32(mapa_u32(smem_u32(&tile_ring[slot]), 1), (uint32_t)t);
          mbar_arrive(&tid_full[slot]);                                   // release (CTA)
          mbar_arrive_cluster(mapa_u32(smem_u32(&tid_full[slot]), 1));   // release (cluster): peer's copy
        } else {
          if (!mbar_wait_cl(&tid_full[slot], (uint32_t)((j / GP_TRING) & 1), p.status)) {
            ok = false;
            break;
          }
          t = tile_ring[slot];
        }
        if (t < 0) break;
        const int mt = t / p.npairs, pair = t - mt * p.npairs;
        const int arow = mt * (2 * GP_BM) + (int)rank * GP_BM;
        const int brow = (2 * pair + (int)rank) * 128;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          if (g >= GP_STAGES && !mbar_wait_cl(&empty[s], ph, p.status)) {
            ok = false;
            break;
          }
          char* st = gsm + (size_t)s * GP_STAGE_BYTES;
          if (leader) mbar_arrive_expect_tx(&full[s], GP_TX_BYTES);
          const uint32_t barc = bar0 + (uint32_t)(s * 8);
          tma_load_2d_pair(st, &p.tmx, kb * GP_BK, arow, barc);
          tma_load_2d_pair(st + GP_A_BYTES, &p.tmw, kb * GP_BK, brow, barc);
          if (++s == GP_STAGES) {  // the next round waits on the releases of this one
            s = 0;
            ++round;
            ph = (uint32_t)((round - 1) & 1);
          }
        }
        // after an expired wait the leader's next turn publishes the end
        // marker (-1), so the readers stop; the peer has nothing to publish
        if (!ok && !leader) break;
      }
      // tail: the stage-release arrivals of the last fills have landed, so no
      // MMA still reads this CTA's stages or arrives on its barriers
      for (int64_t q = (g > GP_STAGES ? g - GP_STAGES : 0); q < g; ++q)
        if (!mbar_wait_cl(&empty[q % GP_STAGES], (uint32_t)((q / GP_STAGES) & 1), p.status)) {
          ok = false;
          break;
        }
      if (!ok) failed = 1;
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA
    if (lane == 0) {
      bool ok = true;
      if (leader) {
        // The stage ring is unrolled, so each stage's barrier addresses are
        // immediates and its operand descriptors (low halves: start address,
        // per stage and K step) sit in registers: an MMA issue needs no
        // arithmetic.  The issuing thread shares its SM sub-partition with an
        // epilogue warp whose comparator networks keep the integer pipe busy,
        // and any integer work here would queue behind them.
        const uint64_t d0 = umma_desc_sw128(smem_u32(gsm));
        const uint32_t d_hi = (uint32_t)(d0 >> 32);
        constexpr uint32_t STAGE_STEP = GP_STAGE_BYTES >> 4, B_STEP = GP_A_BYTES >> 4;
        uint32_t da[GP_STAGES][GP_BK / 16], db[GP_STAGES][GP_BK / 16];
#pragma unroll
        for (int st = 0; st < GP_STAGES; ++st)
#pragma unroll
          for (int kk = 0; kk < GP_BK / 16; ++kk) {  // K = 16 per instruction: 32 bytes along the row
            da[st][kk] = (uint32_t)d0 + (uint32_t)st * STAGE_STEP + 2u * kk;
            db[st][kk] = da[st][kk] + B_STEP;
          }
        const uint32_t full_a = smem_u32(full), empty_a = smem_u32(empty);
        uint32_t ph = 0;  // parity of the full barriers in this round of the ring
        int64_t j = 0;    // tiles begun
        uint32_t dt = 0, tfull_a = 0;
        int kb_left = 0;  // K blocks left in the current tile
        // Starts tile j: its id, then a drained accumulator.  False at the end
        // marker or when a wait expired (ok cleared).
        auto begin_tile = [&]() -> bool {
          if (!mbar_wait_cl(&tid_full[j % GP_TRING], (uint32_t)((j / GP_TRING) & 1), p.status)) {
            ok = false;
            return false;
          }
          if (tile_ring[j % GP_TRING] < 0) return false;
          const int a = (int)(j & 1);
          if (j >= 2 && !mbar_wait_cl(&tempty[a], (uint32_t)(((j >> 1) - 1) & 1), p.status)) {
            ok = false;
            return false;
          }
          tc_fence_after();
          dt = tmem + (uint32_t)(a * GP_BN);
          tfull_a = smem_u32(&tfull[a]);
          kb_left = nkb;
          return true;
        };
        if (begin_tile()) {
          for (;;) {
#pragma unroll
            for (int st = 0; st < GP_STAGES; ++st) {
              if (!mbar_wait_cl(full_a + 8u * st, ph, p.status)) {
                ok = false;
                goto mma_done;
              }
              tc_fence_after();
              {
                const uint32_t acc = kb_left != nkb ? 1u : 0u;  // a tile's first K block overwrites
#pragma unroll
                for (int kk = 0; kk < GP_BK / 16; ++kk) umma_bf16_pair(dt, da[st][kk], db[st][kk], d_hi, kk ? 1u : acc);
              }
              umma_commit_pair(empty_a + 8u * st);
              if (--kb_left == 0) {
                umma_commit_pair(tfull_a);
                ++j;
                if (!begin_tile()) goto mma_done;
              }
            }
            ph ^= 1u;
          }
        }
      mma_done:
        // every MMA issued has completed once this arrives (in both CTAs)
        umma_commit_pair(drain);
      }
      if (!mbar_wait_cl(drain, 0, p.status)) ok = false;
      if (!ok) failed = 1;
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;   // token row within this CTA's half
    const uint32_t tempty0 = mapa_u32(smem_u32(tempty), 0);
    bool ok = true;
    for (int64_t j = 0;; ++j) {
      if (!mbar_wait_cl(&tid_full[j % GP_TRING], (uint32_t)((j / GP_TRING) & 1), p.status)) {
        ok = false;
        break;
      }
      const int t = tile_ring[j % GP_TRING];
      if (t < 0) break;
      const int a = (int)(j & 1);
      if (!mbar_wait_cl(&tfull[a], (uint32_t)((j >> 1) & 1), p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int mt = t / p.npairs, pair = t - mt * p.npairs;
      const int64_t tok = (int64_t)mt * (2 * GP_BM) + (int64_t)rank * GP_BM + row;
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * GP_BN);
      if constexpr (GP_EPI_WARPS == 4) {
        gate_drain_rows<K>(p, tacc, tok, pair);
      } else {
        const int hl = (warp - 2) >> 2;  // warps 2-5: first layer, 6-9: second
        gate_drain_layer<K>(p, tacc + (uint32_t)(hl * 128), tok, 2 * pair + hl);
      }
      // accumulator drained: hand it back to the leader's MMA thread
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + (uint32_t)(a * 8));
    }
    if (!ok && lane == 0) failed = 1;
  }
  __syncthreads();
  if (failed) {
    // a wait expired: give copies still in flight into this CTA time to land
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(GP_TMEM_COLS));
  // neither CTA leaves while the other may still take part in the deallocation
  cluster_sync();
}

// Wt[l*128 + e][h] = W[l][h][e] (bf16 bits), through a 32 x 32 shared tile.
__global__ void gate_transpose_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ wt, int L, int H,
                                      int E) {
  __shared__ uint16_t tile[32][33];
  const int l = blockIdx.z;
  const int h0 = blockIdx.y * 32, e0 = blockIdx.x * 32;
  const uint16_t* src = w + (size_t)l * H * E;
  uint16_t* dst = wt + (size_t)l * E * H;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int h = h0 + i, e = e0 + threadIdx.x;
    tile[i][threadIdx.x] = (h < H && e < E) ? src[(size_t)h * E + e] : 0;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int e = e0 + i, h = h0 + threadIdx.x;
    if (e < E && h < H) dst[(size_t)e * H + h] = tile[threadIdx.x][i];
  }
}

// --------------------------------------------------------------- host side
namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::mutex g_enc_mu;
EncodeTiledFn g_enc = nullptr;

EncodeTiledFn encoder() {
  std::lock_guard<std::mutex> lock(g_enc_mu);
  if (g_enc == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    g_enc = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_enc;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)GP_BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaLaunchConfig_t pair_config(int clusters, cudaStream_t st, cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2u * (unsigned)clusters);
  cfg.blockDim = dim3(GP_THREADS);
  cfg.dynamicSmemBytes = GP_SMEM;
  cfg.stream = st;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of two CTAs that fit on the device at once (one CTA per SM),
// queried once per device.
template <int K>
int pair_max_clusters() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  cudaLaunchAttribute at[1];
  const cudaLaunchConfig_t cfg = pair_config(1, nullptr, at);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gate_pair_kernel<K>, &cfg) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

template <int K>
cudaError_t gate_pair_launch_k(const GateParams& p, cudaStream_t st) {
  static std::atomic<unsigned long long> set{0};
  cudaError_t e = smem_optin(gate_pair_kernel<K>, (int)GP_SMEM, set);
  if (e != cudaSuccess) return e;
  const int maxc = pair_max_clusters<K>();
  if (maxc <= 0) return cudaErrorInvalidConfiguration;
  const int clusters = (int)min64(p.ntiles, maxc);
  cudaLaunchAttribute at[1];
  const cudaLaunchConfig_t cfg = pair_config(clusters, st, at);
  e = cudaLaunchKernelEx(&cfg, gate_pair_kernel<K>, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}
}  // namespace

size_t gate_scratch_bytes(const moer_dims* d, int32_t H) {
  return ((size_t)d->L * 128 * (size_t)H * 2 + 255) / 256 * 256;
}

moer_status gate_topk_launch(const moer_dims* d, const uint16_t* hidden, int64_t T, int32_t H,
                             const uint16_t* w_gate, float* logits, uint8_t* topk, void* ws, cudaStream_t st) {
  uint16_t* wt = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + WS_HEADER);
  dim3 tb(32, 8), tg(128 / 32, (H + 31) / 32, d->L);
  gate_transpose_kernel<<<tg, tb, 0, st>>>(w_gate, wt, d->L, H, 128);
  if (cudaGetLastError() != cudaSuccess) return MOER_ECUDA;
  GateParams p;
  // CTA pairs: 256 tokens per tile, each CTA loads its 128 tokens and one layer's weights
  if (!make_map(&p.tmx, hidden, (uint64_t)T, (uint64_t)H, GP_BM)) return MOER_ECUDA;
  if (!make_map(&p.tmw, wt, (uint64_t)d->L * 128, (uint64_t)H, GP_BN / 2)) return MOER_ECUDA;
  const int64_t tile_tokens = 2 * GP_BM;
  p.T = T;
  p.H = H;
  p.L = d->L;
  p.k = d->k;
  p.npairs = (d->L + 1) / 2;
  p.ntiles = ((T + tile_tokens - 1) / tile_tokens) * p.npairs;
  p.logits = logits;
  p.topk = topk;
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.tile_ctr = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + WS_TILE_CTR);
  const int sms = device_sm_count();
  if (sms <= 0) return MOER_ECUDA;
  // the counter runs past ntiles by at most one fetch per producer
  if (p.ntiles + sms >= (int64_t(1) << 31)) return MOER_ERANGE;
  if (cudaMemsetAsync(p.tile_ctr, 0, sizeof(uint32_t), st) != cudaSuccess) return MOER_ECUDA;
  const cudaError_t e = d->k == 8 ? gate_pair_launch_k<8>(p, st) : gate_pair_launch_k<6>(p, st);
  return e == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
