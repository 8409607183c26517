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
//   * One CTA per SM, persistent over tiles of 128 tokens x 2 layers
//     (M = 128, N = 256 experts), K = H in blocks of 64.  Tiles, token block
//     major, are handed out in order from a global counter, so the grid
//     works on a few token blocks at a time: each hidden-state panel is read
//     from HBM once and shared through L2; the 25 MB of weights stay in L2.
//   * Warp 0 streams both operands with TMA (cp.async.bulk.tensor, 128-byte
//     swizzle) into a 4-stage ring of 48 KB stages (mbarrier full/empty).
//   * Warp 1 owns a 512-column TMEM allocation (two fp32 128 x 256
//     accumulators); one elected thread issues tcgen05.mma.cta_group::1
//     .kind::f16 (4 per K block) and releases stages and accumulators with
//     tcgen05.commit.
//   * Warps 2-5 drain an accumulator with tcgen05.ld while the next tile's
//     MMAs run: each thread owns one token row (one TMEM lane), reads its 128
//     logits per layer, optionally stores them, and selects the row's top-k
//     with the same comparator networks as the logits pass (unique truncated
//     keys; certified, else redone exactly with 40-bit keys).
//   * Every wait is bounded; on expiry the kernel records MOER_ETIMEOUT,
//     drains what it issued and frees its TMEM before returning.
#include <cuda.h>
#include <climits>
#include <mutex>

#include "common.cuh"

namespace moer {

constexpr int GK_BM = 128;   // tokens per tile (UMMA M)
constexpr int GK_BN = 256;   // experts per tile: two layers of 128 (UMMA N)
constexpr int GK_BK = 64;    // K per stage (128 bytes of bf16: one swizzle row)
constexpr int GK_STAGES = 4;
constexpr int GK_A_BYTES = GK_BM * GK_BK * 2;  // 16 KB
constexpr int GK_B_BYTES = GK_BN * GK_BK * 2;  // 32 KB
constexpr int GK_STAGE_BYTES = GK_A_BYTES + GK_B_BYTES;
constexpr int GK_THREADS = 6 * 32;
constexpr int GK_TMEM_COLS = 512;
// Tile ids travel from the producer to the MMA and epilogue warps through a
// ring of GK_TRING slots.  The producer leads the epilogue by at most
// GK_STAGES + 2 tiles (stages in flight, two accumulators), so a slot is never
// rewritten before every reader has taken it.
constexpr int GK_TRING = 16;
static_assert(GK_TRING > GK_STAGES + 2, "tile-id ring shorter than the pipeline's lead");
constexpr size_t GK_OFF_BAR = (size_t)GK_STAGES * GK_STAGE_BYTES;
// barriers (full, empty, tfull, tempty, drain, tile ids), the TMEM address, the tile-id ring
constexpr size_t GK_BAR_BYTES = (2 * GK_STAGES + 2 + 2 + 1 + GK_TRING) * 8 + 16 + GK_TRING * 4;
constexpr size_t GK_SMEM = GK_OFF_BAR + 512 + 1024;  // + barrier area, + 1 KB alignment slack
static_assert(GK_BAR_BYTES <= 512, "barrier area");

struct GateParams {
  CUtensorMap tmx;  // hidden [T][H] bf16, box 64 x 128, 128B swizzle
  CUtensorMap tmw;  // Wt [L*128][H] bf16, box 64 x 256, 128B swizzle
  int64_t T;
  int H, L, k;
  int npairs;       // ceil(L / 2)
  int64_t ntiles;   // ceil(T / 128) * npairs
  float* logits;    // [L][T][128] or nullptr
  uint8_t* topk;    // [L][T][k]
  uint32_t* status;
  uint32_t* tile_ctr;  // next tile to hand out (zeroed before the launch)
};

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(tm), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

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

// Instruction descriptor: D fp32, A and B bf16, both K-major, M = 128, N = 256.
constexpr uint32_t GK_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(GK_BN >> 3) << 17) |
                              ((uint32_t)(GK_BM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t dt, uint64_t a, uint64_t b, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dt),
      "l"(a), "l"(b), "r"(GK_IDESC), "r"(accum));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
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

// ------------------------------------------------------ comparator networks
__device__ __forceinline__ void gcas(int& a, int& b) {
  const int hi = max(a, b), lo = min(a, b);
  a = hi;
  b = lo;
}
__device__ __forceinline__ void gsort8(int (&c)[8]) {
  gcas(c[0], c[2]); gcas(c[1], c[3]); gcas(c[4], c[6]); gcas(c[5], c[7]);
  gcas(c[0], c[4]); gcas(c[1], c[5]); gcas(c[2], c[6]); gcas(c[3], c[7]);
  gcas(c[0], c[1]); gcas(c[2], c[3]); gcas(c[4], c[5]); gcas(c[6], c[7]);
  gcas(c[2], c[4]); gcas(c[3], c[5]);
  gcas(c[1], c[4]); gcas(c[3], c[6]);
  gcas(c[1], c[2]); gcas(c[3], c[4]); gcas(c[5], c[6]);
}
__device__ __forceinline__ void gclean8(int (&m)[8]) {
  gcas(m[0], m[4]); gcas(m[1], m[5]); gcas(m[2], m[6]); gcas(m[3], m[7]);
  gcas(m[0], m[2]); gcas(m[1], m[3]); gcas(m[4], m[6]); gcas(m[5], m[7]);
  gcas(m[0], m[1]); gcas(m[2], m[3]); gcas(m[4], m[5]); gcas(m[6], m[7]);
}

// Folds 32 logits (expert ids e0 .. e0+31) into the running top-8 keys T
// (and the 9th key L9).  Key = upper 24 bits of the float | (255 - expert).
template <bool FIRST>
__device__ __forceinline__ void fold32(const uint32_t (&r)[32], int e0, int (&T)[8], int& L9) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    int c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = ((int)r[8 * g + j] & (int)0xFFFFFF00) | (255 - (e0 + 8 * g + j));
    gsort8(c);
    if (FIRST && g == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) T[i] = c[i];
    } else {
      int m[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        m[i] = max(T[i], c[7 - i]);
        L9 = max(L9, min(T[i], c[7 - i]));
      }
      gclean8(m);
#pragma unroll
      for (int i = 0; i < 8; ++i) T[i] = m[i];
    }
  }
}

// Exact ranking key on 40 bits: order-preserving value key (NaN lowest, -0 ==
// +0) above the inverted expert id (ties to the lower id).
__device__ __forceinline__ uint64_t gexact_key(uint32_t b, int e) {
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) b = 1u;
  else {
    if (b == 0x80000000u) b = 0u;
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  return ((uint64_t)b << 8) | (uint64_t)(255 - e);
}

__device__ __forceinline__ void gcas64(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// ----------------------------------------------------------------- kernel
template <int K>
__global__ void __launch_bounds__(GK_THREADS, 1) gate_topk_kernel(const __grid_constant__ GateParams p) {
  extern __shared__ __align__(1024) char gsm_raw[];
  // 1024-byte alignment of the stage ring (required by the 128-byte swizzle atoms)
  char* gsm = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(gsm + GK_OFF_BAR);
  uint64_t* empty = full + GK_STAGES;
  uint64_t* tfull = empty + GK_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* tid_full = drain + 1;  // [GK_TRING]: slot j % GK_TRING holds tile j's id
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tid_full + GK_TRING);
  int* tile_ring = reinterpret_cast<int*>(tmem_slot + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Tiles are handed out in order from one global counter, so at any moment
  // the grid works on ~gridDim.x consecutive tiles, i.e. on few token blocks:
  // each hidden-state panel comes from HBM once and is shared through L2 by
  // the CTAs on its layers, however unevenly the CTAs progress.
  const int nkb = p.H / GK_BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < GK_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < GK_TRING; ++i) mbar_init(&tid_full[i], 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(GK_TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int64_t g = 0;
      bool ok = true;
      for (int64_t j = 0;; ++j) {
        int t = ok ? (int)atomicAdd(p.tile_ctr, 1u) : -1;
        if (t >= p.ntiles) t = -1;
        tile_ring[j % GK_TRING] = t;
        mbar_arrive(&tid_full[j % GK_TRING]);  // release: the id is visible to the waiters
        if (t < 0) break;
        const int mt = t / p.npairs, pair = t - mt * p.npairs;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = (int)(g % GK_STAGES);
          if (g >= GK_STAGES && !mbar_wait(&empty[s], (uint32_t)((g / GK_STAGES - 1) & 1), p.status)) {
            ok = false;
            break;
          }
          char* st = gsm + (size_t)s * GK_STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], GK_STAGE_BYTES);
          tma_load_2d(st, &p.tmx, kb * GK_BK, mt * GK_BM, &full[s]);
          tma_load_2d(st + GK_A_BYTES, &p.tmw, kb * GK_BK, pair * GK_BN, &full[s]);
        }
      }
      if (!ok) {
        // wait (bounded) for the loads still in flight before leaving
        for (int64_t q = (g > GK_STAGES ? g - GK_STAGES : 0); q < g; ++q)
          mbar_wait(&full[q % GK_STAGES], (uint32_t)((q / GK_STAGES) & 1), nullptr);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA
    if (lane == 0) {
      int64_t g = 0;
      bool ok = true;
      for (int64_t j = 0; ok; ++j) {
        if (!mbar_wait(&tid_full[j % GK_TRING], (uint32_t)((j / GK_TRING) & 1), p.status)) {
          ok = false;
          break;
        }
        if (tile_ring[j % GK_TRING] < 0) break;
        const int a = (int)(j & 1);
        if (j >= 2 && !mbar_wait(&tempty[a], (uint32_t)(((j >> 1) - 1) & 1), p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)(a * GK_BN);
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = (int)(g % GK_STAGES);
          if (!mbar_wait(&full[s], (uint32_t)((g / GK_STAGES) & 1), p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(gsm + (size_t)s * GK_STAGE_BYTES);
          const uint64_t da = umma_desc_sw128(sa), db = umma_desc_sw128(sa + GK_A_BYTES);
#pragma unroll
          for (int kk = 0; kk < GK_BK / 16; ++kk)  // K = 16 per instruction: 32 bytes along the row
            umma_bf16(dt, da + (uint64_t)(2 * kk), db + (uint64_t)(2 * kk), (kb | kk) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (ok) umma_commit(&tfull[a]);
      }
      // all MMAs this thread issued have completed once this commit arrives
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;   // token row within the tile
    for (int64_t j = 0;; ++j) {
      if (!mbar_wait(&tid_full[j % GK_TRING], (uint32_t)((j / GK_TRING) & 1), p.status)) break;
      const int t = tile_ring[j % GK_TRING];
      if (t < 0) break;
      const int a = (int)(j & 1);
      if (!mbar_wait(&tfull[a], (uint32_t)((j >> 1) & 1), p.status)) break;
      tc_fence_after();
      const int mt = t / p.npairs, pair = t - mt * p.npairs;
      const int64_t tok = (int64_t)mt * GK_BM + row;
#pragma unroll 1
      for (int hl = 0; hl < 2; ++hl) {
        const int layer = 2 * pair + hl;
        const bool valid = tok < p.T && layer < p.L;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * GK_BN + hl * 128);
        int T[8], L9 = INT_MIN;
        float* lrow = (p.logits != nullptr && valid) ? p.logits + ((size_t)layer * p.T + tok) * 128 : nullptr;
        {
          uint32_t r[32];
          tmem_ld32(tbase, r);
          tmem_ld_wait();
          if (lrow)
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(lrow + c) = make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]),
                                                                __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
          fold32<true>(r, 0, T, L9);
        }
#pragma unroll 1
        for (int cb = 1; cb < 4; ++cb) {
          uint32_t r[32];
          tmem_ld32(tbase + (uint32_t)(cb * 32), r);
          tmem_ld_wait();
          if (lrow)
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(lrow + cb * 32 + c) =
                  make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]), __uint_as_float(r[c + 2]),
                              __uint_as_float(r[c + 3]));
          fold32<false>(r, cb * 32, T, L9);
        }
        // certification of the truncated-key result
        const int nxt = (K == 8) ? L9 : T[K < 8 ? K : 7];
        bool bad = (T[K - 1] < 256) || (T[0] >= 0x7F800000);
#pragma unroll
        for (int i = 0; i < K; ++i) {
          const int b = (i + 1 < K) ? T[i + 1] : nxt;
          bad = bad || (b >= (T[i] & (int)0xFFFFFF00));
        }
        bad = bad && valid;
        int idx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) idx[i] = 255 - (T[i] & 0xFF);
        if (__any_sync(FULL, bad)) {
          // exact pass for the whole warp (tcgen05.ld is warp-collective); rows
          // that were certified keep their result
          uint64_t X[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) X[i] = 0;
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            uint32_t r[32];
            tmem_ld32(tbase + (uint32_t)(cb * 32), r);
            tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint64_t c[8];
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) c[jj] = gexact_key(r[8 * g + jj], cb * 32 + 8 * g + jj);
              // insertion of 8 keys into the sorted top-8 (descending)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                uint64_t x = c[jj];
#pragma unroll
                for (int i = 0; i < 8; ++i) gcas64(X[i], x);
              }
            }
          }
          if (bad) {
#pragma unroll
            for (int i = 0; i < 8; ++i) idx[i] = 255 - (int)(X[i] & 0xFF);
          }
        }
        if (valid && p.topk != nullptr) {
          uint8_t* o = p.topk + ((size_t)layer * p.T + tok) * K;
          if constexpr (K == 8) {
            const uint32_t lo = (uint32_t)idx[0] | ((uint32_t)idx[1] << 8) | ((uint32_t)idx[2] << 16) |
                                ((uint32_t)idx[3] << 24);
            const uint32_t hi = (uint32_t)idx[4] | ((uint32_t)idx[5] << 8) | ((uint32_t)idx[6] << 16) |
                                ((uint32_t)idx[7] << 24);
            *reinterpret_cast<uint2*>(o) = make_uint2(lo, hi);
          } else {
#pragma unroll
            for (int i = 0; i < K; i += 2) *reinterpret_cast<uint16_t*>(o + i) = (uint16_t)(idx[i] | (idx[i + 1] << 8));
          }
        }
      }
      // accumulator drained: hand it back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(GK_TMEM_COLS));
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
  const cuuint32_t box[2] = {(cuuint32_t)GK_BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int K>
cudaError_t gate_launch_k(const GateParams& p, int grid, cudaStream_t st) {
  static std::atomic<unsigned long long> set{0};
  const cudaError_t e = smem_optin(gate_topk_kernel<K>, (int)GK_SMEM, set);
  if (e != cudaSuccess) return e;
  gate_topk_kernel<K><<<grid, GK_THREADS, GK_SMEM, st>>>(p);
  return cudaGetLastError();
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
  if (!make_map(&p.tmx, hidden, (uint64_t)T, (uint64_t)H, GK_BM)) return MOER_ECUDA;
  if (!make_map(&p.tmw, wt, (uint64_t)d->L * 128, (uint64_t)H, GK_BN)) return MOER_ECUDA;
  p.T = T;
  p.H = H;
  p.L = d->L;
  p.k = d->k;
  p.npairs = (d->L + 1) / 2;
  p.ntiles = ((T + GK_BM - 1) / GK_BM) * p.npairs;
  p.logits = logits;
  p.topk = topk;
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.tile_ctr = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + WS_TILE_CTR);
  const int sms = device_sm_count();
  if (sms <= 0) return MOER_ECUDA;
  const int grid = (int)min64(p.ntiles, sms);
  if (p.ntiles + grid >= (int64_t(1) << 31)) return MOER_ERANGE;
  if (cudaMemsetAsync(p.tile_ctr, 0, sizeof(uint32_t), st) != cudaSuccess) return MOER_ECUDA;
  const cudaError_t e = d->k == 8 ? gate_launch_k<8>(p, grid, st) : gate_launch_k<6>(p, grid, st);
  return e == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
