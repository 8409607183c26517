// block_counts.cu -- per-KV-block expert counts over the signature layers.
//
// ELDR, section "Key idea / structure / operation": the prefill hook records
// the request's expert signature at KV-block granularity -- for each block
// and each layer of the selected mask, how many of the block's tokens picked
// each expert in their top-k.
//
// A segmented histogram over the block table: a persistent grid of warps walks
// the KV blocks; per block the warp reads the block's top-k ids of up to sixteen
// mask layers at once (contiguous uint8, len * k bytes per layer, as 4-byte
// words when k is a multiple of 4), counts them into private shared-memory
// rows of packed 8-bit counters (four experts per 32-bit word; a count never
// exceeds B <= 255) and writes the row out with coalesced 32-bit stores.  No
// global atomics, no pre-zeroing.
//
// Each layer's row is 256 bytes whatever E is, so the counter word of id e
// sits at byte (e & ~3) of the row for every byte value e: an id >= E lands
// in the row's tail, which the checked form reads back as MOER_EDATA instead
// of testing every id.  With 256-byte-aligned rows, the address of an id's
// word is one byte permute of the row base and the id word, and its increment
// (1 << 8 (e & 3)) one funnel shift.  The block table is validated on the fly:
// a block whose length is outside [1, B], that runs past T or that does not
// start where the previous block ends is skipped and recorded as MOER_EDATA.
#include "common.cuh"
#include "pdl.cuh"

namespace moer {

constexpr int BC_WARPS = 8;

struct BcParams {
  const uint8_t* ids;     // top-k ids
  int64_t layer_stride;   // T * k
  int64_t T;
  int k, E, B, m, nblk;
  const int32_t* blk_tab;
  uint8_t* blk_cnt;
  uint32_t* status;
  int16_t layer_row[256];  // ids row-block of mask layer i
};

constexpr int BC_MC = 16;  // mask layers counted together (their loads in flight at once)

constexpr int BC_ROW = 256;  // bytes per layer row of counters (64 words)

// red.shared.add of `inc` at shared address `addr` + IMM
template <int IMM>
__device__ __forceinline__ void bc_add(uint32_t addr, uint32_t inc) {
  asm volatile("red.shared.add.u32 [%0+%1], %2;" ::"r"(addr), "n"(IMM), "r"(inc) : "memory");
}

// The four ids packed in `v` counted into the layer row at `row` (256-aligned).
template <int IMM>
__device__ __forceinline__ void bc_count_word(uint32_t row, uint32_t v) {
  const uint32_t offs = v & 0xFCFCFCFCu;          // byte offset of each id's counter word
  const uint32_t shp = (v << 3) & 0x18181818u;    // 8 (e & 3) in each byte
  // byte j of offs into the low byte of the row base
  const uint32_t a0 = __byte_perm(offs, row, 0x7650), a1 = __byte_perm(offs, row, 0x7651);
  const uint32_t a2 = __byte_perm(offs, row, 0x7652), a3 = __byte_perm(offs, row, 0x7653);
  // 1 << (shift & 31): the wrapping funnel shift reads only the low five bits of its amount
  bc_add<IMM>(a0, __funnelshift_l(0u, 1u, shp));
  bc_add<IMM>(a1, __funnelshift_l(0u, 1u, shp >> 8));
  bc_add<IMM>(a2, __funnelshift_l(0u, 1u, shp >> 16));
  bc_add<IMM>(a3, __funnelshift_l(0u, 1u, shp >> 24));
}

template <int II>
__device__ __forceinline__ void bc_count_layers(uint32_t base, const uint32_t (&v)[BC_MC], int nl, bool in) {
  if constexpr (II < BC_MC) {
    if (II < nl && in) bc_count_word<II * BC_ROW>(base, v[II]);
    bc_count_layers<II + 1>(base, v, nl, in);
  }
}

// CHECK: the ids come from the caller (moer_ids_signature); an id >= E is
// not counted (it lands in the row's tail) and is recorded as MOER_EDATA.
template <bool CHECK>
// Six CTAs per SM (at most 40 registers a thread; 24.8 KB of shared memory at m = 12).
__global__ void __launch_bounds__(BC_WARPS * 32, 6) block_counts_kernel(const __grid_constant__ BcParams p) {
  extern __shared__ uint8_t bc_raw[];  // [BC_WARPS][min(m, BC_MC)][256 bytes], 256-byte aligned
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrows = min(p.m, BC_MC);
  const uint32_t base = ((smem_u32(bc_raw) + (BC_ROW - 1)) & ~(uint32_t)(BC_ROW - 1)) + warp * nrows * BC_ROW;
  uint32_t* cnt = reinterpret_cast<uint32_t*>(bc_raw + (base - smem_u32(bc_raw)));
  constexpr int RW = BC_ROW / 4;  // words per layer row
  const int wpb = p.E / 4;        // words holding the E experts
  const int rw = CHECK ? RW : wpb;  // words written, read back and cleared per row
  for (int w = lane; w < nrows * RW; w += 32) cnt[w] = 0u;
  __syncwarp();
  const int64_t stride = (int64_t)gridDim.x * BC_WARPS;
  // 4-byte loads when every block's id row starts on a 4-byte boundary
  const bool vec = (p.k % 4) == 0;
  uint32_t bad = 0u;
  // persistent warps, one KV block at a time, all mask layers of the block
  for (int64_t bb = (int64_t)blockIdx.x * BC_WARPS + warp; bb < p.nblk; bb += stride) {
    const int b = (int)bb;
    const int t0 = p.blk_tab[2 * b], ln = p.blk_tab[2 * b + 1];
    bool ok = ln >= 1 && ln <= p.B && t0 >= 0 && (int64_t)t0 + ln <= p.T;
    if (b == 0) {
      ok = ok && t0 == 0;
    } else {
      const int pt0 = p.blk_tab[2 * (b - 1)], pln = p.blk_tab[2 * (b - 1) + 1];
      ok = ok && (int64_t)pt0 + pln == (int64_t)t0;
    }
    if (b == p.nblk - 1) ok = ok && (int64_t)t0 + ln == p.T;
    if (!ok) {
      if (lane == 0) atomicOr(p.status, WS_BIT_EDATA);
      continue;
    }
    const int n = ln * p.k;
    for (int i0 = 0; i0 < p.m; i0 += BC_MC) {
      const int nl = min(BC_MC, p.m - i0);
      if (vec) {
        const int nw = n >> 2;
        for (int q0 = 0; q0 < nw; q0 += 32) {
          const int q = q0 + lane;
          uint32_t v[BC_MC];
#pragma unroll
          for (int ii = 0; ii < BC_MC; ++ii) {
            v[ii] = 0u;
            if (ii < nl && q < nw) {
              const uint8_t* src = p.ids + (int64_t)p.layer_row[i0 + ii] * p.layer_stride + (int64_t)t0 * p.k;
              v[ii] = reinterpret_cast<const uint32_t*>(src)[q];
            }
          }
          bc_count_layers<0>(base, v, nl, q < nw);
        }
      } else {
        for (int ii = 0; ii < nl; ++ii) {
          const uint8_t* src = p.ids + (int64_t)p.layer_row[i0 + ii] * p.layer_stride + (int64_t)t0 * p.k;
          const uint32_t row = base + ii * BC_ROW;
          for (int j = lane; j < n; j += 32) {
            const uint32_t e = src[j];
            bc_add<0>(row + (e & ~3u), 1u << ((e & 3u) * 8u));
          }
        }
      }
      __syncwarp();
      for (int ii = 0; ii < nl; ++ii) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.blk_cnt + ((size_t)b * p.m + i0 + ii) * p.E);
        for (int w = lane; w < rw; w += 32) {
          const uint32_t c = cnt[ii * RW + w];
          cnt[ii * RW + w] = 0u;
          if (w < wpb)
            dst[w] = c;
          else
            bad |= c;
        }
      }
      __syncwarp();
    }
  }
  if (CHECK && bad != 0u) atomicOr(p.status, WS_BIT_EDATA);
  pdl_release();
}

// ids: either the caller's [L][T][k] top-k (mask_only = false: row block of
// mask layer i is mask[i]) or a mask-only [m][T][k] buffer (row block i).
// check: ids from outside the library, bounded by E as they are read.
moer_status block_counts_launch(const moer_dims* d, const uint8_t* ids, bool mask_only, int64_t T,
                                const int32_t* blk_tab, int nblk, uint8_t* blk_cnt, uint32_t* status,
                                cudaStream_t st, bool check) {
  BcParams p;
  p.ids = ids;
  p.layer_stride = T * d->k;
  p.T = T;
  p.k = d->k;
  p.E = d->E;
  p.B = d->block;
  p.m = d->m;
  p.nblk = nblk;
  p.blk_tab = blk_tab;
  p.blk_cnt = blk_cnt;
  p.status = status;
  for (int i = 0; i < 256; ++i) p.layer_row[i] = 0;
  for (int i = 0; i < d->m; ++i) p.layer_row[i] = (int16_t)(mask_only ? i : d->mask[i]);
  if (nblk <= 0 || d->m <= 0) return MOER_OK;
  const int sms = device_sm_count();
  if (sms <= 0) return MOER_ECUDA;
  const int64_t grid = min64(((int64_t)nblk + BC_WARPS - 1) / BC_WARPS, (int64_t)sms * 8);
  const size_t smem = (size_t)BC_WARPS * min(d->m, BC_MC) * BC_ROW + BC_ROW;  // + alignment slack
  // a normal launch: the persistent grid's static split wants every SM free when it
  // starts (pdl.cuh); the kernel still releases its successor at its end
  if (check)
    block_counts_kernel<true><<<(unsigned)grid, BC_WARPS * 32, smem, st>>>(p);
  else
    block_counts_kernel<false><<<(unsigned)grid, BC_WARPS * 32, smem, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer

namespace moer {

// Per-layer co-activation counts from top-k ids (the gate path, where the ids
// come out of the GEMM epilogue rather than from a logits pass).  GRACE-MoE,
// section 3 and section 4 / Figure 2(a): A_l[a][b] += #tokens whose top-k
// at layer l holds both a and b.
//
// Persistent grid over (layer, 2048-token chunk) items in layer-major order,
// four token rows per thread with their id loads issued together.  A row's k
// distinct ids, in rank order, add its k(k-1)/2 rank-ordered pairs to a
// shared tile of directed counts D[a][b] (= # rows where a ranks above b).  When the CTA's layer changes
// the tile is folded into the symmetric co-activation -- A[a][b] = D[a][b] +
// D[b][a] off the diagonal, and A[a][a] = (sum over b != a of A[a][b]) /
// (k - 1), since each row holding a holds k - 1 other experts -- and added to
// global memory.  Needs k >= 2.
constexpr int AI_THREADS = 512;
constexpr int AI_U = 4;                      // tokens per thread per item, loads in flight together
constexpr int AI_CHUNK = AI_THREADS * AI_U;  // tokens per work item

// The tile's rows are E + 1 words apart, so the bank of D[a][b] depends on a
// as well as b.  A warp per row a, by warp reductions -- no shared atomics,
// which a row's lanes would all aim at one counter: the diagonal is the sum of
// the row and column of D (D[a][a] is 0: a kept row's ids are distinct) over
// k - 1, and A[a][b] = D[a][b] + D[b][a] goes out with 64-bit reds (two
// neighbouring counts) when the output is 8-byte aligned, else pair by pair.
__device__ void affinity_ids_flush(int* tile, int* rsum, int E, int k, int32_t* dst) {
  (void)rsum;
  const int rs = E + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NW = AI_THREADS / 32;
  if ((reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
    // 8-byte aligned output: a warp adds its row's whole symmetric row, diagonal
    // included, two neighbouring counts per 64-bit red (counts fit in int32, so no
    // carry crosses into the upper count)
    for (int a = warp; a < E; a += NW) {
      int sum = 0;
      for (int b = lane; b < E; b += 32) sum += tile[a * rs + b] + tile[b * rs + a];
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
      const uint32_t diag = (uint32_t)(sum / (k - 1));
      for (int b = 2 * lane; b < E; b += 64) {
        const uint32_t v0 = b == a ? diag : (uint32_t)(tile[a * rs + b] + tile[b * rs + a]);
        const uint32_t v1 = b + 1 == a ? diag : (uint32_t)(tile[a * rs + b + 1] + tile[(b + 1) * rs + a]);
        if ((v0 | v1) != 0u) {
          const unsigned long long v = ((unsigned long long)v1 << 32) | v0;
          asm volatile("red.global.add.u64 [%0], %1;" ::"l"(dst + (size_t)a * E + b), "l"(v) : "memory");
        }
      }
    }
  } else {
    for (int a = warp; a < E - 1; a += NW)
      for (int b = a + 1 + lane; b < E; b += 32) {
        const int v = tile[a * rs + b] + tile[b * rs + a];
        if (v != 0) {
          atomicAdd(&dst[a * E + b], v);
          atomicAdd(&dst[b * E + a], v);
        }
      }
    for (int a = warp; a < E; a += NW) {
      int sum = 0;
      for (int b = lane; b < E; b += 32) sum += tile[a * rs + b] + tile[b * rs + a];
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
      if (lane == 0 && sum != 0) atomicAdd(&dst[a * E + a], sum / (k - 1));
    }
  }
  __syncthreads();  // every read of the tile is done before it is cleared
  for (int c = threadIdx.x; c < E * rs; c += AI_THREADS) tile[c] = 0;
  __syncthreads();
}

// Any byte of x zero: the classic borrow test, exact as an "any" test (a false
// high bit only ever appears above a real zero byte).  Accumulated with OR and
// masked once: acc |= (x - 0x01010101) & ~x.
__device__ __forceinline__ uint32_t zero_byte_acc(uint32_t acc, uint32_t x) {
  return acc | ((x - 0x01010101u) & ~x);
}

// A row of K = 6 or 8 ids packed in two words (ids 0-3 in w0, ids 4.. in w1)
// is usable for the co-activation when every id is below E (<= 128) and the K
// ids are distinct.  Range: per byte, (x | 0x80) - E keeps the high bit only
// when x & 0x7F >= E; x >= 128 is caught by x's own high bit.  Distinctness:
// every pair of bytes compared once by XOR against byte rotations of the
// words (within a word by 8 and 16 bits, across the words by 0, 8, 16 and 24
// bits) and a zero-byte test.  With K = 6 the two unused bytes of w1 hold
// 0xFE and 0xFF, which differ from each other and from every id below E.
template <int K>
__device__ __forceinline__ bool ids_row_ok(uint32_t w0, uint32_t w1, int E) {
  static_assert(K == 6 || K == 8, "rows of 6 or 8 ids");
  if constexpr (K == 6) w1 &= 0xFFFFu;
  const uint32_t E4 = (uint32_t)E * 0x01010101u;
  const uint32_t hi = (((w0 | 0x80808080u) - E4) | w0) | (((w1 | 0x80808080u) - E4) | w1);
  if constexpr (K == 6) w1 |= 0xFFFE0000u;
  uint32_t z = 0u;
  z = zero_byte_acc(z, w0 ^ __funnelshift_l(w0, w0, 8));
  z = zero_byte_acc(z, w0 ^ __funnelshift_l(w0, w0, 16));
  z = zero_byte_acc(z, w1 ^ __funnelshift_l(w1, w1, 8));
  z = zero_byte_acc(z, w1 ^ __funnelshift_l(w1, w1, 16));
  z = zero_byte_acc(z, w0 ^ w1);
  z = zero_byte_acc(z, w0 ^ __funnelshift_l(w1, w1, 8));
  z = zero_byte_acc(z, w0 ^ __funnelshift_l(w1, w1, 16));
  z = zero_byte_acc(z, w0 ^ __funnelshift_l(w1, w1, 24));
  return ((hi | z) & 0x80808080u) == 0u;
}

// CHECK: the ids come from the caller (moer_ids_signature); a row holding an
// id >= E or a repeated id is left out (the diagonal needs k distinct ids)
// and recorded as MOER_EDATA.
template <int K, bool CHECK>
__global__ void __launch_bounds__(AI_THREADS) affinity_ids_kernel(const uint8_t* __restrict__ ids, int64_t T,
                                                                  int E, int L, int nchunks,
                                                                  int32_t* __restrict__ affinity,
                                                                  uint32_t* status) {
  extern __shared__ int ai_tile[];  // [E][E + 1] directed counts, then [E] row sums
  pdl_wait();
  const int rs = E + 1;
  int* rsum = ai_tile + E * rs;
  const uint32_t tile_base = smem_u32(ai_tile);
  const uint32_t row_bytes = (uint32_t)rs * 4u;
  const int64_t nitems = (int64_t)L * nchunks;
  const int64_t i0 = (int64_t)blockIdx.x * nitems / gridDim.x;
  const int64_t i1 = ((int64_t)blockIdx.x + 1) * nitems / gridDim.x;
  for (int c = threadIdx.x; c < E * rs + E; c += AI_THREADS) ai_tile[c] = 0;
  __syncthreads();
  int cur = (int)(i0 / nchunks);
  for (int64_t it = i0; it < i1; ++it) {
    const int l = (int)(it / nchunks);
    if (l != cur) {
      __syncthreads();
      affinity_ids_flush(ai_tile, rsum, E, K, affinity + (size_t)cur * E * E);
      cur = l;
    }
    const int64_t tb = (it - (int64_t)l * nchunks) * AI_CHUNK + threadIdx.x;
    const uint8_t* lay = ids + (size_t)l * T * K;
    uint32_t w[AI_U][(K + 3) / 4];
#pragma unroll
    for (int u = 0; u < AI_U; ++u) {
      const int64_t t = tb + (int64_t)u * AI_THREADS;
      if (t < T) {
        if constexpr (K == 8) {
          const uint2 v = *reinterpret_cast<const uint2*>(lay + (size_t)t * 8);
          w[u][0] = v.x;
          w[u][1] = v.y;
        } else {
          const uint8_t* src = lay + (size_t)t * K;
#pragma unroll
          for (int j = 0; j < K; j += 2) {
            const uint32_t h = *reinterpret_cast<const uint16_t*>(src + j);
            if (j % 4 == 0)
              w[u][j / 4] = h;
            else
              w[u][j / 4] |= h << 16;
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < AI_U; ++u) {
      if (tb + (int64_t)u * AI_THREADS < T) {
        int e[K];
#pragma unroll
        for (int j = 0; j < K; ++j) e[j] = (w[u][j / 4] >> (8 * (j % 4))) & 0xFF;
        if constexpr (CHECK) {
          if (!ids_row_ok<K>(w[u][0], w[u][1], E)) {
            atomicOr(status, WS_BIT_EDATA);
            continue;
          }
        }
        // shared address of D[a][b] = tile + 4 b + a * row pitch: one
        // multiply-add per pair (FMA pipe) rather than integer-ALU adds
        uint32_t colb[K];
#pragma unroll
        for (int j = 1; j < K; ++j) colb[j] = tile_base + 4u * (uint32_t)e[j];
#pragma unroll
        for (int i = 0; i < K - 1; ++i) {
#pragma unroll
          for (int j = i + 1; j < K; ++j) {
            uint32_t addr;
            asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(addr) : "r"((uint32_t)e[i]), "r"(row_bytes), "r"(colb[j]));
            asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(addr) : "memory");
          }
        }
      }
    }
  }
  __syncthreads();
  affinity_ids_flush(ai_tile, rsum, E, K, affinity + (size_t)cur * E * E);
  pdl_release();
}

// ids [L][T][k] (k = 6 or 8, 8-byte aligned rows for k = 8) -> affinity
// [L][E][E] accumulated.
moer_status affinity_ids_launch(const moer_dims* d, const uint8_t* ids, int64_t T, int32_t* affinity,
                                cudaStream_t st, uint32_t* status, bool check) {
  if (d->k != 8 && d->k != 6) return MOER_ERANGE;
  if (d->E > 128) return MOER_ERANGE;
  const int nchunks = (int)((T + AI_CHUNK - 1) / AI_CHUNK);
  const int64_t nitems = (int64_t)d->L * nchunks;
  const int sms = device_sm_count();
  if (sms <= 0) return MOER_ECUDA;
  const size_t smem = ((size_t)d->E * (d->E + 1) + d->E) * sizeof(int);
  static std::atomic<unsigned long long> set8{0}, set6{0}, set8c{0}, set6c{0};
  const int most = (int)((128 * 129 + 128) * sizeof(int));
  if (smem_optin(affinity_ids_kernel<8, false>, most, set8) != cudaSuccess ||
      smem_optin(affinity_ids_kernel<6, false>, most, set6) != cudaSuccess ||
      smem_optin(affinity_ids_kernel<8, true>, most, set8c) != cudaSuccess ||
      smem_optin(affinity_ids_kernel<6, true>, most, set6c) != cudaSuccess)
    return MOER_ECUDA;
  const int grid = (int)min64(nitems, (int64_t)sms * 2);
  auto kernel = d->k == 8 ? (check ? affinity_ids_kernel<8, true> : affinity_ids_kernel<8, false>)
                          : (check ? affinity_ids_kernel<6, true> : affinity_ids_kernel<6, false>);
  // a normal launch, as for the block counts: two CTAs per SM split the items statically
  kernel<<<grid, AI_THREADS, smem, st>>>(ids, T, d->E, d->L, nchunks, affinity, status);
  return cudaGetLastError() == cudaSuccess ? MOER_OK : MOER_ECUDA;
}

}  // namespace moer
