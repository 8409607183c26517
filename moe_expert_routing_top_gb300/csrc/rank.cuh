// rank.cuh -- the ranking of the top-k gate, in one place for every kernel
// that selects experts (the warp-per-row and thread-per-row logits passes and
// the gate GEMM's epilogue).
//
// The order is the standard top-k gate's (ELDR, section "What it tries to
// solve": each token keeps the k experts with the largest router logits),
// made total: larger logit first; equal logits, -0.0 == +0.0 included, rank
// the lower expert id first; NaN ranks below every number, NaNs among
// themselves by expert id.
//
// Two forms of the order live here:
//   * exact keys: rank_key() maps a float to a 32-bit unsigned key whose
//     integer order is the ranking by value (NaN -> 1, the lowest key a
//     value can take; 0 is reserved for "taken"), and rank_key40() appends
//     the inverted expert id so that equal values order by id;
//   * truncated keys for the fast paths: the float's upper bits with an
//     inverted position in the low IDX_BITS bits (8, or 7 when E <= 128),
//     compared as signed ints, sorted by comparator networks.  These agree
//     with the exact order only on positive finite values whose truncations
//     differ, which trunc_top8_uncertain() checks; rows it rejects are
//     redone exactly.
#pragma once

#include <climits>

#include "common.cuh"

namespace moer {

// ------------------------------------------------------------ exact keys
__device__ __forceinline__ uint32_t rank_key_bits(uint32_t b) {
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 1u;  // NaN: below every number
  if (b == 0x80000000u) b = 0u;                      // -0.0 ranks as +0.0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ uint32_t rank_key(float x) { return rank_key_bits(__float_as_uint(x)); }

// 40-bit key: the value key above the inverted expert id (ties to the lower id).
__device__ __forceinline__ uint64_t rank_key40(uint32_t bits, int e) {
  return ((uint64_t)rank_key_bits(bits) << 8) | (uint64_t)(255 - e);
}

// ------------------------------------------------------- truncated keys
// The float's upper 32 - IDX_BITS bits with `low` (an inverted position,
// < 2^IDX_BITS) below.  IDX_BITS = 8 serves any E <= 256; with E <= 128, 7
// bits leave one more mantissa bit to the value, so fewer rows need the
// exact path.  (The thread-per-row pass forms the 8-bit form with a
// multiply-high and a multiply-add, to keep it off the integer ALU pipe.)
template <int IDX_BITS = 8>
__device__ __forceinline__ int trunc_key(uint32_t bits, int low) {
  static_assert(IDX_BITS >= 1 && IDX_BITS <= 8, "index field of 1 to 8 bits");
  return (int)(bits & ~((1u << IDX_BITS) - 1u)) | low;
}

// ---------------------------------------------------- comparator networks
__device__ __forceinline__ void cas(int& a, int& b) {  // a <- max, b <- min
  const int hi = max(a, b), lo = min(a, b);
  a = hi;
  b = lo;
}
__device__ __forceinline__ void cas64(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// Sorts 8 keys in descending order (19 comparators, depth 6).
__device__ __forceinline__ void sort8_desc(int (&c)[8]) {
  cas(c[0], c[2]); cas(c[1], c[3]); cas(c[4], c[6]); cas(c[5], c[7]);
  cas(c[0], c[4]); cas(c[1], c[5]); cas(c[2], c[6]); cas(c[3], c[7]);
  cas(c[0], c[1]); cas(c[2], c[3]); cas(c[4], c[5]); cas(c[6], c[7]);
  cas(c[2], c[4]); cas(c[3], c[5]);
  cas(c[1], c[4]); cas(c[3], c[6]);
  cas(c[1], c[2]); cas(c[3], c[4]); cas(c[5], c[6]);
}

// Sorts a bitonic sequence of 8 keys in descending order (half-cleaners).
__device__ __forceinline__ void clean8_desc(int (&m)[8]) {
  cas(m[0], m[4]); cas(m[1], m[5]); cas(m[2], m[6]); cas(m[3], m[7]);
  cas(m[0], m[2]); cas(m[1], m[3]); cas(m[4], m[6]); cas(m[5], m[7]);
  cas(m[0], m[1]); cas(m[2], m[3]); cas(m[4], m[5]); cas(m[6], m[7]);
}

// One comparator of a descending network whose min output is not needed.
__device__ __forceinline__ void cmax(int& a, int b) { a = max(a, b); }

// T <- top-8 of T and U (both sorted descending), sorted descending; with
// WANT9, L9 <- max(L9, 9th key of T and U).
// Without WANT9: the bitonic split (the maxima of T[i] and U[7 - i]) and a
// half-cleaner network sort the eight winners, 8 + 24 operations.
// With WANT9: Batcher's odd-even merge of the two lists (T on wires 0-7, U
// on wires 8-15; a comparator (i, j) leaves the max on wire i and the min on
// wire j) pruned to its nine leading outputs: comparators that feed none of
// them are dropped and those whose min feeds none keep only the max.  Wires
// 0-7 then hold the new T and wire 8 the 9th key, in 13 full and 7 one-sided
// comparators: 33 operations, against 44 for the split, the cleaner and a
// fold of the split's eight losers.
template <bool WANT9>
__device__ __forceinline__ void merge8(int (&T)[8], const int (&U)[8], int& L9) {
  if constexpr (WANT9) {
    int w[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      w[i] = T[i];
      w[8 + i] = U[i];
    }
    cas(w[0], w[8]);
    cmax(w[4], w[12]);
    cas(w[4], w[8]);
    cas(w[2], w[10]);
    cmax(w[6], w[14]);
    cmax(w[6], w[10]);
    cas(w[2], w[4]);
    cas(w[6], w[8]);
    cas(w[1], w[9]);
    cmax(w[5], w[13]);
    cas(w[5], w[9]);
    cas(w[3], w[11]);
    cmax(w[7], w[15]);
    cmax(w[7], w[11]);
    cas(w[3], w[5]);
    cmax(w[7], w[9]);
    cas(w[1], w[2]);
    cas(w[3], w[4]);
    cas(w[5], w[6]);
    cas(w[7], w[8]);
#pragma unroll
    for (int i = 0; i < 8; ++i) T[i] = w[i];
    L9 = max(L9, w[8]);
  } else {
    int mrg[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mrg[i] = max(T[i], U[7 - i]);
    clean8_desc(mrg);
#pragma unroll
    for (int i = 0; i < 8; ++i) T[i] = mrg[i];
  }
}

// True when the truncated-key top-8 T (descending; L9 the best key outside
// it, used when K == 8) may differ from the exact top-K: a leading key is not
// a positive finite float (zero, negative, NaN and +-inf all land here), or
// two of the K + 1 leading keys share their value bits.
template <int K, int IDX_BITS = 8>
__device__ __forceinline__ bool trunc_top8_uncertain(const int (&T)[8], int L9) {
  static_assert(K >= 1 && K <= 8, "truncated keys serve k <= 8");
  constexpr int VAL = (int)~((1u << IDX_BITS) - 1u);
  const int nxt = (K == 8) ? L9 : T[K < 8 ? K : 7];
  bool bad = (T[K - 1] < (1 << IDX_BITS)) || (T[0] >= 0x7F800000);
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const int b = (i + 1 < K) ? T[i + 1] : nxt;
    bad = bad || (b >= (T[i] & VAL));
  }
  return bad;
}

// ------------------------------------------------------ exact warp path
// Exact top-k of one row of E <= 32 * EPL logits, any k <= 32, by one warp:
// lane l holds experts [l * EPL, l * EPL + EPL); k rounds of a warp maximum
// over exact keys, the lowest lane (hence the lowest id) winning ties.
// Returns, in lane r < k, the id ranked r-th; -1 in the other lanes.
template <int EPL>
__device__ int warp_topk_exact(const float* row, int E, int k, int lane) {
  uint32_t key[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane * EPL + j;
    key[j] = e < E ? rank_key(row[e]) : 0u;
  }
  int myidx = -1;
  for (int r = 0; r < k; ++r) {
    uint32_t best = 0u;
    int bj = 0;
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (key[j] > best) {
        best = key[j];
        bj = j;
      }
    const uint32_t M = __reduce_max_sync(FULL, best);
    const unsigned bal = __ballot_sync(FULL, best == M);
    const int w = __ffs(bal) - 1;
    const int e = __shfl_sync(FULL, lane * EPL + bj, w);
    if (lane == w) {
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (j == bj) key[j] = 0u;
    }
    if (lane == r) myidx = e;
  }
  return myidx;
}

}  // namespace moer
