"""The comparator networks of the top-k kernels (rank.cuh), on the CPU.

The section of rank.cuh that holds the integer comparator networks is plain
C++ apart from its function qualifiers.  This test compiles that section with
g++ (qualifiers defined away, min/max from the standard library) and checks:
  - sort8_desc sorts every one of the 256 inputs of 0s and 1s, which by the
    0-1 principle makes it a sorting network for all inputs;
  - merge8<true> (Batcher's odd-even merge pruned to its nine leading
    outputs) gives the top 8 of two sorted lists and the 9th for every pair of
    sorted 0/1 lists (again the 0-1 principle), and the running 9th key as the
    maximum of the old one and that 9th;
  - merge8<false> (bitonic split and cleaner) gives the top 8 for the same
    inputs;
  - both merges agree with a plain sort on random lists, ties included;
  - trunc_top8_uncertain (7 index bits, as the gate's epilogue uses it) agrees
    with its definition on random sorted keys, close values and negatives
    included.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
RANK = os.path.join(os.path.dirname(HERE), "moe_expert_routing_top_gb300", "csrc", "rank.cuh")
BEGIN = "// ---------------------------------------------------- comparator networks"
END = "// ------------------------------------------------------ exact warp path"

PRE = r"""
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstdio>
#include <random>
#define __device__
#define __forceinline__ inline
using std::max;
using std::min;
static inline uint32_t __vimin3_u32(uint32_t a, uint32_t b, uint32_t c) { return std::min(a, std::min(b, c)); }
"""

DRIVER = r"""
#define CHECK(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

static void sorted_desc(int* v, int n) { std::sort(v, v + n, [](int a, int b) { return a > b; }); }

int main() {
  // sort8_desc on all 0/1 inputs
  for (int m = 0; m < 256; ++m) {
    int c[8];
    for (int i = 0; i < 8; ++i) c[i] = (m >> i) & 1;
    int r[8];
    std::copy(c, c + 8, r);
    sorted_desc(r, 8);
    sort8_desc(c);
    for (int i = 0; i < 8; ++i) CHECK(c[i] == r[i]);
  }
  // both merges on all pairs of sorted 0/1 lists (a ones in T, b ones in U)
  for (int a = 0; a <= 8; ++a)
    for (int b = 0; b <= 8; ++b) {
      int T[8], U[8], all[16];
      for (int i = 0; i < 8; ++i) {
        T[i] = i < a;
        U[i] = i < b;
        all[i] = T[i];
        all[8 + i] = U[i];
      }
      sorted_desc(all, 16);
      for (int l9 : {INT_MIN, 0, 1}) {
        int T9[8], Tb[8];
        std::copy(T, T + 8, T9);
        std::copy(T, T + 8, Tb);
        int L9 = l9, Lb = l9;
        merge8<true>(T9, U, L9);
        merge8<false>(Tb, U, Lb);
        for (int i = 0; i < 8; ++i) CHECK(T9[i] == all[i] && Tb[i] == all[i]);
        CHECK(L9 == std::max(l9, all[8]));
        CHECK(Lb == l9);
      }
    }
  // random lists, ties included
  std::mt19937 rng(12345);
  for (int it = 0; it < 200000; ++it) {
    int v[16];
    const int mode = it % 3;
    for (int i = 0; i < 16; ++i)
      v[i] = mode == 0 ? (int)rng() : (mode == 1 ? (int)(rng() % 5) - 2 : (int)(rng() >> 8));
    int T[8], U[8], all[16];
    std::copy(v, v + 8, T);
    std::copy(v + 8, v + 16, U);
    std::copy(v, v + 16, all);
    sort8_desc(T);
    sort8_desc(U);
    sorted_desc(all, 16);
    int T9[8], Tb[8];
    std::copy(T, T + 8, T9);
    std::copy(T, T + 8, Tb);
    const int l9 = (it % 7 == 0) ? INT_MIN : (int)rng();
    int L9 = l9, Lb = l9;
    merge8<true>(T9, U, L9);
    merge8<false>(Tb, U, Lb);
    for (int i = 0; i < 8; ++i) CHECK(T9[i] == all[i] && Tb[i] == all[i]);
    CHECK(L9 == std::max(l9, all[8]));
  }
  // certification against its definition (a leading key not a positive finite
  // float, or a key at or above its predecessor's value bits)
  for (int it = 0; it < 400000; ++it) {
    int v[16];
    const int mode = it % 4;
    for (int i = 0; i < 16; ++i) {
      const int base = mode == 0 ? (int)rng() : (mode == 1 ? 0x3F800000 + (int)(rng() % 4096) : (int)(rng() % 1024) - 256);
      v[i] = base;
    }
    // distinct keys: the low 7 bits carry a position
    for (int i = 0; i < 16; ++i) v[i] = (int)(((uint32_t)v[i] & ~127u) | (uint32_t)i);
    sorted_desc(v, 16);
    int T[8];
    std::copy(v, v + 8, T);
    const int L9 = v[8];
    for (int K : {6, 8}) {
      const int nxt = K == 8 ? L9 : T[K];
      bool ref = (T[K - 1] < (1 << 7)) || (T[0] >= 0x7F800000);
      for (int i = 0; i < K; ++i) {
        const int b = i + 1 < K ? T[i + 1] : nxt;
        ref = ref || (b >= (int)((uint32_t)T[i] & ~127u));
      }
      const bool got = K == 8 ? trunc_top8_uncertain<8, 7>(T, L9) : trunc_top8_uncertain<6, 7>(T, L9);
      CHECK(got == ref);
    }
  }
  std::printf("OK\n");
  return 0;
}
"""


def test_rank_networks(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    text = open(RANK).read()
    assert BEGIN in text and END in text, "rank.cuh section markers moved"
    section = text[text.index(BEGIN):text.index(END)]
    src = tmp_path / "networks.cpp"
    src.write_text(PRE + "namespace moer {\n" + section + "}  // namespace moer\nusing namespace moer;\n" + DRIVER)
    exe = tmp_path / "networks"
    r = subprocess.run([gxx, "-std=c++17", "-O2", str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr
