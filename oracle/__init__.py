"""Plain, slow CPU oracle of the MoE expert-routing statistics path.

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the
bench's CPU-baseline / reference leg load this package; the library never
does.  The arithmetic lives in `oracle.c` (plain C, double precision); this
module compiles it with gcc and marshals numpy arrays through ctypes.

Every function is pinned by `tests/test_oracle_pins.py` against brute force,
closed forms, invariants and library special cases; building with a mutant
number plants one deliberate mistake, which the pins must reject.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
N_MUTANTS = 10


def so_path(mutant: int = 0) -> str:
    return os.path.join(BUILD, "liboracle.so" if mutant == 0 else f"liboracle_m{mutant}.so")


def build(mutant: int = 0) -> str:
    os.makedirs(BUILD, exist_ok=True)
    out = so_path(mutant)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", f"-DORACLE_MUTANT={mutant}", "-o", out,
           os.path.join(HERE, "oracle.c"), "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


class Oracle:
    """ctypes view of one build of the oracle library."""

    def __init__(self, mutant: int = 0):
        path = so_path(mutant)
        src = os.path.join(HERE, "oracle.c")
        if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(src):
            build(mutant)
        lib = ctypes.CDLL(path)
        vp, i64, i32, f64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        sig = {
            "orc_topk": [vp, i64, i32, i32, vp],
            "orc_num_blocks": [vp, i32, i32],
            "orc_block_counts": [vp, i32, i64, i32, i32, vp, i32, i32, vp, i32, vp],
            "orc_stitch": [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp],
            "orc_signature": [vp, vp, i32, i32, vp],
            "orc_distances": [vp, vp, i32, i32, vp],
            "orc_sig_dist": [vp, i32, vp, i32, i32, vp, i32, vp, vp],
            "orc_route": [vp, i32, i32, f64, vp, i32, vp, vp],
            "orc_affinity": [vp, i32, i64, i32, i32, vp],
            "orc_loads": [vp, i32, i64, i32, i32, vp, i32, vp, vp, vp, vp],
            "orc_idf_fit": [vp, i32, i32, i32, vp],
            "orc_gate_logits": [vp, i64, i32, vp, i32, i32, vp],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ctypes.c_int64 if name == "orc_num_blocks" else None
        self.lib = lib

    # O1
    def topk(self, logits: np.ndarray, k: int) -> np.ndarray:
        x = _c(logits, np.float32)
        E = x.shape[-1]
        rows = x.size // E
        out = np.empty(x.shape[:-1] + (k,), dtype=np.uint8)
        self.lib.orc_topk(_p(x), rows, E, k, _p(out))
        return out

    def num_blocks(self, req_off, B: int) -> int:
        ro = _c(req_off, np.int32)
        return int(self.lib.orc_num_blocks(_p(ro), ro.shape[0] - 1, B))

    # O2
    def block_counts(self, topk, E: int, req_off, B: int, mask) -> np.ndarray:
        tk = _c(topk, np.uint8)
        L, T, k = tk.shape
        ro, mk = _c(req_off, np.int32), _c(mask, np.int32)
        nblk = self.num_blocks(ro, B)
        out = np.empty((nblk, mk.shape[0], E), dtype=np.uint8)
        self.lib.orc_block_counts(_p(tk), L, T, k, E, _p(ro), ro.shape[0] - 1, B, _p(mk),
                                  mk.shape[0], _p(out))
        return out

    # O3
    def stitch(self, blk_cnt, req_off, B: int, cache_idx, req_cache_off, cache, insert_slot):
        bc = _c(blk_cnt, np.uint8)
        _, m, E = bc.shape
        ro = _c(req_off, np.int32)
        R = ro.shape[0] - 1
        ci, rco = _c(cache_idx, np.int32), _c(req_cache_off, np.int32)
        ins = _c(insert_slot, np.int32) if insert_slot is not None else None
        assert cache.dtype == np.uint8 and cache.flags.c_contiguous
        out = np.empty((R, m, E), dtype=np.int32)
        self.lib.orc_stitch(_p(bc), _p(ro), R, B, m, E, _p(ci), _p(rco), _p(cache), _p(ins),
                            _p(out))
        return out

    # O4 + O5
    def signature(self, cnt, idf) -> np.ndarray:
        c, w = _c(cnt, np.int32), _c(idf, np.float32)
        m, E = w.shape
        out = np.empty(m * E, dtype=np.float64)
        self.lib.orc_signature(_p(c), _p(w), m, E, _p(out))
        return out

    def distances(self, s, centroids) -> np.ndarray:
        s, c = _c(s, np.float64), _c(centroids, np.float32)
        D, dim = c.shape
        out = np.empty(D, dtype=np.float64)
        self.lib.orc_distances(_p(s), _p(c), D, dim, _p(out))
        return out

    def sig_dist(self, req_cnt, idf, centroids):
        rc, w, c = _c(req_cnt, np.int32), _c(idf, np.float32), _c(centroids, np.float32)
        R = rc.shape[0]
        m, E = w.shape
        D = c.shape[0]
        sig = np.empty((R, m * E), dtype=np.float64)
        dist = np.empty((R, D), dtype=np.float64)
        self.lib.orc_sig_dist(_p(rc), R, _p(w), m, E, _p(c), D, _p(sig), _p(dist))
        return sig, dist

    # O6
    def route(self, dist, tau: float, loads, live: bool):
        d, ld = _c(dist, np.float64), _c(loads, np.int32)
        R, D = d.shape
        choice = np.empty(R, dtype=np.int32)
        out = np.empty(D, dtype=np.int32)
        self.lib.orc_route(_p(d), R, D, float(tau), _p(ld), int(bool(live)), _p(choice), _p(out))
        return choice, out

    # O7
    def affinity(self, topk, E: int) -> np.ndarray:
        tk = _c(topk, np.uint8)
        L, T, k = tk.shape
        out = np.empty((L, E, E), dtype=np.int64)
        self.lib.orc_affinity(_p(tk), L, T, k, E, _p(out))
        return out

    # O8
    def loads(self, topk, E: int, group_of, G: int):
        tk = _c(topk, np.uint8)
        L, T, k = tk.shape
        go = _c(group_of, np.int32)
        W = np.empty((L, E), dtype=np.int64)
        Wg = np.empty((L, G), dtype=np.int64)
        rg = np.empty(L, dtype=np.float64)
        re = np.empty(L, dtype=np.float64)
        self.lib.orc_loads(_p(tk), L, T, k, E, _p(go), G, _p(W), _p(Wg), _p(rg), _p(re))
        return W, Wg, rg, re

    # O9
    def idf_fit(self, req_cnt) -> np.ndarray:
        rc = _c(req_cnt, np.int32)
        R, m, E = rc.shape
        out = np.empty((m, E), dtype=np.float64)
        self.lib.orc_idf_fit(_p(rc), R, m, E, _p(out))
        return out

    # O10
    def gate_logits(self, hidden_bits, wgate_bits) -> np.ndarray:
        x, w = _c(hidden_bits, np.uint16), _c(wgate_bits, np.uint16)
        T, H = x.shape
        L, H2, E = w.shape
        assert H == H2
        out = np.empty((L, T, E), dtype=np.float32)
        self.lib.orc_gate_logits(_p(x), T, H, _p(w), L, E, _p(out))
        return out


_default = None


def get() -> Oracle:
    """The (unmutated) oracle, built on first use."""
    global _default
    if _default is None:
        _default = Oracle(0)
    return _default
