"""Pins of the CPU oracle against things other than itself.

Each `pin_*` function takes an `oracle.Oracle` and raises AssertionError if
the oracle disagrees with brute force, a library routine, a closed form or an
invariant that the definitions on the pages fix.  `test_oracle_pins.py` runs
them on the real oracle; `test_oracle_mutants.py` runs them on deliberately
broken builds and requires each break to be caught.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

import gen


# ----------------------------------------------------------------- helpers
def _specials_rows(rs, rows, E):
    x = rs.randint(-3, 4, size=(rows, E)).astype(np.float32)
    sp = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0], dtype=np.float32)
    hit = rs.random_sample((rows, E)) < 0.25
    x[hit] = sp[rs.randint(0, len(sp), size=int(hit.sum()))]
    return x


def _outranks(xa, a, xb, b):
    na, nb = math.isnan(xa), math.isnan(xb)
    if na != nb:
        return nb
    if not na and xa != xb:
        return xa > xb
    return a < b


def _brute_topk(x, k):
    E = len(x)
    found = []
    for S in itertools.combinations(range(E), k):
        rest = [b for b in range(E) if b not in S]
        if all(_outranks(x[a], a, x[b], b) for a in S for b in rest):
            found.append(S)
    assert len(found) == 1, "the top-k set must be unique"
    S = found[0]
    beaten = {a: sum(_outranks(x[b], b, x[a], a) for b in S if b != a) for a in S}
    return [a for a in sorted(S, key=lambda a: beaten[a])]


def _small_workload(prefix=False):
    lengths = [20, 35, 40, 70, 18, 50, 33, 64, 17, 1, 16, 32]
    return gen.make_custom(16, 4, 5, lengths, B=16, mask=[0, 2, 3], ndom=2, D=4,
                           prefix_frac=0.8 if prefix else 0.0, seed=777)


# -------------------------------------------------------------------- pins
def pin_topk_bruteforce(orc):
    """O1 equals exhaustive k-subset enumeration on tie-heavy tiny rows."""
    rs = np.random.RandomState(11)
    for E in (1, 3, 5, 8):
        x = _specials_rows(rs, 12, E)
        for k in range(1, E + 1):
            got = orc.topk(x, k)
            for r in range(x.shape[0]):
                assert list(got[r]) == _brute_topk(list(map(float, x[r])), k), (x[r], k, got[r])


def pin_topk_library(orc):
    """O1 equals numpy's stable argsort of the negated logits (same total order)."""
    rs = np.random.RandomState(12)
    for E, rows in ((64, 300), (128, 200), (33, 100)):
        x = _specials_rows(rs, rows, E)
        x[: rows // 2] = rs.standard_normal((rows // 2, E)).astype(np.float32)
        ref = np.argsort(-x, axis=1, kind="stable")
        for k in (1, 6, 8, E):
            assert np.array_equal(orc.topk(x, k), ref[:, :k].astype(np.uint8))


def _wl_topk(orc, wl, batch):
    logits = gen.host_logits(wl, batch.tok_key, batch.tok_dom)
    return orc.topk(logits, wl.k)


def pin_block_counts(orc):
    """O2: each block's counts sum to k*len; blocks of a request sum to its direct count."""
    wl = _small_workload()
    b = wl.batch()
    tk = _wl_topk(orc, wl, b)
    cnt = orc.block_counts(tk, wl.E, b.req_off, wl.B, wl.mask)
    assert cnt.shape == (b.nblk, wl.m, wl.E)
    lens = b.blk_tab[:, 1].astype(np.int64)
    assert np.array_equal(cnt.sum(axis=2, dtype=np.int64), np.repeat(lens[:, None] * wl.k, wl.m, 1))
    for r in range(b.R):
        t0, t1 = b.req_off[r], b.req_off[r + 1]
        blks = cnt[b.req_blk_off[r]:b.req_blk_off[r + 1]].sum(axis=0, dtype=np.int64)
        for i, layer in enumerate(wl.mask):
            direct = np.bincount(tk[layer, t0:t1].reshape(-1), minlength=wl.E)
            assert np.array_equal(blks[i], direct)


def pin_stitch(orc):
    """O3: stitched request counts equal the counts of the full prompt, over two batches."""
    wl = _small_workload(prefix=True)
    assert (wl.cached_blocks > 0).any()
    cache = np.zeros((max(wl.nslots, 1), wl.m, wl.E), dtype=np.uint8)
    half = wl.R // 2
    for r0, r1 in ((0, half), (half, wl.R)):
        b = wl.batch(r0, r1)
        tk = _wl_topk(orc, wl, b)
        cnt = orc.block_counts(tk, wl.E, b.req_off, wl.B, wl.mask)
        req = orc.stitch(cnt, b.req_off, wl.B, b.cache_idx, b.req_cache_off, cache, b.insert_slot)
        for i, r in enumerate(range(r0, r1)):
            keys = wl.prompt_keys(r)
            logits = gen.host_logits(wl, keys, np.full(len(keys), wl.dom[r], np.int32))
            full = orc.topk(logits, wl.k)
            for j, layer in enumerate(wl.mask):
                direct = np.bincount(full[layer].reshape(-1), minlength=wl.E)
                assert np.array_equal(req[i, j], direct), (r, j)
        full_blocks = b.insert_slot >= 0
        assert np.array_equal(cache[b.insert_slot[full_blocks]], cnt[full_blocks])


def pin_signature(orc):
    """O4: unit norm, invariance to scaling idf, one-token indicator / sqrt(m k), zero -> zero."""
    rs = np.random.RandomState(13)
    m, E, k = 3, 16, 4
    cnt = rs.randint(0, 9, size=(m, E)).astype(np.int32)
    idf = (1 + rs.random_sample((m, E))).astype(np.float32)
    s = orc.signature(cnt, idf)
    assert abs(np.sqrt(np.dot(s, s)) - 1.0) < 1e-12
    s2 = orc.signature(cnt, (idf * 4).astype(np.float32))
    assert np.allclose(s, s2, rtol=0, atol=1e-15)
    one = np.zeros((m, E), dtype=np.int32)
    for i in range(m):
        one[i, rs.choice(E, k, replace=False)] = 1
    s1 = orc.signature(one, np.ones((m, E), dtype=np.float32))
    assert np.allclose(s1, one.reshape(-1) / math.sqrt(m * k), rtol=0, atol=1e-15)
    assert not orc.signature(np.zeros((m, E), np.int32), idf).any()


def pin_distance(orc):
    """O5: d^2 = |s|^2 + |c|^2 - 2 s.c, and d(s, s) = 0."""
    rs = np.random.RandomState(14)
    dim, D = 48, 5
    s = rs.standard_normal(dim)
    c = rs.standard_normal((D, dim)).astype(np.float32)
    d = orc.distances(s, c)
    c64 = c.astype(np.float64)
    closed = np.sqrt(np.dot(s, s) + np.einsum("ij,ij->i", c64, c64) - 2 * c64 @ s)
    assert np.allclose(d, closed, rtol=1e-12, atol=1e-12)
    s32 = rs.standard_normal(dim).astype(np.float32)
    assert orc.distances(s32.astype(np.float64), s32[None, :])[0] == 0.0


def pin_route(orc):
    """O6: choice in band and least loaded there; tau=0 -> nearest; tau=inf -> JSQ; live loads."""
    rs = np.random.RandomState(15)
    R, D = 400, 7
    dist = rs.random_sample((R, D)) * 0.5
    loads = rs.randint(0, 5, size=D).astype(np.int32)
    for tau in (0.0, 0.05, 0.1, 0.3):
        ch, out = orc.route(dist, tau, loads, live=False)
        assert np.array_equal(out, loads)
        dmin = dist.min(axis=1)
        inband = dist <= (dmin + tau)[:, None]
        assert inband[np.arange(R), ch].all()
        masked = np.where(inband, loads[None, :], np.iinfo(np.int32).max)
        assert np.array_equal(ch, np.argmin(masked, axis=1))
        if tau == 0.0:
            assert np.array_equal(ch, np.argmin(dist, axis=1))
    ch, _ = orc.route(dist, 1e300, loads, live=False)
    assert np.array_equal(ch, np.full(R, np.argmin(loads)))
    ch, out = orc.route(dist, 0.1, loads, live=True)
    assert np.array_equal(out, loads + np.bincount(ch, minlength=D))
    cur = loads.copy()
    for r in range(R):
        band = np.flatnonzero(dist[r] <= dist[r].min() + 0.1)
        assert ch[r] in band and cur[ch[r]] == cur[band].min()
        assert ch[r] == band[np.argmin(cur[band])]
        cur[ch[r]] += 1
    # undefined distances: a NaN is outside the band and does not define d_min (numpy's
    # nanmin); a request without any finite distance gets -1 and leaves every load alone
    dn = dist[:6].copy()
    dn[0, 0] = np.nan                      # NaN first: d_min from the other six
    dn[1, 3] = np.nan
    dn[2, :] = np.nan                      # no finite distance
    dn[3, :] = np.inf                      # all infinite: every decoder is in the band
    for live in (False, True):
        ch, out = orc.route(dn, 0.1, loads, live=live)
        cur = loads.copy()
        for r in range(6):
            if r == 2:
                assert ch[r] == -1
                continue
            with np.errstate(invalid="ignore"):
                band = np.flatnonzero(dn[r] <= np.nanmin(dn[r]) + 0.1)
            assert ch[r] == band[np.argmin(cur[band])]
            if live:
                cur[ch[r]] += 1
        assert np.array_equal(out, cur)
    assert orc.route(dn[3:4], 0.1, loads, live=False)[0][0] == np.argmin(loads)


def pin_affinity(orc):
    """O7: A = X^T X (X the one-hot selection matrix); symmetric; diagonal = loads."""
    rs = np.random.RandomState(16)
    L, T, E, k = 3, 257, 16, 4
    tk = np.stack([np.stack([rs.choice(E, k, replace=False) for _ in range(T)])
                   for _ in range(L)]).astype(np.uint8)
    A = orc.affinity(tk, E)
    W, _, _, _ = orc.loads(tk, E, np.zeros((L, E), np.int32), 1)
    for l in range(L):
        X = np.zeros((T, E), dtype=np.int64)
        X[np.repeat(np.arange(T), k), tk[l].reshape(-1)] = 1
        assert np.array_equal(A[l], X.T @ X)
        assert np.array_equal(A[l], A[l].T)
        assert np.array_equal(np.diag(A[l]), W[l])
        assert np.array_equal(A[l].sum(axis=1), k * W[l])
    assert A.sum() == L * k * k * T


def pin_loads(orc):
    """O8: sums, rho >= 1, uniform -> 1, a hand example with an empty group, empty layer -> 0."""
    rs = np.random.RandomState(17)
    L, T, E, k, G = 2, 300, 16, 4, 4
    tk = np.stack([np.stack([rs.choice(E, k, replace=False) for _ in range(T)])
                   for _ in range(L)]).astype(np.uint8)
    go = np.stack([rs.permutation(np.arange(E) % G) for _ in range(L)]).astype(np.int32)
    W, Wg, rg, re = orc.loads(tk, E, go, G)
    assert (W.sum(axis=1) == k * T).all() and (Wg.sum(axis=1) == k * T).all()
    assert (rg >= 1).all() and (re >= 1).all()
    for l in range(L):
        assert np.array_equal(Wg[l], np.bincount(go[l], weights=W[l], minlength=G).astype(np.int64))
    # uniform: every expert picked equally often
    uni = np.array([[(np.arange(k) + k * t) % E for t in range(E)]], dtype=np.uint8)
    _, _, rg1, re1 = orc.loads(uni, E, (np.arange(E)[None, :] * G // E).astype(np.int32), G)
    assert rg1[0] == 1.0 and re1[0] == 1.0
    # hand example: E=4, G=4, k=1; tokens pick 0,0,0,1 -> group loads 3,1,0,0
    hand = np.array([[[0], [0], [0], [1]]], dtype=np.uint8)
    W, Wg, rg, re = orc.loads(hand, 4, np.array([[0, 1, 2, 3]], np.int32), 4)
    assert list(Wg[0]) == [3, 1, 0, 0]
    assert rg[0] == 3.0 / (4.0 / 4.0) and re[0] == 3.0
    _, _, rg0, _ = orc.loads(np.zeros((1, 0, 1), np.uint8), 4, np.zeros((1, 4), np.int32), 2)
    assert rg0[0] == 0.0


def pin_idf(orc):
    """O9: df = 0 -> ln(1+N)+1, df = N -> 1, a hand example."""
    N, m, E = 3, 1, 3
    cnt = np.zeros((N, m, E), dtype=np.int32)
    cnt[:, 0, 1] = 5            # term 1 in every request
    cnt[0, 0, 2] = 2            # term 2 in one request
    idf = orc.idf_fit(cnt)
    assert abs(idf[0, 0] - (math.log(4.0) + 1)) < 1e-15
    assert idf[0, 1] == 1.0
    assert abs(idf[0, 2] - (math.log(2.0) + 1)) < 1e-15


def pin_gate(orc):
    """O10: equals a float64 library matmul of the bf16 operands, rounded to fp32 (<= 1 ulp)."""
    T, H, L, E = 7, 96, 2, 16
    x = gen.host_hidden(99, 0, T, H)
    w = gen.host_wgate(99, L, H, E, 0.02)
    got = orc.gate_logits(x, w)

    def f(b):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    ref = np.stack([f(x) @ f(w[l]) for l in range(L)]).astype(np.float32)
    ulp = np.spacing(np.abs(ref))
    assert (np.abs(got.astype(np.float64) - ref) <= ulp).all()


ALL_PINS = [pin_topk_bruteforce, pin_topk_library, pin_block_counts, pin_stitch,
            pin_signature, pin_distance, pin_route, pin_affinity, pin_loads, pin_idf, pin_gate]
