"""Full-size parity, complete, in the launch configuration the bench times.

c3 (Qwen3-30B-A3B shape, 1,000 requests, 1,305,533 tokens x 48 layers): every row's
top-k ids (62.7 M rows), every KV block's counts, all 48 co-activation matrices and the
loads, and every request's stitched counts, signature, distances and decoder choice,
against the oracle.  The GPU's outputs go to .npy files; spawned processes, one per host
core, each regenerate the logits of a range of requests with the host twin of the
generator, run the oracle over it and compare; the parent sums their co-activation and
load partials.  About a minute on 16 host cores.

c5 (the gate GEMM, 524,288 tokens x 48 layers, no logits output, as the bench runs it):
the fp64 gate oracle is ~400x slower per row than the top-k oracle, so every layer of the
first 16 requests (32,768 tokens, 1.57 M rows) is compared -- top-k identical wherever the
oracle's k-th/(k+1)-th margin exceeds 1e-3, ordered where every leading gap does, the
others counted -- and everything downstream of the ids over all 524,288 tokens (block
counts, co-activation, loads, request counts, signatures, distances, choices) against the
oracle applied to the GPU's own ids.
"""
import os
import shutil
import tempfile

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu

REL_TOL, ABS_FLOOR, BAND_EDGE, MARGIN = 1e-5, 1e-7, 1e-5, 1e-3


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import pipeline
    from tests import gpu_util
    return torch, pipeline, gpu_util


def _ncores():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def _pool_map(fn, tasks):
    """fn over tasks in spawned processes (this process holds a CUDA context)."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    with ProcessPoolExecutor(min(_ncores(), len(tasks)), mp_context=mp.get_context("spawn")) as ex:
        return list(ex.map(fn, tasks, timeout=1800))


def _route_checks(orc, rc, idf, centroids, tau, loads0, sig_g, dist_g, ch_g):
    """Oracle signatures, distances and static choices of these requests against the GPU's:
    (entries beyond tolerance, choices differing off the band edge, band-edge requests)."""
    sig, dist = orc.sig_dist(rc, idf, centroids)
    bad = int((np.abs(sig_g.astype(np.float64) - sig) > REL_TOL * np.abs(sig) + ABS_FLOOR).sum())
    bad += int((np.abs(dist_g.astype(np.float64) - dist) > REL_TOL * np.abs(dist) + ABS_FLOOR).sum())
    och, _ = orc.route(dist, tau, loads0, False)
    dmin = dist.min(axis=1, keepdims=True)
    edge = (np.abs(dist - (dmin + tau)) <= BAND_EDGE).any(axis=1)
    return bad, int(((och != ch_g) & ~edge).sum()), int(edge.sum())


def _c3_range(task):
    """Oracle over requests [r0, r1) of c3, four at a time, against the GPU's saved outputs."""
    r0, r1, tmp = task
    orc = oracle.get()
    wl = gen.make_workload("c3")
    meta = np.load(os.path.join(tmp, "meta.npz"))
    g_off, g_boff = meta["req_off"], meta["req_blk_off"]
    topk = np.load(os.path.join(tmp, "topk.npy"), mmap_mode="r")
    blk = np.load(os.path.join(tmp, "blk_cnt.npy"), mmap_mode="r")
    req = np.load(os.path.join(tmp, "req_cnt.npy"), mmap_mode="r")
    sig = np.load(os.path.join(tmp, "sig.npy"), mmap_mode="r")
    dist = np.load(os.path.join(tmp, "dist.npy"), mmap_mode="r")
    ch = np.load(os.path.join(tmp, "choice.npy"), mmap_mode="r")
    E, k, L, B, m = wl.E, wl.k, wl.L, wl.B, wl.m
    aff = np.zeros((L, E, E), dtype=np.int64)
    W = np.zeros((L, E), dtype=np.int64)
    Wg = np.zeros((L, wl.G), dtype=np.int64)
    out = {"rows": 0, "bad_rows": 0, "bad_blocks": 0, "bad_requests": 0, "bad_route_values": 0,
           "bad_choices": 0, "band_edge": 0}
    for a in range(r0, r1, 4):
        z = min(a + 4, r1)
        bb = wl.batch(a, z)
        tk = orc.topk(gen.host_logits(wl, bb.tok_key, bb.tok_dom), k)
        t0, t1 = int(g_off[a]), int(g_off[z])
        out["rows"] += L * (t1 - t0)
        out["bad_rows"] += int((tk != topk[:, t0:t1]).any(axis=2).sum())
        aff += orc.affinity(tk, E)
        w, wg, _, _ = orc.loads(tk, E, wl.group_of, wl.G)
        W += w
        Wg += wg
        bc = orc.block_counts(tk, E, bb.req_off, B, wl.mask)
        b0, b1 = int(g_boff[a]), int(g_boff[z])
        out["bad_blocks"] += int((bc != blk[b0:b1]).any(axis=(1, 2)).sum())
        rc = orc.stitch(bc, bb.req_off, B, np.zeros(0, np.int32), np.zeros(z - a + 1, np.int32),
                        np.zeros((1, m, E), np.uint8), np.full(bc.shape[0], -1, np.int32))
        out["bad_requests"] += int((rc != req[a:z]).any(axis=(1, 2)).sum())
        bad, badc, edge = _route_checks(orc, rc, wl.idf, wl.centroids, wl.tau, wl.loads0,
                                        sig[a:z], dist[a:z], ch[a:z])
        out["bad_route_values"] += bad
        out["bad_choices"] += badc
        out["band_edge"] += edge
    return out, aff.astype(np.int32), W, Wg


def test_qwen3_full_complete(env):
    torch, pipeline, gu = env
    wl = gen.make_workload("c3")
    b = wl.batch()
    bd = pipeline.BatchDev.from_host(b)
    rs = pipeline.RoutingStats.for_workload(wl, max_T=b.T, max_nblk=b.nblk, max_R=b.R)
    logits = gu.device_logits(wl, b)
    rs.step(logits, bd)  # the bench's calls: K1, block counts, stitch, loads, route
    torch.cuda.synchronize()
    assert rs.status() == 0
    del logits
    torch.cuda.empty_cache()
    tmp = tempfile.mkdtemp(prefix="moer_full_")
    try:
        np.save(os.path.join(tmp, "topk.npy"), gu.host(rs.topk_for(b.T)))
        np.save(os.path.join(tmp, "blk_cnt.npy"), gu.host(rs.blk_cnt[:b.nblk]))
        np.save(os.path.join(tmp, "req_cnt.npy"), gu.host(rs.req_cnt[:b.R]))
        np.save(os.path.join(tmp, "sig.npy"), gu.host(rs.sig[:b.R]))
        np.save(os.path.join(tmp, "dist.npy"), gu.host(rs.dist[:b.R]))
        np.save(os.path.join(tmp, "choice.npy"), gu.host(rs.choice[:b.R]))
        np.savez(os.path.join(tmp, "meta.npz"), req_off=b.req_off, req_blk_off=b.req_blk_off)
        cuts = np.linspace(0, b.R, 4 * _ncores() + 1).astype(int)
        res = _pool_map(_c3_range, [(int(a), int(z), tmp) for a, z in zip(cuts[:-1], cuts[1:]) if z > a])
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    tot = {key: sum(r[0][key] for r in res) for key in res[0][0]}
    print(f"c3 full, complete: {tot}")
    assert tot["rows"] == wl.L * b.T
    assert tot["bad_rows"] == 0, "top-k ids"
    assert tot["bad_blocks"] == 0, "block counts"
    assert tot["bad_requests"] == 0, "request counts"
    assert tot["bad_route_values"] == 0, "signatures and distances"
    assert tot["bad_choices"] == 0, "decoder choices off the band edge"
    A = sum(r[1].astype(np.int64) for r in res)
    assert np.array_equal(gu.host(rs.affinity).astype(np.int64), A), "co-activation, all layers"
    W = sum(r[2] for r in res)
    Wg = sum(r[3] for r in res)
    assert np.array_equal(gu.host(rs.W), W) and np.array_equal(gu.host(rs.Wg), Wg), "loads"


def _gate_rows(task):
    """The oracle's fp64 gate logits and top-k of tokens [t0, t1) of c5, every layer."""
    t0, t1 = task
    orc = oracle.get()
    wl = gen.make_workload("c5")
    x = gen.host_hidden(wl.seed, t0, t1 - t0, wl.hidden_dim)
    w = gen.host_wgate(wl.seed, wl.L, wl.hidden_dim, wl.E, wl.wgate_scale)
    ref = orc.gate_logits(x, w)
    srt = -np.sort(-ref.astype(np.float64), axis=-1)[..., :wl.k + 1]
    gaps = srt[..., :-1] - srt[..., 1:]
    return orc.topk(ref, wl.k), (gaps > MARGIN).all(axis=-1), gaps[..., wl.k - 1] > MARGIN


def test_gate_path_full_complete(env):
    torch, pipeline, gu = env
    orc = oracle.get()
    wl = gen.make_workload("c5")
    b = wl.batch()
    H, k, E, L = wl.hidden_dim, wl.k, wl.E, wl.L
    x = torch.empty((b.T, H), dtype=torch.int16, device="cuda")
    w = torch.empty((L, H, E), dtype=torch.int16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    gen.dev_hidden(wl.seed, b.T, H, x, st)
    gen.dev_wgate(wl.seed, L, H, E, wl.wgate_scale, w, st)
    rs = pipeline.RoutingStats.for_workload(wl, max_T=b.T, max_nblk=b.nblk, max_R=b.R)
    bd = pipeline.BatchDev.from_host(b)
    rs.ensure(b.T, b.nblk, b.R, H)
    # the bench's calls: the gate GEMM alone, then the counts from its ids
    rs.gate_topk(x, w, bd, counts=False)
    rs.ids_signature(bd, blk_counts=True, affinity=True)
    rs.block_stitch(bd)
    rs.affinity_load()
    rs.route(b.R)
    torch.cuda.synchronize()
    assert rs.status() == 0
    del x
    tk = gu.host(rs.topk_for(b.T))
    # every layer of the first 16 requests against the fp64 gate oracle
    ntok = 16 * 2048
    cuts = np.linspace(0, ntok, 2 * _ncores() + 1).astype(int)
    parts = _pool_map(_gate_rows, [(int(a), int(z)) for a, z in zip(cuts[:-1], cuts[1:])])
    otk = np.concatenate([p[0] for p in parts], axis=1)
    order_ok = np.concatenate([p[1] for p in parts], axis=1)
    set_ok = np.concatenate([p[2] for p in parts], axis=1)
    got = tk[:, :ntok]
    assert np.array_equal(got[order_ok], otk[order_ok]), "ordered top-k"
    assert np.array_equal(np.sort(got[set_ok], axis=1), np.sort(otk[set_ok], axis=1)), "top-k sets"
    amb = int((~set_ok).sum())
    differ = int((np.sort(got, axis=2) != np.sort(otk, axis=2)).any(axis=2).sum())
    print(f"c5 gate, {ntok} tokens x {L} layers: {amb} rows within the 1e-3 margin, {differ} of them differ")
    # everything downstream of the ids, all tokens, against the oracle on the GPU's own ids
    assert np.array_equal(gu.host(rs.blk_cnt[:b.nblk]), orc.block_counts(tk, E, b.req_off, wl.B, wl.mask))
    assert np.array_equal(gu.host(rs.affinity).astype(np.int64), orc.affinity(tk, E))
    W, Wg, rg, re = orc.loads(tk, E, wl.group_of, wl.G)
    assert np.array_equal(gu.host(rs.W), W) and np.array_equal(gu.host(rs.Wg), Wg)
    assert np.array_equal(gu.host(rs.rho_g), rg) and np.array_equal(gu.host(rs.rho_e), re)
    nb = b.nblk
    rc = orc.stitch(orc.block_counts(tk, E, b.req_off, wl.B, wl.mask), b.req_off, wl.B,
                    np.zeros(0, np.int32), np.zeros(b.R + 1, np.int32), np.zeros((1, wl.m, E), np.uint8),
                    np.full(nb, -1, np.int32))
    assert np.array_equal(gu.host(rs.req_cnt[:b.R]), rc)
    bad, badc, edge = _route_checks(orc, rc, wl.idf, wl.centroids, wl.tau, wl.loads0,
                                    gu.host(rs.sig[:b.R]), gu.host(rs.dist[:b.R]), gu.host(rs.choice[:b.R]))
    assert bad == 0 and badc == 0, (bad, badc, edge)
