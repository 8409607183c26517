"""Full-size workloads in the launch configuration the bench times (the c3 and c5 steps are
compared completely in test_gpu_fullsize_complete.py).

The oracle cannot redo these workloads' rows in seconds, so these tests compare
  * sampled rows (top-k ids) and sampled requests (stitched counts,
    signatures, distances) one by one against the oracle,
  * one whole mask layer (block counts and co-activation) against the oracle,
  * properties that hold at any size on everything else: co-activation
    symmetric with diagonal = loads and row sums = k * loads, every block's
    counts summing to k * len, every live pick valid for the band and loads.
"""
import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import pipeline
    from tests import gpu_util
    return torch, pipeline, gpu_util


def _check_affinity_props(A, W, k, T):
    A = A.astype(np.int64)
    assert np.array_equal(A, A.transpose(0, 2, 1))
    assert np.array_equal(np.diagonal(A, axis1=1, axis2=2), W)
    assert np.array_equal(A.sum(axis=2), k * W)
    assert (W.sum(axis=1) == k * T).all()


def test_deepseek_full(env):
    """The E = 64, k = 6 shape at full size (two 32-expert slices per tile in
    the logits pass): sampled rows, one whole mask layer, invariants everywhere."""
    torch, pipeline, gu = env
    orc = oracle.get()
    wl = gen.make_workload("c2")
    b = wl.batch()
    bd = pipeline.BatchDev.from_host(b)
    logits = gu.device_logits(wl, b)
    rs = pipeline.RoutingStats.for_workload(wl, max_T=b.T, max_nblk=b.nblk, max_R=b.R)
    rs.step(logits, bd)
    torch.cuda.synchronize()
    assert rs.status() == 0
    del logits
    topk = gu.host(rs.topk_for(b.T))
    rng = np.random.RandomState(2)
    layers = rng.randint(0, wl.L, size=4000)
    toks = rng.randint(0, b.T, size=4000)
    rows = gen.host_logit_rows(wl, b.tok_key, b.tok_dom, layers, toks)
    assert np.array_equal(topk[layers, toks], orc.topk(rows, wl.k))
    li = int(rng.randint(0, wl.m))
    layer = int(wl.mask[li])
    lrows = gen.host_logit_rows(wl, b.tok_key, b.tok_dom, np.full(b.T, layer, np.int32),
                                np.arange(b.T))
    tk_l = orc.topk(lrows, wl.k)
    assert np.array_equal(topk[layer], tk_l)
    bc = orc.block_counts(tk_l[None], wl.E, b.req_off, wl.B, np.array([0], np.int32))
    assert np.array_equal(gu.host(rs.blk_cnt[:b.nblk, li]), bc[:, 0])
    A = gu.host(rs.affinity)
    assert np.array_equal(A[layer].astype(np.int64), orc.affinity(tk_l[None], wl.E)[0])
    _check_affinity_props(A, gu.host(rs.W), wl.k, b.T)


def test_online_stream_full(env):
    torch, pipeline, gu = env
    orc = oracle.get()
    wl = gen.make_workload("c4")
    chunks = wl.chunks(300_000)
    cap_T = max(sum(wl.computed_tokens(r) for r in range(a, z)) for a, z in chunks)
    rs = pipeline.RoutingStats.for_workload(wl, max_T=cap_T, max_nblk=cap_T // 8 + 64,
                                            max_R=max(z - a for a, z in chunks))
    flat = torch.empty(wl.L * cap_T * wl.E, dtype=torch.float32, device="cuda")
    rng = np.random.RandomState(2)
    reused = np.flatnonzero(wl.cached_blocks > 0)
    picks = set(rng.choice(reused, size=10, replace=False)) | set(rng.choice(wl.R, size=6, replace=False))
    choices, dists = [], []
    total_T = 0
    got_cnt = {}
    for a, z in chunks:
        b = wl.batch(a, z)
        bd = pipeline.BatchDev.from_host(b)
        view = flat[:wl.L * b.T * wl.E].view(wl.L, b.T, wl.E)
        gu.device_logits(wl, b, out=view)
        rs.step(view, bd, write_topk=False)
        choices.append(gu.host(rs.choice[:b.R]))
        dists.append(gu.host(rs.dist[:b.R]))
        total_T += b.T
        lens = b.blk_tab[:, 1].astype(np.int64)
        assert (gu.host(rs.blk_cnt[:b.nblk]).sum(axis=2, dtype=np.int64) == (wl.k * lens)[:, None]).all()
        req = gu.host(rs.req_cnt[:b.R])
        for r in range(a, z):
            if r in picks:
                got_cnt[r] = req[r - a].copy()
    torch.cuda.synchronize()
    assert rs.status() == 0
    # stitched counts of sampled requests equal the full prompt's counts (cached prefix included)
    for r, cnt in got_cnt.items():
        keys = wl.prompt_keys(r)
        doms = np.full(len(keys), wl.dom[r], np.int32)
        ref = np.zeros((wl.m, wl.E), dtype=np.int32)
        for i, lyr in enumerate(wl.mask):
            rr = gen.host_logit_rows(wl, keys, doms, np.full(len(keys), lyr, np.int32),
                                     np.arange(len(keys)))
            ref[i] = np.bincount(orc.topk(rr, wl.k).reshape(-1), minlength=wl.E)
        assert np.array_equal(cnt, ref), r
    A = gu.host(rs.affinity)
    _check_affinity_props(A, gu.host(rs.W), wl.k, total_T)
    # live routing: every pick valid for the band and the loads at its turn
    ch = np.concatenate(choices)
    dist = np.concatenate(dists).astype(np.float64)
    loads = wl.loads0.astype(np.int64).copy()
    for r in range(wl.R):
        assert gu.valid_choice(int(ch[r]), dist[r], wl.tau, loads), r
        loads[ch[r]] += 1
    assert np.array_equal(gu.host(rs.loads), loads)
