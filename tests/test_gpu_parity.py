"""GPU path (through the C ABI) against the CPU oracle, element by element.

Each workload is run at a size the oracle finishes in seconds, with enough
tokens to span many tiles and a ragged last tile; the streaming workload runs
in several chunks so the signature cache and live loads carry across calls.
"""
import numpy as np
import pytest

import gen
import oracle
from oracle import replication as rp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import pipeline
    from tests import gpu_util
    return torch, pipeline, gpu_util


def test_generator_device_matches_host_twin(env):
    torch, _, gu = env
    wl = gen.make_workload("c1")
    b = wl.batch()
    dev = gu.host(gu.device_logits(wl, b))
    ref = gen.host_logits(wl, b.tok_key, b.tok_dom)
    assert np.array_equal(dev.view(np.uint32), ref.view(np.uint32))


CASES = [("c1", None, 1), ("c2", 48, 1), ("c3", 14, 1), ("c4", 60, 3), ("c5", 3, 1)]


@pytest.mark.parametrize("cfg,R,nchunks", CASES, ids=[c[0] for c in CASES])
def test_path_parity(env, cfg, R, nchunks):
    torch, pipeline, gu = env
    orc = oracle.get()
    wl = gen.make_workload(cfg, R=R)
    total = sum(wl.computed_tokens(r) for r in range(wl.R))
    chunks = wl.chunks(-(-total // nchunks))
    bounds = [wl.batch(a, z) for a, z in chunks]
    rs = pipeline.RoutingStats.for_workload(
        wl, max_T=max(b.T for b in bounds), max_nblk=max(b.nblk for b in bounds),
        max_R=max(b.R for b in bounds))
    cache = np.zeros((max(wl.nslots, 1), wl.m, wl.E), dtype=np.uint8)
    loads = wl.loads0.copy()
    topk_all = []
    edge_total = diff_total = 0
    for b in bounds:
        bd = pipeline.BatchDev.from_host(b)
        logits = gu.device_logits(wl, b)
        rs.step(logits, bd)
        torch.cuda.synchronize()
        assert rs.status() == 0
        lh = gen.host_logits(wl, b.tok_key, b.tok_dom)
        tk = orc.topk(lh, wl.k)
        assert np.array_equal(gu.host(rs.topk_for(b.T)), tk), "top-k ids"
        topk_all.append(tk)
        bc = orc.block_counts(tk, wl.E, b.req_off, wl.B, wl.mask)
        assert np.array_equal(gu.host(rs.blk_cnt[:b.nblk]), bc), "block counts"
        rc = orc.stitch(bc, b.req_off, wl.B, b.cache_idx, b.req_cache_off, cache, b.insert_slot)
        assert np.array_equal(gu.host(rs.req_cnt[:b.R]), rc), "request counts"
        if wl.nslots:
            assert np.array_equal(gu.host(rs.cache), cache[:wl.nslots]), "signature cache"
        tka = np.concatenate(topk_all, axis=1)
        A = orc.affinity(tka, wl.E)
        assert np.array_equal(gu.host(rs.affinity).astype(np.int64), A), "affinity"
        W, Wg, rg, re = orc.loads(tka, wl.E, wl.group_of, wl.G)
        assert np.array_equal(gu.host(rs.W), W) and np.array_equal(gu.host(rs.Wg), Wg)
        assert np.array_equal(gu.host(rs.rho_g), rg) and np.array_equal(gu.host(rs.rho_e), re)
        rs.replication_plan()
        pn, psrc, phot, pdst, pwp = rp.plan(W, wl.group_of, wl.G)
        assert np.array_equal(gu.host(rs.n_rep), pn) and np.array_equal(gu.host(rs.rep_src), psrc)
        assert np.array_equal(gu.host(rs.hot), phot) and np.array_equal(gu.host(rs.rep_dst), pdst)
        assert np.array_equal(gu.host(rs.w_pred), pwp), "replication plan"
        sig, dist = orc.sig_dist(rc, wl.idf, wl.centroids)
        gu.assert_close(gu.host(rs.sig[:b.R]), sig, "signature")
        gu.assert_close(gu.host(rs.dist[:b.R]), dist, "distance")
        och, oloads = orc.route(dist, wl.tau, loads, wl.live)
        ch = gu.host(rs.choice[:b.R])
        if wl.live:
            e, d = gu.check_live_route(ch, dist, wl.tau, loads, och)
            loads = loads + np.bincount(ch, minlength=wl.D).astype(np.int32)
            assert np.array_equal(gu.host(rs.loads), loads)
        else:
            e, d = gu.check_static_route(ch, dist, wl.tau, loads, och)
            assert np.array_equal(gu.host(rs.loads), wl.loads0)
        edge_total += e
        diff_total += d
    print(f"{cfg}: band-edge requests {edge_total}, differing choices {diff_total}")


def test_idf_fit_parity(env):
    torch, _, gu = env
    from moe_expert_routing_top_gb300 import _native as nat
    orc = oracle.get()
    wl = gen.make_workload("c2", R=200)
    rs_ = np.random.RandomState(5)
    cnt = (rs_.poisson(0.4, size=(wl.R, wl.m, wl.E))).astype(np.int32)
    dims = nat.make_dims(wl.E, wl.k, wl.L, wl.mask, wl.B)
    dc = torch.from_numpy(cnt).cuda()
    out = torch.empty((wl.m, wl.E), dtype=torch.float32, device="cuda")
    nat.moer_idf_fit(dims, dc, wl.R, out)
    ref = orc.idf_fit(cnt)
    assert np.array_equal(gu.host(out), ref.astype(np.float32))
