"""The whole path from hidden states: gate GEMM (moer_gate_topk) -> stitch ->
loads -> route, on the gate workload (E=128, k=8, L=48, H=2048, requests of
2,048 tokens) against the oracle.

Reduced size (two requests, 4,096 tokens, 1,536 GEMM tiles over the grid):
the oracle's fp64 gate logits give the reference top-k; the GPU's ids must
equal it wherever the k+1 leading logits are separated by more than 1e-3,
and the downstream results (block counts, stitched counts, co-activation,
loads, signatures, distances, choices) are compared with the oracle's chain
from its own ids -- exactly where no row of the request / layer differs,
within the bound a differing row can move them otherwise.

Full size (256 requests, 524,288 tokens, the bench's launch configuration):
sampled tokens' ids against the oracle, and properties that hold at any size.
"""
import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu

MARGIN = 1e-3


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import pipeline
    from tests import gpu_util
    return torch, pipeline, gpu_util


def _device_inputs(torch, wl, T):
    H = wl.hidden_dim
    x = torch.empty((T, H), dtype=torch.int16, device="cuda")
    w = torch.empty((wl.L, H, wl.E), dtype=torch.int16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    gen.dev_hidden(wl.seed, T, H, x, st)
    gen.dev_wgate(wl.seed, wl.L, H, wl.E, wl.wgate_scale, w, st)
    return x, w


def _margins(ref, k):
    srt = -np.sort(-ref.astype(np.float64), axis=-1)[..., :k + 1]
    gaps = srt[..., :-1] - srt[..., 1:]
    return (gaps > MARGIN).all(axis=-1), gaps[..., k - 1] > MARGIN


def test_gate_path_reduced(env):
    torch, pipeline, gu = env
    orc = oracle.get()
    wl = gen.make_workload("c5", R=2)
    b = wl.batch()
    H, k, E = wl.hidden_dim, wl.k, wl.E
    dx, dw = _device_inputs(torch, wl, b.T)
    x = gen.host_hidden(wl.seed, 0, b.T, H)
    w = gen.host_wgate(wl.seed, wl.L, H, E, wl.wgate_scale)
    # the device twins of the generator reproduce the host's bits
    assert np.array_equal(gu.host(dx).view(np.uint16), x)
    assert np.array_equal(gu.host(dw).view(np.uint16), w)
    rs = pipeline.RoutingStats.for_workload(wl, max_T=b.T, max_nblk=b.nblk, max_R=b.R)
    bd = pipeline.BatchDev.from_host(b)
    rs.gate_step(dx, dw, bd)
    torch.cuda.synchronize()
    assert rs.status() == 0

    ref = gu.oracle_gate_logits(x, w)
    otk = orc.topk(ref, k)
    tk = gu.host(rs.topk_for(b.T))
    order_ok, set_ok = _margins(ref, k)
    assert np.array_equal(tk[order_ok], otk[order_ok]), "ordered top-k"
    assert np.array_equal(np.sort(tk[set_ok], axis=1), np.sort(otk[set_ok], axis=1)), "top-k sets"
    rowdiff = (np.sort(tk, axis=2) != np.sort(otk, axis=2)).any(axis=2)   # [L][T]
    ndiff = rowdiff.sum(axis=1)
    print(f"gate path: ambiguous rows {int((~set_ok).sum())}, differing sets {int(ndiff.sum())}")

    # the oracle's chain from its own ids
    bc = orc.block_counts(otk, E, b.req_off, wl.B, wl.mask)
    cache = np.zeros((max(wl.nslots, 1), wl.m, E), dtype=np.uint8)
    rc = orc.stitch(bc, b.req_off, wl.B, b.cache_idx, b.req_cache_off, cache, b.insert_slot)
    A = orc.affinity(otk, E)
    W, Wg, rg, re = orc.loads(otk, E, wl.group_of, wl.G)
    sig, dist = orc.sig_dist(rc, wl.idf, wl.centroids)
    och, _ = orc.route(dist, wl.tau, wl.loads0, False)

    gA = gu.host(rs.affinity).astype(np.int64)
    gW = gu.host(rs.W)
    for layer in range(wl.L):   # a differing row moves at most 2 k^2 pair counts, 2 loads
        assert np.abs(gA[layer] - A[layer]).sum() <= 2 * k * k * ndiff[layer], layer
        assert np.abs(gW[layer] - W[layer]).sum() <= 2 * ndiff[layer], layer
    gbc = gu.host(rs.blk_cnt[:b.nblk]).astype(np.int64)
    grc = gu.host(rs.req_cnt[:b.R]).astype(np.int64)
    gsig, gdist = gu.host(rs.sig[:b.R]), gu.host(rs.dist[:b.R])
    gch = gu.host(rs.choice[:b.R])
    for i, layer in enumerate(wl.mask):
        for j, (t0, ln) in enumerate(b.blk_tab):
            nd = int(rowdiff[layer, t0:t0 + ln].sum())
            assert np.abs(gbc[j, i] - bc[j, i]).sum() <= 2 * nd, (j, i)
    for r in range(b.R):
        t0, t1 = b.req_off[r], b.req_off[r + 1]
        nd = rowdiff[wl.mask, t0:t1].sum()
        assert np.abs(grc[r] - rc[r]).sum() <= 2 * nd, r
        if nd == 0:
            gu.assert_close(gsig[r], sig[r], "signature")
            gu.assert_close(gdist[r], dist[r], "distance")
            gu.check_static_route(gch[r:r + 1], dist[r:r + 1], wl.tau, wl.loads0, och[r:r + 1])
        assert gu.valid_choice(int(gch[r]), gdist[r].astype(np.float64), wl.tau, wl.loads0), r
    if ndiff.sum() == 0:
        assert np.array_equal(gA, A) and np.array_equal(gW, W)
        assert np.array_equal(gu.host(rs.Wg), Wg)
        assert np.array_equal(gu.host(rs.rho_g), rg) and np.array_equal(gu.host(rs.rho_e), re)
