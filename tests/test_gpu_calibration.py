"""The offline-to-online chain, end to end on the GPU, against the same chain of oracles.

Offline (pipeline.calibrate, on calibration prompts of the served model): top-k ids,
per-block counts and co-activation over every layer -> request counts -> idf fit ->
greedy layer mask -> counts, idf and count.idf signatures over that mask -> balanced
K-means centroids (ELDR, "Key idea / structure / operation": offline calibration,
greedy layer selection, Hungarian-balanced K-means); spectral expert groups of the
co-activation (GRACE-MoE section 4.1).  Online: the served requests routed with that
mask, idf and those centroids, loads and skew over those groups, and the replication
plan (GRACE-MoE sections 4.2-4.3).

The oracle chain runs on the same inputs: O1 -> O2/O3 -> O9 -> the mask oracle ->
O2/O3/O9 -> O4 -> the K-means oracle; O7 -> the grouping oracle; then O1-O8 and the
replication oracle on the served requests.  The calibrated mask, idf, centroids and
groups reach the serving side through the artefact file (save_calibration /
load_calibration), as they would between the offline fit and the server.  Where the greedy mask meets a near-tie (two
layers within 1e-12), the oracle chain adopts the GPU's layer and goes on; K-means runs
on the GPU's fp32 signatures on both sides (they agree with the oracle's to 1e-5), so its
assignments must be identical.
"""
import numpy as np
import pytest

import gen
import oracle
from oracle import grouping as gp
from oracle import kmeans as km
from oracle import mask_select as ms
from oracle import replication as rp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    pytest.importorskip("scipy")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import pipeline
    from tests import gpu_util
    return torch, pipeline, gpu_util


def _mask_agrees(tk, req_off, E, m, idf32, got_order):
    """The GPU's greedy order against the oracle's; a differing step must be a near-tie
    after the same prefix, and from there the GPU's order is adopted."""
    oo, _ = ms.greedy_mask(tk, req_off, E, m, idf32)
    if np.array_equal(oo, got_order):
        return
    c1, c2 = ms.half_counts(tk, req_off, E)
    step = int(np.flatnonzero(oo != got_order)[0])
    prefix = got_order[:step].tolist()
    qa = ms.quality(c1, c2, idf32, prefix + [int(got_order[step])])
    qb = ms.quality(c1, c2, idf32, prefix + [int(oo[step])])
    assert abs(qa - qb) <= 1e-12 * max(1.0, abs(qb)), (step, got_order, oo)


@pytest.mark.parametrize("cfg,ncal,nserve", [("c3", 96, 10), ("c2", 64, 12)])
def test_calibration_chain(env, cfg, ncal, nserve, tmp_path):
    torch, pipeline, gu = env
    orc = oracle.get()
    served = gen.make_workload(cfg, R=nserve)
    cal = gen.make_calibration(served, R=ncal)
    E, k, L, B, D, G = served.E, served.k, served.L, served.B, served.D, served.G
    m = int(served.mask.shape[0])
    cb = cal.batch()
    seed_rows = gen.kmeans_seed_rows(cal.R, D)
    got = pipeline.calibrate(E, k, L, B, gu.device_logits(cal, cb),
                             pipeline.BatchDev.from_host(cb, with_cache=False), cb.req_off,
                             m=m, D=D, G=G, seed_rows=seed_rows, tau=served.tau)
    torch.cuda.synchronize()

    # ---- offline, oracle chain
    tk = orc.topk(gen.host_logits(cal, cb.tok_key, cb.tok_dom), k)
    nb = orc.num_blocks(cb.req_off, B)
    empty_cache = lambda mm: np.zeros((1, mm, E), dtype=np.uint8)  # noqa: E731
    no_cache = (np.zeros(0, np.int32), np.zeros(cal.R + 1, np.int32), np.full(nb, -1, np.int32))
    rc_all = orc.stitch(orc.block_counts(tk, E, cb.req_off, B, np.arange(L)), cb.req_off, B,
                        no_cache[0], no_cache[1], empty_cache(L), no_cache[2])
    idf_all = orc.idf_fit(rc_all).astype(np.float32).astype(np.float64)
    _mask_agrees(tk, cb.req_off, E, m, idf_all, got.mask_order)
    mask = np.sort(got.mask_order)
    assert np.array_equal(mask, got.mask)
    rc_m = orc.stitch(orc.block_counts(tk, E, cb.req_off, B, mask), cb.req_off, B,
                      no_cache[0], no_cache[1], empty_cache(m), no_cache[2])
    idf_m = orc.idf_fit(rc_m)
    assert np.array_equal(gu.host(got.idf), idf_m.astype(np.float32)), "idf of the mask layers"
    sig_o = np.stack([orc.signature(rc_m[r], idf_m.astype(np.float32)) for r in range(cal.R)])
    sig = gu.host(got.sig)
    gu.assert_close(sig, sig_o, "calibration signatures")
    Co, ao, steps, _ = km.balanced_kmeans(sig, sig[seed_rows].astype(np.float64), 100)
    assert np.array_equal(gu.host(got.assign), ao), "K-means assignment"
    assert int(got.kmeans_info[0]) == steps and int(got.kmeans_info[2]) == 0
    cent = gu.host(got.centroids)
    assert np.array_equal(cent, Co.astype(np.float32)) or np.allclose(cent, Co, rtol=2e-7, atol=1e-9)
    A_o = orc.affinity(tk, E)
    assert np.array_equal(gu.host(got.affinity).astype(np.int64), A_o), "calibration co-activation"
    groups = gu.host(got.group_of)
    gapped = 0
    for l in range(L):
        _, w, _ = gp.embedding(A_o[l], G)
        if (w[G - 1] - w[G]) > 1e-6 * abs(w[G - 1]):
            gapped += 1
            og, okn, _, _ = gp.group_layer(A_o[l], G)
            assert okn == got.knee[l] and np.array_equal(og, groups[l]), l
    print(f"{cfg} calibration: mask {mask.tolist()}, K-means {steps} steps, "
          f"{gapped} of {L} layers with a clear eigengap")

    # ---- online, with the calibrated inputs carried through the artefact file
    path = tmp_path / f"{cfg}.cal"
    pipeline.save_calibration(path, got, E=E, k=k, L=L, block=B, G=G, tau=served.tau)
    art = pipeline.load_calibration(path)
    assert (art["E"], art["k"], art["L"], art["m"], art["D"], art["block"]) == (E, k, L, m, D, B)
    assert np.array_equal(art["mask"], mask) and np.array_equal(art["idf"], gu.host(got.idf))
    assert np.array_equal(art["centroids"], cent) and np.array_equal(art["group_of"], groups)
    served.mask, served.idf = art["mask"], art["idf"]
    served.centroids, served.group_of = art["centroids"], art["group_of"]
    b = served.batch()
    rs = pipeline.RoutingStats.for_workload(served, max_T=b.T, max_nblk=b.nblk, max_R=b.R)
    rs.step(gu.device_logits(served, b), pipeline.BatchDev.from_host(b))
    rs.replication_plan()
    torch.cuda.synchronize()
    assert rs.status() == 0
    tks = orc.topk(gen.host_logits(served, b.tok_key, b.tok_dom), k)
    cache = np.zeros((max(served.nslots, 1), m, E), dtype=np.uint8)
    rc = orc.stitch(orc.block_counts(tks, E, b.req_off, B, mask), b.req_off, B, b.cache_idx,
                    b.req_cache_off, cache, b.insert_slot)
    assert np.array_equal(gu.host(rs.req_cnt[:b.R]), rc), "served request counts"
    osig, odist = orc.sig_dist(rc, served.idf, served.centroids)
    gu.assert_close(gu.host(rs.sig[:b.R]), osig, "served signatures")
    gu.assert_close(gu.host(rs.dist[:b.R]), odist, "served distances")
    och, _ = orc.route(odist, served.tau, served.loads0, False)
    gu.check_static_route(gu.host(rs.choice[:b.R]), odist, served.tau, served.loads0, och)
    W, Wg, rg, re = orc.loads(tks, E, groups, G)
    assert np.array_equal(gu.host(rs.W), W) and np.array_equal(gu.host(rs.Wg), Wg)
    assert np.array_equal(gu.host(rs.rho_g), rg) and np.array_equal(gu.host(rs.rho_e), re)
    pn, psrc, phot, pdst, pwp = rp.plan(W, groups, G)
    assert np.array_equal(gu.host(rs.n_rep), pn) and np.array_equal(gu.host(rs.rep_src), psrc)
    assert np.array_equal(gu.host(rs.hot), phot) and np.array_equal(gu.host(rs.rep_dst), pdst)
    assert np.array_equal(gu.host(rs.w_pred), pwp), "replication plan over the spectral groups"
