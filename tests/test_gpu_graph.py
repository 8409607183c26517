"""The step of the path captured as one CUDA graph (RoutingStats.capture_step): a replay
must produce exactly what an eager step produces from the same state -- top-k ids, block
counts, request counts, co-activation, loads, signatures, distances and choices -- and two
replays must accumulate the co-activation twice.
"""
import numpy as np
import pytest

import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import pipeline
    from tests import gpu_util
    return torch, pipeline, gpu_util


def _snap(rs, b):
    return {
        "topk": rs.topk_for(b.T).cpu().numpy(),
        "blk": rs.blk_cnt[:b.nblk].cpu().numpy(),
        "req": rs.req_cnt[:b.R].cpu().numpy(),
        "aff": rs.affinity.cpu().numpy(),
        "W": rs.W.cpu().numpy(),
        "rho": rs.rho_g.cpu().numpy(),
        "sig": rs.sig[:b.R].cpu().numpy(),
        "dist": rs.dist[:b.R].cpu().numpy(),
        "choice": rs.choice[:b.R].cpu().numpy(),
    }


@pytest.mark.parametrize("cfg,R", [("c2", 40), ("c3", 12)])
def test_graph_replay_equals_eager_step(env, cfg, R):
    torch, pipeline, gu = env
    wl = gen.make_workload(cfg, R=R)
    assert not wl.live
    b = wl.batch()
    bd = pipeline.BatchDev.from_host(b)
    logits = gu.device_logits(wl, b)
    rs = pipeline.RoutingStats.for_workload(wl, max_T=b.T, max_nblk=b.nblk, max_R=b.R)
    graph = rs.capture_step(logits, bd)
    assert rs.status() == 0
    rs.reset_stats()
    rs.step(logits, bd)
    torch.cuda.synchronize()
    eager = _snap(rs, b)
    rs.reset_stats()
    graph.replay()
    torch.cuda.synchronize()
    assert rs.status() == 0
    replay = _snap(rs, b)
    for key in eager:
        assert np.array_equal(eager[key], replay[key]), key
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(rs.affinity.cpu().numpy(), 2 * eager["aff"])
