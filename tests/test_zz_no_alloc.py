"""moer_topk_signature_noalloc: the entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc (code inside another framework's memory
pool, plugins that must not grow the device footprint, allocation-free
latency paths).  This entry point takes no workspace; its scratch is a fixed
array inside the library.  These tests call it through the C ABI and check
that two calls in a row give exactly what moer_topk_signature gives with a
caller-allocated workspace: the same top-k ids, block counts and
co-activation counts (all integers, compared bit for bit).  The file sorts
last so that a run stopping at its first failure has run everything else.
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
    from moe_expert_routing_top_gb300 import _native as nat
    from tests import gpu_util
    return torch, nat, gpu_util


def _outputs(torch, wl, b):
    return (torch.zeros((wl.L, b.T, wl.k), dtype=torch.uint8, device="cuda"),
            torch.zeros((b.nblk, wl.m, wl.E), dtype=torch.uint8, device="cuda"),
            torch.zeros((wl.L, wl.E, wl.E), dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("cfg,R", [("c3", 6), ("c2", 20), ("c1", None)])
def test_noalloc_matches_workspace_call(env, cfg, R):
    torch, nat, gu = env
    wl = gen.make_workload(cfg, R=R)
    b = wl.batch()
    dims = nat.make_dims(wl.E, wl.k, wl.L, wl.mask, wl.B)
    logits = gu.device_logits(wl, b)
    tab = torch.from_numpy(b.blk_tab.reshape(-1)).cuda()
    # reference: the workspace entry point
    tk_ref, cnt_ref, aff_ref = _outputs(torch, wl, b)
    wsb = nat.moer_workspace_bytes(dims, b.T, b.nblk, 0, 0)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_topk_signature(dims, logits, b.T, tab, b.nblk, tk_ref, cnt_ref, aff_ref, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    for call in range(2):  # two calls in a row share the library's scratch
        tk, cnt, aff = _outputs(torch, wl, b)
        nat.moer_topk_signature_noalloc(dims, logits, b.T, tab, b.nblk, tk, cnt, aff)
        torch.cuda.synchronize()
        assert torch.equal(tk, tk_ref), call
        assert torch.equal(cnt, cnt_ref), call
        assert torch.equal(aff, aff_ref), call
        # without a top-k buffer the ids are staged in the library's scratch
        _, cnt2, aff2 = _outputs(torch, wl, b)
        nat.moer_topk_signature_noalloc(dims, logits, b.T, tab, b.nblk, None, cnt2, aff2)
        torch.cuda.synchronize()
        assert torch.equal(cnt2, cnt_ref), call
        assert torch.equal(aff2, aff_ref), call


def test_noalloc_rejects_staging_beyond_its_scratch(env):
    torch, nat, _ = env
    # m * T * k above the 32 MiB staging limit, with no top-k buffer given
    E, k, L, T = 128, 8, 16, 300_000
    dims = nat.make_dims(E, k, L, list(range(16)), 16)
    logits = torch.empty((1, 4), dtype=torch.float32, device="cuda")  # never read: rejected first
    tab = torch.zeros(2, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(4, dtype=torch.uint8, device="cuda")
    from moe_expert_routing_top_gb300._native import MoerError
    with pytest.raises(MoerError) as ei:
        nat.moer_topk_signature_noalloc(dims, logits, T, tab, 1, None, cnt, None)
    assert ei.value.code == 5  # MOER_ENOMEM
