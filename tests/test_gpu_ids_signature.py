"""moer_ids_signature (block counts and co-activation from top-k ids computed elsewhere)
against the oracle: the ids are the oracle's own top-k of the workload's logits, so the
block counts must equal O2's and the co-activation O7's, element by element.  Malformed
ids (an id >= E, a row with a repeated id) must be skipped and reported, never read
past the counters.
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
    from moe_expert_routing_top_gb300 import _native as nat
    from tests import gpu_util
    return torch, nat, gpu_util


def _run(env, wl, b, tk, want_aff=True):
    torch, nat, gu = env
    dims = nat.make_dims(wl.E, wl.k, wl.L, wl.mask, wl.B)
    dtk = torch.from_numpy(np.ascontiguousarray(tk)).cuda()
    tab = torch.from_numpy(b.blk_tab.reshape(-1).astype(np.int32)).cuda()
    cnt = torch.full((b.nblk, wl.m, wl.E), 7, dtype=torch.uint8, device="cuda")
    aff = torch.zeros((wl.L, wl.E, wl.E), dtype=torch.int32, device="cuda") if want_aff else None
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    nat.moer_ids_signature(dims, dtk, b.T, tab, b.nblk, cnt, aff, ws, 256)
    status = nat.moer_ws_status(ws)
    return status, gu.host(cnt), (gu.host(aff).astype(np.int64) if want_aff else None)


@pytest.mark.parametrize("cfg,R", [("c1", None), ("c2", 30), ("c3", 6)])
def test_ids_signature_parity(env, cfg, R):
    orc = oracle.get()
    wl = gen.make_workload(cfg, R=R)
    b = wl.batch()
    tk = orc.topk(gen.host_logits(wl, b.tok_key, b.tok_dom), wl.k)
    status, cnt, aff = _run(env, wl, b, tk)
    assert status == 0
    assert np.array_equal(cnt, orc.block_counts(tk, wl.E, b.req_off, wl.B, wl.mask)), "block counts"
    assert np.array_equal(aff, orc.affinity(tk, wl.E)), "co-activation"


def test_ids_signature_matches_fused_call(env):
    """The same ids through moer_topk_signature's fused path and through moer_ids_signature."""
    torch, nat, gu = env
    wl = gen.make_workload("c2", R=12)
    b = wl.batch()
    dims = nat.make_dims(wl.E, wl.k, wl.L, wl.mask, wl.B)
    logits = gu.device_logits(wl, b)
    tab = torch.from_numpy(b.blk_tab.reshape(-1).astype(np.int32)).cuda()
    tk = torch.empty((wl.L, b.T, wl.k), dtype=torch.uint8, device="cuda")
    cnt = torch.empty((b.nblk, wl.m, wl.E), dtype=torch.uint8, device="cuda")
    aff = torch.zeros((wl.L, wl.E, wl.E), dtype=torch.int32, device="cuda")
    wsb = nat.moer_workspace_bytes(dims, b.T, b.nblk, 0, 0)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_topk_signature(dims, logits, b.T, tab, b.nblk, tk, cnt, aff, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    status, cnt2, aff2 = _run(env, wl, b, gu.host(tk))
    assert status == 0
    assert np.array_equal(cnt2, gu.host(cnt)) and np.array_equal(aff2, gu.host(aff).astype(np.int64))


@pytest.mark.parametrize("k", [8, 6])
def test_ids_signature_rejects_bad_ids(env, k):
    """Rows with an id >= E or a repeated id: not in the co-activation, ids >= E not counted,
    MOER_EDATA recorded; every other row counted as usual."""
    orc = oracle.get()
    E, L, B = 64, 2, 16
    wl = gen.make_custom(E, k, L, [40, 25], B=B, mask=[0, 1])
    b = wl.batch()
    tk = orc.topk(gen.host_logits(wl, b.tok_key, b.tok_dom), k)
    bad = tk.copy()
    bad[0, 3, 2] = 200                   # id out of range
    bad[1, 17, 1] = bad[1, 17, 0]        # repeated id
    bad[0, 50, 0] = 64                   # just past E
    status, cnt, aff = _run(env, wl, b, bad)
    assert status == 6                   # MOER_EDATA
    keep = np.ones((L, b.T), dtype=bool)
    keep[0, 3] = keep[1, 17] = keep[0, 50] = False
    # co-activation: the malformed rows are left out
    ref_aff = np.zeros((L, E, E), dtype=np.int64)
    for l in range(L):
        rows = tk[l][keep[l]]
        ref_aff[l] = orc.affinity(rows[None], E)[0]
    assert np.array_equal(aff, ref_aff)
    # block counts: every id below E is counted as given
    ref_cnt = np.zeros_like(cnt, dtype=np.int64)
    for i, layer in enumerate([0, 1]):
        for j, (t0, ln) in enumerate(b.blk_tab):
            ids = bad[layer, t0:t0 + ln].reshape(-1)
            ref_cnt[j, i] = np.bincount(ids[ids < E], minlength=E)
    assert np.array_equal(cnt.astype(np.int64), ref_cnt)
    # the ids alone, no co-activation asked: counts the same, still reported
    status, cnt2, _ = _run(env, wl, b, bad, want_aff=False)
    assert status == 6 and np.array_equal(cnt2, cnt)


@pytest.mark.parametrize("E,k", [(64, 8), (100, 8), (128, 8), (100, 6), (128, 6)])
def test_ids_signature_many_bad_rows(env, E, k):
    """Every slot pair repeated and every slot pushed to E, E + 1 ... 255, across many
    rows and mask layers: the co-activation keeps exactly the good rows, the block counts
    every id below E, and the status reads MOER_EDATA."""
    orc = oracle.get()
    L, B = 3, 16
    wl = gen.make_custom(E, k, L, [300, 77, 161], B=B, mask=[0, 2])
    b = wl.batch()
    tk = orc.topk(gen.host_logits(wl, b.tok_key, b.tok_dom), k)
    bad = tk.copy()
    rs = np.random.RandomState(E * 10 + k)
    keep = np.ones((L, b.T), dtype=bool)
    pairs = [(i, j) for i in range(k) for j in range(k) if i != j]
    rows = rs.choice(b.T, size=(L, 120), replace=False)
    for l in range(L):
        for n, t in enumerate(rows[l]):
            if n < len(pairs):                       # repeated id, every ordered slot pair
                i, j = pairs[n]
                bad[l, t, i] = bad[l, t, j]
            else:                                    # an id at or above E in some slot
                bad[l, t, rs.randint(k)] = rs.choice([E, E + 1, 127 if E < 127 else 255, 128, 255])
            keep[l, t] = False
    status, cnt, aff = _run(env, wl, b, bad)
    assert status == 6
    ref_aff = np.zeros((L, E, E), dtype=np.int64)
    for l in range(L):
        ref_aff[l] = orc.affinity(tk[l][keep[l]][None], E)[0]
    assert np.array_equal(aff, ref_aff)
    ref_cnt = np.zeros_like(cnt, dtype=np.int64)
    for i, layer in enumerate(wl.mask):
        for j, (t0, ln) in enumerate(b.blk_tab):
            ids = bad[layer, t0:t0 + ln].reshape(-1)
            ref_cnt[j, i] = np.bincount(ids[ids < E], minlength=E)
    assert np.array_equal(cnt.astype(np.int64), ref_cnt)
