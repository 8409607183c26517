"""Greedy layer-mask selection on the GPU (moer_mask_select) against the oracle
(oracle/mask_select.py): the layers in the order chosen must be identical, except where
two candidates' qualities agree to 1e-12 (then either is a correct greedy step), and the
qualities must agree to 1e-12 relative.  Inputs: synthetic ids with informative, partly
informative and noise layers; 700 requests (several request slices per layer in a greedy
step); requests of 0 and 1 tokens, a single request, and every layer chosen; and the path's
own top-k over a calibration-shaped batch.
"""
import numpy as np
import pytest

import gen
import oracle
from oracle import mask_select as ms

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import _native as nat
    return torch, nat


def _synthetic(seed, L, E, k, R):
    rs = np.random.RandomState(seed)
    lens = rs.randint(1, 60, size=R)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(off[-1])
    topk = np.zeros((L, T, k), dtype=np.uint8)
    signal = rs.random_sample(L)            # per layer: how often a token follows its request
    for r in range(R):
        pref = [rs.choice(E, size=k, replace=False) for _ in range(L)]
        for t in range(off[r], off[r + 1]):
            for l in range(L):
                topk[l, t] = pref[l] if rs.random_sample() < signal[l] else rs.choice(E, size=k, replace=False)
    return topk, off


def _run(env, topk, off, E, m, idf=None):
    torch, nat = env
    L, T, k = topk.shape
    R = len(off) - 1
    dims = nat.make_dims(E, k, L, [], 16)
    dt = torch.from_numpy(topk).cuda()
    do = torch.from_numpy(off).cuda()
    di = torch.from_numpy(idf.astype(np.float32)).cuda() if idf is not None else None
    mask = torch.full((m,), -1, dtype=torch.int32, device="cuda")
    qual = torch.zeros(m, dtype=torch.float64, device="cuda")
    wsb = nat.moer_mask_select_workspace_bytes(dims, R)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_mask_select(dims, dt, T, do, R, di, m, mask, qual, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    return mask.cpu().numpy(), qual.cpu().numpy()


def _compare(topk, off, E, m, idf, got_mask, got_q):
    om, oq = ms.greedy_mask(topk, off, E, m, None if idf is None else idf.astype(np.float32).astype(np.float64))
    c1, c2 = ms.half_counts(topk, off, E)
    w = np.ones((topk.shape[0], E)) if idf is None else idf.astype(np.float32).astype(np.float64)
    for step in range(m):
        if got_mask[step] != om[step]:
            # a near-tie: both candidates must be equally good after the same prefix
            prefix = om[:step].tolist()
            qa = ms.quality(c1, c2, w, prefix + [int(got_mask[step])])
            qb = ms.quality(c1, c2, w, prefix + [int(om[step])])
            assert abs(qa - qb) <= 1e-12 * max(1.0, abs(qb)), (step, got_mask, om)
            return
        assert abs(got_q[step] - oq[step]) <= 1e-12 * max(1.0, abs(oq[step])), step


def _with_lengths(seed, L, E, k, lens):
    rs = np.random.RandomState(seed)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = max(int(off[-1]), 1)
    topk = np.stack([np.stack([rs.choice(E, size=k, replace=False) for _ in range(T)]) for _ in range(L)])
    return topk.astype(np.uint8), off


def test_several_request_slices_per_layer(env):
    # 700 requests over 8 layers: each greedy step splits every layer's requests over
    # three CTAs, and the last CTA to finish combines their partial sums
    topk, off = _synthetic(4, 8, 32, 4, 700)
    got_m, got_q = _run(env, topk, off, 32, 6)
    _compare(topk, off, 32, 6, None, got_m, got_q)


@pytest.mark.parametrize("case", ["empty_and_one_token", "one_request", "all_layers"])
def test_degenerate_requests_and_masks(env, case):
    # requests of 0 and 1 tokens (both halves, or the first, empty: cosine 0), one
    # request, and m = L (every layer chosen, the last with the only quality left)
    L, E, k = 6, 32, 4
    if case == "empty_and_one_token":
        lens, m = [0, 1, 5, 0, 1, 2, 9, 0], 4
    elif case == "one_request":
        lens, m = [37], 3
    else:
        lens, m = [3, 8, 1, 12, 6], L
    topk, off = _with_lengths(len(case), L, E, k, lens)
    got_m, got_q = _run(env, topk, off, E, m)
    assert sorted(got_m.tolist()) == sorted(set(got_m.tolist())) and (got_m >= 0).all() and (got_m < L).all()
    _compare(topk, off, E, m, None, got_m, got_q)
    if case == "all_layers":
        assert sorted(got_m.tolist()) == list(range(L))


@pytest.mark.parametrize("seed,L,E,k,R,m", [(1, 8, 32, 4, 50, 8), (2, 24, 64, 6, 120, 10), (3, 48, 128, 8, 60, 12)])
def test_synthetic(env, seed, L, E, k, R, m):
    topk, off = _synthetic(seed, L, E, k, R)
    idf = 1.0 + np.random.RandomState(seed + 100).random_sample((L, E)) if seed % 2 else None
    got_m, got_q = _run(env, topk, off, E, m, idf)
    assert len(set(got_m.tolist())) == m and (got_m >= 0).all() and (got_m < L).all()
    _compare(topk, off, E, m, idf, got_m, got_q)


def test_on_the_path_top_k(env):
    torch, nat = env
    from moe_expert_routing_top_gb300 import pipeline
    from tests import gpu_util as gu
    wl = gen.make_workload("c2", R=40)
    b = wl.batch()
    rs = pipeline.RoutingStats.for_workload(wl, max_T=b.T, max_nblk=b.nblk, max_R=b.R)
    bd = pipeline.BatchDev.from_host(b)
    rs.step(gu.device_logits(wl, b), bd)
    torch.cuda.synchronize()
    assert rs.status() == 0
    topk_dev = rs.topk_for(b.T).contiguous()
    off = np.asarray(b.req_off, dtype=np.int32)
    m = 8
    dims = nat.make_dims(wl.E, wl.k, wl.L, [], 16)
    do = torch.from_numpy(off).cuda()
    mask = torch.full((m,), -1, dtype=torch.int32, device="cuda")
    qual = torch.zeros(m, dtype=torch.float64, device="cuda")
    wsb = nat.moer_mask_select_workspace_bytes(dims, b.R)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_mask_select(dims, topk_dev, b.T, do, b.R, None, m, mask, qual, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    # the oracle's chain from the host logits (its own top-k)
    tk = oracle.get().topk(gen.host_logits(wl, b.tok_key, b.tok_dom), wl.k)
    _compare(tk, off, wl.E, m, None, mask.cpu().numpy(), qual.cpu().numpy())


def test_malformed_offsets_are_reported(env):
    torch, nat = env
    topk, off = _synthetic(4, 4, 16, 2, 10)
    bad = off.copy()
    bad[3] = bad[4] + 1          # request 2 runs backwards
    dims = nat.make_dims(16, 2, 4, [], 16)
    mask = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    wsb = nat.moer_mask_select_workspace_bytes(dims, 10)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_mask_select(dims, torch.from_numpy(topk).cuda(), topk.shape[1], torch.from_numpy(bad).cuda(),
                         10, None, 2, mask, None, ws, wsb)
    assert nat.moer_ws_status(ws) == 6


def test_k8_misaligned_view_and_bad_id(env):
    torch, nat = env
    topk, off = _synthetic(5, 6, 64, 8, 40)
    L, T, k = topk.shape
    R = len(off) - 1
    dims = nat.make_dims(64, k, L, [], 16)
    do = torch.from_numpy(off).cuda()

    def run(dt):
        mask = torch.full((4,), -1, dtype=torch.int32, device="cuda")
        qual = torch.zeros(4, dtype=torch.float64, device="cuda")
        wsb = nat.moer_mask_select_workspace_bytes(dims, R)
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        nat.moer_mask_select(dims, dt, T, do, R, None, 4, mask, qual, ws, wsb)
        return mask.cpu().numpy(), qual.cpu().numpy(), nat.moer_ws_status(ws)

    aligned_m, aligned_q, st = run(torch.from_numpy(topk).cuda())
    assert st == 0
    _compare(topk, off, 64, 4, None, aligned_m, aligned_q)
    # the same ids one byte into a buffer: the 8-byte loads are not allowed there
    buf = torch.zeros(topk.size + 8, dtype=torch.uint8, device="cuda")
    buf[1:1 + topk.size] = torch.from_numpy(topk.reshape(-1)).cuda()
    view = buf[1:1 + topk.size]
    assert view.data_ptr() % 8 == 1
    m2, q2, st2 = run(view)
    assert st2 == 0 and np.array_equal(m2, aligned_m) and np.array_equal(q2, aligned_q)
    # an id outside [0, E) is skipped and reported
    bad = topk.copy()
    bad[2, 5, 3] = 64
    _, _, st3 = run(torch.from_numpy(bad).cuda())
    assert st3 == 6
