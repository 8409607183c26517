"""Spectral grouping on the GPU (moer_spectral_groups) against the oracle (oracle/grouping.py).

Planted non-uniform partitions (clear eigengap): the groups at every grid point, the knee
and the utilisation curve must equal the oracle's (utilisation and deviation are ratios of
exact integers, computed the same way on both sides).  The path's own co-activation: the
top-G eigenspace need not be separated from the rest there, so the test checks what holds
for any embedding -- sizes within the bounds, curves equal to the values recomputed from the
returned groups, the knee read off the returned curve -- and requires the oracle's groups
wherever the oracle's eigengap is clear.
"""
import numpy as np
import pytest

import gen
import oracle
from oracle import grouping as gp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    pytest.importorskip("scipy")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import _native as nat
    return torch, nat


def _planted(sizes, inside, outside, noise, seed):
    rs = np.random.RandomState(seed)
    E = sum(sizes)
    lab = rs.permutation(np.repeat(np.arange(len(sizes)), sizes))
    A = np.where(lab[:, None] == lab[None, :], inside, outside).astype(np.int64)
    N = rs.randint(0, noise + 1, size=(E, E))
    A = A + N + N.T
    np.fill_diagonal(A, rs.randint(100, 200, size=E))   # the diagonal (loads) must be ignored
    return A.astype(np.int32), lab


def _run(env, A, G):
    torch, nat = env
    L, E, _ = A.shape
    dims = nat.make_dims(E, 8 if E >= 8 else 1, L, [], 16)
    dA = torch.from_numpy(np.ascontiguousarray(A)).cuda()
    g = torch.full((L, E), -1, dtype=torch.int32, device="cuda")
    k = torch.full((L,), -1, dtype=torch.int32, device="cuda")
    uc = torch.zeros((L, 17), dtype=torch.float64, device="cuda")
    sc = torch.zeros((L, 17), dtype=torch.float64, device="cuda")
    wsb = nat.moer_spectral_workspace_bytes(dims, G)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_spectral_groups(dims, dA, G, g, k, uc, sc, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    return g.cpu().numpy(), k.cpu().numpy(), uc.cpu().numpy(), sc.cpu().numpy()


def _check_properties(A, G, g, k, uc, sc):
    L, E, _ = A.shape
    for l in range(L):
        sz = np.bincount(g[l], minlength=G)
        lo, hi = gp.bounds(E, G, int(k[l]))
        assert (sz >= lo).all() and (sz <= hi).all(), (l, sz, lo, hi)
        Al = A[l].astype(np.int64).copy()
        np.fill_diagonal(Al, 0)
        tot = Al.sum()
        same = Al[g[l][:, None] == g[l][None, :]].sum()
        assert uc[l, k[l]] == (float(same) / float(tot) if tot else 0.0)
        assert sc[l, k[l]] == gp.size_deviation(g[l], G)
        # the knee read off the returned curve
        y = uc[l] - uc[l].min()
        rng = uc[l].max() - uc[l].min()
        y = y / rng if rng > 0 else np.zeros(17)
        x = np.arange(17) / 16.0
        c = (x[-1] - x[0]) * (y - y[0]) - (y[-1] - y[0]) * (x - x[0])
        kk = int(np.argmax(c)) if c.max() > 0 else 0
        assert kk == k[l], l


@pytest.mark.parametrize("E,G", [(128, 8), (64, 4), (128, 16), (128, 31)])
def test_planted_partitions(env, E, G):
    # G = 16 and 31: Bellman-Ford over 17 and 32 nodes (several per warp), swap
    # masks up to bit 30, and the largest shared-memory layout
    profiles = {8: [[24, 20, 16, 16, 16, 12, 12, 12], [16] * 8, [30, 18, 16, 14, 14, 12, 12, 12]],
                4: [[24, 16, 12, 12], [16] * 4, [20, 16, 16, 12]],
                16: [[10, 10, 9, 9, 8, 8, 8, 8, 8, 8, 7, 7, 7, 7, 7, 7], [8] * 16],
                31: [[5] * 4 + [4] * 27, [4] * 30 + [8]]}[G]
    assert all(sum(p) == E for p in profiles)
    layers, labs = [], []
    for i, sizes in enumerate(profiles):
        A, lab = _planted(sizes, inside=30 + 10 * i, outside=1, noise=3,
                          seed=(10 if G <= 8 else 100) * G + i)
        layers.append(A)
        labs.append(lab)
    A = np.stack(layers)
    g, k, uc, sc = _run(env, A, G)
    _check_properties(A, G, g, k, uc, sc)
    for l in range(len(layers)):
        og, ok, ou, os_ = gp.group_layer(A[l], G)
        assert k[l] == ok, (l, k[l], ok)
        assert np.array_equal(g[l], og), l
        assert np.array_equal(uc[l], ou) and np.array_equal(sc[l], os_), l


def test_on_the_path_affinity(env):
    torch, nat = env
    from moe_expert_routing_top_gb300 import pipeline
    from tests import gpu_util as gu
    wl = gen.make_workload("c3", R=10)
    b = wl.batch()
    rs = pipeline.RoutingStats.for_workload(wl, max_T=b.T, max_nblk=b.nblk, max_R=b.R)
    rs.step(gu.device_logits(wl, b), pipeline.BatchDev.from_host(b))
    torch.cuda.synchronize()
    assert rs.status() == 0
    A_gpu = rs.affinity.cpu().numpy()
    G = 8
    g, k, uc, sc = _run(env, A_gpu, G)
    _check_properties(A_gpu, G, g, k, uc, sc)
    # the oracle's own co-activation from its own top-k, and its grouping where the
    # embedding is well defined
    tk = oracle.get().topk(gen.host_logits(wl, b.tok_key, b.tok_dom), wl.k)
    A_orc = oracle.get().affinity(tk, wl.E)
    assert np.array_equal(A_orc, A_gpu.astype(np.int64))
    agree = gapped = 0
    for l in range(wl.L):
        _, w, _ = gp.embedding(A_orc[l], G)
        if (w[G - 1] - w[G]) > 1e-6 * abs(w[G - 1]):
            gapped += 1
            og, ok, _, _ = gp.group_layer(A_orc[l], G)
            if ok == k[l] and np.array_equal(og, g[l]):
                agree += 1
    print(f"path co-activation: {gapped} of {wl.L} layers with a clear eigengap, {agree} identical")
    assert agree == gapped
