"""Balanced K-means on the GPU (moer_kmeans_balanced) against the oracle (oracle/kmeans.py).

Both sides take the assignment decisions in fp64 and reach the exact optimum of each
balanced assignment, so the assignments and the number of steps must be identical; the
fp32 centroids must equal the oracle's fp64 means to fp32 rounding, and the objective
must agree to 1e-9 relative.  Cases: the pages' calibration scale (1,000 signatures of
12 x 128 dims into 16 decoders, and 1,003 so the sizes differ by one), one cluster, one
point per cluster, 32 clusters, a first step that starts far from balance, and a problem
too large for the assignment step's shared-memory staging.
"""
import numpy as np
import pytest

import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    pytest.importorskip("scipy")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import _native as nat
    from oracle import kmeans as km
    return torch, nat, km


def _fit(env, S, C0, max_iter):
    torch, nat, _ = env
    N, dim = S.shape
    D = C0.shape[0]
    ds = torch.from_numpy(S).cuda()
    dc0 = torch.from_numpy(np.ascontiguousarray(C0, dtype=np.float32)).cuda()
    cent = torch.empty((D, dim), dtype=torch.float32, device="cuda")
    assign = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    info = torch.zeros(3, dtype=torch.int32, device="cuda")
    obj = torch.zeros(1, dtype=torch.float64, device="cuda")
    wsb = nat.moer_kmeans_workspace_bytes(N, dim, D)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_kmeans_balanced(ds, N, dim, D, dc0, max_iter, cent, assign, info, obj, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    return cent.cpu().numpy(), assign.cpu().numpy(), info.cpu().numpy(), float(obj.item())


def _check(env, S, C0, max_iter):
    _, _, km = env
    cent, a, info, obj = _fit(env, S, C0, max_iter)
    Co, ao, steps, objo = km.balanced_kmeans(S, C0.astype(np.float64), max_iter)
    N, D = S.shape[0], C0.shape[0]
    assert np.array_equal(np.bincount(a, minlength=D), km.capacities(N, D)), "balance"
    assert np.array_equal(a, ao), f"assignment: {int((a != ao).sum())} points differ"
    assert info[0] == steps and info[2] == 0, (info, steps)
    assert np.array_equal(cent, Co.astype(np.float32)) or np.allclose(cent, Co, rtol=2e-7, atol=1e-9)
    assert abs(obj - objo) <= 1e-9 * max(1.0, abs(objo)), (obj, objo)
    return info


def test_calibration_scale_16_decoders(env):
    S, _ = gen.calib_signatures(1000, 12 * 128, ndom=24)
    rows = gen.kmeans_seed_rows(1000, 16)
    info = _check(env, S, S[rows], 100)
    print(f"N=1000 dim=1536 D=16: steps {info[0]}, cycles cancelled {info[1]}")


def test_uneven_sizes(env):
    S, _ = gen.calib_signatures(1003, 12 * 128, ndom=12, seed=3)
    _check(env, S, S[gen.kmeans_seed_rows(1003, 16, seed=4)], 100)


def test_small_many_clusters(env):
    S, _ = gen.calib_signatures(500, 96, ndom=40, seed=5)
    _check(env, S, S[gen.kmeans_seed_rows(500, 32, seed=6)], 100)


def test_one_cluster(env):
    S, _ = gen.calib_signatures(77, 40, seed=7)
    info = _check(env, S, S[:1], 10)
    assert info[0] == 2


def test_one_point_per_cluster(env):
    S, _ = gen.calib_signatures(20, 24, ndom=20, seed=8)
    _check(env, S, S[::-1].copy(), 10)


def test_far_from_balance_start(env):
    # every initial centroid next to one corner: the greedy start is far from optimal
    rs = np.random.RandomState(9)
    S = rs.standard_normal((300, 16)).astype(np.float32)
    C0 = (np.full((8, 16), 3.0) + 0.01 * rs.standard_normal((8, 16))).astype(np.float32)
    _check(env, S, C0, 60)


def test_large_problem_in_global_memory(env):
    # 2,100 points into 24 clusters: the assignment step's gain rows and member lists
    # (445 KB) do not fit in shared memory and live in the workspace, and the first
    # step's greedy start takes the points in index order (more than 2,048 points)
    S, _ = gen.calib_signatures(2100, 32, ndom=30, seed=12)
    C0 = S[gen.kmeans_seed_rows(2100, 24, seed=13)]
    info = _check(env, S, C0, 8)
    assert info[0] == 8


def test_max_iter_stops_early(env):
    S, _ = gen.calib_signatures(400, 64, ndom=30, seed=10)
    C0 = S[gen.kmeans_seed_rows(400, 8, seed=11)]
    info = _check(env, S, C0, 2)
    assert info[0] == 2
