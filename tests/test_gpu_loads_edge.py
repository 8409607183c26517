"""moer_affinity_load on its edge cases against the oracle (O8), which computes the loads
from the top-k ids rather than from the co-activation: one group (rho = 1), groups left
empty (they count in the mean), group ids outside [0, G) (skipped), and a layer with no
tokens (loads 0, rho 0, checked by hand).  Loads are exact integers; rho is the same fp64
expression on both sides, so it must match exactly.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import _native as nat
    return torch, nat


def _topk(rs, L, T, E, k):
    return np.stack([np.stack([rs.choice(E, size=k, replace=False) for _ in range(T)])
                     for _ in range(L)]).astype(np.uint8)


def _run(env, A, group_of, G):
    torch, nat = env
    L, E, _ = A.shape
    dims = nat.make_dims(E, 8, L, [], 16)
    dA = torch.from_numpy(A.astype(np.int32)).cuda()
    dg = torch.from_numpy(group_of.astype(np.int32)).cuda()
    W = torch.full((L, E), -1, dtype=torch.int64, device="cuda")
    Wg = torch.full((L, G), -1, dtype=torch.int64, device="cuda")
    rg = torch.full((L,), -1.0, dtype=torch.float64, device="cuda")
    re = torch.full((L,), -1.0, dtype=torch.float64, device="cuda")
    nat.moer_affinity_load(dims, dA, dg, G, W, Wg, rg, re)
    torch.cuda.synchronize()
    return W.cpu().numpy(), Wg.cpu().numpy(), rg.cpu().numpy(), re.cpu().numpy()


@pytest.mark.parametrize("case", ["one_group", "empty_groups", "out_of_range", "uneven"])
def test_loads_edge_cases(env, case):
    orc = oracle.get()
    rs = np.random.RandomState(len(case))
    L, T, E, k = 4, 300, 64, 8
    tk = _topk(rs, L, T, E, k)
    if case == "one_group":
        G, go = 1, np.zeros((L, E), np.int32)
    elif case == "empty_groups":
        G, go = 8, np.tile(np.arange(E) % 3, (L, 1)).astype(np.int32)      # groups 3..7 stay empty
    elif case == "out_of_range":
        G = 4
        go = np.tile(np.arange(E) % G, (L, 1)).astype(np.int32)
        go[:, ::7] = -1
        go[:, 3::11] = G                                                      # both skipped
    else:
        G, go = 5, rs.randint(0, 5, size=(L, E)).astype(np.int32)
    A = orc.affinity(tk, E)
    W, Wg, rg, re = _run(env, A, go, G)
    oW, oWg, org, ore = orc.loads(tk, E, go, G)
    assert np.array_equal(W, oW) and np.array_equal(Wg, oWg)
    assert np.array_equal(rg, org) and np.array_equal(re, ore)
    if case == "one_group":
        assert (rg == 1.0).all()
    if case == "empty_groups":
        assert (Wg[:, 3:] == 0).all() and (rg >= 8.0 / 3.0 - 1e-12).all()   # mean over all 8 groups
    if case == "out_of_range":
        assert (Wg.sum(axis=1) < W.sum(axis=1)).all()                         # skipped experts missing


def test_layer_without_tokens(env):
    rs = np.random.RandomState(7)
    L, E, G = 3, 64, 8
    A = oracle.get().affinity(_topk(rs, L, 50, E, 8), E)
    A[1] = 0
    go = np.tile(np.arange(E) % G, (L, 1)).astype(np.int32)
    W, Wg, rg, re = _run(env, A, go, G)
    assert (W[1] == 0).all() and (Wg[1] == 0).all() and rg[1] == 0.0 and re[1] == 0.0
    assert (W[0] == np.diagonal(A[0])).all() and rg[0] >= 1.0
