"""GRACE replication planning on the GPU (moer_replication_plan) against the oracle
(oracle/replication.py), bit for bit: replica counts, sources, hot experts, destinations
and the fp64 predicted loads.  Synthetic loads cover ties, zero layers, one dominant
expert and group counts from 1 to 64; a malformed group map is reported, never a fault.
"""
import numpy as np
import pytest

from oracle import replication as rp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import _native as nat
    return torch, nat


def _layers(rs, L, E, G):
    W = np.zeros((L, E), dtype=np.int64)
    g = np.zeros((L, E), dtype=np.int32)
    for l in range(L):
        g[l] = rs.permutation(np.arange(E) % G)
        kind = l % 5
        if kind == 0:
            W[l] = rs.randint(0, 1000, size=E)
        elif kind == 1:
            W[l] = rs.randint(0, 4, size=E)                  # many ties
        elif kind == 2:
            W[l] = 0                                         # no load
        elif kind == 3:
            W[l] = rs.randint(0, 50, size=E)
            W[l, rs.randint(0, E)] += 100000                 # one dominant expert
        else:
            W[l] = 7                                         # uniform
    return W, g


def _run(env, W, g, G):
    torch, nat = env
    L, E = W.shape
    dims = nat.make_dims(E, 8 if E >= 8 else 1, L, [0], 16)
    dW = torch.from_numpy(W).cuda()
    dg = torch.from_numpy(g).cuda()
    n = torch.full((L,), -7, dtype=torch.int32, device="cuda")
    src = torch.full((L,), -7, dtype=torch.int32, device="cuda")
    hot = torch.full((L, E), 9, dtype=torch.uint8, device="cuda")
    dst = torch.full((L, G), -7, dtype=torch.int32, device="cuda")
    wp = torch.full((L, G), -1.0, dtype=torch.float64, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    nat.moer_replication_plan(dims, dW, dg, G, n, src, hot, dst, wp, ws, 256)
    st = nat.moer_ws_status(ws)
    return st, n.cpu().numpy(), src.cpu().numpy(), hot.cpu().numpy(), dst.cpu().numpy(), wp.cpu().numpy()


@pytest.mark.parametrize("E,G", [(64, 1), (64, 2), (128, 3), (128, 8), (256, 16), (128, 64), (64, 64)])
def test_plan_matches_oracle(env, E, G):
    rs = np.random.RandomState(E * 100 + G)
    W, g = _layers(rs, 40, E, G)
    st, n, src, hot, dst, wp = _run(env, W, g, G)
    assert st == 0
    on, osrc, ohot, odst, owp = rp.plan(W, g, G)
    assert np.array_equal(n, on) and np.array_equal(src, osrc)
    assert np.array_equal(hot, ohot) and np.array_equal(dst, odst)
    assert np.array_equal(wp.view(np.uint64), owp.view(np.uint64)), "predicted loads, bit for bit"


def test_malformed_group_map_is_reported(env):
    rs = np.random.RandomState(1)
    W, g = _layers(rs, 6, 64, 8)
    g[2, 5] = 8          # out of range
    g[4, 0] = -1
    st, n, src, hot, dst, wp = _run(env, W, g, 8)
    assert st == 6       # MOER_EDATA
    assert n[2] == 0 and n[4] == 0 and (dst[2] == -1).all() and hot[2].sum() == 0
    on, osrc, ohot, odst, owp = rp.plan(W[[0, 1, 3, 5]], g[[0, 1, 3, 5]], 8)
    assert np.array_equal(n[[0, 1, 3, 5]], on) and np.array_equal(dst[[0, 1, 3, 5]], odst)
