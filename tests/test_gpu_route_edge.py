"""moer_route on its degenerate settings against the oracle (O4-O6): tau = 0 (the nearest
centroid), a band wider than every distance (join-the-shortest-queue over all decoders),
one decoder, a request whose counts are all zero (signature 0, so every distance is the
centroid's norm), equal loads (ties to the lowest index), and live routing where each
choice raises its decoder's load.  Signatures and distances within the stated tolerance;
choices identical except at the band edge (then any valid pick).
"""
import numpy as np
import pytest

import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import _native as nat
    return torch, nat


def _inputs(seed, R, m, E, D):
    rs = np.random.RandomState(seed)
    cnt = rs.poisson(3.0, size=(R, m, E)).astype(np.int32)
    cnt[0] = 0                                       # an empty request
    cnt[1] = 0
    cnt[1, :, 5] = 7                                 # a single expert per layer
    idf = (1.0 + rs.random_sample((m, E))).astype(np.float32)
    cen = rs.standard_normal((D, m * E)).astype(np.float32)
    cen /= np.linalg.norm(cen, axis=1, keepdims=True).astype(np.float32)
    cen *= np.float32(0.2)
    return cnt, idf, cen


def _run(env, cnt, idf, cen, tau, loads, live):
    torch, nat = env
    R, m, E = cnt.shape
    D = cen.shape[0]
    dims = nat.make_dims(E, 8, m, list(range(m)), 16)
    dc = torch.from_numpy(cnt).cuda()
    di = torch.from_numpy(idf).cuda()
    dcen = torch.from_numpy(cen).cuda()
    dl = torch.from_numpy(np.asarray(loads, dtype=np.int32)).cuda()
    sig = torch.zeros((R, m * E), dtype=torch.float32, device="cuda")
    dist = torch.zeros((R, D), dtype=torch.float32, device="cuda")
    ch = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    wsb = nat.moer_workspace_bytes(dims, 0, 0, R, D)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_route(dims, dc, R, di, dcen, D, tau, dl, 1 if live else 0, sig, dist, ch, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    return sig.cpu().numpy(), dist.cpu().numpy(), ch.cpu().numpy(), dl.cpu().numpy()


CASES = [  # (tau, D, live, equal loads); D > 16 and D > 32 take the wider kernels
    (0.0, 8, False, False),
    (1e6, 8, False, False),
    (0.1, 1, False, False),
    (0.1, 16, False, True),
    (0.05, 16, True, True),
    (1e6, 4, True, False),
    (0.1, 40, False, False),
    (0.1, 40, True, False),
    (0.3, 64, False, True),
    (0.3, 64, True, True),
    (1e6, 64, True, False),
]


@pytest.mark.parametrize("tau,D,live,equal", CASES)
def test_route_degenerate_settings(env, tau, D, live, equal):
    orc = oracle.get()
    R, m, E = 200, 3, 64
    cnt, idf, cen = _inputs(int(tau * 100) + D, R, m, E, D)
    loads0 = np.zeros(D, np.int32) if equal else np.random.RandomState(D).randint(0, 64, size=D).astype(np.int32)
    sig, dist, ch, loads = _run(env, cnt, idf, cen, tau, loads0, live)
    osig, odist = orc.sig_dist(cnt, idf, cen)
    gu.assert_close(sig, osig, "signature")
    gu.assert_close(dist, odist, "distance")
    assert (sig[0] == 0).all()                                   # empty request: zero signature
    assert np.allclose(dist[0], np.linalg.norm(cen.astype(np.float64), axis=1), rtol=1e-5)
    och, oloads = orc.route(odist, tau, loads0, live)
    if live:
        gu.check_live_route(ch, odist, tau, loads0, och)
        assert loads.sum() == loads0.sum() + R                   # every request counted once
        assert np.array_equal(np.bincount(ch, minlength=D) + loads0, loads)
    else:
        gu.check_static_route(ch, odist, tau, loads0, och)
        assert np.array_equal(loads, loads0)                     # static: loads untouched
    if D == 1:
        assert (ch == 0).all()
    if tau == 0.0 and not live:                                  # nearest centroid (off the band edge)
        off = ~gu.band_edge_rows(odist, tau)
        assert (ch[off] == odist.argmin(axis=1)[off]).all()
    if tau >= 1e6 and not live:                                  # least loaded, lowest index on ties
        assert (ch == int(np.lexsort((np.arange(D), loads0))[0])).all()


@pytest.mark.parametrize("live", [False, True])
def test_route_undefined_distances(env, live):
    """Centroids with NaN entries give NaN distances to those decoders: they are outside the band
    and take no part in d_min; with every centroid NaN no decoder is chosen (-1) and no load
    changes.  Static and live mode agree with the oracle on both."""
    orc = oracle.get()
    R, m, E, D = 64, 2, 64, 8
    cnt, idf, cen = _inputs(77, R, m, E, D)
    loads0 = np.random.RandomState(5).randint(0, 8, size=D).astype(np.int32)
    cen_nan = cen.copy()
    cen_nan[0, 3] = np.nan                                       # decoder 0: NaN distance
    cen_nan[5, :] = np.nan                                       # decoder 5: NaN distance
    sig, dist, ch, loads = _run(env, cnt, idf, cen_nan, 0.1, loads0, live)
    assert np.isnan(dist[:, 0]).all() and np.isnan(dist[:, 5]).all()
    _, odist = orc.sig_dist(cnt, idf, cen_nan)
    keep = [q for q in range(D) if q not in (0, 5)]
    gu.assert_close(dist[:, keep], odist[:, keep], "distance")
    och, oloads = orc.route(odist, 0.1, loads0, live)
    assert not np.isin(ch, [0, 5]).any() and (ch >= 0).all()
    if live:
        gu.check_live_route(ch, odist, 0.1, loads0, och)
        assert np.array_equal(np.bincount(ch, minlength=D) + loads0, loads)
    else:
        gu.check_static_route(ch, odist, 0.1, loads0, och)
    # every centroid NaN: no decoder, loads unchanged
    cen_all = np.full_like(cen, np.nan)
    _, dist, ch, loads = _run(env, cnt, idf, cen_all, 0.1, loads0, live)
    assert np.isnan(dist).all()
    assert (ch == -1).all()
    assert np.array_equal(loads, loads0)
    och, oloads = orc.route(dist.astype(np.float64), 0.1, loads0, live)
    assert (och == -1).all() and np.array_equal(oloads, loads0)


@pytest.mark.parametrize("D", [16, 48])
def test_route_live_across_staging_buffers(env, D):
    """5,000 requests in one live call: route_live stages the band masks 2,048 at a time in
    two alternating buffers, so decisions cross two buffer hand-overs.  Loads start unequal;
    every pick must follow the oracle until the first band-edge divergence."""
    orc = oracle.get()
    R, m, E = 5000, 2, 64
    cnt, idf, cen = _inputs(900 + D, R, m, E, D)
    loads0 = np.random.RandomState(D).randint(0, 40, size=D).astype(np.int32)
    sig, dist, ch, loads = _run(env, cnt, idf, cen, 0.1, loads0, True)
    _, odist = orc.sig_dist(cnt, idf, cen)
    gu.assert_close(dist, odist, "distance")
    och, oloads = orc.route(odist, 0.1, loads0, True)
    gu.check_live_route(ch, odist, 0.1, loads0, och)
    assert np.array_equal(np.bincount(ch, minlength=D) + loads0, loads)
    assert loads.sum() == loads0.sum() + R


@pytest.mark.parametrize("D,base", [(16, (1 << 25) - 300), (16, (1 << 25) - 100), (48, (1 << 24) - 300),
                                    (48, (1 << 24) - 100), (16, (1 << 31) - 1000)])
def test_route_live_large_loads(env, D, base):
    """Live routing from large starting loads (around 2^24 and 2^25, and near the int32 limit,
    where 200 requests raise no load past it) gives the oracle's picks and the oracle's final
    loads: the pick compares the loads themselves, however large."""
    orc = oracle.get()
    R, m, E = 200, 2, 64
    cnt, idf, cen = _inputs(31 + D, R, m, E, D)
    loads0 = (base + np.random.RandomState(D).randint(0, 40, size=D)).astype(np.int32)
    tau = 1e6 if base > (1 << 30) else 0.1                       # near int32: every decoder in the band
    _, dist, ch, loads = _run(env, cnt, idf, cen, tau, loads0, True)
    _, odist = orc.sig_dist(cnt, idf, cen)
    och, oloads = orc.route(odist, tau, loads0, True)
    gu.check_live_route(ch, odist, tau, loads0, och)
    assert np.array_equal(np.bincount(ch, minlength=D).astype(np.int64) + loads0, loads.astype(np.int64))
