"""Pins of the spectral-grouping oracle (oracle/grouping.py): size bounds and the bounded
assignment against hand values and brute force, the embedding of a graph of disconnected
cliques (identical rows inside a block, orthogonal rows across blocks), recovery of a planted
non-uniform partition, and hand-computed utilisation, deviation and knee.
"""
import itertools

import numpy as np
import pytest

pytest.importorskip("scipy")
from oracle import grouping as gp  # noqa: E402


def test_bounds():
    assert gp.bounds(128, 8, 0) == (16, 16)
    assert gp.bounds(128, 8, 16) == (1, 32)
    assert gp.bounds(128, 8, 4) == (12, 20)
    assert gp.bounds(100, 8, 0) == (12, 13)       # 12.5 experts per group: 12 or 13
    for E, G in [(64, 8), (128, 8), (100, 7), (64, 3)]:
        for j in range(gp.NGRID):
            lo, hi = gp.bounds(E, G, j)
            assert 1 <= lo <= hi and G * lo <= E <= G * hi


@pytest.mark.parametrize("N,G,lo,hi,seed", [(7, 3, 1, 4, 0), (8, 3, 2, 3, 1), (6, 2, 1, 5, 2), (9, 4, 2, 3, 3)])
def test_bounded_assign_against_brute_force(N, G, lo, hi, seed):
    rs = np.random.RandomState(seed)
    cost = rs.random_sample((N, G))
    best, arg = np.inf, None
    for a in itertools.product(range(G), repeat=N):
        sz = np.bincount(a, minlength=G)
        if (sz >= lo).all() and (sz <= hi).all():
            c = cost[np.arange(N), a].sum()
            if c < best:
                best, arg = c, np.array(a)
    got = gp.bounded_assign(cost, lo, hi)
    sz = np.bincount(got, minlength=G)
    assert (sz >= lo).all() and (sz <= hi).all()
    assert abs(cost[np.arange(N), got].sum() - best) < 1e-9
    assert np.array_equal(got, arg)


def _blocks(sizes, inside=50, outside=0, noise=0, seed=0):
    rs = np.random.RandomState(seed)
    E = sum(sizes)
    lab = np.repeat(np.arange(len(sizes)), sizes)
    A = np.where(lab[:, None] == lab[None, :], inside, outside).astype(np.int64)
    if noise:
        N = rs.randint(0, noise + 1, size=(E, E))
        A = A + N + N.T
    np.fill_diagonal(A, 0)
    return A, lab


def test_embedding_of_disconnected_cliques():
    A, lab = _blocks([5, 3, 4])
    U, w, deg = gp.embedding(A, 3)
    assert np.allclose(w[:3], 1.0) and w[3] < 1.0 - 1e-9
    for a in range(12):
        for b in range(12):
            dot = float(U[a] @ U[b])
            assert abs(dot - (1.0 if lab[a] == lab[b] else 0.0)) < 1e-9


def _same_partition(g, lab):
    pairs = {}
    for x, y in zip(g, lab):
        if pairs.setdefault(x, y) != y:
            return False
    return len(set(pairs.values())) == len(pairs)


def test_planted_nonuniform_partition():
    sizes = [24, 20, 16, 16, 16, 12, 12, 12]
    A, lab = _blocks(sizes, inside=40, outside=1, noise=3, seed=5)
    g, k, Uc, Sc = gp.group_layer(A, 8)
    lo, hi = gp.bounds(128, 8, k)
    assert lo <= 12 and hi >= 24                   # the knee admits the planted sizes
    assert _same_partition(g, lab)
    assert Uc[0] < Uc[k] and Sc[0] == 0.0          # uniform groups split some blocks
    assert abs(Uc[k] - gp.utilisation(A, lab)) < 1e-15


def test_bounded_kmeans_respects_bounds():
    rs = np.random.RandomState(9)
    U = rs.standard_normal((60, 4))
    C0 = U[[0, 1, 2, 3]]
    for lo, hi in [(15, 15), (10, 20), (1, 60)]:
        a = gp.bounded_kmeans(U, C0, lo, hi)
        sz = np.bincount(a, minlength=4)
        assert (sz >= lo).all() and (sz <= hi).all()


def test_utilisation_and_deviation_by_hand():
    A = np.array([[0, 3, 1, 0], [3, 0, 0, 2], [1, 0, 0, 5], [0, 2, 5, 0]])
    g = np.array([0, 0, 1, 1])
    assert gp.utilisation(A, g) == (3 + 3 + 5 + 5) / (2 * (3 + 1 + 2 + 5))
    assert gp.size_deviation(np.array([0, 0, 0, 1]), 2) == np.sqrt(((3 - 2) ** 2 + (1 - 2) ** 2) / 2) / 2
    assert gp.utilisation(np.zeros((3, 3)), np.array([0, 1, 2])) == 0.0


def test_size_deviation_against_the_definition_in_high_precision():
    # S = sqrt(mean_g (size_g - E/G)^2) / (E/G) evaluated with 50 significant digits
    # from the sizes themselves (non-integer means included), against the oracle's
    # double: within one unit in the last place
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    rs = np.random.RandomState(21)
    for E, G in [(128, 31), (128, 8), (100, 7), (64, 3), (128, 2)]:
        for _ in range(20):
            g = rs.randint(0, G, size=E)
            sizes = np.bincount(g, minlength=G)
            mean = Decimal(E) / Decimal(G)
            var = sum((Decimal(int(x)) - mean) ** 2 for x in sizes) / Decimal(G)
            exact = var.sqrt() / mean
            got = gp.size_deviation(g, G)
            assert abs(Decimal(got) - exact) <= Decimal(np.spacing(got)), (E, G, got, exact)
    # balanced sizes give 0 exactly
    assert gp.size_deviation(np.repeat(np.arange(8), 16), 8) == 0.0


def test_knee_by_hand():
    r = np.linspace(0, 1, 17)
    Uc = 1 - (1 - r) ** 6                          # steep rise, then flat: knee early
    k = gp.knee(Uc)
    y = (Uc - Uc.min()) / (Uc.max() - Uc.min())
    d = [(r[-1] - r[0]) * (y[j] - y[0]) - (y[-1] - y[0]) * (r[j] - r[0]) for j in range(17)]
    assert k == int(np.argmax(d)) and 0 < k < 8
    assert gp.knee(r.copy()) == 0                  # a straight line has no knee
    assert gp.knee(np.zeros(17)) == 0
    plateau = np.minimum(r, 0.5)                   # linear up to r = 0.5, then flat
    assert gp.knee(plateau) == 8
