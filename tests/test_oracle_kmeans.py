"""Pins of the balanced K-means oracle (oracle/kmeans.py) against things other than itself:
brute force over every balanced assignment of tiny inputs, closed cases (one cluster, one
point per cluster, well-separated blobs), exact balance, and a non-increasing objective.
"""
import itertools

import numpy as np
import pytest

pytest.importorskip("scipy")
from oracle import kmeans as km  # noqa: E402


def _brute_best(cost, caps):
    """Minimum summed cost over all assignments with the given cluster sizes."""
    N, D = cost.shape
    best, arg = np.inf, None
    for a in itertools.product(range(D), repeat=N):
        if np.array_equal(np.bincount(a, minlength=D), caps):
            c = cost[np.arange(N), a].sum()
            if c < best - 1e-12:
                best, arg = c, np.array(a)
    return best, arg


def test_capacities():
    assert km.capacities(10, 3).tolist() == [4, 3, 3]
    assert km.capacities(16, 16).tolist() == [1] * 16
    assert km.capacities(1000, 16).sum() == 1000
    assert km.capacities(1000, 16).max() - km.capacities(1000, 16).min() == 1


@pytest.mark.parametrize("N,D,seed", [(6, 2, 0), (7, 3, 1), (8, 4, 2), (7, 2, 3), (9, 3, 4)])
def test_assignment_against_brute_force(N, D, seed):
    rs = np.random.RandomState(seed)
    S = rs.standard_normal((N, 3))
    C = rs.standard_normal((D, 3))
    cost = km.sq_distances(S, C)
    caps = km.capacities(N, D)
    best, arg = _brute_best(cost, caps)
    a = km.balanced_assign(cost, caps)
    assert np.array_equal(np.bincount(a, minlength=D), caps)
    assert abs(cost[np.arange(N), a].sum() - best) < 1e-9
    assert np.array_equal(a, arg)  # generic costs: the optimum is unique


def test_sq_distances_by_hand():
    S = np.array([[0.0, 0.0], [1.0, 2.0]])
    C = np.array([[1.0, 1.0]])
    assert km.sq_distances(S, C).ravel().tolist() == [2.0, 1.0]


def test_one_cluster_is_the_mean():
    rs = np.random.RandomState(5)
    S = rs.standard_normal((50, 7))
    C, a, steps, obj = km.balanced_kmeans(S, S[:1], 10)
    assert (a == 0).all() and steps == 2
    assert np.allclose(C[0], S.mean(axis=0), rtol=0, atol=1e-12)
    assert abs(obj - ((S - S.mean(axis=0)) ** 2).sum()) < 1e-9


def test_one_point_per_cluster():
    rs = np.random.RandomState(6)
    S = rs.standard_normal((5, 4))
    C0 = S[[3, 1, 4, 0, 2]] + 0.01 * rs.standard_normal((5, 4))
    C, a, steps, obj = km.balanced_kmeans(S, C0, 10)
    assert a.tolist() == [3, 1, 4, 0, 2]
    assert np.allclose(C[a], S) and obj < 1e-20


def test_separated_blobs_are_recovered():
    rs = np.random.RandomState(7)
    D, per, dim = 4, 25, 16
    centers = 10.0 * rs.standard_normal((D, dim))
    S = np.concatenate([centers[d] + 0.1 * rs.standard_normal((per, dim)) for d in range(D)])
    truth = np.repeat(np.arange(D), per)
    C0 = S[[5, 30, 55, 80]] + 0.5   # one point of each blob, shifted
    C, a, steps, obj = km.balanced_kmeans(S, C0, 20)
    assert np.array_equal(a, truth) and steps == 2
    for d in range(D):
        assert np.allclose(C[d], S[truth == d].mean(axis=0))


def test_balance_is_enforced_against_a_dominant_centroid():
    rs = np.random.RandomState(8)
    S = rs.standard_normal((40, 5)) * 0.1
    C0 = np.stack([np.zeros(5), np.full(5, 50.0), np.full(5, -50.0), np.full(5, 80.0)])
    _, a, _, _ = km.balanced_kmeans(S, C0, 30)
    assert np.bincount(a, minlength=4).tolist() == [10, 10, 10, 10]


def test_objective_never_increases():
    rs = np.random.RandomState(9)
    S = rs.standard_normal((120, 6))
    S /= np.linalg.norm(S, axis=1, keepdims=True)
    C0 = S[rs.choice(120, 7, replace=False)]
    objs = [km.balanced_kmeans(S, C0, it)[3] for it in range(1, 9)]
    assert all(b <= a + 1e-12 for a, b in zip(objs, objs[1:]))


def test_no_improving_swap():
    rs = np.random.RandomState(10)
    S = rs.standard_normal((60, 4))
    C = rs.standard_normal((5, 4))
    cost = km.sq_distances(S, C)
    a = km.balanced_assign(cost, km.capacities(60, 5))
    for i in range(60):
        for j in range(i + 1, 60):
            if a[i] != a[j]:
                assert cost[i, a[j]] + cost[j, a[i]] >= cost[i, a[i]] + cost[j, a[j]] - 1e-12
