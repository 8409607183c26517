"""Balanced K-means of calibration signatures into D decoder centroids -- the oracle.

TEST INFRASTRUCTURE ONLY: only `tests/`, `__graft_entry__.smoke()` and the bench's
CPU-baseline / reference leg use it; the library never does.

ELDR, section "Key idea / structure / operation": offline, the signatures of the
calibration prompts are split into D clusters, one per decode worker, by K-means with a
balance constraint (solved with the Hungarian method), because plain K-means can pile
requests onto one decoder.  Plain reading, written out here in fp64:

* capacities: cluster d holds floor(N/D) points, plus one for d < N mod D;
* assignment step: given centroids C, minimise sum_i ||s_i - c_a(i)||^2 over the
  assignments a with exactly cap_d points in cluster d -- the Hungarian method on the
  N x N cost matrix whose columns repeat centroid d cap_d times (the library routine
  `scipy.optimize.linear_sum_assignment` is that step);
* update step: c_d = mean of the signatures assigned to d (no renormalisation);
* start from the given initial centroids; stop after the first assignment step that
  changes nothing (no update follows it), or after `max_iter` assignment steps;
* the objective is sum_i ||s_i - c_a(i)||^2 for the returned centroids and assignment.
"""
from __future__ import annotations

import numpy as np
from scipy.optimize import linear_sum_assignment


def capacities(N: int, D: int) -> np.ndarray:
    caps = np.full(D, N // D, dtype=np.int64)
    caps[: N % D] += 1
    return caps


def sq_distances(S, C) -> np.ndarray:
    """cost[i][d] = ||s_i - c_d||^2 in fp64."""
    S = np.asarray(S, dtype=np.float64)
    C = np.asarray(C, dtype=np.float64)
    return ((S[:, None, :] - C[None, :, :]) ** 2).sum(axis=2)


def balanced_assign(cost, caps) -> np.ndarray:
    """The assignment with cap_d points per cluster minimising the summed cost."""
    cost = np.asarray(cost, dtype=np.float64)
    N, D = cost.shape
    cols = np.repeat(np.arange(D), caps)
    assert len(cols) == N, "capacities must add up to N"
    rows, picked = linear_sum_assignment(cost[:, cols])
    a = np.empty(N, dtype=np.int64)
    a[rows] = cols[picked]
    return a


def means(S, a, D) -> np.ndarray:
    S = np.asarray(S, dtype=np.float64)
    return np.stack([S[a == d].mean(axis=0) for d in range(D)])


def objective(S, C, a) -> float:
    cost = sq_distances(S, C)
    return float(cost[np.arange(len(a)), a].sum())


def balanced_kmeans(S, C0, max_iter: int):
    """Returns (centroids fp64 [D][dim], assignment [N], assignment steps, objective)."""
    S = np.asarray(S, dtype=np.float64)
    C = np.asarray(C0, dtype=np.float64).copy()
    N, D = S.shape[0], C.shape[0]
    assert 1 <= D <= N
    caps = capacities(N, D)
    a = None
    steps = 0
    while steps < max_iter:
        steps += 1
        a_new = balanced_assign(sq_distances(S, C), caps)
        if a is not None and np.array_equal(a_new, a):
            break
        a = a_new
        C = means(S, a, D)
    return C, a, steps, objective(S, C, a)
