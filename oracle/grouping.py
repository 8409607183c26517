"""Spectral grouping of experts per layer with a controlled size tolerance -- the oracle.

TEST INFRASTRUCTURE ONLY: only `tests/` and the bench's CPU leg use it.

GRACE-MoE, section 4.1 (expert grouping, communication first): spectral clustering of the
affinity matrix puts experts that co-activate on the same GPU; fully non-uniform groups
minimise communication but worsen load balance, so group sizes are held within
[E_bar - delta, E_bar + delta], delta = E_bar * r (E_bar: the mean group size), and r is
chosen at the knee point of the affinity utilisation U(r) against the size deviation S(r).
Plain reading for one node of G GPUs, in fp64:

* similarity: the layer's co-activation counts A with the diagonal set to 0; degree
  d_a = sum_b A[a][b]; M = D^-1/2 A D^-1/2 (rows and columns of a zero-degree expert are 0);
* embedding: the eigenvectors of the G largest eigenvalues of M (numpy eigh, the library
  routine for this step), each expert's row scaled to unit length (a zero row stays 0);
* size bounds for r = j/16, j = 0..16: lo = max(1, floor(E (16 - j) / (16 G))),
  hi = min(E, ceil(E (16 + j) / (16 G)));
* K-means on the embedding rows with every group size in [lo, hi]: seeds are the expert of
  largest degree, then repeatedly the expert farthest (largest minimum squared distance)
  from the seeds so far (ties: lower expert id); each step assigns at the least total squared
  distance under the bounds (Hungarian method on N x G*hi slots, the first lo slots of every
  group made mandatory), then moves each centroid to the mean of its rows; stop after a step
  that changes nothing, or after max_iter steps;
* U(r) = sum of A over distinct experts in the same group / sum of A over distinct experts
  (0 when the layer has none); S(r) = sqrt(mean_g (size_g - E/G)^2) / (E/G);
* knee: U(r) over r, both scaled to [0, 1] over the grid (a zero range scales to 0); the
  knee is the grid point farthest above the chord from r = 0 to r = 1 (largest positive cross
  product; ties: smaller r; none above the chord: r = 0) -- where widening the size tolerance
  stops buying affinity.  S(r) is reported with it: with S rising in r, the same point is where
  more size deviation stops paying (on the (S, U) curve itself both saturate together once the
  natural group sizes are admitted, which leaves no knee).
"""
from __future__ import annotations

import numpy as np
from scipy.optimize import linear_sum_assignment

NGRID = 17


def bounds(E: int, G: int, j: int):
    lo = max(1, (E * (16 - j)) // (16 * G))
    hi = min(E, -((-E * (16 + j)) // (16 * G)))
    return lo, hi


def embedding(A, G):
    A = np.array(A, dtype=np.float64)
    np.fill_diagonal(A, 0.0)
    d = A.sum(axis=1)
    inv = np.where(d > 0, 1.0 / np.sqrt(np.where(d > 0, d, 1.0)), 0.0)
    M = inv[:, None] * A * inv[None, :]
    w, V = np.linalg.eigh(M)
    U = V[:, ::-1][:, :G].copy()                  # G largest eigenvalues, descending
    n = np.linalg.norm(U, axis=1, keepdims=True)
    U = np.where(n > 0, U / np.where(n > 0, n, 1.0), 0.0)
    return U, w[::-1], d


def seeds(U, deg, G):
    chosen = [int(np.argmax(deg))]                # first maximum: the lower id on ties
    mind = ((U - U[chosen[0]]) ** 2).sum(axis=1)
    for _ in range(1, G):
        nxt = int(np.argmax(mind))
        chosen.append(nxt)
        mind = np.minimum(mind, ((U - U[nxt]) ** 2).sum(axis=1))
    return chosen


def bounded_assign(cost, lo, hi):
    """Assignment with every group size in [lo, hi] minimising the summed cost."""
    cost = np.asarray(cost, dtype=np.float64)
    N, G = cost.shape
    assert G * lo <= N <= G * hi
    cols = np.repeat(np.arange(G), hi)
    mandatory = np.tile(np.arange(hi) < lo, G)
    big = 1.0 + 4.0 * (np.abs(cost).max() + 1.0) * N
    rows, picked = linear_sum_assignment(cost[:, cols] - big * mandatory[None, :])
    a = np.empty(N, dtype=np.int64)
    a[rows] = cols[picked]
    return a


def bounded_kmeans(U, C0, lo, hi, max_iter=100):
    U = np.asarray(U, dtype=np.float64)
    C = np.asarray(C0, dtype=np.float64).copy()
    G = C.shape[0]
    a = None
    for _ in range(max_iter):
        cost = ((U[:, None, :] - C[None, :, :]) ** 2).sum(axis=2)
        a_new = bounded_assign(cost, lo, hi)
        if a is not None and np.array_equal(a_new, a):
            break
        a = a_new
        C = np.stack([U[a == g].mean(axis=0) for g in range(G)])
    return a


def utilisation(A, groups) -> float:
    A = np.array(A, dtype=np.int64)
    np.fill_diagonal(A, 0)
    total = int(A.sum())
    if total == 0:
        return 0.0
    same = groups[:, None] == groups[None, :]
    return float(int(A[same].sum())) / float(total)


def size_deviation(groups, G) -> float:
    """S(r) = sqrt(mean_g (size_g - E/G)^2) / (E/G).  Since sum_g size_g = E, the mean of
    the squared deviations is (G * sum_g size_g^2 - E^2) / G^2, so S = sqrt(G * sum_g
    size_g^2 - E^2) / E: an exact integer under the root, rounded only by the root and the
    division (a floating-point sum of the squared deviations would depend on its order)."""
    E = len(groups)
    sizes = np.bincount(groups, minlength=G).astype(np.int64)
    num = int(G) * int((sizes * sizes).sum()) - E * E
    return float(np.sqrt(float(num)) / float(E))


def knee(Uc) -> int:
    Uc = np.asarray(Uc, dtype=np.float64)
    n = len(Uc)
    rng = Uc.max() - Uc.min()
    y = (Uc - Uc.min()) / rng if rng > 0 else np.zeros_like(Uc)
    x = np.arange(n, dtype=np.float64) / (n - 1)
    dx, dy = x[-1] - x[0], y[-1] - y[0]
    best, bc = 0, 0.0
    for j in range(n):
        c = dx * (y[j] - y[0]) - dy * (x[j] - x[0])
        if c > bc:
            best, bc = j, c
    return best


def group_layer(A, G, max_iter=100):
    """Returns (groups at the knee [E], knee index j, U curve [17], S curve [17])."""
    A = np.asarray(A)
    E = A.shape[0]
    U, _, deg = embedding(A, G)
    s = seeds(U, deg, G)
    C0 = U[s]
    Ucur, Scur, allg = [], [], []
    for j in range(NGRID):
        lo, hi = bounds(E, G, j)
        g = bounded_kmeans(U, C0, lo, hi, max_iter)
        allg.append(g)
        Ucur.append(utilisation(A, g))
        Scur.append(size_deviation(g, G))
    k = knee(Ucur)
    return allg[k], k, np.array(Ucur), np.array(Scur)
