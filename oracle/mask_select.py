"""Greedy signature layer-mask selection -- the oracle.

TEST INFRASTRUCTURE ONLY: only `tests/` and the bench's CPU leg use it.

ELDR, section "Key idea / structure / operation": the signature does not use every MoE
layer; a greedy layer selection keeps the subset of layers whose signature quality is
highest.  The pages do not print the quality objective (the paper relates prefill
signatures to the experts reused in decode, which needs decode traces).  The plain,
labelled proxy used here: each calibration prompt is split into its first half
(tokens [0, floor(len/2))) and its second half; the count.idf signature of the first half
should predict that of the second half.

* counts c1[r][l][e], c2[r][l][e]: tokens of request r's first / second half whose top-k at
  layer l holds expert e;
* w = c * idf[l][e] (idf = 1 when not given);
* quality(M) = mean over all R requests of cos_r(M), where cos_r(M) is the cosine between
  the first-half and second-half signatures restricted to the layers in M (concatenated),
  and 0 when either is the zero vector;
* greedy: M starts empty; m times, add the layer outside M that gives the largest
  quality(M + {l}) (ties: the lower layer index).

Returns the layers in the order chosen and the quality after each addition (fp64).
"""
from __future__ import annotations

import numpy as np


def half_counts(topk, req_off, E):
    """topk [L][T][k] uint8, req_off [R+1] -> c1, c2 [R][L][E] int64."""
    topk = np.asarray(topk)
    L, T, k = topk.shape
    R = len(req_off) - 1
    c1 = np.zeros((R, L, E), dtype=np.int64)
    c2 = np.zeros((R, L, E), dtype=np.int64)
    for r in range(R):
        t0, t1 = int(req_off[r]), int(req_off[r + 1])
        mid = t0 + (t1 - t0) // 2
        for l in range(L):
            c1[r, l] = np.bincount(topk[l, t0:mid].reshape(-1), minlength=E)
            c2[r, l] = np.bincount(topk[l, mid:t1].reshape(-1), minlength=E)
    return c1, c2


def quality(c1, c2, idf, layers) -> float:
    """Mean over requests of the cosine of the two halves' signatures over `layers`."""
    R = c1.shape[0]
    if len(layers) == 0:
        return 0.0
    layers = list(layers)
    w1 = (c1[:, layers, :] * idf[layers][None]).reshape(R, -1)
    w2 = (c2[:, layers, :] * idf[layers][None]).reshape(R, -1)
    total = 0.0
    for r in range(R):
        n1, n2 = np.linalg.norm(w1[r]), np.linalg.norm(w2[r])
        if n1 > 0 and n2 > 0:
            total += float(np.dot(w1[r], w2[r]) / (n1 * n2))
    return total / R


def greedy_mask(topk, req_off, E, m, idf=None):
    topk = np.asarray(topk)
    L = topk.shape[0]
    idf = np.ones((L, E)) if idf is None else np.asarray(idf, dtype=np.float64)
    c1, c2 = half_counts(topk, req_off, E)
    chosen, qual = [], []
    for _ in range(m):
        best, bq = -1, -np.inf
        for l in range(L):
            if l in chosen:
                continue
            q = quality(c1, c2, idf, chosen + [l])
            if q > bq:
                best, bq = l, q
        chosen.append(best)
        qual.append(bq)
    return np.array(chosen, dtype=np.int32), np.array(qual, dtype=np.float64)
