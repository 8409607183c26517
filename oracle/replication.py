"""GRACE replication planning per MoE layer -- the oracle.

TEST INFRASTRUCTURE ONLY: only `tests/` and the bench's CPU leg use it.

GRACE-MoE, section 4.2 (expert replication, load-balance first) and section 4.3
(predicted load, equation 3: W' = W - W_r + W_p).  Each expert group sits on one GPU, so
there are G GPUs.  Per layer, plain reading:

* the source is the group with the largest load W_max (ties: the lower group index);
  skew rho = W_max / mean_g W_g (mean over all G groups);
* n_replica = min(max(1, floor(rho)), G - 1), floor(rho) taken exactly in integers as
  floor(W_max * G / sum_g W_g); a layer with no load, or G = 1, plans nothing (n_replica = 0);
* hot experts: the source group's experts in descending load (ties: lower expert id); the hot
  set is the shortest such prefix whose cumulative load exceeds W_max * n / (1 + n) -- the
  expert whose load carries the sum past that threshold is the last one in;
* replicas go to the n least-loaded other groups (ascending load, ties: lower index), in
  that order;
* predicted loads: the hot load H is split evenly over the original and its n copies, so the
  source keeps W_max - H * n / (1 + n) and each replica group receives H / (1 + n); the other
  groups keep their load.  In fp64: W_max - (H n) / (1 + n) and W_g + H / (1 + n), each an
  exact integer converted, then one correctly rounded division and one subtraction or sum.
"""
from __future__ import annotations

import numpy as np


def plan_layer(W_e, group_of, G):
    """W_e [E] int loads, group_of [E] -> (n, src, hot [E] u8, dst [G] i32, w_pred [G] f64)."""
    W_e = np.asarray(W_e, dtype=np.int64)
    group_of = np.asarray(group_of, dtype=np.int64)
    E = len(W_e)
    Wg = np.zeros(G, dtype=np.int64)
    for e in range(E):
        Wg[group_of[e]] += W_e[e]
    hot = np.zeros(E, dtype=np.uint8)
    dst = np.full(G, -1, dtype=np.int32)
    w_pred = Wg.astype(np.float64)
    src = 0
    for g in range(1, G):
        if Wg[g] > Wg[src]:
            src = g
    wmax = int(Wg[src])
    if G < 2 or wmax == 0:
        return 0, src, hot, dst, w_pred
    # floor(rho) = floor(W_max / (sum / G)) in integers
    n = min(max(1, (wmax * G) // int(Wg.sum())), G - 1)
    members = [e for e in range(E) if group_of[e] == src]
    members.sort(key=lambda e: (-W_e[e], e))
    acc = 0
    for e in members:
        hot[e] = 1
        acc += int(W_e[e])
        if acc * (1 + n) > wmax * n:  # cumulative load > W_max * n / (1 + n), in integers
            break
    H = acc
    others = sorted((g for g in range(G) if g != src), key=lambda g: (Wg[g], g))
    dst[:n] = others[:n]
    share = float(H) / float(1 + n)
    w_pred[src] = float(wmax) - float(H * n) / float(1 + n)
    for g in others[:n]:
        w_pred[g] = float(Wg[g]) + share
    return n, src, hot, dst, w_pred


def plan(W, group_of, G):
    """Per layer: W [L][E] int64 expert loads, group_of [L][E] -> arrays over layers."""
    W = np.asarray(W)
    L, E = W.shape
    n = np.zeros(L, dtype=np.int32)
    src = np.zeros(L, dtype=np.int32)
    hot = np.zeros((L, E), dtype=np.uint8)
    dst = np.full((L, G), -1, dtype=np.int32)
    w_pred = np.zeros((L, G), dtype=np.float64)
    for l in range(L):
        n[l], src[l], hot[l], dst[l], w_pred[l] = plan_layer(W[l], group_of[l], G)
    return n, src, hot, dst, w_pred
