"""Pins of the GRACE replication-planning oracle (oracle/replication.py): a worked example
done by hand, closed cases (uniform loads, one group, no load), ties, and invariants on
random layers checked against independent computations (float skew, sorted groups,
conservation of load, minimality of the hot set).
"""
import numpy as np

from oracle import replication as rp


def test_hand_example():
    # groups of 2 experts: loads [10+30, 5+5, 5+5, 20+0] = [40, 10, 10, 20], mean 20, rho 2
    W = [10, 30, 5, 5, 5, 5, 20, 0]
    g = [0, 0, 1, 1, 2, 2, 3, 3]
    n, src, hot, dst, wp = rp.plan_layer(W, g, 4)
    assert (n, src) == (2, 0)
    assert hot.tolist() == [0, 1, 0, 0, 0, 0, 0, 0]   # 30 > 40 * 2/3, so expert 1 alone
    assert dst.tolist() == [1, 2, -1, -1]              # the two least-loaded other groups
    assert wp.tolist() == [20.0, 20.0, 20.0, 20.0]     # 40 - 30*2/3, 10 + 10, 10 + 10, 20


def test_threshold_needs_two_experts():
    # group 0 = [12, 10, 8] = 30; others 10, 10: mean 50/3, rho 1.8 -> n 1, threshold 15
    W = [12, 10, 8, 6, 4, 5, 5]
    g = [0, 0, 0, 1, 1, 2, 2]
    n, src, hot, dst, wp = rp.plan_layer(W, g, 3)
    assert (n, src) == (1, 0)
    assert hot.tolist() == [1, 1, 0, 0, 0, 0, 0]      # 12 <= 15 < 22
    assert dst.tolist() == [1, -1, -1]                 # groups 1 and 2 tie at 10: lower index
    assert wp.tolist() == [30 - 22 / 2, 10 + 11.0, 10.0]


def test_uniform_loads_replicate_once():
    W = np.full(16, 7)
    g = np.repeat(np.arange(4), 4)
    n, src, hot, dst, wp = rp.plan_layer(W, g, 4)
    assert (n, src) == (1, 0)                          # rho = 1, ties to group 0
    assert hot.tolist() == [1, 1, 1] + [0] * 13        # 21 > 28/2 after three experts
    assert dst.tolist() == [1, -1, -1, -1]


def test_single_group_and_empty_layer_plan_nothing():
    n, _, hot, dst, wp = rp.plan_layer([3, 4], [0, 0], 1)
    assert n == 0 and hot.sum() == 0 and (dst == -1).all() and wp.tolist() == [7.0]
    n, _, hot, dst, wp = rp.plan_layer([0, 0, 0, 0], [0, 0, 1, 1], 2)
    assert n == 0 and hot.sum() == 0 and wp.tolist() == [0.0, 0.0]


def test_expert_ties_go_to_the_lower_id():
    # group 0 = three experts of 9 (27), group 1 = 2: n = 1, threshold 13.5, so two of the
    # three tied experts are hot -- the two lower ids
    n, src, hot, dst, wp = rp.plan_layer([9, 9, 9, 1, 1], [0, 0, 0, 1, 1], 2)
    assert (n, src) == (1, 0)
    assert hot.tolist() == [1, 1, 0, 0, 0]
    assert dst.tolist() == [1, -1]
    assert wp.tolist() == [27 - 18 / 2, 2 + 9.0]


def test_invariants_on_random_layers():
    rs = np.random.RandomState(3)
    for trial in range(300):
        G = int(rs.randint(2, 9))
        E = G * int(rs.randint(1, 9))
        g = rs.permutation(np.repeat(np.arange(G), E // G))
        W = rs.randint(0, 50, size=E) * (rs.random_sample(E) < 0.9)
        W[rs.randint(0, E)] += int(rs.randint(0, 400))   # one hot expert now and then
        n, src, hot, dst, wp = rp.plan_layer(W, g, G)
        Wg = np.bincount(g, weights=W, minlength=G)
        if Wg.max() == 0:
            assert n == 0
            continue
        assert Wg[src] == Wg.max() and src == int(np.argmax(Wg))
        rho = Wg.max() / Wg.mean()
        if abs(rho - round(rho)) > 1e-9:                 # away from integer boundaries
            assert n == min(max(1, int(np.floor(rho))), G - 1)
        hot_e = np.flatnonzero(hot)
        assert (g[hot_e] == src).all() and len(hot_e) >= 1
        H = W[hot_e].sum()
        thr = Wg.max() * n / (1 + n)
        assert H > thr - 1e-9                            # the hot load passes the threshold
        assert H - W[hot_e].min() <= thr + 1e-9          # ... and no hot expert is spare
        rest = W[(g == src) & (hot == 0)]
        assert rest.size == 0 or rest.max() <= W[hot_e].min()
        others = [x for x in range(G) if x != src]
        order = sorted(others, key=lambda x: (Wg[x], x))
        assert dst[:n].tolist() == order[:n] and (dst[n:] == -1).all()
        assert abs(wp.sum() - Wg.sum()) <= 1e-9 * max(1.0, Wg.sum())
        assert abs(wp[src] - (Wg[src] - H * n / (1 + n))) <= 1e-9 * max(1.0, Wg[src])
