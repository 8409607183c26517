"""Pins of the greedy layer-mask oracle (oracle/mask_select.py): hand-computed cosines,
closed cases (identical halves, disjoint halves, one-token requests), invariance to the idf
scale, informative layers chosen before noise layers, ties to the lower layer, and each
greedy step checked as the best single addition.
"""
import numpy as np

from oracle import mask_select as ms


def test_hand_cosines():
    # one request of 4 tokens, k = 1, E = 4
    same = np.array([[[0], [1], [0], [1]]], dtype=np.uint8)       # halves {0,1} and {0,1}
    apart = np.array([[[0], [0], [1], [1]]], dtype=np.uint8)      # halves {0,0} and {1,1}
    mixed = np.array([[[0], [1], [0], [2]]], dtype=np.uint8)      # [1,1,0,0] vs [1,0,1,0]
    off = np.array([0, 4])
    c1, c2 = ms.half_counts(same, off, 4)
    assert c1.tolist() == [[[1, 1, 0, 0]]] and c2.tolist() == [[[1, 1, 0, 0]]]
    assert abs(ms.quality(c1, c2, np.ones((1, 4)), [0]) - 1.0) < 1e-15
    c1, c2 = ms.half_counts(apart, off, 4)
    assert ms.quality(c1, c2, np.ones((1, 4)), [0]) == 0.0
    c1, c2 = ms.half_counts(mixed, off, 4)
    assert abs(ms.quality(c1, c2, np.ones((1, 4)), [0]) - 0.5) < 1e-15   # 1 / (sqrt2 sqrt2)


def test_odd_lengths_and_one_token_requests():
    topk = np.array([[[3], [1], [1], [2]]], dtype=np.uint8)
    # request 0 = token 0 (halves: {} and {3}); request 1 = tokens 1..3 (halves {1} and {1, 2})
    c1, c2 = ms.half_counts(topk, np.array([0, 1, 4]), 4)
    assert c1[0, 0].tolist() == [0, 0, 0, 0] and c2[0, 0].tolist() == [0, 0, 0, 1]
    assert c1[1, 0].tolist() == [0, 1, 0, 0] and c2[1, 0].tolist() == [0, 1, 1, 0]
    q = ms.quality(c1, c2, np.ones((1, 4)), [0])
    assert abs(q - (0.0 + 1 / np.sqrt(2)) / 2) < 1e-15


def _domain_case(seed=0):
    """Layers 0, 2, 4 carry a per-request expert set (the same in both halves); layers
    1, 3, 5 pick experts at random per token."""
    rs = np.random.RandomState(seed)
    L, E, k, R = 6, 16, 2, 40
    lens = rs.randint(4, 30, size=R)
    off = np.concatenate([[0], np.cumsum(lens)])
    T = off[-1]
    topk = np.zeros((L, T, k), dtype=np.uint8)
    for r in range(R):
        pref = rs.choice(E, size=k, replace=False)
        for t in range(off[r], off[r + 1]):
            for l in range(L):
                topk[l, t] = pref if l % 2 == 0 else rs.choice(E, size=k, replace=False)
    return topk, off, E


def test_informative_layers_first():
    topk, off, E = _domain_case()
    chosen, qual = ms.greedy_mask(topk, off, E, 6)
    assert sorted(chosen[:3].tolist()) == [0, 2, 4]
    assert abs(qual[0] - 1.0) < 1e-12          # a consistent layer alone: cosine 1 everywhere
    assert qual[3] < qual[2]                   # a noise layer can only dilute it


def test_greedy_steps_are_best_single_additions():
    topk, off, E = _domain_case(3)
    idf = 1.0 + np.random.RandomState(4).random_sample((6, E))
    chosen, qual = ms.greedy_mask(topk, off, E, 4, idf)
    c1, c2 = ms.half_counts(topk, off, E)
    for step in range(4):
        prefix = chosen[:step].tolist()
        cands = {l: ms.quality(c1, c2, idf, prefix + [l]) for l in range(6) if l not in prefix}
        best = max(cands.values())
        assert cands[int(chosen[step])] == best
        assert int(chosen[step]) == min(l for l, q in cands.items() if q == best)
        assert qual[step] == best


def test_idf_scale_invariance_and_ties():
    topk, off, E = _domain_case(5)
    idf = 1.0 + np.random.RandomState(6).random_sample((6, E))
    a, qa = ms.greedy_mask(topk, off, E, 3, idf)
    b, qb = ms.greedy_mask(topk, off, E, 3, 7.0 * idf)
    assert np.array_equal(a, b) and np.allclose(qa, qb, rtol=1e-12)
    # two identical layers tie at every step: the lower index goes first
    dup = np.concatenate([topk[:1], topk[:1], topk[1:2]])
    c, _ = ms.greedy_mask(dup, off, E, 2)
    assert c.tolist() == [0, 1]


def test_identical_halves_give_quality_one():
    rs = np.random.RandomState(7)
    L, E, k = 3, 8, 2
    first = rs.randint(0, E, size=(L, 5, k)).astype(np.uint8)
    topk = np.concatenate([first, first], axis=1)   # one request: second half repeats the first
    chosen, qual = ms.greedy_mask(topk, np.array([0, 10]), E, 3)
    assert np.allclose(qual, 1.0, atol=1e-12)
