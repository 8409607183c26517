"""Host-side logic of the synthetic workloads: block tables, cache slots, generator twin."""
import numpy as np
import pytest

import gen


@pytest.mark.parametrize("cfg,R", [("c1", None), ("c2", 40), ("c3", 30), ("c4", 300), ("c5", 3)])
def test_batch_structure(cfg, R):
    wl = gen.make_workload(cfg, R=R)
    b = wl.batch()
    B = wl.B
    # blocks tile every request's computed tokens in order, B tokens each but the last
    tok = 0
    for r in range(b.R):
        n = b.req_off[r + 1] - b.req_off[r]
        blks = b.blk_tab[b.req_blk_off[r]:b.req_blk_off[r + 1]]
        assert len(blks) == (n + B - 1) // B
        for j, (t0, ln) in enumerate(blks):
            assert t0 == tok and 1 <= ln <= B and (ln == B or j == len(blks) - 1)
            tok += ln
    assert tok == b.T
    # only full blocks get a slot; slots are used once; cached slots were inserted earlier
    full = b.blk_tab[:, 1] == B
    assert (b.insert_slot[~full] == -1).all()
    ins = b.insert_slot[b.insert_slot >= 0]
    assert len(np.unique(ins)) == len(ins)
    first_block_of = {}
    for r in range(b.R):
        for bb in range(b.req_blk_off[r], b.req_blk_off[r + 1]):
            if b.insert_slot[bb] >= 0:
                first_block_of[int(b.insert_slot[bb])] = r
    for r in range(b.R):
        for c in b.cache_idx[b.req_cache_off[r]:b.req_cache_off[r + 1]]:
            assert first_block_of[int(c)] < r


def test_chunks_cover_requests():
    wl = gen.make_workload("c4", R=500)
    ch = wl.chunks(100_000)
    assert ch[0][0] == 0 and ch[-1][1] == wl.R
    assert all(a[1] == b[0] for a, b in zip(ch, ch[1:]))


def test_prefix_tokens_share_donor_keys():
    wl = gen.make_workload("c4", R=400)
    r = int(np.flatnonzero(wl.cached_blocks > 0)[0])
    d = int(wl.donor[r])
    n = int(wl.cached_blocks[r]) * wl.B
    assert np.array_equal(wl.prompt_keys(r)[:n], wl.prompt_keys(d)[:n])
    assert wl.dom[r] == wl.dom[d]


def test_generator_twin_rows_and_moments():
    wl = gen.make_workload("c3", R=3)
    b = wl.batch()
    full = gen.host_logits(wl, b.tok_key[:50], b.tok_dom[:50])
    rows = gen.host_logit_rows(wl, b.tok_key, b.tok_dom, [0, 5, 47], [0, 10, 49])
    assert np.array_equal(rows, full[[0, 5, 47], [0, 10, 49]])
    # unbiased experts: N(0,1) moments; values are multiples of 2^-16 within [-6, 6)
    biased = wl.bias_mask[b.tok_dom[:50]].transpose(1, 0, 2)  # [L][50][E]
    x = full[biased == 0]
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    assert np.all(x * 65536 == np.rint(x * 65536)) and x.min() >= -6 and x.max() < 6
