"""Edge cases of the fused top-k / block-count / co-activation call against the oracle.

Shapes off the fast path (E from 4 to 256, k from 1 to 32), tie-heavy and
special-valued logits (NaN, +-inf, -0.0/+0.0), length-1 requests, partial
blocks, B = 1 and B = 255, an empty layer mask, a single token, and
malformed block tables (the bad blocks are skipped and reported through
the workspace status, never a fault).
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import _native as nat
    return torch, nat


def _blocks(lengths, B):
    req_off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    tab = []
    for r in range(len(lengths)):
        for t0 in range(req_off[r], req_off[r + 1], B):
            tab.append((t0, min(B, req_off[r + 1] - t0)))
    return req_off, np.array(tab, dtype=np.int32).reshape(-1, 2)


def _logits(rs, kind, L, T, E):
    if kind == "normal":
        x = rs.standard_normal((L, T, E)).astype(np.float32)
    elif kind == "ties":
        x = rs.randint(-2, 3, size=(L, T, E)).astype(np.float32)
    elif kind == "equal":
        x = np.full((L, T, E), 0.5, dtype=np.float32)
    else:  # specials mixed into small integers
        x = rs.randint(-3, 4, size=(L, T, E)).astype(np.float32)
        sp = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0, 1e-45, -1e-45], dtype=np.float32)
        hit = rs.random_sample(x.shape) < 0.2
        x[hit] = sp[rs.randint(0, len(sp), size=int(hit.sum()))]
    return x


def _run(env, x, k, lengths, B, mask, want_aff=True, want_topk=True):
    torch, nat = env
    L, T, E = x.shape
    req_off, tab = _blocks(lengths, B)
    dims = nat.make_dims(E, k, L, mask, B)
    m = len(mask)
    dx = torch.from_numpy(x).cuda()
    dtab = torch.from_numpy(tab.reshape(-1)).cuda()
    topk = torch.full((L, T, k), 255, dtype=torch.uint8, device="cuda")
    cnt = torch.full((max(len(tab), 1), max(m, 1), E), 77, dtype=torch.uint8, device="cuda")
    aff = torch.zeros((L, E, E), dtype=torch.int32, device="cuda") if want_aff else None
    wsb = nat.moer_workspace_bytes(dims, T, len(tab), 0, 0)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_topk_signature(dims, dx, T, dtab, len(tab), topk if want_topk else None,
                            cnt if m else None, aff, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    orc = oracle.get()
    tk = orc.topk(x, k)
    if want_topk:
        assert np.array_equal(topk.cpu().numpy(), tk)
    else:
        assert (topk == 255).all()
    if m:
        bc = orc.block_counts(tk, E, req_off, B, mask)
        assert np.array_equal(cnt.cpu().numpy()[:len(tab)], bc)
    if want_aff:
        assert np.array_equal(aff.cpu().numpy().astype(np.int64), orc.affinity(tk, E))


SHAPES = [  # (E, k, L)
    (4, 1, 2), (8, 8, 2), (12, 5, 3), (32, 32, 2), (64, 8, 3), (64, 6, 3), (64, 1, 2),
    (64, 32, 2), (100, 7, 2), (128, 8, 3), (128, 2, 2), (128, 32, 2), (200, 9, 2), (256, 8, 2),
    (256, 32, 2),
]


@pytest.mark.parametrize("E,k,L", SHAPES, ids=[f"E{e}k{k}" for e, k, _ in SHAPES])
@pytest.mark.parametrize("kind", ["normal", "ties", "specials"])
def test_shapes_and_values(env, E, k, L, kind):
    rs = np.random.RandomState(E * 131 + k * 7 + L)
    lengths = [1, 17, 16, 3, 40, 1, 129, 64, 2]
    T = sum(lengths)
    x = _logits(rs, kind, L, T, E)
    mask = list(range(0, L, 2))
    _run(env, x, k, lengths, 16, mask)


@pytest.mark.parametrize("E,k", [(128, 8), (64, 6), (64, 8)])
def test_all_equal_logits(env, E, k):
    rs = np.random.RandomState(3)
    x = _logits(rs, "equal", 2, 300, E)
    _run(env, x, k, [100, 200], 16, [1])


@pytest.mark.parametrize("B", [1, 5, 64, 255])
def test_block_sizes(env, B):
    rs = np.random.RandomState(B)
    lengths = [1, 300, 255, 256, 7, 512]
    x = _logits(rs, "normal", 2, sum(lengths), 128)
    _run(env, x, 8, lengths, B, [0, 1])


def test_single_token_and_empty_mask(env):
    rs = np.random.RandomState(9)
    _run(env, _logits(rs, "normal", 3, 1, 128), 8, [1], 16, [2])
    _run(env, _logits(rs, "normal", 3, 50, 64), 6, [50], 16, [])
    _run(env, _logits(rs, "normal", 3, 50, 64), 6, [20, 30], 16, [0, 1, 2], want_aff=False)


@pytest.mark.parametrize("E,k", [(128, 8), (64, 6), (100, 5)])
def test_block_counts_without_topk_output(env, E, k):
    rs = np.random.RandomState(31 + E)
    lengths = [5, 33, 16, 90]
    x = _logits(rs, "normal", 4, sum(lengths), E)
    _run(env, x, k, lengths, 16, [1, 3], want_topk=False)


def test_many_tiles_ragged_tail(env):
    rs = np.random.RandomState(21)
    lengths = list(rs.randint(1, 200, size=60))
    x = _logits(rs, "normal", 5, sum(lengths), 128)
    _run(env, x, 8, lengths, 16, [0, 3, 4])


def test_malformed_block_table_is_reported(env):
    torch, nat = env
    E, k, L, T = 128, 8, 2, 64
    dims = nat.make_dims(E, k, L, [0], 16)
    x = torch.randn((L, T, E), device="cuda")
    bad = torch.tensor([0, 16, 16, 16, 40, 16, 48, 16], dtype=torch.int32, device="cuda")  # gap at 32
    cnt = torch.full((4, 1, E), 7, dtype=torch.uint8, device="cuda")
    topk = torch.full((L, T, k), 255, dtype=torch.uint8, device="cuda")
    wsb = nat.moer_workspace_bytes(dims, T, 4, 0, 0)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_topk_signature(dims, x, T, bad, 4, topk, cnt, None, ws, wsb)
    assert nat.moer_ws_status(ws) == 6  # MOER_EDATA
    # the malformed blocks are skipped; the good ones and the top-k are produced
    c = cnt.cpu().numpy().astype(np.int64)
    assert (c[2:] == 7).all()
    assert (c[:2].sum(axis=2) == k * 16).all()
    tk = oracle.get().topk(x.cpu().numpy(), k)
    assert np.array_equal(topk.cpu().numpy(), tk)
    # the status word is cleared by the read; a good call afterwards succeeds
    good = torch.tensor([0, 16, 16, 16, 32, 16, 48, 16], dtype=torch.int32, device="cuda")
    nat.moer_topk_signature(dims, x, T, good, 4, topk, cnt, None, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    assert (cnt.cpu().numpy().astype(np.int64).sum(axis=2) == k * 16).all()


def test_stitch_bad_slot_is_reported(env):
    torch, nat = env
    E, m = 64, 1
    dims = nat.make_dims(E, 8, 1, [0], 16)
    blk = torch.ones((2, m, E), dtype=torch.uint8, device="cuda")
    tab = torch.tensor([0, 16, 16, 16], dtype=torch.int32, device="cuda")
    rbo = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    cache = torch.zeros((3, m, E), dtype=torch.uint8, device="cuda")
    cidx = torch.tensor([5], dtype=torch.int32, device="cuda")      # out of range
    rco = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    ins = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    out = torch.empty((1, m, E), dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    nat.moer_block_stitch(dims, blk, tab, 2, rbo, 1, cidx, 1, rco, cache, 3, ins, out, ws, 256)
    assert nat.moer_ws_status(ws) == 6
    assert (out == 2).all()


@pytest.mark.parametrize("rco_vals", [[0, 5], [-1, 1], [1, 0]])
def test_stitch_bad_cache_offsets_are_reported(env, rco_vals):
    """A request whose cached-prefix range is not within [0, ncached) has its cached part
    skipped (its computed blocks are still summed) and MOER_EDATA is recorded; no cache_idx
    entry outside the buffer is read."""
    torch, nat = env
    E, m = 64, 1
    dims = nat.make_dims(E, 8, 1, [0], 16)
    blk = torch.ones((2, m, E), dtype=torch.uint8, device="cuda")
    tab = torch.tensor([0, 16, 16, 16], dtype=torch.int32, device="cuda")
    rbo = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    cache = torch.full((3, m, E), 9, dtype=torch.uint8, device="cuda")
    cidx = torch.tensor([1], dtype=torch.int32, device="cuda")      # one cached block
    rco = torch.tensor(rco_vals, dtype=torch.int32, device="cuda")
    out = torch.empty((1, m, E), dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    nat.moer_block_stitch(dims, blk, tab, 2, rbo, 1, cidx, 1, rco, cache, 3, None, out, ws, 256)
    assert nat.moer_ws_status(ws) == 6
    assert (out == 2).all()                                         # computed blocks only
    # the well-formed range sums the cached block too, and reports nothing
    rco = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    nat.moer_block_stitch(dims, blk, tab, 2, rbo, 1, cidx, 1, rco, cache, 3, None, out, ws, 256)
    assert nat.moer_ws_status(ws) == 0
    assert (out == 11).all()


@pytest.mark.parametrize("m,E", [(26, 128), (3, 4), (2, 8), (12, 128)])
def test_stitch_record_shapes(env, m, E):
    """moer_block_stitch against O3 on records of every launch shape: 26 x 128 counts
    (3,328 B: two thread groups per request), 3 x 4 and 2 x 8 (12 and 16 B: 4-byte words /
    16-byte words with one word per record), and 12 x 128 (the path's).  Ragged requests,
    cached prefixes read from pre-filled slots, full blocks inserted into fresh slots."""
    torch, nat = env
    orc = oracle.get()
    B, R = 16, 50
    rs = np.random.RandomState(m * 1000 + E)
    lens = rs.randint(1, 120, size=R)
    req_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tab, rbo = [], [0]
    for r in range(R):
        for t0 in range(req_off[r], req_off[r + 1], B):
            tab.append((t0, min(B, req_off[r + 1] - t0)))
        rbo.append(len(tab))
    tab = np.array(tab, dtype=np.int32)
    nblk = len(tab)
    blk = rs.randint(0, B + 1, size=(nblk, m, E)).astype(np.uint8)
    npre = 40
    ncache = rs.randint(0, 6, size=R)
    rco = np.concatenate([[0], np.cumsum(ncache)]).astype(np.int32)
    cidx = rs.randint(0, npre, size=int(rco[-1])).astype(np.int32)
    full = tab[:, 1] == B
    ins = np.full(nblk, -1, dtype=np.int32)
    ins[full] = npre + np.arange(int(full.sum()))
    ins[rs.random_sample(nblk) < 0.2] = -1                 # some full blocks are not cached
    nslots = npre + int(full.sum())
    cache0 = np.zeros((nslots, m, E), dtype=np.uint8)
    cache0[:npre] = rs.randint(0, B + 1, size=(npre, m, E))
    dims = nat.make_dims(E, 1, m, list(range(m)), B)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    cache = d(cache0)
    out = torch.empty((R, m, E), dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    nat.moer_block_stitch(dims, d(blk), d(tab.reshape(-1)), nblk, d(np.array(rbo, np.int32)), R,
                          d(cidx), len(cidx), d(rco), cache, nslots, d(ins), out, ws, 256)
    assert nat.moer_ws_status(ws) == 0
    ocache = cache0.copy()
    ref = orc.stitch(blk, req_off, B, cidx, rco, ocache, ins)
    assert np.array_equal(out.cpu().numpy(), ref)
    assert np.array_equal(cache.cpu().numpy(), ocache)
