"""The tensor-core gate GEMM with fused top-k (moer_gate_topk) against the oracle.

Logits: |gpu - oracle| <= 1e-2 |oracle| + 1e-3 rms(row) (the oracle sums the
bf16 products in double).  Top-k ids: identical to the oracle's wherever the
oracle's logits order the k+1 leading experts with gaps above 1e-3; where
only the k-th / (k+1)-th gap exceeds 1e-3 the sets must agree; elsewhere the
GPU's ids must be a valid top-k of the GPU's own logits (checked with
numpy).  Block counts and co-activation counts must equal the oracle's on
the GPU's ids' own definition (counted here with numpy) and the oracle's
wherever the top-k is unambiguous.
"""
import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu

MARGIN = 1e-3


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import _native as nat
    return torch, nat


def _run(env, T, H, L, k, mask, lengths=None, seed=5, want_logits=True):
    torch, nat = env
    E, B = 128, 16
    x = gen.host_hidden(seed, 0, T, H)
    w = gen.host_wgate(seed, L, H, E, 0.02)
    dims = nat.make_dims(E, k, L, mask, B)
    lengths = lengths or [T]
    req_off = np.concatenate([[0], np.cumsum(lengths)])
    tab = np.array([(t0, min(B, req_off[r + 1] - t0)) for r in range(len(lengths))
                    for t0 in range(req_off[r], req_off[r + 1], B)], dtype=np.int32)
    dx = torch.from_numpy(x.view(np.int16)).cuda()
    dw = torch.from_numpy(w.view(np.int16)).cuda()
    dtab = torch.from_numpy(tab.reshape(-1)).cuda()
    logits = torch.empty((L, T, E), dtype=torch.float32, device="cuda") if want_logits else None
    topk = torch.full((L, T, k), 255, dtype=torch.uint8, device="cuda")
    cnt = torch.zeros((len(tab), len(mask), E), dtype=torch.uint8, device="cuda")
    aff = torch.zeros((L, E, E), dtype=torch.int32, device="cuda")
    wsb = nat.moer_gate_workspace_bytes(dims, H)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_gate_topk(dims, dx, T, H, dw, dtab, len(tab), logits, topk, cnt, aff, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    return x, w, req_off, tab, (logits.cpu().numpy() if want_logits else None), topk.cpu().numpy(), \
        cnt.cpu().numpy(), aff.cpu().numpy()


def _check(env, T, H, L, k, mask, lengths=None, rows=None):
    x, w, req_off, tab, lg, tk, cnt, aff = _run(env, T, H, L, k, mask, lengths)
    orc = oracle.get()
    ref = orc.gate_logits(x, w)                                   # [L][T][E] fp32 of fp64 sums
    rms = np.sqrt((ref.astype(np.float64) ** 2).mean(axis=2, keepdims=True))
    err = np.abs(lg.astype(np.float64) - ref)
    assert (err <= 1e-2 * np.abs(ref) + 1e-3 * rms).all(), f"logits: worst {err.max():.3e}"
    otk = orc.topk(ref, k)
    srt = -np.sort(-ref.astype(np.float64), axis=2)[:, :, :k + 1]
    gaps = srt[:, :, :-1] - srt[:, :, 1:]
    order_ok = (gaps > MARGIN).all(axis=2)
    set_ok = gaps[:, :, k - 1] > MARGIN
    assert np.array_equal(tk[order_ok], otk[order_ok]), "ordered top-k"
    assert np.array_equal(np.sort(tk[set_ok], axis=1), np.sort(otk[set_ok], axis=1)), "top-k sets"
    # every row: a valid top-k of the GPU's own fp32 logits (ties to the lower id)
    own = np.argsort(-lg, axis=2, kind="stable")[:, :, :k].astype(np.uint8)
    assert np.array_equal(tk, own), "top-k of own logits"
    # counts and co-activation from the GPU's ids, by definition
    for i, layer in enumerate(mask):
        for b, (t0, ln) in enumerate(tab):
            assert np.array_equal(cnt[b, i], np.bincount(tk[layer, t0:t0 + ln].reshape(-1), minlength=128))
    for layer in range(L):
        X = np.zeros((T, 128), dtype=np.int64)
        X[np.repeat(np.arange(T), k), tk[layer].reshape(-1)] = 1
        assert np.array_equal(aff[layer].astype(np.int64), X.T @ X)
    return int((~set_ok).sum())


@pytest.mark.parametrize("T,H,L,k", [(128, 64, 2, 8), (300, 256, 3, 8), (200, 128, 2, 6), (1024, 2048, 4, 8)])
def test_gate_small(env, T, H, L, k):
    amb = _check(env, T, H, L, k, mask=list(range(0, L, 2)), lengths=None)
    print(f"T={T} H={H} L={L} k={k}: ambiguous rows {amb}")


def test_gate_ragged_requests(env):
    _check(env, 777, 512, 3, 8, mask=[1], lengths=[5, 100, 16, 300, 356])


def _bf16_bits(a):
    """Small integers as bf16 bit patterns (exact)."""
    return (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("lo,hi,k", [(0, 3, 8), (-2, 3, 8), (0, 2, 6), (-1, 2, 6)])
def test_gate_integer_ties(env, lo, hi, k):
    """Hidden states and weights that are small integers give exact integer logits with many
    ties, so the GPU must reproduce the oracle's ranking on every row: equal logits rank the
    lower expert first.  Rows of zeros and negative values reach the full exact pass; positive
    ties reach the candidate-filtered one."""
    torch, nat = env
    T, H, L, E = 520, 128, 3, 128
    rs = np.random.RandomState(100 + lo * 10 + hi + k)
    xi = rs.randint(lo, hi, size=(T, H))
    xi[:40] = 0                                                 # all-zero rows: every logit ties at 0
    wi = rs.randint(0, 2, size=(L, H, E)) * rs.randint(-1 if lo < 0 else 0, 2, size=(L, H, E))
    x, w = _bf16_bits(xi), _bf16_bits(wi)
    dims = nat.make_dims(E, k, L, [0], 16)
    dx = torch.from_numpy(x.view(np.int16)).cuda()
    dw = torch.from_numpy(w.view(np.int16)).cuda()
    tab = np.array([(t0, min(16, T - t0)) for t0 in range(0, T, 16)], dtype=np.int32)
    dtab = torch.from_numpy(tab.reshape(-1)).cuda()
    logits = torch.empty((L, T, E), dtype=torch.float32, device="cuda")
    topk = torch.full((L, T, k), 255, dtype=torch.uint8, device="cuda")
    cnt = torch.zeros((len(tab), 1, E), dtype=torch.uint8, device="cuda")
    wsb = nat.moer_gate_workspace_bytes(dims, H)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    nat.moer_gate_topk(dims, dx, T, H, dw, dtab, len(tab), logits, topk, cnt, None, ws, wsb)
    assert nat.moer_ws_status(ws) == 0
    ref = oracle.get().gate_logits(x, w)
    lg = logits.cpu().numpy()
    assert np.array_equal(lg, ref.astype(np.float32)), "integer logits are exact"
    assert np.array_equal(topk.cpu().numpy(), oracle.get().topk(ref, k))
