"""Helpers shared by the GPU parity tests (imported lazily, GPU only)."""
from __future__ import annotations

import numpy as np
import torch

import gen

REL_TOL = 1e-5    # signatures and distances: relative tolerance (fp32 path vs fp64 oracle)
ABS_FLOOR = 1e-7  # absolute floor for entries close to zero
BAND_EDGE = 1e-5  # decoder choices may differ only where a distance is this close to the band edge


def stream_handle():
    return torch.cuda.current_stream().cuda_stream


def device_logits(wl, b, out=None):
    """The batch's logits [L][T][E], filled on the GPU by the generator's device twin."""
    tk = torch.from_numpy(np.ascontiguousarray(b.tok_key)).cuda()
    td = torch.from_numpy(np.ascontiguousarray(b.tok_dom)).cuda()
    bm = torch.from_numpy(np.ascontiguousarray(wl.bias_mask.reshape(-1))).cuda()
    if out is None:
        out = torch.empty((wl.L, b.T, wl.E), dtype=torch.float32, device="cuda")
    gen.dev_logits(wl, tk, td, out, bm, stream=stream_handle())
    return out


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_close(gpu, ref, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    lim = REL_TOL * np.abs(ref) + ABS_FLOOR
    bad = err > lim
    assert not bad.any(), f"{what}: {int(bad.sum())} entries beyond tolerance, worst {err.max():.3e}"


def band_edge_rows(dist_ref, tau):
    """Requests whose oracle distances put some decoder within BAND_EDGE of the band edge
    (NaN distances are outside every band and do not define the minimum)."""
    with np.errstate(invalid="ignore"):
        dmin = np.fmin.reduce(dist_ref, axis=1, keepdims=True)
    return (np.abs(dist_ref - (dmin + tau)) <= BAND_EDGE).any(axis=1)


def valid_choice(q, dist_row, tau, loads):
    """True if q is the tau-band least-loaded pick for some band between the edge tolerances."""
    if q < 0:
        return bool(np.isnan(dist_row).all())
    dmin = np.fmin.reduce(dist_row)
    hi = dist_row <= dmin + tau + BAND_EDGE
    lo = dist_row <= dmin + tau - BAND_EDGE
    if not hi[q]:
        return False
    for d in np.flatnonzero(lo):
        if (loads[d], d) < (loads[q], q):
            return False
    return True


def check_static_route(choice, dist_ref, tau, loads, oracle_choice):
    edge = band_edge_rows(dist_ref, tau)
    diff = choice != oracle_choice
    assert not (diff & ~edge).any(), f"decoder choices differ off the band edge: {np.flatnonzero(diff & ~edge)[:10]}"
    for r in np.flatnonzero(diff):
        assert valid_choice(int(choice[r]), dist_ref[r], tau, loads), r
    return int(edge.sum()), int(diff.sum())


def check_live_route(choice, dist_ref, tau, loads0, oracle_choice):
    """Exact match up to the first band-edge divergence; valid picks after it."""
    edge = band_edge_rows(dist_ref, tau)
    diff = np.flatnonzero(choice != oracle_choice)
    if len(diff) == 0:
        return int(edge.sum()), 0
    first = int(diff[0])
    assert edge[first], f"live routing diverged off the band edge at request {first}"
    loads = np.array(loads0, dtype=np.int64)
    for r in range(len(choice)):
        q = int(choice[r])
        if r >= first:
            assert valid_choice(q, dist_ref[r], tau, loads), f"invalid live pick at request {r}"
        loads[q] += 1
    return int(edge.sum()), len(diff)


def _gate_rows(args):
    import oracle
    x, w = args
    return oracle.get().gate_logits(x, w)


def oracle_gate_logits(x, w, nproc=None):
    """The oracle's gate logits [L][T][E], token ranges spread over spawned worker processes
    (the oracle itself is single-threaded; spawn, because this process holds a CUDA context;
    an executor, so a worker that dies raises instead of leaving the pool waiting)."""
    import multiprocessing as mp
    import os
    from concurrent.futures import ProcessPoolExecutor
    T = x.shape[0]
    nproc = nproc or max(1, min(16, os.cpu_count() or 1))
    cuts = np.linspace(0, T, min(nproc, T) + 1).astype(int)
    parts = [(x[a:z], w) for a, z in zip(cuts[:-1], cuts[1:]) if z > a]
    if len(parts) == 1:
        return _gate_rows(parts[0])
    with ProcessPoolExecutor(len(parts), mp_context=mp.get_context("spawn")) as ex:
        outs = list(ex.map(_gate_rows, parts, timeout=900))
    return np.concatenate(outs, axis=1)
