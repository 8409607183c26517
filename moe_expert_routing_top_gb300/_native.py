"""ctypes binding of libmoeroute's C ABI (argument marshalling only).

Every function here has the name of the C entry point it calls and forwards
device pointers (torch tensors' `data_ptr()`), sizes and the CUDA stream
handle.  There is no fallback: if the shared library is missing the import
fails, and a non-zero status raises `MoerError`.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("MOER_LIBRARY", os.path.join(HERE, "_build", "libmoeroute.so"))

STATUS = {0: "MOER_OK", 1: "MOER_EINVAL", 2: "MOER_ESHAPE", 3: "MOER_ERANGE", 4: "MOER_ECUDA",
          5: "MOER_ENOMEM", 6: "MOER_EDATA", 7: "MOER_ETIMEOUT", 8: "MOER_EEXTENT"}


class MoerError(RuntimeError):
    def __init__(self, fn: str, code: int, text: str):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({text})")
        self.code = code


class moer_dims(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("k", ctypes.c_int32), ("L", ctypes.c_int32),
                ("m", ctypes.c_int32), ("mask", ctypes.POINTER(ctypes.c_int32)),
                ("block", ctypes.c_int32)]


def make_dims(E: int, k: int, L: int, mask, block: int = 16) -> moer_dims:
    """Builds the dims struct; the mask array is kept alive on the struct."""
    mask = [int(x) for x in mask]
    arr = (ctypes.c_int32 * max(len(mask), 1))(*mask)
    d = moer_dims(E, k, L, len(mask), ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32)), block)
    d._mask_keepalive = arr
    return d


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoeroute is not built ({LIB_PATH} missing); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
    dp = ctypes.POINTER(moer_dims)
    sigs = {
        "moer_workspace_bytes": ([dp, i64, i32, i32, i32], sz),
        "moer_topk_signature": ([dp, vp, i64, vp, i32, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "moer_topk_signature_noalloc": ([dp, vp, i64, vp, i32, vp, vp, vp, vp], ctypes.c_int),
        "moer_block_stitch": ([dp, vp, vp, i32, vp, i32, vp, i32, vp, vp, i32, vp, vp, vp, sz, vp],
                              ctypes.c_int),
        "moer_affinity_load": ([dp, vp, vp, i32, vp, vp, vp, vp, vp], ctypes.c_int),
        "moer_route": ([dp, vp, i32, vp, vp, i32, f32, vp, i32, vp, vp, vp, vp, sz, vp],
                       ctypes.c_int),
        "moer_idf_fit": ([dp, vp, i32, vp, vp], ctypes.c_int),
        "moer_gate_workspace_bytes": ([dp, i32], sz),
        "moer_gate_topk": ([dp, vp, i64, i32, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "moer_ids_signature": ([dp, vp, i64, vp, i32, vp, vp, vp, sz, vp], ctypes.c_int),
        "moer_spectral_workspace_bytes": ([dp, i32], sz),
        "moer_spectral_groups": ([dp, vp, i32, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "moer_mask_select_workspace_bytes": ([dp, i32], sz),
        "moer_mask_select": ([dp, vp, i64, vp, i32, vp, i32, vp, vp, vp, sz, vp], ctypes.c_int),
        "moer_replication_plan": ([dp, vp, vp, i32, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "moer_kmeans_workspace_bytes": ([i32, i32, i32], sz),
        "moer_kmeans_balanced": ([vp, i32, i32, i32, vp, i32, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "moer_ws_status": ([vp, vp], ctypes.c_int),
        "moer_wait_selftest": ([vp, sz, ctypes.c_uint32, vp], ctypes.c_int),
        "moer_status_str": ([ctypes.c_int], ctypes.c_char_p),
        "moer_version": ([], ctypes.c_int32),
        "moer_set_extent_checks": ([i32], None),
        "moer_extent_checks": ([], ctypes.c_int32),
        "moer_buffer_holds": ([vp, sz], ctypes.c_int32),
    }
    for name, (args, res) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


LIB = _load()
EXPORTS = ("moer_workspace_bytes", "moer_topk_signature", "moer_topk_signature_noalloc",
           "moer_block_stitch", "moer_affinity_load",
           "moer_route", "moer_idf_fit", "moer_gate_workspace_bytes", "moer_gate_topk",
           "moer_ids_signature",
           "moer_replication_plan", "moer_kmeans_workspace_bytes", "moer_kmeans_balanced",
           "moer_mask_select_workspace_bytes", "moer_mask_select", "moer_spectral_workspace_bytes",
           "moer_spectral_groups",
           "moer_ws_status", "moer_wait_selftest",
           "moer_status_str", "moer_version", "moer_set_extent_checks", "moer_extent_checks",
           "moer_buffer_holds")


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return s if isinstance(s, int) else s.cuda_stream


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise MoerError(fn, code, LIB.moer_status_str(code).decode())


def moer_workspace_bytes(dims, T: int = 0, nblk: int = 0, R: int = 0, D: int = 0) -> int:
    return int(LIB.moer_workspace_bytes(ctypes.byref(dims), T, nblk, R, D))


def moer_topk_signature(dims, logits, T, blk_tab, nblk, topk, blk_cnt, affinity, ws, ws_bytes,
                        stream=None) -> None:
    _check("moer_topk_signature", LIB.moer_topk_signature(
        ctypes.byref(dims), _ptr(logits), int(T), _ptr(blk_tab), int(nblk), _ptr(topk),
        _ptr(blk_cnt), _ptr(affinity), _ptr(ws), int(ws_bytes), _stream(stream)))


def moer_topk_signature_noalloc(dims, logits, T, blk_tab, nblk, topk, blk_cnt, affinity,
                                stream=None) -> None:
    """moer_topk_signature without a workspace: the scratch is a fixed array inside the library,
    for callers that cannot allocate device memory (see include/moeroute.h)."""
    _check("moer_topk_signature_noalloc", LIB.moer_topk_signature_noalloc(
        ctypes.byref(dims), _ptr(logits), int(T), _ptr(blk_tab), int(nblk), _ptr(topk),
        _ptr(blk_cnt), _ptr(affinity), _stream(stream)))


def moer_block_stitch(dims, blk_cnt, blk_tab, nblk, req_blk_off, R, cache_idx, ncached, req_cache_off,
                      cache, nslots, insert_slot, req_cnt, ws, ws_bytes, stream=None) -> None:
    _check("moer_block_stitch", LIB.moer_block_stitch(
        ctypes.byref(dims), _ptr(blk_cnt), _ptr(blk_tab), int(nblk), _ptr(req_blk_off), int(R),
        _ptr(cache_idx), int(ncached), _ptr(req_cache_off), _ptr(cache), int(nslots), _ptr(insert_slot),
        _ptr(req_cnt), _ptr(ws), int(ws_bytes), _stream(stream)))


def moer_affinity_load(dims, affinity, group_of, G, W_expert, W_group, rho_group, rho_expert,
                       stream=None) -> None:
    _check("moer_affinity_load", LIB.moer_affinity_load(
        ctypes.byref(dims), _ptr(affinity), _ptr(group_of), int(G), _ptr(W_expert),
        _ptr(W_group), _ptr(rho_group), _ptr(rho_expert), _stream(stream)))


def moer_route(dims, req_cnt, R, idf, centroids, D, tau, loads, live, sig, dist, choice, ws,
               ws_bytes, stream=None) -> None:
    _check("moer_route", LIB.moer_route(
        ctypes.byref(dims), _ptr(req_cnt), int(R), _ptr(idf), _ptr(centroids), int(D),
        float(tau), _ptr(loads), int(live), _ptr(sig), _ptr(dist), _ptr(choice), _ptr(ws),
        int(ws_bytes), _stream(stream)))


def moer_idf_fit(dims, req_cnt, R, idf, stream=None) -> None:
    _check("moer_idf_fit", LIB.moer_idf_fit(ctypes.byref(dims), _ptr(req_cnt), int(R), _ptr(idf),
                                            _stream(stream)))


def moer_spectral_workspace_bytes(dims, G: int) -> int:
    return int(LIB.moer_spectral_workspace_bytes(ctypes.byref(dims), int(G)))


def moer_spectral_groups(dims, affinity, G, group_of, knee, u_curve, s_curve, ws, ws_bytes,
                         stream=None) -> None:
    _check("moer_spectral_groups", LIB.moer_spectral_groups(
        ctypes.byref(dims), _ptr(affinity), int(G), _ptr(group_of), _ptr(knee), _ptr(u_curve),
        _ptr(s_curve), _ptr(ws), int(ws_bytes), _stream(stream)))


def moer_mask_select_workspace_bytes(dims, R: int) -> int:
    return int(LIB.moer_mask_select_workspace_bytes(ctypes.byref(dims), int(R)))


def moer_mask_select(dims, topk, T, req_off, R, idf, m, mask_out, quality_out, ws, ws_bytes,
                     stream=None) -> None:
    _check("moer_mask_select", LIB.moer_mask_select(
        ctypes.byref(dims), _ptr(topk), int(T), _ptr(req_off), int(R), _ptr(idf), int(m),
        _ptr(mask_out), _ptr(quality_out), _ptr(ws), int(ws_bytes), _stream(stream)))


def moer_replication_plan(dims, W, group_of, G, n_rep, src, hot, dst, w_pred, ws, ws_bytes,
                          stream=None) -> None:
    _check("moer_replication_plan", LIB.moer_replication_plan(
        ctypes.byref(dims), _ptr(W), _ptr(group_of), int(G), _ptr(n_rep), _ptr(src), _ptr(hot),
        _ptr(dst), _ptr(w_pred), _ptr(ws), int(ws_bytes), _stream(stream)))


def moer_kmeans_workspace_bytes(N: int, dim: int, D: int) -> int:
    return int(LIB.moer_kmeans_workspace_bytes(int(N), int(dim), int(D)))


def moer_kmeans_balanced(sig, N, dim, D, init_centroids, max_iter, centroids, assign, info, objective,
                         ws, ws_bytes, stream=None) -> None:
    _check("moer_kmeans_balanced", LIB.moer_kmeans_balanced(
        _ptr(sig), int(N), int(dim), int(D), _ptr(init_centroids), int(max_iter), _ptr(centroids),
        _ptr(assign), _ptr(info), _ptr(objective), _ptr(ws), int(ws_bytes), _stream(stream)))


def moer_gate_workspace_bytes(dims, H: int) -> int:
    return int(LIB.moer_gate_workspace_bytes(ctypes.byref(dims), int(H)))


def moer_gate_topk(dims, hidden, T, H, w_gate, blk_tab, nblk, logits, topk, blk_cnt, affinity, ws,
                   ws_bytes, stream=None) -> None:
    _check("moer_gate_topk", LIB.moer_gate_topk(
        ctypes.byref(dims), _ptr(hidden), int(T), int(H), _ptr(w_gate), _ptr(blk_tab), int(nblk),
        _ptr(logits), _ptr(topk), _ptr(blk_cnt), _ptr(affinity), _ptr(ws), int(ws_bytes),
        _stream(stream)))


def moer_ids_signature(dims, topk, T, blk_tab, nblk, blk_cnt, affinity, ws, ws_bytes, stream=None) -> None:
    _check("moer_ids_signature", LIB.moer_ids_signature(
        ctypes.byref(dims), _ptr(topk), int(T), _ptr(blk_tab), int(nblk), _ptr(blk_cnt), _ptr(affinity),
        _ptr(ws), int(ws_bytes), _stream(stream)))


def moer_ws_status(ws, stream=None) -> int:
    """Waits for the stream and returns (and clears) the workspace status code."""
    return int(LIB.moer_ws_status(_ptr(ws), _stream(stream)))


def moer_wait_selftest(ws, ws_bytes, limit_us, stream=None) -> None:
    """One kernel whose bounded wait cannot complete: it gives up after limit_us and
    records MOER_ETIMEOUT in ws (read it with moer_ws_status)."""
    _check("moer_wait_selftest", LIB.moer_wait_selftest(_ptr(ws), int(ws_bytes), int(limit_us), _stream(stream)))


def moer_status_str(code: int) -> str:
    return LIB.moer_status_str(int(code)).decode()


def moer_version() -> int:
    return int(LIB.moer_version())


def moer_set_extent_checks(on: bool) -> None:
    LIB.moer_set_extent_checks(1 if on else 0)


def moer_extent_checks() -> bool:
    return bool(LIB.moer_extent_checks())


def moer_buffer_holds(p, nbytes: int) -> bool:
    """Host-side: whether one device allocation holds [p, p + nbytes)."""
    return bool(LIB.moer_buffer_holds(_ptr(p), nbytes))
