"""One routing-statistics step over a batch, through the C ABI.

`RoutingStats` owns the caller-side buffers the C ABI expects (PyTorch
allocates them; the library allocates nothing) and issues, on one CUDA
stream:

  moer_topk_signature  top-k + per-KV-block counts + co-activation (one pass)
  moer_block_stitch    prefix-cache stitching into per-request counts
  moer_affinity_load   expert / group loads and skew from the co-activation
  moer_route           signatures, centroid distances, tau-band decoder choice

or, when the router logits are not materialised, `moer_gate_topk` (the bf16
gate GEMM with top-k, block counts and co-activation fused behind it) in
place of the first call.  `moer_ids_signature` derives the block counts and
co-activation from top-k ids already produced (the bench uses it to time the
dominant kernel's call alone).

`calibrate` runs the offline half (idf, greedy layer mask, balanced K-means
centroids, spectral expert groups) call by call on the GPU, and
`save_calibration` / `load_calibration` carry its result to the serving side.

This module only marshals arguments and orders calls; every step of the
path runs in the library's kernels.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from . import _native as nat


@dataclasses.dataclass
class BatchDev:
    """Device copies of one batch's metadata (see gen.workloads.Batch)."""
    T: int
    R: int
    nblk: int
    blk_tab: torch.Tensor
    req_blk_off: torch.Tensor
    cache_idx: Optional[torch.Tensor]
    req_cache_off: Optional[torch.Tensor]
    insert_slot: Optional[torch.Tensor]
    ncached: int = 0

    @staticmethod
    def from_host(b, device="cuda", with_cache=True, pin=False) -> "BatchDev":
        def t(a, dt=torch.int32):
            x = torch.from_numpy(np.ascontiguousarray(a)).to(dt)
            if pin:
                x = x.pin_memory()
            return x.to(device, non_blocking=pin)
        ci = t(b.cache_idx) if with_cache and len(b.cache_idx) else None
        return BatchDev(T=b.T, R=b.R, nblk=b.nblk, blk_tab=t(b.blk_tab.reshape(-1)),
                        req_blk_off=t(b.req_blk_off),
                        cache_idx=ci if with_cache else None,
                        req_cache_off=t(b.req_cache_off) if with_cache else None,
                        insert_slot=t(b.insert_slot) if with_cache else None,
                        ncached=int(len(b.cache_idx)) if with_cache else 0)


class RoutingStats:
    """Holds the model/serving state of the path and runs steps over batches."""

    def __init__(self, E, k, L, mask, block, *, D, tau, centroids, idf, loads, live, G, group_of,
                 nslots=0, max_T=0, max_nblk=0, max_R=0, device="cuda", stream=None):
        self.dims = nat.make_dims(E, k, L, list(mask), block)
        self.E, self.k, self.L, self.m, self.B = E, k, L, len(mask), block
        self.D, self.tau, self.live, self.G = D, float(tau), bool(live), G
        dev = torch.device(device)
        self.device = dev
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        f32, i32 = torch.float32, torch.int32
        self.centroids = torch.as_tensor(np.asarray(centroids), dtype=f32).to(dev).contiguous()
        self.idf = torch.as_tensor(np.asarray(idf), dtype=f32).to(dev).contiguous()
        self.loads = torch.as_tensor(np.asarray(loads), dtype=i32).to(dev).contiguous()
        self.group_of = torch.as_tensor(np.asarray(group_of), dtype=i32).to(dev).contiguous()
        self.affinity = torch.zeros((L, E, E), dtype=i32, device=dev)
        self.W = torch.empty((L, E), dtype=torch.int64, device=dev)
        self.Wg = torch.empty((L, G), dtype=torch.int64, device=dev)
        self.rho_g = torch.empty(L, dtype=torch.float64, device=dev)
        self.rho_e = torch.empty(L, dtype=torch.float64, device=dev)
        self.n_rep = torch.empty(L, dtype=i32, device=dev)
        self.rep_src = torch.empty(L, dtype=i32, device=dev)
        self.hot = torch.empty((L, E), dtype=torch.uint8, device=dev)
        self.rep_dst = torch.empty((L, G), dtype=i32, device=dev)
        self.w_pred = torch.empty((L, G), dtype=torch.float64, device=dev)
        self.cache = (torch.zeros((nslots, self.m, E), dtype=torch.uint8, device=dev)
                      if nslots > 0 else None)
        self.nslots = nslots
        self.gate_H = 0
        self._alloc(max_T, max_nblk, max_R)

    def _alloc(self, T, nblk, R):
        dev, E, k, L, m, D = self.device, self.E, self.k, self.L, self.m, self.D
        self.cap = (T, nblk, R)
        self.topk = torch.empty(L * max(T, 1) * k, dtype=torch.uint8, device=dev)
        self.blk_cnt = torch.empty((max(nblk, 1), m, E), dtype=torch.uint8, device=dev)
        self.req_cnt = torch.empty((max(R, 1), m, E), dtype=torch.int32, device=dev)
        self.sig = torch.empty((max(R, 1), m * E), dtype=torch.float32, device=dev)
        self.dist = torch.empty((max(R, 1), D), dtype=torch.float32, device=dev)
        self.choice = torch.empty(max(R, 1), dtype=torch.int32, device=dev)
        self.ws_bytes = nat.moer_workspace_bytes(self.dims, T, nblk, R, D)
        if self.gate_H:
            self.ws_bytes = max(self.ws_bytes, nat.moer_gate_workspace_bytes(self.dims, self.gate_H))
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)

    def ensure(self, T, nblk, R, H=0):
        grow_gate = H > self.gate_H
        if grow_gate:
            self.gate_H = H
        if grow_gate or T > self.cap[0] or nblk > self.cap[1] or R > self.cap[2]:
            self._alloc(max(T, self.cap[0]), max(nblk, self.cap[1]), max(R, self.cap[2]))

    def topk_for(self, T: int) -> torch.Tensor:
        """The top-k ids of the last batch of T tokens, as [L][T][k]."""
        return self.topk[:self.L * T * self.k].view(self.L, T, self.k)

    def reset_stats(self):
        self.affinity.zero_()

    # ------------------------------------------------------------ the step
    def topk_signature(self, logits, bd: BatchDev, write_topk=True, blk_counts=True):
        """Top-k ids and co-activation, plus the block counts unless ``blk_counts`` is False
        (then ``ids_signature`` can produce them from the ids)."""
        nat.moer_topk_signature(self.dims, logits, bd.T, bd.blk_tab, bd.nblk,
                                self.topk if write_topk else None,
                                self.blk_cnt if blk_counts else None, self.affinity,
                                self.ws, self.ws_bytes, self.stream)

    def gate_topk(self, hidden, w_gate, bd: BatchDev, logits=None, counts=True):
        """hidden bf16 [T][H] x w_gate bf16 [L][H][E] -> top-k and, unless ``counts`` is False,
        block counts and co-activation (else ``ids_signature`` produces them from the ids)."""
        H = hidden.shape[-1]
        nat.moer_gate_topk(self.dims, hidden, bd.T, H, w_gate, bd.blk_tab, bd.nblk, logits,
                           self.topk, self.blk_cnt if counts else None,
                           self.affinity if counts else None, self.ws, self.ws_bytes,
                           self.stream)

    def ids_signature(self, bd: BatchDev, blk_counts=True, affinity=False):
        """Block counts (and, if asked, co-activation) from the top-k ids in ``self.topk``."""
        T = bd.T
        nat.moer_ids_signature(self.dims, self.topk, T, bd.blk_tab, bd.nblk,
                               self.blk_cnt if blk_counts else None,
                               self.affinity if affinity else None, self.ws, self.ws_bytes, self.stream)

    def block_stitch(self, bd: BatchDev):
        use_cache = self.cache is not None and bd.req_cache_off is not None
        nat.moer_block_stitch(self.dims, self.blk_cnt, bd.blk_tab, bd.nblk, bd.req_blk_off, bd.R,
                              bd.cache_idx if use_cache else None,
                              bd.ncached if use_cache else 0,
                              bd.req_cache_off if use_cache else None,
                              self.cache if use_cache else None, self.nslots,
                              bd.insert_slot if use_cache else None, self.req_cnt, self.ws,
                              self.ws_bytes, self.stream)

    def affinity_load(self):
        nat.moer_affinity_load(self.dims, self.affinity, self.group_of, self.G, self.W, self.Wg,
                               self.rho_g, self.rho_e, self.stream)

    def replication_plan(self):
        """GRACE replication plan per layer from the current loads (after affinity_load)."""
        nat.moer_replication_plan(self.dims, self.W, self.group_of, self.G, self.n_rep, self.rep_src,
                                  self.hot, self.rep_dst, self.w_pred, self.ws, self.ws_bytes,
                                  self.stream)

    def route(self, R, write_sig=True):
        nat.moer_route(self.dims, self.req_cnt, R, self.idf, self.centroids, self.D, self.tau,
                       self.loads, int(self.live), self.sig if write_sig else None, self.dist,
                       self.choice, self.ws, self.ws_bytes, self.stream)

    def step(self, logits, bd: BatchDev, write_topk=True, write_sig=True):
        """All rows of the path over one batch (loads and co-activation accumulate)."""
        self.ensure(bd.T, bd.nblk, bd.R)
        self.topk_signature(logits, bd, write_topk)
        self.block_stitch(bd)
        self.affinity_load()
        self.route(bd.R, write_sig)

    def gate_step(self, hidden, w_gate, bd: BatchDev, write_sig=True):
        """All rows of the path over one batch, starting from hidden states (gate GEMM)."""
        self.ensure(bd.T, bd.nblk, bd.R, hidden.shape[-1])
        self.gate_topk(hidden, w_gate, bd)
        self.block_stitch(bd)
        self.affinity_load()
        self.route(bd.R, write_sig)

    def capture_step(self, logits, bd: BatchDev, write_topk=True, write_sig=True):
        """A CUDA graph of one ``step`` on these buffers and inputs (their device addresses
        are baked in): ``replay()`` runs the whole step again with no per-call host work.

        One eager step runs first, on the pipeline's stream, so that the library's one-time
        set-up (kernel attributes, the tensor-map encoder) and any buffer growth happen
        outside the capture; its counts accumulate like any step's.  The capture itself
        runs on a side stream (the legacy default stream cannot be captured)."""
        self.step(logits, bd, write_topk, write_sig)
        torch.cuda.synchronize(self.affinity.device)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=self.affinity.device)
        own = self.stream
        self.stream = side
        try:
            with torch.cuda.graph(graph, stream=side):
                self.step(logits, bd, write_topk, write_sig)
        finally:
            self.stream = own
        return graph

    def status(self) -> int:
        return nat.moer_ws_status(self.ws, self.stream)

    @staticmethod
    def for_workload(wl, *, max_T=0, max_nblk=0, max_R=0, device="cuda", stream=None):
        return RoutingStats(wl.E, wl.k, wl.L, wl.mask, wl.B, D=wl.D, tau=wl.tau,
                            centroids=wl.centroids, idf=wl.idf, loads=wl.loads0, live=wl.live,
                            G=wl.G, group_of=wl.group_of, nslots=wl.nslots, max_T=max_T,
                            max_nblk=max_nblk, max_R=max_R, device=device, stream=stream)


@dataclasses.dataclass
class Calibration:
    """What the offline half of the method hands to serving (device tensors unless noted)."""
    mask: np.ndarray          # host [m] sorted layer ids: the signature's layer mask
    mask_order: np.ndarray    # host [m] the layers in the order the greedy selection chose them
    quality: np.ndarray       # host [m] fp64 proxy quality after each addition
    idf: torch.Tensor         # [m][E] fp32 idf of the mask layers
    sig: torch.Tensor         # [N][m*E] fp32 signatures of the calibration prompts
    centroids: torch.Tensor   # [D][m*E] fp32 balanced K-means centroids: one per decoder
    assign: torch.Tensor      # [N] int32 cluster of each calibration prompt
    kmeans_info: np.ndarray   # host [3] steps, cancellations, step-bound flag
    affinity: torch.Tensor    # [L][E][E] int32 co-activation over the calibration prompts
    group_of: torch.Tensor    # [L][E] int32 spectral expert groups
    knee: np.ndarray          # host [L] knee grid point of each layer's grouping


def calibrate(E, k, L, block, logits, bd: BatchDev, req_off, *, m, D, G, seed_rows, max_iter=100,
              tau=0.1, device="cuda", stream=None) -> Calibration:
    """The offline calibration on the GPU, call by call: the prompts' top-k ids, per-block
    counts and co-activation over every layer (moer_topk_signature), their request counts
    (moer_block_stitch) and idf (moer_idf_fit); the greedy layer mask (moer_mask_select);
    the counts, idf and count.idf signatures over that mask (moer_ids_signature,
    moer_block_stitch, moer_idf_fit, moer_route with one zero centroid, whose choice is
    not used); the balanced K-means centroids from the rows `seed_rows` of those
    signatures (moer_kmeans_balanced); and the spectral expert groups of the
    co-activation (moer_spectral_groups).  This function orders calls and holds buffers;
    the arithmetic is the library's.

    logits [L][T][E] fp32 (device) and bd / req_off (host [R+1]) describe the calibration
    prompts, one request each, without prefix reuse."""
    dev = torch.device(device)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    f32, i32, u8 = torch.float32, torch.int32, torch.uint8
    T, R, nblk = bd.T, bd.R, bd.nblk
    d_all = nat.make_dims(E, k, L, list(range(L)), block)
    topk = torch.empty((L, T, k), dtype=u8, device=dev)
    blk_all = torch.empty((nblk, L, E), dtype=u8, device=dev)
    aff = torch.zeros((L, E, E), dtype=i32, device=dev)
    wsb = nat.moer_workspace_bytes(d_all, T, nblk, R, 1)
    ws = torch.zeros(wsb, dtype=u8, device=dev)
    nat.moer_topk_signature(d_all, logits, T, bd.blk_tab, nblk, topk, blk_all, aff, ws, wsb, st)
    req_all = torch.empty((R, L, E), dtype=i32, device=dev)
    nat.moer_block_stitch(d_all, blk_all, bd.blk_tab, nblk, bd.req_blk_off, R, None, 0, None, None, 0,
                          None, req_all, ws, wsb, st)
    del blk_all
    idf_all = torch.empty((L, E), dtype=f32, device=dev)
    nat.moer_idf_fit(d_all, req_all, R, idf_all, st)
    del req_all
    # the greedy layer mask
    d_sel = nat.make_dims(E, k, L, [], block)
    mask_order = torch.empty(m, dtype=i32, device=dev)
    quality = torch.empty(m, dtype=torch.float64, device=dev)
    msb = nat.moer_mask_select_workspace_bytes(d_sel, R)
    ms_ws = torch.zeros(msb, dtype=u8, device=dev)
    off = torch.as_tensor(np.asarray(req_off, dtype=np.int32)).to(dev)
    nat.moer_mask_select(d_sel, topk, T, off, R, idf_all, m, mask_order, quality, ms_ws, msb, st)
    order = mask_order.cpu().numpy()
    mask = np.sort(order)  # the dims take the mask as a sorted host array
    # counts, idf and signatures over the mask
    d_m = nat.make_dims(E, k, L, mask.tolist(), block)
    blk_m = torch.empty((nblk, m, E), dtype=u8, device=dev)
    nat.moer_ids_signature(d_m, topk, T, bd.blk_tab, nblk, blk_m, None, ws, wsb, st)
    req_m = torch.empty((R, m, E), dtype=i32, device=dev)
    nat.moer_block_stitch(d_m, blk_m, bd.blk_tab, nblk, bd.req_blk_off, R, None, 0, None, None, 0, None,
                          req_m, ws, wsb, st)
    idf_m = torch.empty((m, E), dtype=f32, device=dev)
    nat.moer_idf_fit(d_m, req_m, R, idf_m, st)
    sig = torch.empty((R, m * E), dtype=f32, device=dev)
    zero_c = torch.zeros((1, m * E), dtype=f32, device=dev)
    zero_l = torch.zeros(1, dtype=i32, device=dev)
    unused = torch.empty(R, dtype=i32, device=dev)
    nat.moer_route(d_m, req_m, R, idf_m, zero_c, 1, tau, zero_l, 0, sig, None, unused, None, 0, st)
    # balanced K-means from the caller's seed rows
    init = sig.index_select(0, torch.as_tensor(np.asarray(seed_rows, dtype=np.int64)).to(dev)).contiguous()
    cent = torch.empty((D, m * E), dtype=f32, device=dev)
    assign = torch.empty(R, dtype=i32, device=dev)
    info = torch.zeros(3, dtype=i32, device=dev)
    kmb = nat.moer_kmeans_workspace_bytes(R, m * E, D)
    km_ws = torch.zeros(kmb, dtype=u8, device=dev)
    nat.moer_kmeans_balanced(sig, R, m * E, D, init, max_iter, cent, assign, info, None, km_ws, kmb, st)
    # spectral expert groups of the co-activation
    group_of = torch.empty((L, E), dtype=i32, device=dev)
    knee = torch.empty(L, dtype=i32, device=dev)
    u = torch.empty((L, 17), dtype=torch.float64, device=dev)
    s = torch.empty((L, 17), dtype=torch.float64, device=dev)
    spb = nat.moer_spectral_workspace_bytes(d_all, G)
    sp_ws = torch.zeros(spb, dtype=u8, device=dev)
    nat.moer_spectral_groups(d_all, aff, G, group_of, knee, u, s, sp_ws, spb, st)
    for w in (ws, ms_ws, km_ws, sp_ws):
        code = nat.moer_ws_status(w, st)
        if code != 0:
            raise nat.MoerError("calibrate", code, nat.moer_status_str(code))
    return Calibration(mask=mask, mask_order=order, quality=quality.cpu().numpy(), idf=idf_m, sig=sig,
                       centroids=cent, assign=assign, kmeans_info=info.cpu().numpy(), affinity=aff,
                       group_of=group_of, knee=knee.cpu().numpy())


# ---------------------------------------------------------------- artefacts
CALIB_MAGIC = b"MOERCAL1"
CALIB_VERSION = 1
_CALIB_HEADER = "<8s8Id"  # magic, version, E, k, L, m, D, G, block, tau


def save_calibration(path, cal: Calibration, *, E, k, L, block, G, tau) -> None:
    """Writes what serving needs from a calibration, as little-endian binary: a header
    (magic, version, E, k, L, m, D, G, block, tau), then the mask int32 [m], idf fp32 [m][E],
    centroids fp32 [D][m*E] and expert groups int32 [L][E], then a CRC-32 of all of it.
    The calibration must be refitted when the model, the traffic or the decoder count changes;
    the file only carries it from the offline fit to the serving process."""
    import struct
    import zlib
    mask = np.ascontiguousarray(cal.mask, dtype="<i4")
    idf = np.ascontiguousarray(cal.idf.cpu().numpy() if torch.is_tensor(cal.idf) else cal.idf, dtype="<f4")
    cen = np.ascontiguousarray(cal.centroids.cpu().numpy() if torch.is_tensor(cal.centroids) else cal.centroids,
                               dtype="<f4")
    grp = np.ascontiguousarray(cal.group_of.cpu().numpy() if torch.is_tensor(cal.group_of) else cal.group_of,
                               dtype="<i4")
    m, D = int(mask.shape[0]), int(cen.shape[0])
    if idf.shape != (m, E) or cen.shape != (D, m * E) or grp.shape != (L, E):
        raise ValueError("calibration arrays do not match E, L and the mask")
    if grp.size and (grp.min() < 0 or grp.max() >= G):
        raise ValueError("expert group ids outside [0, G)")
    body = struct.pack(_CALIB_HEADER, CALIB_MAGIC, CALIB_VERSION, E, k, L, m, D, G, block, float(tau))
    body += mask.tobytes() + idf.tobytes() + cen.tobytes() + grp.tobytes()
    with open(path, "wb") as f:
        f.write(body + struct.pack("<I", zlib.crc32(body)))


def load_calibration(path) -> dict:
    """Reads a file written by save_calibration; raises ValueError when the magic, the
    version, the sizes or the CRC do not match.  Returns the header fields and host arrays
    (mask, idf, centroids, group_of), ready for RoutingStats."""
    import struct
    import zlib
    with open(path, "rb") as f:
        data = f.read()
    hs = struct.calcsize(_CALIB_HEADER)
    if len(data) < hs + 4:
        raise ValueError("calibration file too short")
    magic, ver, E, k, L, m, D, G, block, tau = struct.unpack_from(_CALIB_HEADER, data, 0)
    if magic != CALIB_MAGIC or ver != CALIB_VERSION:
        raise ValueError("not a calibration file of this version")
    sizes = [m * 4, m * E * 4, D * m * E * 4, L * E * 4]
    if len(data) != hs + sum(sizes) + 4:
        raise ValueError("calibration file size does not match its header")
    (crc,) = struct.unpack_from("<I", data, len(data) - 4)
    if zlib.crc32(data[:-4]) != crc:
        raise ValueError("calibration file checksum mismatch")
    off = hs
    out = {"E": E, "k": k, "L": L, "m": m, "D": D, "G": G, "block": block, "tau": tau}
    for name, n, dt, shape in (("mask", sizes[0], "<i4", (m,)), ("idf", sizes[1], "<f4", (m, E)),
                               ("centroids", sizes[2], "<f4", (D, m * E)), ("group_of", sizes[3], "<i4", (L, E))):
        out[name] = np.frombuffer(data, dtype=dt, count=n // 4, offset=off).reshape(shape).astype(dt[1:])
        off += n
    return out
