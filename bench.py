#!/usr/bin/env python3
"""Bench of the MoE expert-routing statistics path (libmoeroute) on GB300.

One step = one pass of the whole path over one batch of the Qwen3-30B-A3B-shaped
workload (E=128, k=8, L=48, 1,000 requests, ~1.3 M tokens, 12-layer signature
mask, D=16 decoders, tau=0.1, 8 expert groups):

    moer_topk_signature  ->  moer_block_stitch  ->  moer_affinity_load  ->  moer_route

Inputs are seeded and synthetic (counter-based generator, filled on the GPU
outside the timed region); the ~32.6 GB logits tensor is larger than L2, so no
explicit L2 flush is needed between steps.

The same line carries `gate_path`: the path from hidden states on the gate
workload (bf16 hidden [524288, 2048] x 48 bf16 W_gate [2048, 128], 256
requests of 2,048 tokens), whose first call is the tensor-core gate GEMM
with the top-k fused behind it:

    moer_gate_topk  ->  moer_block_stitch  ->  moer_affinity_load  ->  moer_route

`--config c5` makes that path the line's main measurement.

Output: one JSON line (rank 0).  `--impl reference` times the plain CPU oracle
on host cores over a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "routed token·layers/s (top-k+signature+affinity); HBM GB/s vs GB300 peak"
UNIT = "token·layers/s"
WORKLOAD = {
    "c1": "OLMoE-shaped tiny (E=64,k=8,L=16,R=32)",
    "c2": "DeepSeek-V2-Lite-shaped calibration (E=64,k=6,L=26,R=1000)",
    "c3": "Qwen3-30B-A3B-shaped (E=128,k=8,L=48,R=1000,mask=12,D=16,G=8)",
    "c4": "online routing stream (E=128,k=8,L=48,R=14000, 30% cached prefixes, live loads, D=16)",
    "c5": "gate GEMM then path (bf16 hidden T=524288 x H=2048, E=128,k=8,L=48,R=256x2048)",
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
STREAM_TAU = 0.1  # the online stream's locality band


def sources_sha(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, config: str, rows: float):
    """DRAM bytes of one launch over `rows` token x layer pairs, from the committed ncu record
    of a small case of the same workload scaled by rows (the part that does not grow with
    rows, `fixed_bytes`, kept once); None when the record is missing or the kernel's
    sources changed since it was taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            tr = json.loads(ln)
            if tr.get("kernel") == kernel and tr.get("config") == config:
                try:
                    if sources_sha(tr["sources"]) != tr.get("kernel_sha"):
                        return None
                except OSError:
                    return None
                fixed = tr.get("fixed_bytes", 0.0)
                case = tr["dram_bytes_read"] + tr["dram_bytes_write"] - fixed
                return case * rows / tr["case_rows"] + fixed
    return None


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi every 50 ms while the bench runs; samples are timestamped, and those taken
    between mark_start() and mark_stop() (the timed region) are the ones reported."""
    FIELDS = ["timestamp", "index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None
        self.path = os.path.join("/tmp", f"moer_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark_start(self):
        import datetime
        self.t0 = datetime.datetime.now()

    def mark_stop(self):
        import datetime
        self.t1 = datetime.datetime.now()

    def stop(self) -> dict:
        import datetime
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)  # one more sample after the region
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for ln in f:
                c = [x.strip() for x in ln.split(",")]
                if len(c) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(c[0], "%Y/%m/%d %H:%M:%S.%f")
                    rows.append((ts, float(c[2]), float(c[3]), float(c[4]),
                                 {n for n, v in zip(names, c[6:10]) if v.lower().startswith("active")}))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None
                  and self.t0 <= r[0] <= self.t1 + datetime.timedelta(milliseconds=50)]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = sorted(set().union(*[r[4] for r in use]))
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "power_w_max": max(r[3] for r in use), "samples": len(use),
                "samples_in_timed_region": len(inside), "reasons": reasons}


# ------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if ws > 1 else None


def max_over_ranks(dist, x: float, device) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float, device) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def pinned_on_all_ranks(shape, dtype, dist, device):
    """A pinned host buffer, or None on every rank when any rank cannot pin its own (each
    replica pins its full step input; a node's host memory may not hold them all)."""
    import torch
    try:
        buf = torch.empty(shape, dtype=dtype, pin_memory=True)
        ok = 1.0
    except RuntimeError:
        buf, ok = None, 0.0
    if dist is not None:
        ok = -max_over_ranks(dist, -ok, device)  # the minimum over ranks
    return buf if ok >= 1.0 else None


# ------------------------------------------------------------ CPU oracle arm
def oracle_pass(orc, wl, b, logits):
    """The plain oracle over one batch: every row of the path, as it stands.  Returns the
    oracle's distances and decoder choices (the parity sample of the bench line)."""
    tk = orc.topk(logits, wl.k)
    bc = orc.block_counts(tk, wl.E, b.req_off, wl.B, wl.mask)
    cache = np.zeros((max(wl.nslots, 1), wl.m, wl.E), dtype=np.uint8)
    rc = orc.stitch(bc, b.req_off, wl.B, b.cache_idx, b.req_cache_off, cache, b.insert_slot)
    orc.affinity(tk, wl.E)
    orc.loads(tk, wl.E, wl.group_of, wl.G)
    _, dist = orc.sig_dist(rc, wl.idf, wl.centroids)
    choice, _ = orc.route(dist, wl.tau, wl.loads0, wl.live)
    return dist, choice


def cpu_sample(wl, nreq):
    import gen
    b = wl.batch(0, nreq)
    logits = gen.host_logits(wl, b.tok_key, b.tok_dom)
    return b, logits


def oracle_gate_pass(orc, wl, x, w):
    """The plain oracle over the gate path for one request made of the given tokens."""
    ntok = x.shape[0]
    tk = orc.topk(orc.gate_logits(x, w), wl.k)
    req_off = np.array([0, ntok], dtype=np.int32)
    nblk = -(-ntok // wl.B)
    bc = orc.block_counts(tk, wl.E, req_off, wl.B, wl.mask)
    cache = np.zeros((1, wl.m, wl.E), dtype=np.uint8)
    rc = orc.stitch(bc, req_off, wl.B, np.zeros(0, np.int32), np.zeros(2, np.int32), cache,
                    np.full(nblk, -1, np.int32))
    orc.affinity(tk, wl.E)
    orc.loads(tk, wl.E, wl.group_of, wl.G)
    _, dist = orc.sig_dist(rc, wl.idf, wl.centroids)
    orc.route(dist, wl.tau, wl.loads0, wl.live)


def _ref_worker(cfg, i, share, nrounds, barrier, results):
    """One host core of the reference arm: its share of the sample (requests, or c5
    tokens through the fp64 gate) is made first, untimed; then each round starts at the
    common barrier and runs the oracle over the share once."""
    import gen
    import oracle
    orc = oracle.get()
    wl = gen.make_workload(cfg)
    if cfg == "c5":
        x = gen.host_hidden(wl.seed, i * share, share, wl.hidden_dim)
        w = gen.host_wgate(wl.seed, wl.L, wl.hidden_dim, wl.E, wl.wgate_scale)
        units = share
        run = lambda: oracle_gate_pass(orc, wl, x, w)  # noqa: E731
    else:
        b = wl.batch(i * share, (i + 1) * share)
        logits = gen.host_logits(wl, b.tok_key, b.tok_dom)
        units = b.T
        run = lambda: oracle_pass(orc, wl, b, logits)  # noqa: E731
    for _ in range(nrounds):
        barrier.wait()
        run()
        results.put(units)


def run_reference(args):
    """The oracle, as it stands, on every host core: one spawned process per core, each with
    its own share of a bounded sample (args.ref_requests requests of the config, or
    args.ref_tokens c5 tokens through the fp64 gate); a step is one round of all shares,
    timed from their common start to the last one's end."""
    import multiprocessing as mp
    import oracle
    import gen
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    oracle.get()  # built once here, so the workers only load it
    cfg = args.config
    wl = gen.make_workload(cfg)
    try:
        ncores = len(os.sched_getaffinity(0))
    except AttributeError:
        ncores = os.cpu_count() or 1
    share = args.ref_tokens if cfg == "c5" else args.ref_requests
    limit = (int(np.sum(wl.prompt_len)) if cfg == "c5" else wl.R) // share  # shares the workload holds
    ncores = max(1, min(ncores, limit))
    nrounds = args.warmup + args.steps
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(ncores + 1)
    results = ctx.Queue()
    procs = [ctx.Process(target=_ref_worker, args=(cfg, i, share, nrounds, barrier, results))
             for i in range(ncores)]
    for pr in procs:
        pr.start()
    try:
        total_t, total_units = 0.0, 0
        for r in range(nrounds):
            barrier.wait(timeout=600)
            t0 = time.perf_counter()
            units = sum(results.get(timeout=600) for _ in procs)
            dt = time.perf_counter() - t0
            if r >= args.warmup:
                total_t += dt
                total_units += units
    finally:
        for pr in procs:
            pr.join(timeout=60)
    v = wl.L * total_units / total_t
    per = total_units // max(args.steps, 1)
    if cfg == "c5":
        sample = (f"{share} c5 tokens per process through the fp64 gate on {ncores} host cores "
                  f"({per} tokens x {wl.L} layers) per step")
    else:
        sample = (f"first {ncores * share} requests of {cfg}, {share} per process on {ncores} host "
                  f"cores ({per} tokens x {wl.L} layers) per step")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD.get(cfg, cfg), "sample": sample},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": ncores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------- decoder-choice reporting
BAND_EDGE = 1e-5  # a distance this close to d_min + tau may fall on either side


def _edge_rows(dist, tau):
    d = np.asarray(dist, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        dmin = np.fmin.reduce(d, axis=1, keepdims=True)
        return (np.abs(d - (dmin + tau)) <= BAND_EDGE).any(axis=1)


def band_report(dist, tau):
    """On the timed step's own distances: the requests with a decoder within BAND_EDGE of
    the band edge, and the histogram of band sizes (entry i: requests whose band holds
    i + 1 decoders)."""
    d = np.asarray(dist, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        dmin = np.fmin.reduce(d, axis=1, keepdims=True)
        size = (d <= dmin + tau).sum(axis=1)
    hist = np.bincount(size, minlength=d.shape[1] + 1)[1:].tolist()
    return int(_edge_rows(d, tau).sum()), hist


def choice_parity(gpu_choice, parity, tau, live):
    """The GPU's decoder choices against the oracle's (on the oracle's own distances) over
    the CPU-baseline sample: requests compared, choices that differ, and how many of the
    sample's requests lie within BAND_EDGE of the band edge.  In live mode a difference
    at the band edge changes the loads every later choice sees."""
    if not parity or not parity.get("oracle"):
        return None
    n = diff = edge = off_edge = 0
    first = None
    for r0, od, oc in sorted(parity["oracle"], key=lambda x: x[0]):
        g = np.asarray(gpu_choice[r0:r0 + len(oc)])
        e = _edge_rows(od, tau)
        dd = g != np.asarray(oc)
        n += len(oc)
        diff += int(dd.sum())
        edge += int(e.sum())
        off_edge += int((dd & ~e).sum())
        if first is None and dd.any():
            first = r0 + int(np.flatnonzero(dd)[0])
    out = {"requests": n, "choice_diff": diff, "band_edge": edge, "choice_diff_off_band_edge": off_edge}
    if live:
        out["first_diff"] = first
    return out


# ------------------------------------------------------ the online stream
def measure_stream(args, device, dist, stream, with_e2e=False, parity=None):
    """The online routing stream (c4): 14,000 requests, ~13 M computed tokens, 320 GB of
    logits, far more than HBM, so it runs in chunks of whole requests (about 8 GB of logits
    each).  Per chunk the generator fills the logits on the device, untimed; the timed path
    is moer_topk_signature (K1, top-k ids and co-activation), moer_ids_signature (block
    counts), moer_block_stitch (signature cache carried across chunks: prefixes hit blocks
    inserted by earlier chunks), moer_affinity_load and moer_route in live mode (loads
    carried across chunks).  Per-chunk CUDA-event times are summed."""
    import torch
    import gen
    from moe_expert_routing_top_gb300 import pipeline
    sh = stream.cuda_stream
    wl = gen.make_workload("c4", R=args.stream_requests)
    chunks = wl.chunks(args.stream_chunk_tokens)
    batches = [wl.batch(a, z) for a, z in chunks]
    cap_T = max(x.T for x in batches)
    rs = pipeline.RoutingStats.for_workload(wl, max_T=cap_T, max_nblk=max(x.nblk for x in batches),
                                            max_R=max(x.R for x in batches), device=device,
                                            stream=stream)
    flat = torch.empty(wl.L * cap_T * wl.E, dtype=torch.float32, device=device)
    bias = torch.from_numpy(wl.bias_mask.reshape(-1)).to(device)
    # warm-up on a throwaway copy of the state, so the timed stream starts from an empty
    # signature cache and the initial loads
    b0 = batches[0]
    bd0 = pipeline.BatchDev.from_host(b0, device=device)
    v0 = flat[:wl.L * b0.T * wl.E].view(wl.L, b0.T, wl.E)
    gen.dev_logits(wl, torch.from_numpy(b0.tok_key).to(device), torch.from_numpy(b0.tok_dom).to(device),
                   v0, bias, sh)
    rs_w = pipeline.RoutingStats.for_workload(wl, max_T=b0.T, max_nblk=b0.nblk, max_R=b0.R, device=device,
                                              stream=stream)
    for _ in range(max(args.warmup, 3)):
        rs_w.topk_signature(v0, bd0, blk_counts=False)
        rs_w.ids_signature(bd0)
        rs_w.block_stitch(bd0)
        rs_w.affinity_load()
        rs_w.route(b0.R)
    torch.cuda.synchronize()
    if rs_w.status() != 0:
        raise RuntimeError("device-side status after the stream warm-up is not OK")
    del rs_w
    choice = np.empty(wl.R, dtype=np.int32)
    gdist = np.empty((wl.R, wl.D), dtype=np.float32)
    choice_host = torch.empty(max(x.R for x in batches), dtype=torch.int32, pin_memory=True)
    pinned = pinned_on_all_ranks(wl.L * cap_T * wl.E, torch.float32, dist, device) if with_e2e else None
    e2e_unavailable = with_e2e and pinned is None
    with_e2e = with_e2e and pinned is not None
    # per chunk: start, K1 start (after the host copy in the end-to-end run), K1 end, route
    # start, end
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in batches]
    clocks = ClockSampler(device.index or 0)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    clocks.mark_start()
    for i, (b, (a, z)) in enumerate(zip(batches, chunks)):
        bd = pipeline.BatchDev.from_host(b, device=device)
        view = flat[:wl.L * b.T * wl.E].view(wl.L, b.T, wl.E)
        gen.dev_logits(wl, torch.from_numpy(b.tok_key).to(device), torch.from_numpy(b.tok_dom).to(device),
                       view, bias, sh)
        if with_e2e:  # the chunk's inputs in pinned host memory, untimed
            pinned[:view.numel()].copy_(view.reshape(-1))
        rs.ensure(b.T, b.nblk, b.R)
        e = ev[i]
        e[0].record(stream)
        if with_e2e:
            view.reshape(-1).copy_(pinned[:view.numel()], non_blocking=True)
        e[1].record(stream)
        rs.topk_signature(view, bd, blk_counts=False)
        e[2].record(stream)
        rs.ids_signature(bd)
        rs.block_stitch(bd)
        rs.affinity_load()
        e[3].record(stream)
        rs.route(b.R)
        choice_host[:b.R].copy_(rs.choice[:b.R], non_blocking=True)
        e[4].record(stream)
        torch.cuda.synchronize()
        choice[a:z] = choice_host[:b.R].numpy()
        gdist[a:z] = rs.dist[:b.R].cpu().numpy()
    clocks.mark_stop()
    clk = clocks.stop()
    if rs.status() != 0:
        raise RuntimeError("device-side status after the stream is not OK")
    k1 = sum(x[1].elapsed_time(x[2]) for x in ev)
    path = sum(x[1].elapsed_time(x[4]) for x in ev)
    route = sum(x[3].elapsed_time(x[4]) for x in ev)
    e2e_ms = sum(x[0].elapsed_time(x[4]) for x in ev) if with_e2e else None
    T = sum(x.T for x in batches)
    units = wl.L * T
    alg = wl.L * T * (4 * wl.E + wl.k)
    peaks = measured_peaks()
    ms_total = max_over_ranks(dist, path, device)
    achieved = alg / (k1 / 1e3) / 1e9
    edge, hist = band_report(gdist, wl.tau)
    out = {
        "workload": WORKLOAD["c4"] if args.stream_requests is None else f"c4, first {wl.R} requests",
        "value": sum_over_ranks(dist, units, device) / (ms_total / 1e3), "unit": UNIT,
        "ms_per_step": ms_total, "steps": 1, "chunks": len(batches), "tokens": T, "layers": wl.L,
        "requests": wl.R, "kv_blocks": sum(x.nblk for x in batches),
        "cached_blocks": int(sum(len(x.cache_idx) for x in batches)),
        "logits_gb": wl.L * T * wl.E * 4 / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": recorded_traffic("k1_tpr_kernel", "c3", units / len(batches)),
                     "kernel": "k1_tpr_kernel (moer_topk_signature calls, summed over the chunks)",
                     "kernel_ms": k1, "algorithmic_bytes_per_launch": alg / len(batches),
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"},
        "route_live_ms": route, "route_live_share": route / path,
        "band_edge": edge, "band_size_hist": hist,
        "gpu_launches": len(batches) * (1 + 1 + 2 + 1 + 2),
        "clocks": clk,
        "l2": "inputs larger than L2 (logits %.1f GB per chunk)" % (wl.L * cap_T * wl.E * 4 / 1e9),
        "gpu_choice": choice,
    }
    if e2e_unavailable:
        out["e2e"] = {"unavailable": "pinned host memory for a chunk's input (%.1f GB per replica) could not be "
                                     "allocated on every rank" % (wl.L * cap_T * wl.E * 4 / 1e9)}
    if with_e2e:
        h2d = wl.L * T * wl.E * 4
        out["e2e"] = {"value": units / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                      "d2h_bytes_per_step": int(wl.R * 4), "ms_per_step": e2e_ms,
                      "h2d_gbs": h2d / (e2e_ms / 1e3) / 1e9,
                      "note": "per chunk: host logits -> device, the path, choices -> host; sequential"}
    return out


def run_stream_main(args, ws, rank, local, device, dist, stream):
    import gen
    parity = {}
    g = measure_stream(args, device, dist, stream, with_e2e=args.e2e, parity=parity)
    cpu = cpu1 = None
    if rank == 0 and not args.no_cpu_baseline:
        wl4 = gen.make_workload("c4", R=args.stream_requests)
        cpu1 = cpu_baseline(wl4, args.cpu_requests, parity)
        cpu = cpu_baseline_all_cores("c4", wl4, args.cpu_requests)
    if rank == 0:
        line = {
            "metric": METRIC, "value": g["value"], "unit": UNIT, "n_gpus": ws,
            "steps": 1, "warmup": args.warmup, "ms_per_step": g["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
            "data": "synthetic (seeded counter-based generator; stands in for the pages' datasets)",
            "config": {"workload": g["workload"], "tokens": g["tokens"], "layers": g["layers"],
                       "requests": g["requests"], "kv_blocks": g["kv_blocks"], "chunks": g["chunks"],
                       "parallelism": f"replicas x{ws}", "l2": g["l2"]},
            "roofline": g["roofline"], "gpu_launches": g["gpu_launches"], "clocks": g["clocks"],
            "e2e": g.get("e2e"), "cpu_baseline": cpu, "cpu_baseline_1core": cpu1,
            "band_edge": g["band_edge"], "band_size_hist": g["band_size_hist"],
            "choice_parity": choice_parity(g["gpu_choice"], parity, STREAM_TAU, True),
            "choice_diff": None,
            "route_live_ms": g["route_live_ms"], "route_live_share": g["route_live_share"],
        }
        if line["choice_parity"]:
            line["choice_diff"] = line["choice_parity"]["choice_diff"]
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------ offline calibration
def calibrate_workload(args, wl, device, stream):
    """The offline half before the served step (untimed for the line's value): calibration
    prompts of the same model (same logit stream and expert biases, new prompts) go
    through pipeline.calibrate -- top-k and co-activation, idf, greedy layer mask,
    signatures, balanced K-means, spectral groups -- and the served workload takes the
    resulting mask, idf, centroids and expert groups.  Returns a summary for the line and
    the arrays the oracle workers need (overrides)."""
    import torch
    import gen
    from moe_expert_routing_top_gb300 import pipeline
    cal = gen.make_calibration(wl, R=args.calib_requests)
    cb = cal.batch()
    logits = torch.empty((wl.L, cb.T, wl.E), dtype=torch.float32, device=device)
    gen.dev_logits(cal, torch.from_numpy(cb.tok_key).to(device), torch.from_numpy(cb.tok_dom).to(device),
                   logits, torch.from_numpy(cal.bias_mask.reshape(-1)).to(device), stream.cuda_stream)
    seed_rows = gen.kmeans_seed_rows(cal.R, wl.D)
    cbd = pipeline.BatchDev.from_host(cb, device=device, with_cache=False)

    def run():
        return pipeline.calibrate(wl.E, wl.k, wl.L, wl.B, logits, cbd, cb.req_off, m=int(wl.mask.shape[0]),
                                  D=wl.D, G=wl.G, seed_rows=seed_rows, tau=wl.tau, device=device,
                                  stream=stream)
    # one untimed pass first: a fresh process pays its one-time costs there (module loading,
    # the allocator's first device allocations, first-use set-up), which are not the
    # calibration's work; the timed pass gives the same results
    run()
    torch.cuda.synchronize()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    got = run()
    z.record(stream)
    torch.cuda.synchronize()
    del logits
    torch.cuda.empty_cache()
    over = {"mask": got.mask.astype(np.int32), "idf": got.idf.cpu().numpy(),
            "centroids": got.centroids.cpu().numpy(), "group_of": got.group_of.cpu().numpy()}
    apply_overrides(wl, over)
    sizes = np.bincount(got.assign.cpu().numpy(), minlength=wl.D)
    summary = {"prompts": cal.R, "tokens": cb.T, "ms": a.elapsed_time(z),
               "mask_in_order": got.mask_order.tolist(), "mask": got.mask.tolist(),
               "kmeans_steps": int(got.kmeans_info[0]), "cluster_sizes": sizes.tolist(),
               "group_knee_j": got.knee.tolist()}
    return summary, over


def apply_overrides(wl, over):
    """The served workload takes the calibrated mask, idf, centroids and expert groups."""
    if over:
        wl.mask, wl.idf = over["mask"], over["idf"]
        wl.centroids, wl.group_of = over["centroids"], over["group_of"]


# --------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch
    import gen
    from moe_expert_routing_top_gb300 import pipeline
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(ws, "nccl")
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    if args.config == "c5":
        return run_gate_main(args, ws, rank, local, device, dist, stream)
    if args.config == "c4":
        return run_stream_main(args, ws, rank, local, device, dist, stream)
    if args.kmeans_only:
        if rank == 0:
            print(json.dumps({"kmeans_fit": measure_kmeans(args, device, stream, rank)}), flush=True)
        return 0

    wl = gen.make_workload(args.config, R=args.requests)
    calib, over = (calibrate_workload(args, wl, device, stream)
                   if args.calibrate and args.config in ("c2", "c3") else (None, None))
    b = wl.batch()
    bd = pipeline.BatchDev.from_host(b, device=device)
    logits = torch.empty((wl.L, b.T, wl.E), dtype=torch.float32, device=device)
    gen.dev_logits(wl, torch.from_numpy(b.tok_key).to(device),
                   torch.from_numpy(b.tok_dom).to(device), logits,
                   torch.from_numpy(wl.bias_mask.reshape(-1)).to(device), sh)
    rs = pipeline.RoutingStats.for_workload(wl, max_T=b.T, max_nblk=b.nblk, max_R=b.R,
                                            device=device, stream=stream)
    units = wl.L * b.T
    # the timed kernel is K1 alone (its call runs without block counts): the logits read and
    # the top-k ids written; the block counts follow from the ids in the same step
    alg_bytes = wl.L * b.T * (4 * wl.E + wl.k)
    launches_per_step = 2 + (2 if rs.cache is not None else 1) + 1 + (2 if wl.live else 1)

    for _ in range(max(args.warmup, 0)):
        rs.step(logits, bd)
    torch.cuda.synchronize()
    if rs.status() != 0:
        raise RuntimeError("device-side status after warm-up is not OK")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    clocks.mark_start()
    start.record(stream)
    for i in range(args.steps):
        rs.ensure(bd.T, bd.nblk, bd.R)
        ev[i][0].record(stream)
        rs.topk_signature(logits, bd, blk_counts=False)
        ev[i][1].record(stream)
        rs.ids_signature(bd)
        rs.block_stitch(bd)
        rs.affinity_load()
        rs.route(bd.R)
    stop.record(stream)
    torch.cuda.synchronize()
    clocks.mark_stop()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    ms_total = start.elapsed_time(stop)
    k1_ms = statistics.mean(a.elapsed_time(z) for a, z in ev)
    ms_total = max_over_ranks(dist, ms_total, device)
    ms_step = ms_total / args.steps
    total_units = sum_over_ranks(dist, units * args.steps, device)
    value = total_units / (ms_total / 1e3)

    # decoder choices of the timed step: band-edge requests and band sizes on its own distances
    gpu_choice = rs.choice[:b.R].cpu().numpy()
    band_edge, band_hist = band_report(rs.dist[:b.R].cpu().numpy(), wl.tau)

    # end-to-end through the public API: pinned host logits -> device, step, results -> host
    e2e = run_e2e(args, wl, b, bd, rs, logits, stream, device, dist) if args.e2e else None

    cpu = cpu1 = None
    parity = {}
    if rank == 0 and not args.no_cpu_baseline:
        cpu1 = cpu_baseline(wl, args.cpu_requests, parity)
        cpu = cpu_baseline_all_cores(args.config, wl, args.cpu_requests, parity, over)

    logits_gb = logits.numel() * 4 / 1e9
    # GRACE replication plan from this step's loads (per layer, after moer_affinity_load)
    rp_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(10)]
    for a, z in rp_ev:
        a.record(stream)
        rs.replication_plan()
        z.record(stream)
    torch.cuda.synchronize()
    if rs.status() != 0:
        raise RuntimeError("device-side status after the replication plan is not OK")
    replication = {"ms": statistics.median(x.elapsed_time(y) for x, y in rp_ev), "layers": wl.L,
                   "groups": wl.G, "replicas_per_layer": rs.n_rep.cpu().tolist()}
    mask_sel = measure_mask_select(args, wl, b, bd, rs, device, stream, rank)
    spectral = measure_spectral(args, wl, rs, device, stream, rank)
    kmeans = measure_kmeans(args, device, stream, rank) if args.kmeans else None
    gate = stream_line = None
    if args.gate or args.stream:
        del logits, rs
        torch.cuda.empty_cache()
    if args.gate:
        gate = measure_gate(args, device, dist, stream, args.gate_steps, with_e2e=False)
    if args.stream:
        sparity = {}
        stream_line = measure_stream(args, device, dist, stream, with_e2e=False)
        if rank == 0 and not args.no_cpu_baseline:
            wl4 = gen.make_workload("c4", R=args.stream_requests)
            stream_line["cpu_baseline_1core"] = cpu_baseline(wl4, args.cpu_requests, sparity)
            stream_line["choice_parity"] = choice_parity(stream_line["gpu_choice"], sparity, wl4.tau, True)
            if stream_line["choice_parity"]:
                stream_line["choice_diff"] = stream_line["choice_parity"]["choice_diff"]
        del stream_line["gpu_choice"]
        torch.cuda.empty_cache()

    peaks = measured_peaks()
    achieved = alg_bytes / (k1_ms / 1e3) / 1e9
    traffic = recorded_traffic("k1_tpr_kernel", "c3", units) if args.config == "c3" else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
            "data": "synthetic (seeded counter-based generator; stands in for the pages' datasets)",
            "config": {"workload": WORKLOAD.get(args.config, args.config), "tokens": b.T,
                       "layers": wl.L, "requests": b.R, "kv_blocks": b.nblk,
                       "parallelism": f"replicas x{ws}",
                       "l2": "inputs larger than L2 (logits %.1f GB per step)" % logits_gb},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "frac_of_8tbs": achieved / 8000.0,
                         "kernel": "k1_tpr_kernel (moer_topk_signature call, block counts "
                                   "after it by moer_ids_signature)", "kernel_ms": k1_ms,
                         "algorithmic_bytes_per_launch": alg_bytes,
                         "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "cpu_baseline_1core": cpu1,
        }
        if calib is not None:
            line["calibration"] = calib
            line["config"]["mask"] = "greedy selection on %d calibration prompts" % calib["prompts"]
            line["config"]["centroids"] = "balanced K-means of the calibration signatures"
            line["config"]["groups"] = "spectral grouping of the calibration co-activation"
        line["band_edge"] = band_edge
        line["band_size_hist"] = band_hist
        line["choice_parity"] = choice_parity(gpu_choice, parity, wl.tau, wl.live)
        line["choice_diff"] = line["choice_parity"]["choice_diff"] if line["choice_parity"] else None
        line["replication_plan"] = replication
        line["mask_select"] = mask_sel
        line["spectral_groups"] = spectral
        if kmeans is not None:
            line["kmeans_fit"] = kmeans
        if gate is not None:
            line["gate_path"] = {key: gate[key] for key in
                                 ("workload", "value", "unit", "ms_per_step", "steps", "roofline",
                                  "gpu_launches", "clocks")}
        if stream_line is not None:
            line["online_stream"] = stream_line
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


GATE_LAUNCHES_PER_CALL = 4   # W_gate transpose, GEMM + top-k; co-activation, block counts


def measure_gate(args, device, dist, stream, steps, with_e2e):
    """The path from hidden states on the gate workload: per step moer_gate_topk (GEMM
    with fused top-k, then co-activation and block counts from the ids), stitch, loads,
    route.  The tensor roofline is taken on the moer_gate_topk call's duration (CUDA
    events on the launching stream around the call, so the three short kernels behind
    the GEMM count against it)."""
    import torch
    import gen
    from moe_expert_routing_top_gb300 import pipeline
    sh = stream.cuda_stream
    wl = gen.make_workload("c5", R=args.requests)
    b = wl.batch()
    H = wl.hidden_dim
    bd = pipeline.BatchDev.from_host(b, device=device)
    hidden = torch.empty((b.T, H), dtype=torch.int16, device=device)
    w_gate = torch.empty((wl.L, H, wl.E), dtype=torch.int16, device=device)
    gen.dev_hidden(wl.seed, b.T, H, hidden, sh)
    gen.dev_wgate(wl.seed, wl.L, H, wl.E, wl.wgate_scale, w_gate, sh)
    rs = pipeline.RoutingStats.for_workload(wl, max_T=b.T, max_nblk=b.nblk, max_R=b.R,
                                            device=device, stream=stream)
    rs.ensure(b.T, b.nblk, b.R, H)
    flops = 2.0 * b.T * H * wl.E * wl.L
    launches = (GATE_LAUNCHES_PER_CALL + (2 if rs.cache is not None else 1) + 1
                + (2 if wl.live else 1))
    for _ in range(max(args.warmup, 3)):
        rs.gate_step(hidden, w_gate, bd)
    torch.cuda.synchronize()
    if rs.status() != 0:
        raise RuntimeError("device-side status after gate warm-up is not OK")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device.index or 0)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    clocks.mark_start()
    start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        rs.gate_topk(hidden, w_gate, bd, counts=False)
        ev[i][1].record(stream)
        rs.ids_signature(bd, blk_counts=True, affinity=True)
        rs.block_stitch(bd)
        rs.affinity_load()
        rs.route(bd.R)
    stop.record(stream)
    torch.cuda.synchronize()
    clocks.mark_stop()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    if rs.status() != 0:
        raise RuntimeError("device-side status after the timed gate steps is not OK")
    ms_total = max_over_ranks(dist, start.elapsed_time(stop), device)
    call_ms = statistics.mean(a.elapsed_time(z) for a, z in ev)
    units = sum_over_ranks(dist, wl.L * b.T * steps, device)
    peaks = measured_peaks()
    achieved = flops / (call_ms / 1e3) / 1e12
    out = {
        "workload": WORKLOAD["c5"] if args.requests is None else f"c5 with {b.R} requests",
        "value": units / (ms_total / 1e3), "unit": UNIT, "ms_per_step": ms_total / steps,
        "steps": steps, "tokens": b.T, "layers": wl.L, "requests": b.R, "kv_blocks": b.nblk,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "traffic": recorded_traffic("gate_pair_kernel", "c5", wl.L * b.T),
                     "kernel": "gate_pair_kernel (moer_gate_topk call: W_gate transpose and the "
                               "GEMM with fused top-k; counts after it by moer_ids_signature)",
                     "kernel_ms": call_ms,
                     "algorithmic_flops_per_launch": flops,
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json bf16_tflops, burst)"},
        "gpu_launches": launches * steps,
        "clocks": clk,
        "l2": "inputs larger than L2 (hidden %.1f GB per step)" % (hidden.numel() * 2 / 1e9),
    }
    if with_e2e:
        out["e2e"] = run_gate_e2e(args, wl, b, rs, hidden, w_gate, stream, device, dist)
    return out


def run_gate_main(args, ws, rank, local, device, dist, stream):
    import gen
    g = measure_gate(args, device, dist, stream, args.steps, with_e2e=args.e2e)
    cpu = cpu1 = None
    if rank == 0 and not args.no_cpu_baseline:
        wl5 = gen.make_workload("c5")
        cpu1 = gate_cpu_baseline(wl5, args.cpu_tokens)
        cpu = gate_cpu_baseline_all_cores(wl5, args.cpu_tokens)
    if rank == 0:
        line = {
            "metric": METRIC, "value": g["value"], "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": g["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded counter-based generator; stands in for the pages' datasets)",
            "config": {"workload": g["workload"], "tokens": g["tokens"], "layers": g["layers"],
                       "requests": g["requests"], "kv_blocks": g["kv_blocks"],
                       "parallelism": f"replicas x{ws}", "l2": g["l2"]},
            "roofline": g["roofline"], "gpu_launches": g["gpu_launches"], "clocks": g["clocks"],
            "e2e": g.get("e2e"), "cpu_baseline": cpu, "cpu_baseline_1core": cpu1,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_gate_e2e(args, wl, b, rs, hidden, w_gate, stream, device, dist):
    """The gate path with host buffers: per step the hidden states go host -> device in
    request chunks on a copy stream (W_gate stays resident, as model weights do),
    overlapped with the path on the compute stream; the choices come back to the host."""
    import torch
    from moe_expert_routing_top_gb300 import pipeline
    nch = args.e2e_chunks
    bounds = np.linspace(0, wl.R, nch + 1).astype(int)
    batches = [wl.batch(int(a), int(z)) for a, z in zip(bounds[:-1], bounds[1:])]
    H = wl.hidden_dim
    pinned = pinned_on_all_ranks((b.T, H), torch.int16, dist, device)
    if pinned is None:
        return {"unavailable": "pinned host memory for the step input (%.1f GB per replica) could not be "
                               "allocated on every rank" % (b.T * H * 2 / 1e9)}
    pinned.copy_(hidden)  # untimed: the host copy of the same inputs
    offs = np.concatenate([[0], np.cumsum([x.T for x in batches])]).astype(int)
    copy_streams = [torch.cuda.Stream(device) for _ in range(max(args.e2e_copy_streams, 1))]
    maxT = max(x.T for x in batches)
    dev_bufs = [torch.empty((maxT, H), dtype=torch.int16, device=device) for _ in range(2)]
    bds = [pipeline.BatchDev.from_host(bb, device=device) for bb in batches]
    choice_host = torch.empty(wl.R, dtype=torch.int32, pin_memory=True)

    def one_step():
        freed = [torch.cuda.Event() for _ in range(nch)]
        for i, bb in enumerate(batches):
            dst = dev_bufs[i % 2][:bb.T]
            cuts = np.linspace(0, bb.T, len(copy_streams) + 1).astype(int)
            for j, cs in enumerate(copy_streams):  # contiguous row ranges over the copy streams
                with torch.cuda.stream(cs):
                    if i >= 2:
                        cs.wait_event(freed[i - 2])
                    a, z = int(cuts[j]), int(cuts[j + 1])
                    dst[a:z].copy_(pinned[offs[i] + a:offs[i] + z], non_blocking=True)
                    done = torch.cuda.Event()
                    done.record(cs)
                stream.wait_event(done)
            rs.gate_step(dst, w_gate, bds[i])
            freed[i].record(stream)
            r0 = int(bounds[i])
            choice_host[r0:r0 + bb.R].copy_(rs.choice[:bb.R], non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        one_step()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        one_step()
    dt = (time.perf_counter() - t0) / args.e2e_steps
    dt = max_over_ranks(dist, dt, device)
    units = sum_over_ranks(dist, wl.L * b.T, device)
    return {"value": units / dt, "unit": UNIT, "h2d_bytes_per_step": int(b.T * H * 2),
            "d2h_bytes_per_step": int(wl.R * 4), "ms_per_step": dt * 1e3, "chunks": nch,
            "copy_streams": len(copy_streams), "h2d_gbs": b.T * H * 2 / dt / 1e9,
            "steps": args.e2e_steps}


def gate_cpu_baseline(wl, ntok):
    """The oracle's gate logits + top-k over the first `ntok` tokens (every layer), the
    dominant CPU cost of the gate path, single thread."""
    import oracle
    import gen
    orc = oracle.get()
    H = wl.hidden_dim
    x = gen.host_hidden(wl.seed, 0, ntok, H)
    w = gen.host_wgate(wl.seed, wl.L, H, wl.E, wl.wgate_scale)
    t0 = time.perf_counter()
    orc.topk(orc.gate_logits(x, w), wl.k)
    dt = time.perf_counter() - t0
    return {"value": wl.L * ntok / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"gate logits (fp64 sums) + top-k of the first {ntok} tokens x {wl.L} "
                      f"layers, one pass, {dt:.1f} s, single thread"}


def _gate_cpu_worker(t0_tok, ntok, barrier, results):
    import gen
    import oracle
    orc = oracle.get()
    wl = gen.make_workload("c5")
    H = wl.hidden_dim
    x = gen.host_hidden(wl.seed, t0_tok, ntok, H)
    w = gen.host_wgate(wl.seed, wl.L, H, wl.E, wl.wgate_scale)
    barrier.wait()
    t0 = time.perf_counter()
    orc.topk(orc.gate_logits(x, w), wl.k)
    results.put((ntok, time.perf_counter() - t0))


def gate_cpu_baseline_all_cores(wl, ntok_per_core):
    """gate_cpu_baseline on every host core: token ranges over spawned processes, timed
    from a common start barrier to the last worker's end."""
    import multiprocessing as mp
    import oracle
    oracle.get()
    try:
        ncores = len(os.sched_getaffinity(0))
    except AttributeError:
        ncores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(ncores + 1)
    results = ctx.Queue()
    procs = [ctx.Process(target=_gate_cpu_worker,
                         args=(i * ntok_per_core, ntok_per_core, barrier, results))
             for i in range(ncores)]
    for pr in procs:
        pr.start()
    try:
        barrier.wait(timeout=600)
        t0 = time.perf_counter()
        got = [results.get(timeout=600) for _ in procs]
        wall = time.perf_counter() - t0
    finally:
        for pr in procs:
            pr.join(timeout=60)
    tokens = sum(t for t, _ in got)
    return {"value": wl.L * tokens / wall, "unit": UNIT, "cores": ncores, "kind": "oracle",
            "sample": f"gate logits (fp64 sums) + top-k of the first {tokens} tokens x {wl.L} "
                      f"layers, {ntok_per_core} per process on {ncores} host cores, one pass, "
                      f"{wall:.1f} s wall"}


def measure_mask_select(args, wl, b, bd, rs, device, stream, rank):
    """Greedy layer-mask selection (12 of the 48 layers) over the whole batch's top-k ids
    from the step just timed, with CUDA events; the oracle on the first 16 requests."""
    import torch
    from moe_expert_routing_top_gb300 import _native as nat
    m = 12
    dims = nat.make_dims(wl.E, wl.k, wl.L, [], wl.B)
    topk = rs.topk_for(b.T)
    off = torch.from_numpy(np.asarray(b.req_off, dtype=np.int32)).to(device)
    mask = torch.empty(m, dtype=torch.int32, device=device)
    qual = torch.empty(m, dtype=torch.float64, device=device)
    wsb = nat.moer_mask_select_workspace_bytes(dims, b.R)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=device)
    times = []
    for _ in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        nat.moer_mask_select(dims, topk, b.T, off, b.R, None, m, mask, qual, ws, wsb, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if nat.moer_ws_status(ws, stream) != 0:
        raise RuntimeError("device-side status after the mask selection is not OK")
    out = {"workload": f"greedy mask, {m} of {wl.L} layers, {b.R} requests ({b.T} tokens)",
           "ms": statistics.median(times[1:]), "mask_in_order": mask.cpu().tolist(),
           "quality": qual.cpu().tolist()}
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        from oracle import mask_select as ms
        nreq = 16
        bs, logits = cpu_sample(wl, nreq)
        tk = oracle.get().topk(logits, wl.k)
        t0 = time.perf_counter()
        ms.greedy_mask(tk, bs.req_off, wl.E, m)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"ms_per_request": dt * 1e3 / nreq, "cores": 1, "kind": "oracle",
                               "sample": f"first {nreq} requests ({bs.T} tokens), {dt:.1f} s"}
        out["gpu_ms_per_request"] = out["ms"] / b.R
    return out


def measure_spectral(args, wl, rs, device, stream, rank):
    """Spectral grouping of the step's 48 co-activation matrices into 8 groups (17 size
    tolerances each, knee), with CUDA events; the oracle per layer on the first 4 layers."""
    import torch
    from moe_expert_routing_top_gb300 import _native as nat
    G = wl.G
    dims = nat.make_dims(wl.E, wl.k, wl.L, [], wl.B)
    g = torch.empty((wl.L, wl.E), dtype=torch.int32, device=device)
    k = torch.empty(wl.L, dtype=torch.int32, device=device)
    uc = torch.empty((wl.L, 17), dtype=torch.float64, device=device)
    sc = torch.empty((wl.L, 17), dtype=torch.float64, device=device)
    wsb = nat.moer_spectral_workspace_bytes(dims, G)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=device)
    times = []
    for _ in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        nat.moer_spectral_groups(dims, rs.affinity, G, g, k, uc, sc, ws, wsb, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if nat.moer_ws_status(ws, stream) != 0:
        raise RuntimeError("device-side status after the spectral grouping is not OK")
    out = {"workload": f"spectral grouping, {wl.L} layers, E={wl.E} into G={G}, 17 size tolerances",
           "ms": statistics.median(times[1:]), "knee_j": k.cpu().tolist()}
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import grouping as gp
        A = rs.affinity.cpu().numpy()
        t0 = time.perf_counter()
        for l in range(4):
            gp.group_layer(A[l], G)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"ms_per_layer": dt * 1e3 / 4, "cores": 1, "kind": "oracle",
                               "sample": "4 layers (numpy eigh + scipy Hungarian per step)"}
        out["gpu_ms_per_layer"] = out["ms"] / wl.L
    return out


def measure_kmeans(args, device, stream, rank):
    """The calibration fit (balanced K-means of 1,000 signatures of 12 x 128 dims into 16
    decoders), timed with CUDA events after one untimed fit, beside the oracle's fit of
    the same inputs on one host core."""
    import torch
    import gen
    from moe_expert_routing_top_gb300 import _native as nat
    N, dim, D, max_iter = 1000, 12 * 128, 16, 100
    S, _ = gen.calib_signatures(N, dim, ndom=24)
    C0 = S[gen.kmeans_seed_rows(N, D)]
    ds = torch.from_numpy(S).to(device)
    dc0 = torch.from_numpy(np.ascontiguousarray(C0)).to(device)
    cent = torch.empty((D, dim), dtype=torch.float32, device=device)
    assign = torch.empty(N, dtype=torch.int32, device=device)
    info = torch.zeros(3, dtype=torch.int32, device=device)
    obj = torch.zeros(1, dtype=torch.float64, device=device)
    wsb = nat.moer_kmeans_workspace_bytes(N, dim, D)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=device)

    def fit():
        nat.moer_kmeans_balanced(ds, N, dim, D, dc0, max_iter, cent, assign, info, obj, ws, wsb,
                                 stream)

    fit()
    torch.cuda.synchronize()
    times = []
    for _ in range(max(args.kmeans_reps, 1)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fit()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if nat.moer_ws_status(ws, stream) != 0:
        raise RuntimeError("device-side status after the K-means fit is not OK")
    inf = info.cpu().tolist()
    out = {"workload": f"balanced K-means, N={N} signatures, dim={dim}, D={D}, max_iter={max_iter}",
           "ms": statistics.median(times), "steps": inf[0], "cycles_cancelled": inf[1],
           "launches": 3 * max_iter + 3, "objective": float(obj.item())}
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import kmeans as km
        t0 = time.perf_counter()
        _, a_o, steps_o, obj_o = km.balanced_kmeans(S, C0.astype(np.float64), max_iter)
        out["cpu_baseline"] = {"ms": (time.perf_counter() - t0) * 1e3, "cores": 1, "kind": "oracle",
                               "sample": "the same fit (scipy Hungarian assignment per step)"}
        out["matches_oracle"] = bool(np.array_equal(assign.cpu().numpy(), a_o) and steps_o == inf[0])
    return out


def run_e2e(args, wl, b, bd, rs, logits, stream, device, dist):
    """Same metric through the public API with host buffers: per step the logits go
    host -> device in request chunks on a copy stream, overlapped with the path on
    the compute stream; the decoder choices and loads come back to the host."""
    import torch
    from moe_expert_routing_top_gb300 import pipeline
    nch = args.e2e_chunks
    bounds = np.linspace(0, wl.R, nch + 1).astype(int)
    batches = [wl.batch(int(a), int(z)) for a, z in zip(bounds[:-1], bounds[1:])]
    host_bytes = logits.numel() * 4
    pinned = pinned_on_all_ranks((wl.L, b.T, wl.E), torch.float32, dist, device)
    if pinned is None:
        return {"unavailable": "pinned host memory for the step input (%.1f GB per replica) could not be "
                               "allocated on every rank" % (host_bytes / 1e9)}
    pinned.copy_(logits)  # untimed: the host copy of the same inputs
    chunk_views, off = [], 0
    for bb in batches:
        chunk_views.append((off, bb.T))
        off += bb.T
    copy_streams = [torch.cuda.Stream(device) for _ in range(max(args.e2e_copy_streams, 1))]
    dev_bufs = [torch.empty((wl.L, max(x.T for x in batches), wl.E), dtype=torch.float32,
                            device=device) for _ in range(2)]
    bds = [pipeline.BatchDev.from_host(bb, device=device) for bb in batches]
    choice_host = torch.empty(wl.R, dtype=torch.int32, pin_memory=True)
    h2d = host_bytes
    d2h = wl.R * 4

    def one_step():
        freed = [torch.cuda.Event() for _ in range(nch)]
        for i, (o, t) in enumerate(chunk_views):
            buf = dev_bufs[i % 2]
            dst = buf[:, :t]
            # [L][T][E]: one contiguous row range per layer, spread over the copy streams
            for j, cs in enumerate(copy_streams):
                with torch.cuda.stream(cs):
                    if i >= 2:
                        cs.wait_event(freed[i - 2])
                    for l in range(j, wl.L, len(copy_streams)):
                        dst[l].copy_(pinned[l, o:o + t], non_blocking=True)
                    done = torch.cuda.Event()
                    done.record(cs)
                stream.wait_event(done)
            rs.step(dst, bds[i])
            freed[i].record(stream)
            r0 = int(bounds[i])
            choice_host[r0:r0 + batches[i].R].copy_(rs.choice[:batches[i].R], non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        one_step()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        one_step()
    dt = (time.perf_counter() - t0) / args.e2e_steps
    dt = max_over_ranks(dist, dt, device)
    units = sum_over_ranks(dist, wl.L * b.T, device)
    return {"value": units / dt, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": dt * 1e3, "chunks": nch,
            "copy_streams": len(copy_streams), "h2d_gbs": h2d / dt / 1e9, "steps": args.e2e_steps}


def cpu_baseline(wl, nreq, parity=None):
    """The oracle single-threaded over the first `nreq` requests.  With `parity` (a dict),
    the oracle's distances and choices of those requests are left in it as
    parity["oracle"] = [(r0, dist, choice)]."""
    import oracle
    orc = oracle.get()
    b, logits = cpu_sample(wl, nreq)
    t0 = time.perf_counter()
    dist, choice = oracle_pass(orc, wl, b, logits)
    dt = time.perf_counter() - t0
    if parity is not None:
        parity.setdefault("oracle", []).append((0, dist, choice))
    return {"value": wl.L * b.T / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {nreq} requests ({b.T} tokens x {wl.L} layers), one pass, "
                      f"{dt:.1f} s, single thread"}


def _cpu_worker(cfg, r0, r1, barrier, results, over=None):
    """One host core's share of the all-cores oracle run: its requests' inputs are made
    first (untimed), then every worker starts the oracle pass at the same barrier."""
    import gen
    import oracle
    orc = oracle.get()
    wl = gen.make_workload(cfg)
    apply_overrides(wl, over)
    b = wl.batch(r0, r1)
    logits = gen.host_logits(wl, b.tok_key, b.tok_dom)
    barrier.wait()
    t0 = time.perf_counter()
    dist, choice = oracle_pass(orc, wl, b, logits)
    results.put((b.T, time.perf_counter() - t0, r0, dist, choice))


def cpu_baseline_all_cores(cfg, wl, nreq_per_core, parity=None, over=None):
    """The oracle on every host core: request ranges split over spawned processes (the
    oracle itself is single-threaded and unchanged), timed from a common start barrier to
    the last worker's end.  With `parity`, each range's oracle distances and choices are
    added to parity["oracle"] (static routing only: a live range would start from the
    initial loads)."""
    import multiprocessing as mp
    import oracle
    oracle.get()  # built once here, so the workers only load it
    try:
        ncores = len(os.sched_getaffinity(0))
    except AttributeError:
        ncores = os.cpu_count() or 1
    ncores = max(1, min(ncores, wl.R // max(nreq_per_core, 1)))
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(ncores + 1)
    results = ctx.Queue()
    procs = [ctx.Process(target=_cpu_worker,
                         args=(cfg, i * nreq_per_core, (i + 1) * nreq_per_core, barrier, results, over))
             for i in range(ncores)]
    for pr in procs:
        pr.start()
    try:
        barrier.wait(timeout=600)
        t0 = time.perf_counter()
        got = [results.get(timeout=600) for _ in procs]
        wall = time.perf_counter() - t0
    finally:
        for pr in procs:
            pr.join(timeout=60)
    tokens = sum(g[0] for g in got)
    if parity is not None and not wl.live:
        parity.setdefault("oracle", []).extend((g[2], g[3], g[4]) for g in got)
    return {"value": wl.L * tokens / wall, "unit": UNIT, "cores": ncores, "kind": "oracle",
            "sample": f"first {ncores * nreq_per_core} requests ({tokens} tokens x {wl.L} layers), "
                      f"{nreq_per_core} per process on {ncores} host cores, one pass, "
                      f"{wall:.1f} s wall"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["own", "reference"], default="own")
    ap.add_argument("--config", default="c3", choices=["c1", "c2", "c3", "c4", "c5"])
    ap.add_argument("--requests", type=int, default=None,
                    help="run a reduced workload with this many requests (profiling)")
    ap.add_argument("--cpu-requests", type=int, default=16)
    ap.add_argument("--ref-requests", type=int, default=4)
    ap.add_argument("--ref-tokens", type=int, default=32,
                    help="gate path reference arm: tokens per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e", dest="e2e", action="store_true", default=True)
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--e2e-chunks", type=int, default=8)
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="copy streams for the host-to-device copies (1 measured as fast as 2-8)")
    ap.add_argument("--gate", dest="gate", action="store_true", default=True,
                    help="also measure the gate path (moer_gate_topk first) into gate_path")
    ap.add_argument("--no-gate", dest="gate", action="store_false")
    ap.add_argument("--gate-steps", type=int, default=30)
    ap.add_argument("--kmeans", dest="kmeans", action="store_true", default=True,
                    help="also time the calibration fit (balanced K-means) into kmeans_fit")
    ap.add_argument("--no-kmeans", dest="kmeans", action="store_false")
    ap.add_argument("--kmeans-reps", type=int, default=5)
    ap.add_argument("--kmeans-only", action="store_true",
                    help="time only the calibration fit (one JSON object, for profiling)")
    ap.add_argument("--calibrate", dest="calibrate", action="store_true", default=True,
                    help="c2/c3: calibrate mask, idf, centroids and expert groups on the GPU first")
    ap.add_argument("--no-calibrate", dest="calibrate", action="store_false")
    ap.add_argument("--calib-requests", type=int, default=1000,
                    help="calibration prompts (lognormal lengths, median 512)")
    ap.add_argument("--stream", dest="stream", action="store_true", default=True,
                    help="also run the online routing stream (c4, chunked) into online_stream")
    ap.add_argument("--no-stream", dest="stream", action="store_false")
    ap.add_argument("--stream-requests", type=int, default=None,
                    help="online stream: the first this many requests only (profiling)")
    ap.add_argument("--stream-chunk-tokens", type=int, default=320_000,
                    help="online stream: computed tokens per chunk (48 x 128 x 4 B each)")
    ap.add_argument("--cpu-tokens", type=int, default=512,
                    help="gate path: tokens in the oracle's CPU-baseline sample")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "own":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
