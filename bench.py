#!/usr/bin/env python3
"""Bench of the MoE expert-routing statistics path (libmoeroute) on GB300.

One step = one pass of the whole path over one batch of the Qwen3-30B-A3B-shaped
workload (E=128, k=8, L=48, 1,000 requests, ~1.3 M tokens, 12-layer signature
mask, D=16 decoders, tau=0.1, 8 expert groups):

    moer_topk_signature  ->  moer_block_stitch  ->  moer_affinity_load  ->  moer_route

Inputs are seeded and synthetic (counter-based generator, filled on the GPU
outside the timed region); the ~32.6 GB logits tensor is larger than L2, so no
explicit L2 flush is needed between steps.

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
}
KERNEL_SOURCES = ["moe_expert_routing_top_gb300/csrc/topk_signature.cu",
                  "moe_expert_routing_top_gb300/csrc/common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "k1_dram_traffic.json")


def kernel_sha() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moer_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for ln in f:
                c = [x.strip() for x in ln.split(",")]
                if len(c) < 9:
                    continue
                try:
                    sm.append(float(c[1]))
                    smax.append(float(c[2]))
                except ValueError:
                    continue
                for n, v in zip(names, c[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


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


# ------------------------------------------------------------ CPU oracle arm
def oracle_pass(orc, wl, b, logits):
    """The plain oracle over one batch: every row of the path, as it stands."""
    tk = orc.topk(logits, wl.k)
    bc = orc.block_counts(tk, wl.E, b.req_off, wl.B, wl.mask)
    cache = np.zeros((max(wl.nslots, 1), wl.m, wl.E), dtype=np.uint8)
    rc = orc.stitch(bc, b.req_off, wl.B, b.cache_idx, b.req_cache_off, cache, b.insert_slot)
    orc.affinity(tk, wl.E)
    orc.loads(tk, wl.E, wl.group_of, wl.G)
    _, dist = orc.sig_dist(rc, wl.idf, wl.centroids)
    orc.route(dist, wl.tau, wl.loads0, wl.live)


def cpu_sample(wl, nreq):
    import gen
    b = wl.batch(0, nreq)
    logits = gen.host_logits(wl, b.tok_key, b.tok_dom)
    return b, logits


def run_reference(args):
    import oracle
    import gen
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = gen.make_workload(args.config)
    orc = oracle.get()
    b, logits = cpu_sample(wl, args.ref_requests)
    units = wl.L * b.T
    for _ in range(args.warmup):
        oracle_pass(orc, wl, b, logits)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(orc, wl, b, logits)
    dt = (time.perf_counter() - t0) / args.steps
    v = units / dt
    sample = f"first {args.ref_requests} requests of {args.config} ({b.T} tokens x {wl.L} layers) per step"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD.get(args.config, args.config),
                                            "sample": sample},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


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

    wl = gen.make_workload(args.config, R=args.requests)
    b = wl.batch()
    bd = pipeline.BatchDev.from_host(b, device=device)
    logits = torch.empty((wl.L, b.T, wl.E), dtype=torch.float32, device=device)
    gen.dev_logits(wl, torch.from_numpy(b.tok_key).to(device),
                   torch.from_numpy(b.tok_dom).to(device), logits,
                   torch.from_numpy(wl.bias_mask.reshape(-1)).to(device), sh)
    rs = pipeline.RoutingStats.for_workload(wl, max_T=b.T, max_nblk=b.nblk, max_R=b.R,
                                            device=device, stream=stream)
    units = wl.L * b.T
    alg_bytes = wl.L * b.T * (4 * wl.E + wl.k) + b.nblk * wl.m * wl.E
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
    start.record(stream)
    for i in range(args.steps):
        rs.ensure(bd.T, bd.nblk, bd.R)
        ev[i][0].record(stream)
        rs.topk_signature(logits, bd)
        ev[i][1].record(stream)
        rs.block_stitch(bd)
        rs.affinity_load()
        rs.route(bd.R)
    stop.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    ms_total = start.elapsed_time(stop)
    k1_ms = statistics.mean(a.elapsed_time(z) for a, z in ev)
    ms_total = max_over_ranks(dist, ms_total, device)
    ms_step = ms_total / args.steps
    total_units = sum_over_ranks(dist, units * args.steps, device)
    value = total_units / (ms_total / 1e3)

    # end-to-end through the public API: pinned host logits -> device, step, results -> host
    e2e = run_e2e(args, wl, b, bd, rs, logits, stream, device, dist) if args.e2e else None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_requests)

    peaks = measured_peaks()
    achieved = alg_bytes / (k1_ms / 1e3) / 1e9
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        if tr.get("kernel_sha") == kernel_sha() and tr.get("config") == args.config:
            traffic = tr.get("dram_bytes_per_launch")
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
            "data": "synthetic (seeded counter-based generator; stands in for the pages' datasets)",
            "config": {"workload": WORKLOAD.get(args.config, args.config), "tokens": b.T,
                       "layers": wl.L, "requests": b.R, "kv_blocks": b.nblk,
                       "parallelism": f"replicas x{ws}",
                       "l2": "inputs larger than L2 (logits %.1f GB per step)" % (logits.numel() * 4 / 1e9)},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "kernel": "k1_kernel (moer_topk_signature)", "kernel_ms": k1_ms,
                         "algorithmic_bytes_per_launch": alg_bytes,
                         "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


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
    pinned = torch.empty((wl.L, b.T, wl.E), dtype=torch.float32, pin_memory=True)
    pinned.copy_(logits)  # untimed: the host copy of the same inputs
    chunk_views, off = [], 0
    for bb in batches:
        chunk_views.append((off, bb.T))
        off += bb.T
    copy_stream = torch.cuda.Stream(device)
    dev_bufs = [torch.empty((wl.L, max(x.T for x in batches), wl.E), dtype=torch.float32,
                            device=device) for _ in range(2)]
    bds = [pipeline.BatchDev.from_host(bb, device=device) for bb in batches]
    choice_host = torch.empty(wl.R, dtype=torch.int32, pin_memory=True)
    h2d = host_bytes
    d2h = wl.R * 4

    def one_step():
        copied = [torch.cuda.Event() for _ in range(nch)]
        freed = [torch.cuda.Event() for _ in range(nch)]
        for i, (o, t) in enumerate(chunk_views):
            buf = dev_bufs[i % 2]
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(freed[i - 2])
                dst = buf[:, :t]
                for l in range(wl.L):  # [L][T][E]: one contiguous row range per layer
                    dst[l].copy_(pinned[l, o:o + t], non_blocking=True)
                copied[i].record(copy_stream)
            stream.wait_event(copied[i])
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
            "steps": args.e2e_steps}


def cpu_baseline(wl, nreq):
    import oracle
    orc = oracle.get()
    b, logits = cpu_sample(wl, nreq)
    t0 = time.perf_counter()
    oracle_pass(orc, wl, b, logits)
    dt = time.perf_counter() - t0
    return {"value": wl.L * b.T / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {nreq} requests ({b.T} tokens x {wl.L} layers), one pass, "
                      f"{dt:.1f} s, single thread"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["own", "reference"], default="own")
    ap.add_argument("--config", default="c3", choices=["c1", "c2", "c3"])
    ap.add_argument("--requests", type=int, default=None,
                    help="run a reduced workload with this many requests (profiling)")
    ap.add_argument("--cpu-requests", type=int, default=16)
    ap.add_argument("--ref-requests", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e", dest="e2e", action="store_true", default=True)
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--e2e-chunks", type=int, default=8)
    ap.add_argument("--e2e-steps", type=int, default=3)
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "own":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
