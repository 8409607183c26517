"""The bench's multi-rank host logic on CPU: two gloo ranks.

`bench.py --gpus N` runs N independent replicas (the path has no collective); what it
shares across ranks is the rendezvous, the barrier, the maximum of the per-rank times and
the sum of the per-rank units.  These run here as two processes over gloo on 127.0.0.1,
and the reference arm is launched under torchrun with two ranks (rank 0 prints, rank 1
exits quietly).
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import torch
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    dist = bench.init_dist(ws, "gloo")
    dev = torch.device("cpu")
    t = bench.max_over_ranks(dist, 10.0 + rank, dev)
    u = bench.sum_over_ranks(dist, 100.0 * (rank + 1), dev)
    dist.barrier()
    dist.destroy_process_group()
    out.put((r, ws, t, u))


def test_max_and_sum_over_two_gloo_ranks():
    torch = pytest.importorskip("torch")
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 11.0, 300.0), (1, 2, 11.0, 300.0)]
    assert torch is not None


def test_reference_arm_under_torchrun_two_ranks():
    pytest.importorskip("torch")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "c1", "--gpus", "2", "--steps", "1", "--warmup", "1",
           "--ref-requests", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1                      # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def _pin_rank(rank, world, port, fail_rank, out):
    import torch
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    real_empty = torch.empty

    def fake_empty(*a, pin_memory=False, **k):
        # this host has no GPU: a "pinned" buffer is a plain one, except on the failing rank
        if pin_memory and rank == fail_rank:
            raise RuntimeError("cannot pin")
        return real_empty(*a, **k)

    torch.empty = fake_empty
    ws, r, local = bench.dist_env()
    dist = bench.init_dist(ws, "gloo")
    buf = bench.pinned_on_all_ranks((16,), torch.float32, dist, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()
    out.put((r, buf is None))


@pytest.mark.parametrize("fail_rank", [-1, 1])
def test_pinned_input_agreed_over_ranks(fail_rank):
    """The end-to-end legs pin each replica's whole step input; when one rank cannot, every
    rank drops the leg together (none is left waiting in a collective)."""
    pytest.importorskip("torch")
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_pin_rank, args=(r, 2, port, fail_rank, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    none = fail_rank >= 0
    assert got == [(0, none), (1, none)]
