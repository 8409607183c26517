"""Checked mode (moer_set_extent_checks / MOER_CHECK_EXTENTS) on the GPU.

Run in a child process with PyTorch's caching allocator off, so that every
tensor is its own device allocation and the driver's ranges are the tensors'
own.  Checked:
  - moer_buffer_holds on exact allocations: the whole buffer and its last
    byte pass; an extent running 64 MiB past the end, a host pointer and a
    pointer in no allocation fail;
  - entry points refuse an extent their buffers cannot hold with
    MOER_EEXTENT and launch nothing.  Every refused call here is one that
    would stay in bounds even if it had been launched (an overstated
    workspace size, an overstated cache slot count with no slot used), so
    the test cannot fault a GPU whatever the check does;
  - the whole step of a small workload runs with checked mode on and gives
    the same results as with it off.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import numpy as np
import torch
import gen
from moe_expert_routing_top_gb300 import _native as nat, pipeline

assert nat.moer_extent_checks(), "MOER_CHECK_EXTENTS=1 turns checked mode on"
dev = torch.device("cuda", 0)

# ---- the query on exact allocations
a = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
p = a.data_ptr()
assert nat.moer_buffer_holds(p, 1 << 20)
assert nat.moer_buffer_holds(p + (1 << 20) - 1, 1)
assert nat.moer_buffer_holds(p + 4096, 0)
assert not nat.moer_buffer_holds(p, (1 << 20) + (64 << 20))
assert not nat.moer_buffer_holds(p + (1 << 20) - 16, 64 << 20)
host = torch.empty(4096, dtype=torch.uint8)
assert not nat.moer_buffer_holds(host.data_ptr(), 16)
assert not nat.moer_buffer_holds(None, 16)

def refused(fn, *args):
    try:
        fn(*args)
    except nat.MoerError as e:
        assert e.code == 8, e
        return
    raise AssertionError(fn.__name__ + " was not refused")

# ---- refused calls (each would stay in bounds if launched)
ws = torch.zeros(256, dtype=torch.uint8, device=dev)
refused(nat.moer_wait_selftest, ws, 64 << 20, 1000)

wl = gen.make_custom(64, 8, 2, [40, 25], B=16, mask=[0, 1])
b = wl.batch()
dims = nat.make_dims(wl.E, wl.k, wl.L, wl.mask, wl.B)
logits = torch.from_numpy(gen.host_logits(wl, b.tok_key, b.tok_dom).astype(np.float32)).to(dev)
tab = torch.from_numpy(b.blk_tab.reshape(-1).astype(np.int32)).to(dev)
tk = torch.empty((wl.L, b.T, wl.k), dtype=torch.uint8, device=dev)
cnt = torch.empty((b.nblk, wl.m, wl.E), dtype=torch.uint8, device=dev)
wsb = nat.moer_workspace_bytes(dims, b.T, b.nblk, 0, 0)
ws2 = torch.zeros(wsb, dtype=torch.uint8, device=dev)
refused(nat.moer_topk_signature, dims, logits, b.T, tab, b.nblk, tk, cnt, None, ws2, wsb + (64 << 20))
nat.moer_topk_signature(dims, logits, b.T, tab, b.nblk, tk, cnt, None, ws2, wsb)
assert nat.moer_ws_status(ws2) == 0

off = torch.from_numpy(np.array([0, b.nblk], dtype=np.int32)).to(dev)
req = torch.empty((1, wl.m, wl.E), dtype=torch.int32, device=dev)
cache = torch.zeros((4, wl.m, wl.E), dtype=torch.uint8, device=dev)
coff = torch.zeros(2, dtype=torch.int32, device=dev)
ins = torch.full((b.nblk,), -1, dtype=torch.int32, device=dev)
refused(nat.moer_block_stitch, dims, cnt, tab, b.nblk, off, 1, None, 0, coff, cache, 1 << 20, ins, req, ws2, wsb)
nat.moer_block_stitch(dims, cnt, tab, b.nblk, off, 1, None, 0, coff, cache, 4, ins, req, ws2, wsb)
assert nat.moer_ws_status(ws2) == 0

# ---- a whole step, checked and unchecked
def step():
    w = gen.make_workload("c1", R=6)
    bb = w.batch()
    rs = pipeline.RoutingStats.for_workload(w, max_T=bb.T, max_nblk=bb.nblk, max_R=bb.R)
    rs.step(torch.from_numpy(gen.host_logits(w, bb.tok_key, bb.tok_dom).astype(np.float32)).to(dev),
            pipeline.BatchDev.from_host(bb))
    rs.replication_plan()
    torch.cuda.synchronize()
    assert rs.status() == 0
    return [t.cpu().clone() for t in (rs.topk, rs.blk_cnt, rs.req_cnt, rs.affinity, rs.choice, rs.W)]

on = step()
nat.moer_set_extent_checks(False)
off_ = step()
for x, y in zip(on, off_):
    assert torch.equal(x, y)
print("checked mode ok")
"""


def test_checked_mode():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, PYTORCH_NO_CUDA_MEMORY_CACHING="1", MOER_CHECK_EXTENTS="1")
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "checked mode ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
