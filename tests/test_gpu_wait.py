"""The expiry path of the bounded device waits (moer_wait_selftest): a wait that can never
complete gives up after its limit, the status word reports MOER_ETIMEOUT, the kernel ends
normally and the context keeps working.  Nothing faults, traps or spins without a bound.
"""
import time

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

MOER_ETIMEOUT = 7


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_routing_top_gb300 import _native as nat
    return torch, nat


def test_expired_wait_is_reported_and_context_survives(env):
    torch, nat = env
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    nat.moer_wait_selftest(ws, 256, 2000)           # 2 ms
    assert nat.moer_ws_status(ws) == MOER_ETIMEOUT
    elapsed = time.perf_counter() - t0
    gave_up = int(ws.view(torch.int32)[2].item())
    assert gave_up == 1
    assert elapsed < 5.0
    # the status was cleared by the read, and the device still runs work
    assert nat.moer_ws_status(ws) == 0
    x = torch.arange(1 << 20, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == float(np.arange(1 << 20, dtype=np.float64).sum())
