"""The C-ABI library without a GPU: it loads, exports every declared entry point and
rejects bad arguments on the host with the documented status codes (nothing is launched)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if fn.endswith(".h"):
            src = open(os.path.join(inc, fn)).read()
            names += re.findall(r"MOER_API\s+[\w\s\*]+?\b(moer_\w+)\s*\(", src)
    return names


@pytest.fixture(scope="module")
def nat():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "moer_libbuild", os.path.join(ROOT, "moe_expert_routing_top_gb300", "build.py"))
    build = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build)
    if not os.path.exists(build.LIB):
        build.build()
    from moe_expert_routing_top_gb300 import _native
    return _native


def test_exports_every_declared_symbol(nat):
    names = _declared()
    assert len(names) >= 9
    lib = ctypes.CDLL(nat.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(nat.EXPORTS)


def test_version_and_status_strings(nat):
    assert nat.moer_version() >= 100
    for code in range(8):
        assert nat.moer_status_str(code)


def _code(fn, *args):
    from moe_expert_routing_top_gb300._native import MoerError
    with pytest.raises(MoerError) as ei:
        fn(*args)
    return ei.value.code


BADPTR = 0x1001  # misaligned, never dereferenced: validation rejects it first


@pytest.mark.parametrize("E,k,L,mask,B,code", [
    (3, 1, 2, [0], 16, 3), (260, 8, 2, [0], 16, 3), (64, 0, 2, [0], 16, 3), (64, 33, 2, [0], 16, 3),
    (8, 9, 2, [0], 16, 3), (64, 8, 0, [], 16, 3), (64, 8, 2, [1, 0], 16, 1), (64, 8, 2, [2], 16, 3),
    (64, 8, 2, [0], 0, 3), (64, 8, 2, [0], 256, 3)])
def test_bad_dims(nat, E, k, L, mask, B, code):
    d = nat.make_dims(E, k, L, mask, B)
    assert _code(nat.moer_topk_signature, d, 64, 10, None, 0, None, None, None, 64, 4096, 0) == code


def test_bad_pointers_and_sizes(nat):
    d = nat.make_dims(128, 8, 4, [0, 2], 16)
    ws = nat.moer_workspace_bytes(d, 1000, 70, 0, 0)
    assert ws >= 256
    f = nat.moer_topk_signature
    assert _code(f, d, BADPTR, 1000, 64, 70, None, 64, None, 64, ws, 0) == 1      # misaligned logits
    assert _code(f, d, 64, 1000, None, 70, None, 64, None, 64, ws, 0) == 1        # no block table
    assert _code(f, d, 64, 1000, 64, 0, None, 64, None, 64, ws, 0) == 2           # no blocks
    assert _code(f, d, 64, 1000, 64, 70, None, 64, None, 64, ws - 4, 0) == 5      # workspace
    assert _code(f, d, 64, -1, 64, 70, None, 64, None, 64, ws, 0) == 3
    r = nat.moer_route
    assert _code(r, d, 64, 10, 64, 64, 0, 0.1, 64, 0, None, None, 64, None, 0, 0) == 3   # D = 0
    assert _code(r, d, 64, 10, 64, 64, 65, 0.1, 64, 0, None, None, 64, None, 0, 0) == 3  # D > 64
    assert _code(r, d, 64, 10, 64, 64, 16, -1.0, 64, 0, None, None, 64, None, 0, 0) == 3
    assert _code(r, d, 64, 10, 64, 64, 16, 0.1, 64, 2, None, None, 64, None, 0, 0) == 1
    assert _code(r, d, 64, 10, 64, 64, 16, 0.1, 64, 1, None, None, 64, None, 0, 0) == 1  # live, no ws
    s = nat.moer_block_stitch
    assert _code(s, d, 64, 64, 10, None, 5, None, 0, None, None, 0, None, 64, None, 0, 0) == 1
    assert _code(s, d, 64, 64, 10, 64, 5, 64, 1, None, None, 0, None, 64, None, 0, 0) == 1  # idx w/o cache
    assert _code(s, d, 64, 64, 10, 64, 5, None, 3, 64, 64, 4, None, 64, None, 0, 0) == 1   # ncached, no idx
    assert _code(s, d, 64, 64, 10, 64, 5, 64, -1, 64, 64, 4, None, 64, None, 0, 0) == 3    # ncached < 0
    assert _code(s, d, 64, 64, 10, 64, 5, None, 2, None, None, 0, None, 64, None, 0, 0) == 1  # ncached w/o cache
    nat.moer_topk_signature(d, 64, 0, None, 0, None, None, None, 64, ws, 0)  # T = 0: no-op


def test_workspace_size_covers_calls(nat):
    d = nat.make_dims(128, 8, 48, list(range(12)), 16)
    t = nat.moer_workspace_bytes(d, 1305533, 82065, 0, 0)
    r = nat.moer_workspace_bytes(d, 0, 0, 14000, 16)
    both = nat.moer_workspace_bytes(d, 1305533, 82065, 14000, 16)
    assert both == max(t, r) and t >= 256 + 4 * (1305533 // 64)


def test_gate_arguments(nat):
    d = nat.make_dims(128, 8, 4, [0], 16)
    g = nat.moer_gate_topk
    ws = nat.moer_gate_workspace_bytes(d, 256)
    assert _code(g, nat.make_dims(64, 8, 4, [0], 16), 64, 128, 256, 64, None, 0, None, 64, None, None, 256, ws, 0) == 3
    assert _code(g, nat.make_dims(128, 7, 4, [0], 16), 64, 128, 256, 64, None, 0, None, 64, None, None, 256, ws, 0) == 3
    assert _code(g, d, 64, 128, 100, 64, None, 0, None, 64, None, None, 256, ws, 0) == 3        # H % 64
    assert _code(g, d, None, 128, 256, 64, None, 0, None, 64, None, None, 256, ws, 0) == 1     # no hidden
    assert _code(g, d, 64, 128, 256, 64, None, 0, None, None, None, None, 256, ws, 0) == 1     # no top-k
    assert _code(g, d, BADPTR, 128, 256, 64, None, 0, None, 64, None, None, 256, ws, 0) == 1   # misaligned
    assert _code(g, d, 64, 128, 256, 64, None, 0, None, 64, None, None, 256, ws - 256, 0) == 5
    g(d, 64, 0, 256, 64, None, 0, None, 64, None, None, 256, ws, 0)                            # T = 0: no-op


def test_kmeans_arguments(nat):
    k = nat.moer_kmeans_balanced
    ws = nat.moer_kmeans_workspace_bytes(100, 32, 4)
    assert ws > 256
    assert _code(k, 64, 100, 32, 0, 64, 10, 64, 64, None, None, 256, ws, 0) == 3    # D = 0
    assert _code(k, 64, 100, 32, 33, 64, 10, 64, 64, None, None, 256, ws, 0) == 3   # D > 32
    assert _code(k, 64, 3, 32, 4, 64, 10, 64, 64, None, None, 256, ws, 0) == 3      # N < D
    assert _code(k, 64, 100, 0, 4, 64, 10, 64, 64, None, None, 256, ws, 0) == 3     # dim = 0
    assert _code(k, 64, 100, 32, 4, 64, 0, 64, 64, None, None, 256, ws, 0) == 3     # max_iter = 0
    assert _code(k, None, 100, 32, 4, 64, 10, 64, 64, None, None, 256, ws, 0) == 1  # no signatures
    assert _code(k, 64, 100, 32, 4, 64, 10, 64, 64, None, BADPTR, 256, ws, 0) == 1  # misaligned objective
    assert _code(k, 64, 100, 32, 4, 64, 10, 64, 64, None, None, 256, ws - 8, 0) == 5


def test_replication_arguments(nat):
    d = nat.make_dims(128, 8, 4, [0], 16)
    r = nat.moer_replication_plan
    assert _code(r, d, 64, 64, 0, 64, 64, 64, 64, 64, 256, 256, 0) == 3      # G = 0
    assert _code(r, d, 64, 64, 65, 64, 64, 64, 64, 64, 256, 256, 0) == 3     # G > 64
    assert _code(r, d, None, 64, 8, 64, 64, 64, 64, 64, 256, 256, 0) == 1    # no loads
    assert _code(r, d, BADPTR, 64, 8, 64, 64, 64, 64, 64, 256, 256, 0) == 1  # misaligned loads
    assert _code(r, d, 64, 64, 8, 64, 64, 64, 64, 64, 256, 128, 0) == 5      # workspace


def test_mask_select_arguments(nat):
    d = nat.make_dims(128, 8, 4, [], 16)
    m = nat.moer_mask_select
    ws = nat.moer_mask_select_workspace_bytes(d, 10)
    assert _code(m, d, 64, 100, 64, 10, None, 0, 64, None, 256, ws, 0) == 3     # m = 0
    assert _code(m, d, 64, 100, 64, 10, None, 5, 64, None, 256, ws, 0) == 3     # m > L
    assert _code(m, d, 64, 100, 64, 0, None, 2, 64, None, 256, ws, 0) == 3      # R = 0
    assert _code(m, d, None, 100, 64, 10, None, 2, 64, None, 256, ws, 0) == 1   # no top-k
    assert _code(m, d, 64, 100, 64, 10, None, 2, 64, None, 256, ws - 8, 0) == 5


def test_spectral_arguments(nat):
    s = nat.moer_spectral_groups
    d = nat.make_dims(128, 8, 4, [], 16)
    ws = nat.moer_spectral_workspace_bytes(d, 8)
    big = nat.make_dims(256, 8, 4, [], 16)
    assert _code(s, big, 64, 8, 64, 64, 64, 64, 256, ws, 0) == 3     # E > 128
    assert _code(s, d, 64, 1, 64, 64, 64, 64, 256, ws, 0) == 3       # G < 2
    assert _code(s, d, 64, 32, 64, 64, 64, 64, 256, ws, 0) == 3      # G > 31
    assert _code(s, nat.make_dims(16, 8, 4, [], 16), 64, 17, 64, 64, 64, 64, 256, ws, 0) == 3  # G > E
    assert _code(s, d, None, 8, 64, 64, 64, 64, 256, ws, 0) == 1     # no co-activation
    assert _code(s, d, 64, 8, 64, 64, BADPTR, 64, 256, ws, 0) == 1   # misaligned curve
    assert _code(s, d, 64, 8, 64, 64, 64, 64, 256, ws - 8, 0) == 5


def test_wait_selftest_arguments(nat):
    t = nat.LIB.moer_wait_selftest
    assert t(None, 256, 1000, None) == 1
    assert t(BADPTR, 256, 1000, None) == 1
    assert t(64, 100, 1000, None) == 5
    assert t(64, 256, 0, None) == 3
    assert t(64, 256, 1000001, None) == 3


def test_ids_signature_arguments(nat):
    """Host-side validation of moer_ids_signature (no device work: every call is rejected)."""
    f = nat.moer_ids_signature
    d = nat.make_dims(128, 8, 4, [0, 2], 16)
    assert _code(f, d, None, 100, 64, 7, 64, None, 64, 256, 0) == 1          # no ids
    assert _code(f, d, BADPTR, 100, 64, 7, 64, None, 64, 256, 0) == 1        # misaligned ids
    assert _code(f, d, 64, 100, None, 7, 64, None, 64, 256, 0) == 1          # counts without a block table
    assert _code(f, d, 64, 100, 64, 0, 64, None, 64, 256, 0) == 2            # no blocks
    assert _code(f, d, 64, 100, 64, 7, 64, None, 64, 255, 0) == 5            # status word
    assert _code(f, d, 64, -1, 64, 7, 64, None, 64, 256, 0) == 3
    d6 = nat.make_dims(256, 8, 4, [0], 16)
    assert _code(f, d6, 64, 100, 64, 7, None, 64, 64, 256, 0) == 3           # co-activation needs E <= 128
    d5 = nat.make_dims(128, 5, 4, [0], 16)
    assert _code(f, d5, 64, 100, 64, 7, None, 64, 64, 256, 0) == 3           # and k in {6, 8}
    nat.moer_ids_signature(d, 64, 0, None, 0, None, None, 64, 256, 0)       # T = 0: no-op
