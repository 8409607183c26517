"""Workload shapes and constants against the values the pages print (tests/golden/)."""
import os

import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_model_shapes_match_page_table():
    shapes = {r[0]: tuple(int(v) for v in r[1:4]) for r in _rows("model_shapes.txt")}
    for cfg, model in (("c1", "OLMoE"), ("c2", "DeepSeek-V2-Lite-chat"), ("c3", "Qwen3-30B-A3B"),
                       ("c4", "Qwen3-30B-A3B"), ("c5", "Qwen3-30B-A3B")):
        wl = gen.make_workload(cfg, R=4)
        assert (wl.k, wl.E, wl.L) == shapes[model], cfg


def test_eldr_constants():
    c = {r[0]: float(r[1]) for r in _rows("eldr_constants.txt")}
    for cfg in ("c2", "c3", "c4"):
        wl = gen.make_workload(cfg, R=4)
        assert wl.tau == c["tau"] and wl.D == c["decoders"]
    # the printed ~12 KiB per-request signature record is one 16-bit count per
    # (layer, expert) of Qwen3-30B-A3B: 48 * 128 * 2 bytes
    wl = gen.make_workload("c3", R=4)
    assert wl.L * wl.E * 2 == c["record_kib"] * 1024
