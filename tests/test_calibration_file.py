"""Calibration artefacts written and read back (CPU): exact round trip, and every kind of
damage (another magic, a wrong size, a flipped byte) refused."""
import numpy as np
import pytest

pipeline = pytest.importorskip("moe_expert_routing_top_gb300.pipeline")


def _cal(E=64, L=6, m=3, D=5, G=4, seed=1):
    rs = np.random.RandomState(seed)
    return pipeline.Calibration(
        mask=np.sort(rs.choice(L, m, replace=False)).astype(np.int32), mask_order=None, quality=None,
        idf=(1 + rs.random_sample((m, E))).astype(np.float32), sig=None,
        centroids=rs.standard_normal((D, m * E)).astype(np.float32), assign=None, kmeans_info=None,
        affinity=None, group_of=rs.randint(0, G, size=(L, E)).astype(np.int32), knee=None)


def test_round_trip(tmp_path):
    cal = _cal()
    p = tmp_path / "cal.bin"
    pipeline.save_calibration(p, cal, E=64, k=8, L=6, block=16, G=4, tau=0.1)
    got = pipeline.load_calibration(p)
    assert (got["E"], got["k"], got["L"], got["m"], got["D"], got["block"]) == (64, 8, 6, 3, 5, 16)
    assert got["tau"] == 0.1 and got["G"] == 4
    for name in ("mask", "idf", "centroids", "group_of"):
        assert np.array_equal(got[name], getattr(cal, name)), name
        assert got[name].dtype == getattr(cal, name).dtype


def test_damage_is_refused(tmp_path):
    p = tmp_path / "cal.bin"
    pipeline.save_calibration(p, _cal(), E=64, k=8, L=6, block=16, G=4, tau=0.1)
    good = p.read_bytes()
    for bad in (b"XXXXXXXX" + good[8:],            # another magic
                good[:-10],                          # truncated
                good[:100] + bytes([good[100] ^ 1]) + good[101:]):  # one flipped bit
        p.write_bytes(bad)
        with pytest.raises(ValueError):
            pipeline.load_calibration(p)


def test_shapes_must_match(tmp_path):
    with pytest.raises(ValueError):
        pipeline.save_calibration(tmp_path / "c.bin", _cal(), E=32, k=8, L=6, block=16, G=4, tau=0.1)


def test_group_ids_must_fit(tmp_path):
    with pytest.raises(ValueError):
        pipeline.save_calibration(tmp_path / "c.bin", _cal(G=4), E=64, k=8, L=6, block=16, G=3, tau=0.1)
