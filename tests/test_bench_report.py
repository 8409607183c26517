"""The bench's decoder-choice report on hand-made distances (CPU): band sizes, band-edge
requests and the choice comparison against an oracle sample."""
import numpy as np

import bench


def test_band_report_counts_sizes_and_edges():
    tau = 0.1
    dist = np.array([
        [0.50, 0.55, 0.70, 0.90],        # band {0, 1}: size 2
        [0.30, 0.40 + 5e-6, 0.90, 0.90],  # decoder 1 within 1e-5 of the edge: size 1, edge
        [0.20, 0.20, 0.20, 0.20],        # every decoder in the band: size 4
        [np.nan, 0.80, 0.85, 1.50],      # NaN outside the band: {1, 2}, size 2
    ], dtype=np.float32)
    edge, hist = bench.band_report(dist, tau)
    assert edge == 1
    assert hist == [1, 2, 0, 1]


def test_choice_parity_counts_differences_and_edges():
    tau = 0.1
    od = np.array([[0.3, 0.9], [0.3, 0.4], [0.5, 0.5]])  # request 1 sits on the band edge
    oc = np.array([0, 1, 0], dtype=np.int32)
    gpu = np.array([7, 7, 0, 0, 0], dtype=np.int32)      # requests 2..4 of the stream
    par = {"oracle": [(2, od, oc)]}
    out = bench.choice_parity(gpu, par, tau, live=True)
    assert out["requests"] == 3 and out["choice_diff"] == 1 and out["band_edge"] == 1
    assert out["choice_diff_off_band_edge"] == 0 and out["first_diff"] == 3
    assert bench.choice_parity(gpu, {}, tau, live=False) is None
