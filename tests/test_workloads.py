"""The seeded input generators: determinism, shapes and the stated structure."""
import numpy as np

import workloads


def test_determinism_and_independent_streams():
    a1, b1 = workloads.nvfp4_pair(8, 8, 64, seed=3)
    a2, b2 = workloads.nvfp4_pair(8, 8, 64, seed=3)
    assert np.array_equal(a1, a2) and np.array_equal(b1, b2)
    a3, _ = workloads.nvfp4_pair(8, 8, 64, seed=4)
    assert not np.array_equal(a1, a3)


def test_tiny_has_worked_row_and_outlier_count():
    a, b = workloads.tiny()
    assert a.shape == (16, 512) and b.shape == (256, 512) and a.dtype == np.float32
    assert np.array_equal(a[0, :8], workloads.WORKED_ROW) and np.all(a[0, 8:16] == 0)
    big = np.abs(b) >= 0.5
    assert big.sum() == round(1e-3 * b.size)  # N(0, 0.02) never reaches 0.5


def test_channel_outliers_count():
    a, _ = workloads.mxfp4_pair(64, 8, 7168, seed=9)
    col_rms = np.sqrt((a.astype(np.float64) ** 2).mean(0))
    assert (col_rms > 5).sum() == 36  # round(0.5% * 7168)


def test_routing_structure():
    offs, rt = workloads.route_top_k(4096, 64, 8, seed=workloads.SEED_BASE + 5)
    counts = np.diff(offs)
    assert offs[-1] == 4096 * 8 and counts[63] == 0
    assert counts[:63].min() > 100 and counts.max() < 1300
    for e in (0, 17):
        seg = rt[offs[e]:offs[e + 1]]
        assert np.all(np.diff(seg) > 0)  # ascending tokens, no token twice per expert
    assert np.all(np.bincount(rt, minlength=4096) == 8)
