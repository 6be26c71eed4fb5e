"""The seeded workload generators: shapes and the stated point counts (the
recipes are in the generators' docstrings; these counts are what the parity
tests and the benchmark run on)."""
import numpy as np
import pytest

from depth_weighted_scatter_gb300 import workloads


@pytest.mark.parametrize("name,kept,C", [
    ("canonical", 209077, 80), ("table1_small", 104871, 80), ("table1_large", 571762, 80),
    ("table1_very_large", 1279954, 80), ("wide_c128", 209466, 128), ("wide_c256", 210000, 256)])
def test_ring_workloads(name, kept, C):
    wl = workloads.make(name)
    assert wl.n_kept == kept and wl.C == C
    assert wl.cell_ids.max() < wl.n_cells and wl.feat.shape == (wl.NC, wl.H, wl.W, C)


def test_fp8_variants_quantise_the_same_map():
    a = workloads.make("wide_c128")
    b = workloads.make("wide_c128_fp8")
    assert np.array_equal(a.cell_ids, b.cell_ids) and b.dtype == "e4m3"
    assert b.depth_scale > 0 and b.feat_scale > 0


def test_unknown_name():
    with pytest.raises(KeyError):
        workloads.make("no_such_workload")
