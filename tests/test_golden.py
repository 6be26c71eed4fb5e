"""The oracle still reproduces the stored tiny-workload values.

tests/golden/tiny_map.txt and tiny_forward.txt were written by
tests/golden/make_golden.py from the oracle alone; a change to the oracle's
arithmetic shows up here and must be justified by the passage it follows."""
import os

import numpy as np

import oracle
from depth_weighted_scatter_gb300 import workloads

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_map():
    out = {}
    with open(os.path.join(HERE, "tiny_map.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = np.array([int(v) for v in vals], dtype=np.int32)
    return out


def test_tiny_map_golden():
    wl = workloads.tiny()
    m = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    g = _read_map()
    assert m["n_points"] == int(g["n_points"][0]) and m["n_intervals"] == int(g["n_intervals"][0])
    for key in ["ranks_depth", "ranks_feat", "ranks_bev", "interval_starts", "interval_lengths"]:
        assert np.array_equal(m[key], g[key]), key


def test_tiny_forward_golden():
    wl = workloads.tiny()
    out = oracle.forward("f16", wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, wl.depth, wl.feat)
    want = np.loadtxt(os.path.join(HERE, "tiny_forward.txt"))
    assert np.array_equal(out, want)
