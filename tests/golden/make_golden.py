"""Writes the stored expected values under tests/golden/ from the oracle alone.

Run from the repository root:  python tests/golden/make_golden.py
It imports only ``oracle`` and the seeded workload generator; nothing here
comes from the CUDA path."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from depth_weighted_scatter_gb300 import workloads  # noqa: E402


def main():
    wl = workloads.tiny()
    m = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    with open(os.path.join(HERE, "tiny_map.txt"), "w") as f:
        f.write("# tiny workload (seed 0) scatter map written by tests/golden/make_golden.py from the oracle\n")
        f.write(f"n_points {m['n_points']}\nn_intervals {m['n_intervals']}\n")
        for key in ["ranks_depth", "ranks_feat", "ranks_bev", "interval_starts", "interval_lengths"]:
            f.write(key + " " + " ".join(str(int(v)) for v in m[key]) + "\n")
    out = oracle.forward("f16", wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, wl.depth, wl.feat)
    np.savetxt(os.path.join(HERE, "tiny_forward.txt"), out, fmt="%.17g",
               header="tiny workload (seed 0) FP64 forward [256 cells x 8 channels], "
                      "written by tests/golden/make_golden.py from the oracle")


if __name__ == "__main__":
    main()
