"""bench.py's pipelined end-to-end loop (two frames in flight on two streams,
host buffers through the C ABI) on small workloads: the output read back for
the last frame equals the device-side forward's (the loop checks it and
raises otherwise)."""
import os
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("name,out_dtype", [("tiny", "f16"), ("table1_small", "f16"),
                                            ("table1_small_nvfp4", "e4m3")])
def test_pipelined_e2e_reads_back_the_forward(name, out_dtype):
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    from depth_weighted_scatter_gb300 import bevpool, workloads

    dev = torch.device("cuda")
    wl = workloads.make(name)
    dt = {"f16": bevpool.BEVPOOL_F16, "e4m3": bevpool.BEVPOOL_E4M3, "nvfp4": bevpool.BEVPOOL_NVFP4}[wl.dtype]
    view = np.uint16 if dt == bevpool.BEVPOOL_F16 else np.uint8
    depth_h = torch.from_numpy(np.ascontiguousarray(wl.depth).reshape(-1).view(view).copy()).pin_memory()
    feat_h = torch.from_numpy(np.ascontiguousarray(wl.feat).reshape(-1).view(view).copy()).pin_memory()
    block_h = (torch.from_numpy(np.ascontiguousarray(wl.feat_block).reshape(-1).copy()).pin_memory()
               if wl.feat_block is not None else None)
    m = bevpool.build_map(torch.from_numpy(wl.cell_ids).to(dev), *wl.dims(), wl.n_cells)
    cap = (m.n_points, m.n_intervals)
    depth, feat = depth_h.to(dev), feat_h.to(dev)
    block = block_h.to(dev) if block_h is not None else None
    out_scale = 0.05 if out_dtype == "e4m3" else None
    l0 = bevpool.bevpool_kernel_launches()
    ref = bevpool.forward(m, depth, feat, wl.C, dtype=dt, depth_scale=wl.depth_scale, feat_scale=wl.feat_scale,
                          capacity=cap, out_scale=out_scale, feat_block=block)
    torch.cuda.synchronize()
    per_forward = bevpool.bevpool_kernel_launches() - l0
    assert per_forward >= 1
    launches0 = bevpool.bevpool_kernel_launches()
    us = bench.pipelined_e2e_us(bevpool, m, wl, dt, cap, out_scale, ref, depth_h, feat_h, block_h, 7,
                                torch.cuda.current_stream())
    assert us > 0
    assert bevpool.bevpool_kernel_launches() - launches0 == 24 * per_forward   # 3 untimed + 3 x 7 timed frames
