"""Helpers shared by the GPU parity tests: upload a workload, run the C ABI,
compare with the oracle.  Tolerances are the stated bar for this path:
fp16 inputs |gpu - ref| <= 1e-2*max|ref| + 1e-3, E4M3 inputs <= 6e-2*max|ref|,
with ref the FP64 oracle on the very values the GPU received."""
import numpy as np

MAP_KEYS = ["ranks_depth", "ranks_feat", "ranks_bev", "interval_starts", "interval_lengths"]


def tolerance(wl, ref):
    m = float(np.abs(ref).max()) if ref.size else 0.0
    return (1e-2 * m + 1e-3) if wl.dtype == "f16" else 6e-2 * m


def dtype_code(wl):
    from depth_weighted_scatter_gb300 import bevpool

    return bevpool.BEVPOOL_F16 if wl.dtype == "f16" else bevpool.BEVPOOL_E4M3


def upload(wl, device="cuda"):
    import torch

    view = np.uint16 if wl.dtype == "f16" else np.uint8
    cells = torch.from_numpy(np.ascontiguousarray(wl.cell_ids)).to(device)
    depth = torch.from_numpy(np.ascontiguousarray(wl.depth).reshape(-1).view(view).copy()).to(device)
    feat = torch.from_numpy(np.ascontiguousarray(wl.feat).reshape(-1).view(view).copy()).to(device)
    return cells, depth, feat


def oracle_forward(wl):
    import oracle

    return oracle.forward(wl.dtype, wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, wl.depth, wl.feat,
                          wl.depth_scale, wl.feat_scale)


def gpu_forward(wl, m, depth, feat, out=None, **kw):
    from depth_weighted_scatter_gb300 import bevpool

    return bevpool.forward(m, depth, feat, wl.C, dtype=dtype_code(wl), depth_scale=wl.depth_scale,
                           feat_scale=wl.feat_scale, out=out, **kw)


def assert_forward_close(wl, got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape
    assert np.all(np.isfinite(g)), "non-finite output (a row left unwritten?)"
    err = np.abs(g - ref).max() if ref.size else 0.0
    tol = tolerance(wl, ref)
    assert err <= tol, f"{wl.name}: max abs err {err:.3g} above tolerance {tol:.3g}"
    return err
