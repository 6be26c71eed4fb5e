"""Helpers shared by the GPU parity tests: upload a workload, run the C ABI,
compare with the oracle.  Tolerances are the stated bar for this path:
fp16 inputs |gpu - ref| <= 1e-2*max|ref| + 1e-3, E4M3 inputs <= 6e-2*max|ref|,
with ref the FP64 oracle on the very values the GPU received.  NVFP4
features take the fp16 bar: their products are exact in the kernel, so only
the FP32 sum and the fp16 rounding of the output differ from the oracle."""
import numpy as np

MAP_KEYS = ["ranks_depth", "ranks_feat", "ranks_bev", "interval_starts", "interval_lengths"]


def tolerance(wl, ref):
    m = float(np.abs(ref).max()) if ref.size else 0.0
    return (1e-2 * m + 1e-3) if wl.dtype in ("f16", "nvfp4") else 6e-2 * m


def dtype_code(wl):
    from depth_weighted_scatter_gb300 import bevpool

    return {"f16": bevpool.BEVPOOL_F16, "e4m3": bevpool.BEVPOOL_E4M3, "nvfp4": bevpool.BEVPOOL_NVFP4}[wl.dtype]


def upload(wl, device="cuda"):
    """cell ids, depth and feat on the device (NVFP4: feat is the packed
    E2M1 bytes; its block scales are in upload_block)."""
    import torch

    view = np.uint16 if wl.dtype == "f16" else np.uint8
    cells = torch.from_numpy(np.ascontiguousarray(wl.cell_ids)).to(device)
    depth = torch.from_numpy(np.ascontiguousarray(wl.depth).reshape(-1).view(view).copy()).to(device)
    feat = torch.from_numpy(np.ascontiguousarray(wl.feat).reshape(-1).view(view).copy()).to(device)
    return cells, depth, feat


def upload_block(wl, device="cuda"):
    import torch

    if wl.feat_block is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(wl.feat_block).reshape(-1).copy()).to(device)


def oracle_values(wl, absolute=False):
    """The oracle's FP64 forward of any workload; with absolute=True, of
    |depth| and |feat| (sign bits cleared), for error bounds."""
    import oracle

    d, f = wl.depth, wl.feat
    if absolute:
        if wl.dtype == "f16":
            d = np.ascontiguousarray(d).view(np.uint16) & np.uint16(0x7FFF)
            f = np.ascontiguousarray(f).view(np.uint16) & np.uint16(0x7FFF)
        elif wl.dtype == "e4m3":
            d = np.ascontiguousarray(d).view(np.uint8) & np.uint8(0x7F)
            f = np.ascontiguousarray(f).view(np.uint8) & np.uint8(0x7F)
        else:                                           # E2M1 sign is bit 3 of each nibble
            d = np.ascontiguousarray(d).view(np.uint8) & np.uint8(0x7F)
            f = np.ascontiguousarray(f).view(np.uint8) & np.uint8(0x77)
    if wl.dtype == "nvfp4":
        return oracle.forward_nvfp4(wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, d, f, wl.feat_block,
                                    wl.depth_scale, wl.feat_scale)
    return oracle.forward(wl.dtype, wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, d, f, wl.depth_scale,
                          wl.feat_scale)


def oracle_forward(wl):
    return oracle_values(wl)


def gpu_forward(wl, m, depth, feat, out=None, **kw):
    from depth_weighted_scatter_gb300 import bevpool

    if wl.dtype == "nvfp4" and "feat_block" not in kw:
        kw["feat_block"] = upload_block(wl, feat.device)
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


# ---------------------------------------------------------------- E4M3 output

def oracle_e4m3_out(wl, out_scale):
    """(codes, exact values v = value / out_scale, FP32 error window) for the
    E4M3-output forward.  The window bounds |v_fp32 - v| for a GPU that sums
    exact products in FP32 (one rounding per point, per partial-row combine
    and for the scale): (2L + 8) * 2^-24 * sum|d f| * scale, L the longest
    interval."""
    import oracle

    if wl.dtype == "nvfp4":
        v = oracle_values(wl) / out_scale
        codes = oracle.e4m3_from_double(v)
    else:
        codes, v = oracle.forward_e4m3_out(wl.dtype, wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, wl.depth,
                                           wl.feat, wl.depth_scale, wl.feat_scale, out_scale)
    s_abs = oracle_values(wl, absolute=True) / out_scale
    kept = wl.cell_ids[wl.cell_ids >= 0]
    L = int(np.bincount(kept).max()) if kept.size else 0
    window = (2 * L + 8) * 2.0 ** -24 * np.abs(s_abs)
    return codes, v, window


def assert_e4m3_out_matches(wl, got, out_scale):
    """Every E4M3 code equals the oracle's nearest code, except where the exact
    value lies within the FP32 error window of the midpoint between that code
    and the GPU's (adjacent) one."""
    import oracle

    g = got.cpu().numpy().reshape(wl.n_cells, wl.C)
    codes, v, window = oracle_e4m3_out(wl, out_scale)
    gv = oracle.e4m3_to_double(g)
    wv = oracle.e4m3_to_double(codes)
    assert not np.isnan(gv).any(), "NaN code in the output"
    diff = gv != wv
    if diff.any():
        vi, gi, wi, win = v[diff], gv[diff], wv[diff], window[diff]
        mid = (gi + wi) / 2
        # adjacent codes: nothing representable strictly between them
        lo, hi = np.minimum(gi, wi), np.maximum(gi, wi)
        all_vals = np.unique(oracle.e4m3_to_double(np.arange(256, dtype=np.uint16).astype(np.uint8)))
        all_vals = all_vals[~np.isnan(all_vals)]
        between = np.array([np.any((all_vals > a) & (all_vals < b)) for a, b in zip(lo, hi)])
        near_mid = np.abs(vi - mid) <= win
        bad = between | ~near_mid
        assert not bad.any(), (f"{wl.name}: {int(bad.sum())} codes off the nearest one "
                               f"(first at value {vi[bad][0]!r}: got {gi[bad][0]!r}, want {wi[bad][0]!r})")
    return int(diff.sum())
