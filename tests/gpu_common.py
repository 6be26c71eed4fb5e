"""Helpers shared by the GPU parity tests: upload a workload, run the C ABI,
compare with the oracle.  Tolerances are the stated bar for this path:
fp16 inputs |gpu - ref| <= 1e-2*max|ref| + 1e-3, E4M3 inputs <= 6e-2*max|ref|,
with ref the FP64 oracle on the very values the GPU received.  NVFP4
features take the fp16 bar: their products are exact in the kernel, so only
the FP32 sum and the fp16 rounding of the output differ from the oracle.

The stated bar is global (a fraction of the largest output), which is wider
than one scatter point's contribution on the full workloads.  So every fp16
output is also held, element by element, to the error an FP32 sum of exact
products can make: |gpu - ref| <= (2L + 8) * 2^-24 * sum|d f| + 1/2 ulp_fp16,
L the longest interval, sum|d f| the oracle's forward of |depth| and |feat|
(scales included).  A dropped or doubled point of ordinary size fails it."""
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


def oracle_values(wl, absolute=False, cell_ids=None):
    """The oracle's FP64 forward of any workload (of cell_ids in place of the
    workload's own, if given); with absolute=True, of |depth| and |feat| (sign
    bits cleared), for error bounds."""
    import oracle

    d, f = wl.depth, wl.feat
    cid = wl.cell_ids if cell_ids is None else cell_ids
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
        return oracle.forward_nvfp4(cid, *wl.dims(), wl.n_cells, wl.C, d, f, wl.feat_block,
                                    wl.depth_scale, wl.feat_scale)
    return oracle.forward(wl.dtype, cid, *wl.dims(), wl.n_cells, wl.C, d, f, wl.depth_scale,
                          wl.feat_scale)


def oracle_forward(wl):
    return oracle_values(wl)


def gpu_forward(wl, m, depth, feat, out=None, **kw):
    from depth_weighted_scatter_gb300 import bevpool

    if wl.dtype == "nvfp4" and "feat_block" not in kw:
        kw["feat_block"] = upload_block(wl, feat.device)
    return bevpool.forward(m, depth, feat, wl.C, dtype=dtype_code(wl), depth_scale=wl.depth_scale,
                           feat_scale=wl.feat_scale, out=out, **kw)


def longest_interval(cell_ids):
    kept = cell_ids[cell_ids >= 0]
    return int(np.bincount(kept).max()) if kept.size else 0


def fp32_window(s_abs, L):
    """Bound on |FP32 sum - exact sum| for sums of at most L exact products in
    any order, with partial rows combined and one scale multiply:
    (2L + 8) * 2^-24 * sum|d f|."""
    return (2 * L + 8) * 2.0 ** -24 * np.abs(s_abs)


def half_ulp_fp16(a, b):
    """Half the fp16 spacing at the larger of |a| and |b| (element-wise): the
    most that rounding one FP32 value to fp16 moves it."""
    m = np.maximum(np.abs(np.asarray(a, np.float64)), np.abs(np.asarray(b, np.float64)))
    _, e = np.frexp(np.maximum(m, 2.0 ** -14))       # m = f * 2^e, f in [0.5, 1): binade 2^(e-1)
    return np.ldexp(0.5, e - 11)                      # half of 2^(e-1-10), the fp16 spacing there


def window_violations(got, ref, s_abs, L):
    """Mask of elements outside the per-element window around ref."""
    g = np.asarray(got, np.float64)
    return np.abs(g - ref) > fp32_window(s_abs, L) + half_ulp_fp16(g, ref)


def assert_forward_close(wl, got, ref, cell_ids=None):
    """The stated global tolerance, then the per-element FP32 window (cell_ids:
    the frustum the expected output was computed from, if not the workload's)."""
    g = got.float().cpu().numpy().astype(np.float64) if hasattr(got, "cpu") else np.asarray(got, np.float64)
    assert g.shape == ref.shape
    assert np.all(np.isfinite(g)), "non-finite output (a row left unwritten?)"
    err = np.abs(g - ref).max() if ref.size else 0.0
    tol = tolerance(wl, ref)
    assert err <= tol, f"{wl.name}: max abs err {err:.3g} above tolerance {tol:.3g}"
    cid = wl.cell_ids if cell_ids is None else cell_ids
    if ref.size:
        bad = window_violations(g, ref, oracle_values(wl, absolute=True, cell_ids=cid), longest_interval(cid))
        if bad.any():
            cell, ch = np.argwhere(bad)[0]
            raise AssertionError(f"{wl.name}: {int(bad.sum())} elements outside the FP32 window "
                                 f"(first at cell {cell}, channel {ch}: got {g[cell, ch]!r}, "
                                 f"want {ref[cell, ch]!r})")
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
    window = fp32_window(s_abs, longest_interval(wl.cell_ids))
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
