"""Pins for the oracle's FP64 forward.

The forward is the scatter-reduce of "Accelerating BEV Pooling on NVIDIA
GPUs for Physical AI Applications", section "Eliminate redundant scatter
traffic":  out[ranks_bev[t], c] += depth[ranks_depth[t]] * feat[ranks_feat[t], c].

Pins, none of which calls the oracle's own arithmetic twice:
  * a dense one-hot scatter-matrix product S @ (diag(d) F) (numpy matmul);
  * a CSR sparse product A @ F with A[cell, row] = sum of depth (torch.sparse);
  * closed forms: all-ones inputs give the per-cell point count (bincount),
    one point per cell with D=1 gives a plain row gather, one-hot depth
    gives a segment sum of feature rows;
  * invariants: untouched cells are exactly 0, the per-channel total equals
    sum_p d_p * f_p, and relabelling the cameras does not change the result;
  * E4M3 codes decoded by torch and scaled agree with the E4M3 oracle.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore:Sparse invariant checks")

import oracle
from depth_weighted_scatter_gb300 import workloads


def _decoded(wl):
    if wl.dtype == "f16":
        return wl.depth.astype(np.float64).reshape(-1), wl.feat.astype(np.float64).reshape(wl.n_feat_rows, wl.C)
    import torch

    dec = lambda a: torch.from_numpy(a.reshape(-1)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return dec(wl.depth) * wl.depth_scale, (dec(wl.feat) * wl.feat_scale).reshape(wl.n_feat_rows, wl.C)


def _rows(wl):
    p = np.arange(wl.n_frustum)
    nc, _, h, w = np.unravel_index(p, wl.dims())
    return np.ravel_multi_index((nc, h, w), (wl.NC, wl.H, wl.W))


def _run(wl):
    return oracle.forward(wl.dtype, wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, wl.depth, wl.feat,
                          wl.depth_scale, wl.feat_scale)


def _dense_reference(wl):
    d, F = _decoded(wl)
    kept = wl.cell_ids >= 0
    S = np.zeros((wl.n_cells, wl.n_frustum))
    S[wl.cell_ids[kept], np.nonzero(kept)[0]] = 1.0
    return S @ (d[:, None] * F[_rows(wl)])


def check_forward_pins(out, wl, rtol=1e-12):
    """Dense product + invariants; returns violated pins (used on planted mistakes too)."""
    bad = []
    ref = _dense_reference(wl)
    scale = max(np.abs(ref).max(), 1e-300)
    if out.shape != ref.shape or np.abs(out - ref).max() > rtol * scale:
        bad.append("dense one-hot product")
    hit = np.zeros(wl.n_cells, bool)
    hit[wl.cell_ids[wl.cell_ids >= 0]] = True
    if np.any(out[~hit] != 0.0):
        bad.append("untouched cell not zero")
    d, F = _decoded(wl)
    kept = wl.cell_ids >= 0
    total = (d[kept, None] * F[_rows(wl)[kept]]).sum(axis=0)
    if np.abs(out.sum(axis=0) - total).max() > 1e-9 * max(np.abs(total).max(), 1.0):
        bad.append("channel totals")
    return bad


def test_tiny_dense_product():
    wl = workloads.tiny()
    assert check_forward_pins(_run(wl), wl) == []


@pytest.mark.parametrize("name", ["canonical", "bevdet"])
def test_sparse_product(name, wl_cache):
    torch = pytest.importorskip("torch")
    wl = wl_cache(name)
    out = _run(wl)
    d, F = _decoded(wl)
    kept = np.nonzero(wl.cell_ids >= 0)[0]
    rows = _rows(wl)[kept]
    idx = torch.from_numpy(np.stack([wl.cell_ids[kept].astype(np.int64), rows.astype(np.int64)]))
    A = torch.sparse_coo_tensor(idx, torch.from_numpy(d[kept]), (wl.n_cells, wl.n_feat_rows)).coalesce()
    ref = torch.sparse.mm(A, torch.from_numpy(F)).numpy()
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()


def test_all_ones_gives_bincount():
    NC, D, H, W, C, cells = 2, 3, 4, 5, 8, 11
    rng = np.random.default_rng(7)
    cid = rng.integers(-1, cells, size=NC * D * H * W).astype(np.int32)
    wl = workloads.custom(NC, D, H, W, C, cells, cid, depth=np.ones((NC, D, H, W), np.float16),
                          feat=np.ones((NC, H, W, C), np.float16))
    out = _run(wl)
    want = np.bincount(cid[cid >= 0], minlength=cells).astype(np.float64)
    assert np.array_equal(out, np.repeat(want[:, None], C, axis=1))


def test_one_point_per_cell_is_row_gather():
    NC, D, H, W, C = 2, 1, 3, 4, 16
    nf = NC * D * H * W
    rng = np.random.default_rng(8)
    cid = rng.permutation(nf).astype(np.int32)       # a bijection: one point per cell
    wl = workloads.custom(NC, D, H, W, C, nf, cid, seed=8)
    out = _run(wl)
    d = wl.depth.astype(np.float64).reshape(-1)
    F = wl.feat.astype(np.float64).reshape(-1, C)
    # with D == 1 the feature row of frustum point p is p itself
    want = np.empty((nf, C))
    want[cid] = d[:, None] * F
    assert np.array_equal(out, want)                  # single products of fp16 values are exact


def test_one_hot_depth_is_segment_sum():
    NC, D, H, W, C, cells = 1, 4, 3, 5, 8, 6
    rng = np.random.default_rng(9)
    cid = rng.integers(0, cells, size=NC * D * H * W).astype(np.int32)
    depth = np.zeros((NC, D, H, W), np.float16)
    depth[0, 2] = 1.0                                 # only depth bin 2 carries weight
    wl = workloads.custom(NC, D, H, W, C, cells, cid, depth=depth, seed=9)
    out = _run(wl)
    F = wl.feat.astype(np.float64).reshape(H * W, C)
    want = np.zeros((cells, C))
    for hw in range(H * W):                           # bin-2 points are p = 2*H*W + hw
        want[cid[2 * H * W + hw]] += F[hw]
    assert np.array_equal(out, want)


def test_camera_relabelling_invariance():
    wl = workloads.bevdet()
    out = _run(wl)
    perm = np.array([3, 0, 5, 1, 4, 2])
    cid = wl.cell_ids.reshape(wl.NC, -1)[perm].reshape(-1)
    wl2 = workloads.custom(wl.NC, wl.D, wl.H, wl.W, wl.C, wl.n_cells, cid,
                           depth=wl.depth[perm], feat=wl.feat[perm])
    out2 = _run(wl2)
    assert np.abs(out - out2).max() <= 1e-12 * np.abs(out).max()


def test_e4m3_against_library_decode(wl_cache):
    wl = workloads.custom(2, 5, 4, 6, 16, 30, np.random.default_rng(3).integers(-1, 30, 240).astype(np.int32),
                          seed=3, dtype="e4m3")
    assert wl.dtype == "e4m3"
    assert check_forward_pins(_run(wl), wl) == []


def test_canonical_fp8_totals(wl_cache):
    wl = wl_cache("canonical_fp8")
    out = _run(wl)
    d, F = _decoded(wl)
    kept = wl.cell_ids >= 0
    total = (d[kept, None] * F[_rows(wl)[kept]]).sum(axis=0)
    assert np.abs(out.sum(axis=0) - total).max() <= 1e-9 * np.abs(total).max()


def test_out_of_range_cell_rejected():
    cid = np.zeros(8, np.int32)
    cid[2] = 9
    wl = workloads.custom(1, 2, 2, 2, 8, 4, cid)
    with pytest.raises(oracle.OracleError):
        _run(wl)


def test_pins_catch_planted_mistakes():
    """Mistakes planted in oracle outputs (on the CPU) must fail a pin."""
    wl = workloads.tiny()
    out = _run(wl)
    assert check_forward_pins(out, wl) == []
    d, F = _decoded(wl)
    rows = _rows(wl)
    p = int(np.nonzero(wl.cell_ids >= 0)[0][-1])
    c = int(wl.cell_ids[p])
    plants = []
    dropped = out.copy()
    dropped[c] -= d[p] * F[rows[p]]                   # a dropped term
    plants.append(dropped)
    flipped = out.copy()
    flipped[c] = -flipped[c]                          # a wrong sign
    plants.append(flipped)
    plants.append(out[:, ::-1].copy())                # transposed channel order
    shifted = np.roll(out, 1, axis=0)                 # off-by-one cell index
    plants.append(shifted)
    wrong_row = out.copy()
    other = rows[p] ^ 1
    wrong_row[c] += d[p] * (F[other] - F[rows[p]])    # h/w mix-up: wrong feature row
    plants.append(wrong_row)
    for bad in plants:
        assert check_forward_pins(bad, wl) != []


def test_e4m3_output_closed_form():
    """E4M3 output with out_scale 0.5 of all-ones inputs: the codes decode to
    exactly 2 x the per-cell point count (even integers up to 32 are E4M3
    values), and untouched cells are the zero code."""
    NC, D, H, W, C, cells = 2, 3, 4, 5, 16, 40
    rng = np.random.default_rng(17)
    cid = rng.integers(-1, cells, size=NC * D * H * W).astype(np.int32)
    wl = workloads.custom(NC, D, H, W, C, cells, cid, depth=np.ones((NC, D, H, W), np.float16),
                          feat=np.ones((NC, H, W, C), np.float16))
    codes, v = oracle.forward_e4m3_out("f16", wl.cell_ids, *wl.dims(), wl.n_cells, C, wl.depth, wl.feat,
                                       1.0, 1.0, 0.5)
    count = np.bincount(cid[cid >= 0], minlength=cells).astype(np.float64)
    assert count.max() <= 16
    assert np.array_equal(oracle.e4m3_to_double(codes), np.repeat(2 * count[:, None], C, axis=1))
    assert np.array_equal(v, np.repeat(2 * count[:, None], C, axis=1))


def test_e4m3_output_rejects_bad_scale():
    wl = workloads.tiny()
    with pytest.raises(oracle.OracleError):
        oracle.forward_e4m3_out(wl.dtype, wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, wl.depth, wl.feat,
                                1.0, 1.0, 0.0)


# ---------------------------------------------------------------- NVFP4 features

def _nvfp4_decoded_feat(wl, swap_nibbles=False, block_shift=0):
    """Feature values of an NVFP4 workload decoded independently of the
    oracle: the E2M1 magnitudes table of the OCP format and the library's
    E4M3 decode of the block scales."""
    torch = pytest.importorskip("torch")
    packed = wl.feat.reshape(wl.n_feat_rows, wl.C // 2)
    lo, hi = packed & 0xF, packed >> 4
    if swap_nibbles:
        lo, hi = hi, lo
    codes = np.empty((wl.n_feat_rows, wl.C), dtype=np.uint8)
    codes[:, 0::2], codes[:, 1::2] = lo, hi
    val = workloads.E2M1_VALUES[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    blocks = torch.from_numpy(wl.feat_block.reshape(wl.n_feat_rows, wl.C // 16).copy()).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    blocks = np.roll(blocks, block_shift, axis=1)
    return val * np.repeat(blocks, 16, axis=1) * wl.feat_scale


def _nvfp4_dense(wl, F):
    torch = pytest.importorskip("torch")
    d = torch.from_numpy(wl.depth.reshape(-1).copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    d = d * wl.depth_scale
    kept = wl.cell_ids >= 0
    S = np.zeros((wl.n_cells, wl.n_frustum))
    S[wl.cell_ids[kept], np.nonzero(kept)[0]] = 1.0
    return S @ (d[:, None] * F[_rows(wl)])


def _nvfp4_run(wl):
    return oracle.forward_nvfp4(wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, wl.depth, wl.feat, wl.feat_block,
                                wl.depth_scale, wl.feat_scale)


def _small_nvfp4(C=32, seed=12):
    NC, D, H, W, cells = 2, 3, 4, 5, 30
    rng = np.random.default_rng(seed)
    cid = rng.integers(-1, cells, size=NC * D * H * W).astype(np.int32)
    return workloads._to_nvfp4(workloads.custom(NC, D, H, W, C, cells, cid, seed=seed), "small_nvfp4")


def test_e2m1_decode_matches_format_table():
    got = oracle.e2m1_to_double(np.arange(16, dtype=np.uint8))
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]          # OCP MX E2M1 value set
    assert np.array_equal(got[:8], mags) and np.array_equal(got[8:], [-m for m in mags])


def test_nvfp4_forward_is_dense_product():
    wl = _small_nvfp4()
    out = _nvfp4_run(wl)
    ref = _nvfp4_dense(wl, _nvfp4_decoded_feat(wl))
    assert np.abs(out - ref).max() <= 1e-12 * max(np.abs(ref).max(), 1e-300)


def test_nvfp4_pins_catch_planted_mistakes():
    """Swapped nibble order or a shifted block-scale index in the decoding
    that the oracle is compared with must be detected."""
    wl = _small_nvfp4()
    out = _nvfp4_run(wl)
    for F in (_nvfp4_decoded_feat(wl, swap_nibbles=True), _nvfp4_decoded_feat(wl, block_shift=1)):
        ref = _nvfp4_dense(wl, F)
        assert np.abs(out - ref).max() > 1e-6 * np.abs(ref).max()


def test_nvfp4_quantisation_round_trip_is_close():
    """The generator's two-level quantisation keeps every value within one
    E2M1 step of its block (a pin on the inputs, not on the oracle)."""
    wl = workloads.make("canonical_nvfp4")
    base = workloads.canonical()
    F = _nvfp4_decoded_feat(wl)
    f = base.feat.astype(np.float64).reshape(wl.n_feat_rows, wl.C)
    blocks = np.abs(f).reshape(wl.n_feat_rows, wl.C // 16, 16).max(axis=2)
    assert np.all(np.abs(F - f) <= np.repeat(blocks, 16, axis=1) * 0.26 + 1e-3)
