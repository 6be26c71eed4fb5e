"""GPU parity: libbevpool (through the C ABI) against the FP64 oracle.

Scatter maps must match bit-exactly; forward outputs within the fp16 / E4M3
tolerances of tests/gpu_common.py.  Every workload below is seeded; the full
configurations run at their full sizes in the launch configuration the
benchmark times."""
import numpy as np
import pytest

from gpu_common import MAP_KEYS, assert_forward_close, gpu_forward, oracle_forward, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bp():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from depth_weighted_scatter_gb300 import bevpool

    return bevpool


def _gpu_map(bp, wl, cells, sync=True):
    return bp.build_map(cells, *wl.dims(), wl.n_cells, sync=sync)


def _check_map(bp, wl, m):
    import oracle

    ref = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    got = m.host()
    assert got["n_points"] == ref["n_points"] and got["n_intervals"] == ref["n_intervals"]
    for k in MAP_KEYS:
        assert np.array_equal(got[k], ref[k]), f"{wl.name}: {k} differs"
    assert bp.validate_map(m) == 0
    return ref


CONFIGS = ["tiny", "canonical", "canonical_fp8", "bevdet", "dram_batch"]


@pytest.mark.parametrize("name", CONFIGS)
def test_full_config_parity(bp, name, wl_cache):
    wl = wl_cache(name)
    cells, depth, feat = upload(wl)
    m = _gpu_map(bp, wl, cells)
    _check_map(bp, wl, m)
    out = torch.full((wl.n_cells, wl.C), float("nan"), dtype=torch.float16, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out)
    torch.cuda.synchronize()
    assert_forward_close(wl, out, oracle_forward(wl))


@pytest.mark.parametrize("name", ["canonical", "bevdet"])
def test_forward_is_deterministic(bp, name, wl_cache):
    wl = wl_cache(name)
    cells, depth, feat = upload(wl)
    m = _gpu_map(bp, wl, cells)
    a = gpu_forward(wl, m, depth, feat)
    b = gpu_forward(wl, m, depth, feat)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_device_counts_path_matches_host_counts(bp, wl_cache):
    """build_map without a host sync, forward reading the counts on the device.

    With capacities equal to the counts the launch is the same, so the bits
    are; with larger capacities the interval chunking (and with it the split
    points of long intervals) may differ, so only the tolerance holds."""
    wl = wl_cache("canonical")
    cells, depth, feat = upload(wl)
    m_sync = _gpu_map(bp, wl, cells)
    m_async = _gpu_map(bp, wl, cells, sync=False)
    a = gpu_forward(wl, m_sync, depth, feat)
    b = gpu_forward(wl, m_async, depth, feat, capacity=(m_sync.n_points, m_sync.n_intervals))
    c = gpu_forward(wl, m_async, depth, feat, capacity=(m_sync.n_points + 1000, m_sync.n_intervals + 5000))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert_forward_close(wl, c, oracle_forward(wl))


def test_forward_on_oracle_map(bp, wl_cache):
    """The forward alone, fed the oracle's map (independent of the GPU map builder)."""
    import oracle

    wl = wl_cache("bevdet")
    cells, depth, feat = upload(wl)
    ref_map = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    m = bp.ScatterMap.allocate(*wl.dims(), wl.n_cells)
    for k in MAP_KEYS:
        getattr(m, k)[: len(ref_map[k])].copy_(torch.from_numpy(ref_map[k]))
    m.n_points, m.n_intervals = ref_map["n_points"], ref_map["n_intervals"]
    out = gpu_forward(wl, m, depth, feat)
    torch.cuda.synchronize()
    assert_forward_close(wl, out, oracle_forward(wl))


# ---------------------------------------------------------------- channel counts and dtypes

SUPPORTED_C = [8, 16, 32, 64, 80, 96, 128, 160, 192, 256]


def _check_interval_mix(m, intervals):
    """The kernel variant depends on the mean interval length (fewer than 8
    points per interval counts as short): check the case is on the intended side."""
    n_pts, n_int = m.n_points, m.n_intervals
    assert (n_pts < 8 * n_int) == (intervals == "short"), (n_pts, n_int)


@pytest.mark.parametrize("intervals", ["short", "long"])
@pytest.mark.parametrize("dtype", ["f16", "e4m3"])
@pytest.mark.parametrize("C", SUPPORTED_C)
def test_every_channel_count(bp, C, dtype, intervals):
    """Every channel count, with intervals of about 3 points (short) and of
    about 60 (long): the two select different fp16 kernel variants."""
    from depth_weighted_scatter_gb300 import workloads

    NC, D, H, W, cells = 3, 17, 6, 11, 700
    rng = np.random.default_rng(C * 7 + (dtype == "e4m3") + 1000 * (intervals == "long"))
    nf = NC * D * H * W
    cid = rng.integers(0, cells if intervals == "short" else 40, nf).astype(np.int32)
    cid[rng.random(nf) < 0.3] = -1
    cid[rng.random(nf) < 0.08] = 123                 # one long interval (several owners share it)
    wl = workloads.custom(NC, D, H, W, C, cells, cid, seed=C, dtype=dtype, name=f"C{C}_{dtype}_{intervals}")
    c_d, depth, feat = upload(wl)
    m = _gpu_map(bp, wl, c_d)
    _check_interval_mix(m, intervals)
    _check_map(bp, wl, m)
    out = torch.full((cells, C), float("nan"), dtype=torch.float16, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out)
    torch.cuda.synchronize()
    assert_forward_close(wl, out, oracle_forward(wl))


# ---------------------------------------------------------------- edge cases

def _edge(bp, cid, NC, D, H, W, C, cells, name, dtype="f16", seed=0):
    from depth_weighted_scatter_gb300 import workloads

    wl = workloads.custom(NC, D, H, W, C, cells, np.asarray(cid, np.int32), seed=seed, dtype=dtype, name=name)
    c_d, depth, feat = upload(wl)
    m = _gpu_map(bp, wl, c_d)
    _check_map(bp, wl, m)
    out = torch.full((cells, C), float("nan"), dtype=torch.float16, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out)
    torch.cuda.synchronize()
    assert_forward_close(wl, out, oracle_forward(wl))
    return m, out


def test_edge_all_dropped(bp):
    m, out = _edge(bp, np.full(2 * 3 * 4 * 5, -1), 2, 3, 4, 5, 64, 50, "all_dropped")
    assert m.n_points == 0 and m.n_intervals == 0
    assert torch.count_nonzero(out) == 0


def test_edge_single_cell_grid(bp):
    _edge(bp, np.zeros(1 * 6 * 5 * 7), 1, 6, 5, 7, 80, 1, "one_cell")


def test_edge_one_interval_of_20000_points(bp):
    NC, D, H, W = 2, 50, 10, 20                       # 20,000 frustum points, all in cell 5
    _edge(bp, np.full(NC * D * H * W, 5), NC, D, H, W, 80, 9, "long_interval")


def test_edge_run_lengths_at_sort_boundaries(bp):
    """Runs whose lengths sit on either side of every sort boundary of the
    map build: 16 / 17 points (one thread's registers / a warp's slice),
    32 / 33 (one slice / two), 8192 / 8193 (256 slices / the frustum scan),
    placed at random frustum positions so the order inside each run is
    checked against the oracle's (cell, p) order."""
    NC, D, H, W = 2, 30, 20, 25                       # 30,000 frustum points
    nf = NC * D * H * W
    lengths = [16, 17, 32, 33, 64, 65, 128, 129, 8191, 8192, 8193]
    rng = np.random.default_rng(31)
    cid = np.full(nf, -1, np.int64)
    pos = rng.permutation(nf)
    at = 0
    for cell, L in enumerate(lengths):
        cid[pos[at:at + L]] = cell
        at += L
    rest = pos[at:]
    cid[rest] = np.where(rng.random(rest.size) < 0.5, rng.integers(len(lengths), 400, rest.size), -1)
    m, _ = _edge(bp, cid, NC, D, H, W, 64, 400, "sort_boundaries")
    got = np.bincount(m.ranks_bev[:m.n_points].cpu().numpy(), minlength=400)[:len(lengths)]
    assert got.tolist() == lengths


def test_edge_every_cell_hit_once(bp):
    NC, D, H, W = 2, 1, 16, 32
    nf = NC * D * H * W
    _edge(bp, np.random.default_rng(4).permutation(nf), NC, D, H, W, 64, nf, "bijection")


def test_edge_largest_output(bp):
    """n_cells * C just under 2^31 (the largest output the forward accepts, a
    4 GB fp16 grid): points in the first and in the last cells, so rows at the
    far end of the output (byte offsets near 4 GiB) are written and checked.
    The expected rows come from the oracle run on the same points with the
    occupied cells numbered compactly; every other row must be zero."""
    from depth_weighted_scatter_gb300 import workloads

    C = 256
    cells = (2 ** 31 - 1) // C
    NC, D, H, W = 1, 8, 8, 16
    nf = NC * D * H * W
    rng = np.random.default_rng(41)
    cid = np.where(rng.random(nf) < 0.5, rng.integers(0, 60, nf), rng.integers(cells - 60, cells, nf))
    cid[rng.random(nf) < 0.2] = -1
    wl = workloads.custom(NC, D, H, W, C, cells, cid.astype(np.int32), seed=41, name="largest_output")
    c_d, depth, feat = upload(wl)
    m = _gpu_map(bp, wl, c_d)
    _check_map(bp, wl, m)
    out = torch.full((cells, C), float("nan"), dtype=torch.float16, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out)
    torch.cuda.synchronize()
    used = np.unique(cid[cid >= 0])
    compact = np.where(cid >= 0, np.searchsorted(used, cid), -1).astype(np.int32)
    wl_c = workloads.custom(NC, D, H, W, C, len(used), compact, name="largest_output_compact", depth=wl.depth,
                            feat=wl.feat)
    assert_forward_close(wl_c, out[torch.from_numpy(used).cuda()], oracle_forward(wl_c))
    assert not bool(torch.isnan(out).any())
    rows_nonzero = int((out != 0).any(dim=1).sum())
    assert rows_nonzero <= len(used)
    assert used.max() >= cells - 60                    # the far end of the grid is among the checked rows


def test_edge_ragged_tiles_and_many_cells(bp):
    """Frustum not a multiple of the 4096-point tile; cell ids need 31 bits (3 radix passes)."""
    NC, D, H, W = 1, 37, 13, 11                       # 5291 points: one full tile + a ragged one
    rng = np.random.default_rng(11)
    cells = (1 << 31) - 1
    cid = rng.integers(0, 40, NC * D * H * W).astype(np.int64) * 50_000_000 + rng.integers(0, 3, NC * D * H * W)
    cid[rng.random(cid.size) < 0.2] = -1
    from depth_weighted_scatter_gb300 import workloads
    import oracle

    wl = workloads.custom(NC, D, H, W, 8, cells, cid.astype(np.int32), seed=11, name="wide_keys")
    c_d, depth, feat = upload(wl)
    m = _gpu_map(bp, wl, c_d)
    _check_map(bp, wl, m)


def test_edge_radix_path_just_above_counting_limit(bp):
    """A grid one cell bigger than the counting-sort limit takes the radix path (25-bit keys)."""
    from depth_weighted_scatter_gb300 import workloads

    NC, D, H, W = 2, 9, 17, 19
    nf = NC * D * H * W
    cells = (1 << 24) + 1
    rng = np.random.default_rng(21)
    cid = np.where(rng.random(nf) < 0.5, rng.integers(0, 300, nf), rng.integers(cells - 300, cells, nf))
    cid[rng.random(nf) < 0.1] = -1
    wl = workloads.custom(NC, D, H, W, 8, cells, cid.astype(np.int32), seed=21, name="radix_path")
    c_d, _, _ = upload(wl)
    _check_map(bp, wl, _gpu_map(bp, wl, c_d))


def test_edge_out_of_range_ids_flagged(bp):
    NC, D, H, W, cells = 1, 4, 8, 8, 64
    rng = np.random.default_rng(12)
    cid = rng.integers(0, cells, NC * D * H * W).astype(np.int32)
    cid[[3, 77, 200]] = [-5, cells, 1 << 30]
    c_d = torch.from_numpy(cid).cuda()
    with pytest.raises(bp.BevpoolError) as ei:
        bp.build_map(c_d, NC, D, H, W, cells)
    assert ei.value.status == bp.BEVPOOL_ERR_OUT_OF_RANGE
    m = bp.build_map(c_d, NC, D, H, W, cells, sync=False)
    counts = m.d_counts.cpu().numpy()
    assert counts[2] == 3                             # three invalid ids, treated as dropped
    import oracle

    good = cid.copy()
    good[[3, 77, 200]] = -1
    ref = oracle.build_map(good, NC, D, H, W, cells)
    got = m.host()
    for k in MAP_KEYS:
        assert np.array_equal(got[k], ref[k])


def test_validate_map_flags_corruption(bp, wl_cache):
    wl = wl_cache("tiny")
    cells, _, _ = upload(wl)
    m = _gpu_map(bp, wl, cells)
    assert bp.validate_map(m) == 0
    m.interval_lengths[0] += 1
    assert bp.validate_map(m) & (1 | 2)
    m.interval_lengths[0] -= 1
    m.ranks_feat[0] = wl.n_feat_rows
    assert bp.validate_map(m) & 32


def test_forward_rejects_bad_arguments(bp, wl_cache):
    wl = wl_cache("tiny")
    cells, depth, feat = upload(wl)
    m = _gpu_map(bp, wl, cells)
    with pytest.raises(bp.BevpoolError) as ei:
        bp.forward(m, depth, feat, 24)
    assert ei.value.status == bp.BEVPOOL_ERR_UNSUPPORTED
    out = torch.empty(wl.n_cells * wl.C + 8, dtype=torch.float16, device="cuda")
    with pytest.raises(bp.BevpoolError) as ei:
        bp.forward(m, depth, feat, wl.C, out=out[1:])     # misaligned output
    assert ei.value.status == bp.BEVPOOL_ERR_INVALID_ARG


@pytest.mark.parametrize("intervals", ["short", "long"])
@pytest.mark.parametrize("dtype", ["f16", "e4m3"])
@pytest.mark.parametrize("C", [8, 80, 256])
def test_streaming_regime_channel_counts(bp, C, dtype, intervals):
    """A grid big enough that the output streams past L2 selects the kernels
    for that regime (evict-first stores; the variants with four CTAs per SM,
    one for short intervals and one for long): parity on every row, the few
    occupied ones and the many zeros."""
    from depth_weighted_scatter_gb300 import workloads

    cells = (72 << 20) // (2 * C) + 1                   # > 72 MiB of fp16 output
    NC, D, H, W = 2, 11, 9, 13
    rng = np.random.default_rng(C + 77 + 1000 * (intervals == "long"))
    nf = NC * D * H * W
    cid = rng.integers(0, cells, nf).astype(np.int32)
    hot = rng.random(nf) < (0.3 if intervals == "short" else 0.97)
    cid[hot] = rng.integers(0, 50, int(hot.sum()))      # a dense corner with long intervals
    cid[rng.random(nf) < 0.2] = -1
    wl = workloads.custom(NC, D, H, W, C, cells, cid, seed=C, dtype=dtype,
                          name=f"stream_C{C}_{dtype}_{intervals}")
    c_d, depth, feat = upload(wl)
    m = _gpu_map(bp, wl, c_d)
    _check_interval_mix(m, intervals)
    _check_map(bp, wl, m)
    out = torch.full((cells, C), float("nan"), dtype=torch.float16, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out)
    torch.cuda.synchronize()
    assert_forward_close(wl, out, oracle_forward(wl))


def test_forward_skips_out_of_range_entries(bp, wl_cache):
    """A map with out-of-range entries, as the forward's contract states:
    a point whose ranks_depth / ranks_feat is outside the tensors adds
    nothing, an interval whose cell is outside [0, n_cells) is not written
    (its old cell is then written as zeros).  The expected output is the
    oracle's on the same frustum with those points dropped, which gives the
    same rows.  Runs the checked walk (skipped points) and the no-cell path."""
    import oracle

    wl = wl_cache("canonical")
    cells, depth, feat = upload(wl)
    m = _gpu_map(bp, wl, cells)
    h = m.host()
    n = h["n_points"]
    rng = np.random.default_rng(5)
    rd0 = h["ranks_depth"]
    rd, rf, rb = rd0.copy(), h["ranks_feat"].copy(), h["ranks_bev"].copy()
    bad_d = rng.choice(n, 300, replace=False)
    bad_f = rng.choice(n, 300, replace=False)
    rd[bad_d[:150]] = -3
    rd[bad_d[150:]] = wl.n_frustum + 11
    rf[bad_f[:150]] = -1
    rf[bad_f[150:]] = wl.n_feat_rows
    s, ln = h["interval_starts"], h["interval_lengths"]
    first = np.arange(s[0], s[0] + ln[0])
    last = np.arange(s[-1], s[-1] + ln[-1])
    rb[first] = -7                                   # still ascending
    rb[last] = wl.n_cells + 5
    dropped = np.unique(np.concatenate([rd0[bad_d], rd0[bad_f], rd0[first], rd0[last]]))
    m.ranks_depth[:n].copy_(torch.from_numpy(rd))
    m.ranks_feat[:n].copy_(torch.from_numpy(rf))
    m.ranks_bev[:n].copy_(torch.from_numpy(rb))
    out = torch.full((wl.n_cells, wl.C), float("nan"), dtype=torch.float16, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out)
    torch.cuda.synchronize()
    cid = wl.cell_ids.copy()
    cid[dropped] = -1
    ref = oracle.forward(wl.dtype, cid, *wl.dims(), wl.n_cells, wl.C, wl.depth, wl.feat, wl.depth_scale,
                         wl.feat_scale)
    assert_forward_close(wl, out, ref, cell_ids=cid)
    g = out.float().cpu().numpy()
    assert np.all(g[int(h["ranks_bev"][s[0]])] == 0) and np.all(g[int(h["ranks_bev"][s[-1]])] == 0)

