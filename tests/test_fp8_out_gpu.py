"""GPU parity of the E4M3-output forward (bevpool_forward_e4m3_out) against
the FP64 oracle's nearest E4M3 codes; see gpu_common.assert_e4m3_out_matches
for the criterion (exact except at rounding midpoints within the FP32 error
bound)."""
import numpy as np
import pytest

from gpu_common import assert_e4m3_out_matches, dtype_code, oracle_forward, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bp():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from depth_weighted_scatter_gb300 import bevpool

    return bevpool


def _run(bp, wl, out_scale, sync=True):
    cells, depth, feat = upload(wl)
    m = bp.build_map(cells, *wl.dims(), wl.n_cells, sync=sync)
    out = torch.full((wl.n_cells, wl.C), 0x7F, dtype=torch.uint8, device="cuda")    # NaN code: unwritten rows show
    bp.forward(m, depth, feat, wl.C, dtype=dtype_code(wl), depth_scale=wl.depth_scale,
               feat_scale=wl.feat_scale, out=out, out_scale=out_scale)
    torch.cuda.synchronize()
    return out, m


def _calibrated_scale(wl):
    ref = oracle_forward(wl)
    return float(np.abs(ref).max()) / 448.0


@pytest.mark.parametrize("name", ["canonical_fp8", "canonical", "bevdet"])
def test_full_config_e4m3_out(bp, name, wl_cache):
    wl = wl_cache(name)
    s = _calibrated_scale(wl)
    out, _ = _run(bp, wl, s)
    assert_e4m3_out_matches(wl, out, s)


def test_dram_batch_e4m3_out_sampled(bp, wl_cache):
    """Full DRAM batch in the launch configuration of the benchmark; checked
    on 4096 sampled cells (every output row written, codes near the oracle's)."""
    import oracle

    wl = wl_cache("dram_batch")
    ref = oracle_forward(wl)
    s = float(np.abs(ref).max()) / 448.0
    out, _ = _run(bp, wl, s)
    g = out.cpu().numpy()
    rng = np.random.default_rng(3)
    rows = rng.choice(wl.n_cells, 4096, replace=False)
    gv = oracle.e4m3_to_double(g[rows])
    v = ref[rows] / s
    assert not np.isnan(gv).any()
    # within one E4M3 step of the exact value (3 mantissa bits: half-ulp 2^-4 relative, plus subnormals)
    assert np.all(np.abs(gv - v) <= np.maximum(np.abs(v) * 2.0 ** -3, 2.0 ** -9))


@pytest.mark.parametrize("intervals", ["short", "long"])
@pytest.mark.parametrize("dtype", ["f16", "e4m3"])
@pytest.mark.parametrize("C", [16, 32, 64, 80, 96, 128, 160, 192, 256])
def test_every_channel_count_e4m3_out(bp, C, dtype, intervals):
    """Intervals of about 3 points (short) and of about 60 (long) select
    different fp16 kernel variants."""
    from depth_weighted_scatter_gb300 import workloads

    NC, D, H, W, cells = 3, 17, 6, 11, 700
    rng = np.random.default_rng(C * 11 + (dtype == "e4m3") + 1000 * (intervals == "long"))
    nf = NC * D * H * W
    cid = rng.integers(0, cells if intervals == "short" else 40, nf).astype(np.int32)
    cid[rng.random(nf) < 0.3] = -1
    cid[rng.random(nf) < 0.08] = 123
    wl = workloads.custom(NC, D, H, W, C, cells, cid, seed=C + 1, dtype=dtype, name=f"C{C}_{dtype}_{intervals}_q")
    s = _calibrated_scale(wl)
    out, m = _run(bp, wl, s)
    assert (m.n_points < 8 * m.n_intervals) == (intervals == "short"), (m.n_points, m.n_intervals)
    assert_e4m3_out_matches(wl, out, s)


@pytest.mark.parametrize("intervals", ["short", "long"])
@pytest.mark.parametrize("dtype", ["f16", "e4m3"])
def test_streaming_regime_e4m3_out(bp, dtype, intervals):
    """An E4M3 output larger than half of L2 takes the streaming kernels (four
    CTAs per SM; for fp16 rows one variant for short intervals and one for
    long): every row checked, the few occupied ones and the many zeros."""
    from depth_weighted_scatter_gb300 import workloads

    C = 128
    cells = (72 << 20) // C + 1                          # > 72 MiB of E4M3 output
    NC, D, H, W = 2, 11, 9, 13
    rng = np.random.default_rng(91 + (dtype == "e4m3") + 1000 * (intervals == "long"))
    nf = NC * D * H * W
    cid = rng.integers(0, cells, nf).astype(np.int32)
    hot = rng.random(nf) < (0.3 if intervals == "short" else 0.97)
    cid[hot] = rng.integers(0, 50, int(hot.sum()))
    cid[rng.random(nf) < 0.2] = -1
    wl = workloads.custom(NC, D, H, W, C, cells, cid, seed=5, dtype=dtype, name=f"stream_q_{dtype}_{intervals}")
    s = _calibrated_scale(wl)
    out, m = _run(bp, wl, s)
    assert (m.n_points < 8 * m.n_intervals) == (intervals == "short"), (m.n_points, m.n_intervals)
    assert_e4m3_out_matches(wl, out, s)


def test_e4m3_out_saturates_and_zero_fills(bp):
    """A small out_scale drives most values past 448: they saturate (no NaN
    codes); cells without points hold the zero code."""
    from depth_weighted_scatter_gb300 import workloads

    NC, D, H, W, C, cells = 2, 9, 5, 7, 64, 400
    rng = np.random.default_rng(23)
    cid = rng.integers(0, cells // 2, NC * D * H * W).astype(np.int32)     # upper half of the grid empty
    wl = workloads.custom(NC, D, H, W, C, cells, cid, seed=23, name="saturate")
    s = _calibrated_scale(wl) / 50.0
    out, _ = _run(bp, wl, s)
    assert_e4m3_out_matches(wl, out, s)
    g = out.cpu().numpy()
    assert np.all(g[cells // 2:] == 0)
    assert np.any((g & 0x7F) == 0x7E)                     # some saturated codes


def test_e4m3_out_device_counts_and_determinism(bp, wl_cache):
    wl = wl_cache("canonical_fp8")
    s = _calibrated_scale(wl)
    a, _ = _run(bp, wl, s)
    b, _ = _run(bp, wl, s)
    assert torch.equal(a, b)
    cells, depth, feat = upload(wl)
    m = bp.build_map(cells, *wl.dims(), wl.n_cells, sync=False)
    n_pts = int(m.d_counts[0].item())
    n_int = int(m.d_counts[1].item())
    c = bp.forward(m, depth, feat, wl.C, dtype=dtype_code(wl), depth_scale=wl.depth_scale,
                   feat_scale=wl.feat_scale, out_scale=s, capacity=(n_pts, n_int))
    torch.cuda.synchronize()
    assert torch.equal(a, c)


def test_e4m3_out_all_dropped(bp):
    from depth_weighted_scatter_gb300 import workloads

    wl = workloads.custom(2, 3, 4, 5, 32, 50, np.full(2 * 3 * 4 * 5, -1, np.int32), name="dropped_q")
    out, m = _run(bp, wl, 1.0)
    assert m.n_points == 0
    assert torch.count_nonzero(out) == 0


def test_e4m3_out_rejects_bad_arguments(bp, wl_cache):
    wl = wl_cache("tiny")                                   # C = 8: not a multiple of 16
    cells, depth, feat = upload(wl)
    m = bp.build_map(cells, *wl.dims(), wl.n_cells)
    with pytest.raises(bp.BevpoolError) as ei:
        bp.forward(m, depth, feat, wl.C, out_scale=1.0)
    assert ei.value.status == bp.BEVPOOL_ERR_UNSUPPORTED
