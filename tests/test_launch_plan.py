"""The forward's launch plan (bevpool_forward_plan): the kernel variant, the
compute-CTA count and the fill tiling chosen on the host, checked without a
GPU against the rules the kernel header states.  The plan is asked for an
explicit GPU (SM count, L2 size), so no device is needed."""
import itertools

import numpy as np
import pytest

from depth_weighted_scatter_gb300 import bevpool as bp

SMS = 152
L2 = 135_528_448                      # GB300 l2CacheSize
DEFAULT, LEAN, SHORT, LEAN_SHORT = 0, 1, 2, 3
CANON = dict(NC=6, D=118, H=32, W=88)


def plan(dtype, C, n_points, n_intervals, n_cells, *, dims=CANON, e4m3_out=False, on_device=False, sms=SMS, l2=L2):
    return bp.forward_plan(dtype, C, dims["NC"], dims["D"], dims["H"], dims["W"], n_points, n_intervals, n_cells,
                           e4m3_out=e4m3_out, counts_on_device=on_device, sm_count=sms, l2_bytes=l2)


def footprint(dtype, C, n_points, n_intervals, n_cells, dims=CANON, e4m3_out=False):
    """Bytes a forward touches once: ranks, intervals, depth, features, output."""
    nf = dims["NC"] * dims["D"] * dims["H"] * dims["W"]
    rows = dims["NC"] * dims["H"] * dims["W"]
    eb = 2 if dtype == bp.BEVPOOL_F16 else 1
    feat = rows * (C // 2 + C // 16) if dtype == bp.BEVPOOL_NVFP4 else rows * C * eb
    return 12 * n_points + 8 * n_intervals + nf * eb + feat + n_cells * C * (1 if e4m3_out else 2)


def expected_fill_cells(n_cells, n_points, row_bytes, streaming, sms=SMS):
    """Output in L2: the largest power of two in [128, 1024] with at most 80 KB
    of rows, at most 1024 points on average and at least one tile per SM.
    Streaming: 256 doubled while the grid exceeds four tiles per SM, at most 1024."""
    if streaming:
        f = 256
        while f < 1024 and n_cells > f * 4 * sms:
            f *= 2
        return f
    f = 1024
    while f > 128 and (f * row_bytes > 80 * 1024 or n_points * f > 1024 * n_cells or -(-n_cells // f) < sms):
        f //= 2
    return f


# ------------------------------------------------------------------ the configurations

def test_plans_of_the_five_configurations():
    """The plans the benchmarked workloads get (regression pins of the rules below)."""
    canon = plan(bp.BEVPOOL_F16, 80, 209_077, 57_403, 129_600)
    assert (canon["variant"], canon["ctas_per_sm"], canon["n_compute"], canon["fill_cells"], canon["n_fill"],
            canon["streaming"]) == (SHORT, 2, 304, 512, 254, 0)
    fp8 = plan(bp.BEVPOOL_E4M3, 80, 209_077, 57_403, 129_600)
    assert (fp8["variant"], fp8["n_compute"], fp8["streaming"]) == (DEFAULT, 304, 0)
    bevdet = plan(bp.BEVPOOL_F16, 64, 182_660, 9_452, 16_384, dims=dict(NC=6, D=59, H=16, W=44))
    assert (bevdet["variant"], bevdet["n_compute"], bevdet["fill_cells"], bevdet["n_fill"]) == (DEFAULT, 304, 128, 128)
    dram = plan(bp.BEVPOOL_F16, 128, 2_198_618, 738_763, 1 << 20, dims=dict(NC=24, D=118, H=32, W=88))
    assert (dram["variant"], dram["ctas_per_sm"], dram["n_compute"], dram["fill_cells"], dram["n_fill"],
            dram["streaming"]) == (LEAN_SHORT, 4, 1824, 1024, 1024, 1)
    assert dram["round"] == 1280 and canon["round"] == 1024 and bevdet["round"] == 1280 and fp8["round"] == 1024
    tiny = plan(bp.BEVPOOL_F16, 8, 190, 150, 256, dims=dict(NC=1, D=8, H=4, W=8))
    assert tiny["n_compute"] == 1 and tiny["n_fill"] == 2 and tiny["streaming"] == 0


# ------------------------------------------------------------------ variant rules

@pytest.mark.parametrize("C", [64, 80, 128, 256])
def test_fp16_variant_rules(C):
    """fp16: lean when the output streams past the L2 or there are at least
    2^17 point-channels per SM; lean-short / short when intervals average
    under 8 points (host counts); the default otherwise."""
    n_cells = 129_600
    for n, per_interval in itertools.product([20_000, 209_077, 400_000, 900_000], [2.5, 7.9, 8.0, 19.0]):
        n_int = max(1, int(n / per_interval))
        p = plan(bp.BEVPOOL_F16, C, n, n_int, n_cells)
        streaming = footprint(bp.BEVPOOL_F16, C, n, n_int, n_cells) > L2 // 2
        much = n * C >= (1 << 17) * SMS
        short = n < 8 * n_int
        assert p["streaming"] == int(streaming)
        if streaming or much:
            want = LEAN_SHORT if short else LEAN
        else:
            want = SHORT if short else DEFAULT
        assert p["variant"] == want, (C, n, n_int, p)
        assert p["ctas_per_sm"] == (4 if want in (LEAN, LEAN_SHORT) else (3 if streaming else 2))


def test_lean_threshold_is_point_channels_per_sm():
    """The work rule switches exactly at n_points * C = 2^17 * SMs."""
    C = 80
    n_edge = -(-(1 << 17) * SMS // C)          # the smallest count at or above the threshold
    below = plan(bp.BEVPOOL_F16, C, n_edge - 1, (n_edge - 1) // 20, 129_600)
    at = plan(bp.BEVPOOL_F16, C, n_edge, n_edge // 20, 129_600)
    assert below["variant"] == DEFAULT and at["variant"] == LEAN
    other = plan(bp.BEVPOOL_F16, C, n_edge, n_edge // 20, 129_600, sms=148)
    assert other["variant"] == LEAN            # fewer SMs: more work per SM


def test_short_interval_threshold_is_eight_points():
    for n_int, want in [(26_134, DEFAULT), (26_135, SHORT)]:       # 209_077 < 8 * 26_135
        assert plan(bp.BEVPOOL_F16, 80, 209_077, n_int, 129_600)["variant"] == want


def test_e4m3_and_nvfp4_variants():
    """E4M3 rows take the lean variant only when the output streams; NVFP4
    rows always take the default one."""
    for dtype in (bp.BEVPOOL_E4M3, bp.BEVPOOL_NVFP4):
        small = plan(dtype, 80, 209_077, 57_403, 129_600)
        assert small["variant"] == DEFAULT and small["streaming"] == 0
        big = plan(dtype, 128, 2_198_618, 738_763, 1 << 20, dims=dict(NC=24, D=118, H=32, W=88))
        assert big["streaming"] == 1
        assert big["variant"] == (LEAN if dtype == bp.BEVPOOL_E4M3 else DEFAULT)
        assert big["ctas_per_sm"] == (4 if dtype == bp.BEVPOOL_E4M3 else 3)


def test_memory_regime_boundary_is_half_the_l2():
    """The output streams past the L2 exactly when the footprint exceeds half of it."""
    args = (bp.BEVPOOL_F16, 80, 209_077, 57_403, 129_600)
    fp = footprint(*args)
    assert plan(*args, l2=2 * fp)["streaming"] == 0
    assert plan(*args, l2=2 * fp - 2)["streaming"] == 1
    e4 = (bp.BEVPOOL_E4M3, 80, 209_077, 57_403, 129_600)
    assert plan(*e4, e4m3_out=True, l2=2 * footprint(*e4, e4m3_out=True))["streaming"] == 0
    assert plan(*e4, e4m3_out=True, l2=2 * footprint(*e4, e4m3_out=True) - 2)["streaming"] == 1


def test_counts_on_device_with_the_whole_frustum_as_capacity():
    """A capacity equal to the frustum says nothing about the frame's points:
    no work or interval-length rule, one wave of compute CTAs at most."""
    nf = 6 * 118 * 32 * 88
    p = plan(bp.BEVPOOL_F16, 80, nf, 129_600, 129_600, on_device=True, l2=(1 << 31) - 1)
    assert p["variant"] == DEFAULT and p["n_compute"] <= SMS * p["ctas_per_sm"]
    # a tight capacity with the counts on the device is planned like host counts
    q = plan(bp.BEVPOOL_F16, 80, 209_077, 57_403, 129_600, on_device=True)
    r = plan(bp.BEVPOOL_F16, 80, 209_077, 57_403, 129_600)
    assert q == r


# ------------------------------------------------------------------ compute CTAs

@pytest.mark.parametrize("dtype,C", [(bp.BEVPOOL_F16, 80), (bp.BEVPOOL_F16, 128), (bp.BEVPOOL_E4M3, 80),
                                     (bp.BEVPOOL_NVFP4, 64), (bp.BEVPOOL_F16, 8)])
def test_compute_cta_count(dtype, C):
    """One wave (SMs x CTAs per SM) at most, and at least a batch of points per
    owner, unless one round per CTA needs more: then whole waves of CTAs of at
    most a round less 64 points."""
    for n in [1, 100, 5_000, 60_000, 209_077, 700_000, 2_200_000]:
        n_int = max(1, n // 3)
        p = plan(dtype, C, n, n_int, 1 << 20, dims=dict(NC=24, D=118, H=32, W=88))
        slots = SMS * p["ctas_per_sm"]
        one_wave = min(-(-n // (p["owners"] * p["batch"])), slots)
        want = -(-n // (p["round"] - 64))
        if want > one_wave:
            assert p["n_compute"] % slots == 0 and p["n_compute"] == slots * -(-want // slots)
            assert -(-n // p["n_compute"]) <= p["round"] - 64
        else:
            assert p["n_compute"] == max(1, one_wave)
        assert p["round"] % 256 == 0 and 256 <= p["round"] <= (1280 if dtype == bp.BEVPOOL_F16 else 1024)


def test_rounds_fit_the_shared_memory_of_wide_rows():
    """Rows of 256 channels leave room for full rounds: 1280 points for the fp16
    default and lean-short variants, 1024 for the other variants and dtypes."""
    for dtype in (bp.BEVPOOL_F16, bp.BEVPOOL_E4M3, bp.BEVPOOL_NVFP4):
        p = plan(dtype, 256, 210_000, 57_000, 129_600)
        wide = dtype == bp.BEVPOOL_F16 and p["variant"] in (DEFAULT, LEAN_SHORT)
        assert p["round"] == (1280 if wide else 1024)
    assert plan(bp.BEVPOOL_F16, 256, 210_000, 20_000, 129_600)["round"] == 1024      # the plain lean variant


# ------------------------------------------------------------------ fill tiles

@pytest.mark.parametrize("n_cells", [1, 255, 256, 4_096, 16_384, 129_600, 155_648, 155_649, 311_296, 311_297,
                                     1 << 20, 4 << 20])
@pytest.mark.parametrize("points_per_cell", [0.01, 1.6, 8.0, 11.0])
def test_fill_tiles(n_cells, points_per_cell):
    """Cells per fill CTA by the two rules (the output in L2 or streaming past
    it); the fill CTAs cover the grid exactly once."""
    dims = dict(NC=96, D=118, H=32, W=88)                       # room for every point count below
    for C in (8, 80, 256):
        if n_cells * C >= 1 << 31:
            continue
        n = min(int(n_cells * points_per_cell), 96 * 118 * 32 * 88)
        p = plan(bp.BEVPOOL_F16, C, n, max(0, min(n, n_cells) // 2), n_cells, dims=dims)
        assert p["fill_cells"] == expected_fill_cells(n_cells, n, 2 * C, p["streaming"] == 1), (n_cells, n, C, p)
        assert p["n_fill"] == -(-n_cells // p["fill_cells"])
        assert (p["n_fill"] - 1) * p["fill_cells"] < n_cells <= p["n_fill"] * p["fill_cells"]


def test_fill_tiles_follow_the_sm_count_and_the_regime():
    # output in L2: at least one fill CTA per SM
    assert plan(bp.BEVPOOL_F16, 80, 100, 50, 200_000, sms=152)["fill_cells"] == 512
    assert plan(bp.BEVPOOL_F16, 80, 100, 50, 200_000, sms=256)["fill_cells"] == 512
    assert plan(bp.BEVPOOL_F16, 80, 100, 50, 100_000, sms=256)["fill_cells"] == 256
    # streaming: four fill CTAs per SM
    assert plan(bp.BEVPOOL_F16, 80, 100, 50, 200_000, sms=152, l2=1 << 20)["fill_cells"] == 512
    assert plan(bp.BEVPOOL_F16, 80, 100, 50, 200_000, sms=256, l2=1 << 20)["fill_cells"] == 256


# ------------------------------------------------------------------ refusals

def test_plan_refuses_what_the_forward_refuses():
    plan_arr = np.zeros(9, dtype=np.int32)
    call = lambda dtype, C, e4m3_out=0, n_pts=10, n_int=5, n_cells=100: bp.bevpool_forward_plan(
        dtype, C, e4m3_out, 1, 2, 3, 4, n_pts, n_int, 0, n_cells, SMS, L2, plan_arr)
    assert call(bp.BEVPOOL_F16, 81) == bp.BEVPOOL_ERR_UNSUPPORTED
    assert call(bp.BEVPOOL_F16, 8, e4m3_out=1) == bp.BEVPOOL_ERR_UNSUPPORTED      # E4M3 output needs C % 16 == 0
    assert call(bp.BEVPOOL_NVFP4, 8) == bp.BEVPOOL_ERR_UNSUPPORTED
    assert call(bp.BEVPOOL_F16, 80, n_pts=25) == bp.BEVPOOL_ERR_INVALID_ARG        # more points than the frustum
    assert call(bp.BEVPOOL_F16, 80, n_int=11) == bp.BEVPOOL_ERR_INVALID_ARG        # more intervals than points
    assert call(bp.BEVPOOL_F16, 80, n_cells=0) == bp.BEVPOOL_ERR_INVALID_ARG
    assert bp.bevpool_forward_plan(bp.BEVPOOL_F16, 80, 0, 1, 2, 3, 4, 10, 5, 0, 100, SMS, L2, None) == \
        bp.BEVPOOL_ERR_INVALID_ARG
    assert call(bp.BEVPOOL_F16, 80) == bp.BEVPOOL_OK


@pytest.mark.gpu
def test_plan_for_the_current_device_uses_its_sm_count_and_l2():
    """With no GPU named, the plan is the one for the current device."""
    import torch

    props = torch.cuda.get_device_properties(0)
    args = (bp.BEVPOOL_F16, 80, 6, 118, 32, 88, 209_077, 57_403, 129_600)
    assert bp.forward_plan(*args) == bp.forward_plan(*args, sm_count=props.multi_processor_count,
                                                     l2_bytes=props.L2_cache_size)
