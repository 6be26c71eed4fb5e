"""GPU parity of the NVFP4-feature forward (bevpool_forward_nvfp4: E2M1
features with E4M3 block scales, E4M3 depth) against the FP64 oracle, with
fp16 and E4M3 outputs, at full size on the canonical and Table-1 shapes."""
import numpy as np
import pytest

from gpu_common import (MAP_KEYS, assert_e4m3_out_matches, assert_forward_close, gpu_forward, oracle_forward,
                        upload)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from depth_weighted_scatter_gb300 import workloads  # noqa: E402


@pytest.fixture(scope="module")
def bp():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from depth_weighted_scatter_gb300 import bevpool

    return bevpool


NAMES = ["canonical_nvfp4"] + [n + "_nvfp4" for n in workloads.TABLE1]


@pytest.mark.parametrize("name", NAMES)
def test_nvfp4_full_shape(bp, name, wl_cache):
    wl = wl_cache(name)
    cells, depth, feat = upload(wl)
    m = bp.build_map(cells, *wl.dims(), wl.n_cells)
    out = torch.full((wl.n_cells, wl.C), float("nan"), dtype=torch.float16, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out)
    torch.cuda.synchronize()
    assert_forward_close(wl, out, oracle_forward(wl))


@pytest.mark.parametrize("C", [64, 80, 96, 128, 160, 192, 256])
def test_nvfp4_every_channel_count(bp, C):
    NC, D, H, W, cells = 3, 17, 6, 11, 700
    rng = np.random.default_rng(C * 13)
    nf = NC * D * H * W
    cid = rng.integers(0, cells, nf).astype(np.int32)
    cid[rng.random(nf) < 0.3] = -1
    cid[rng.random(nf) < 0.08] = 123
    wl = workloads._to_nvfp4(workloads.custom(NC, D, H, W, C, cells, cid, seed=C + 2), f"C{C}_nvfp4")
    cells_d, depth, feat = upload(wl)
    m = bp.build_map(cells_d, *wl.dims(), wl.n_cells)
    out = torch.full((cells, C), float("nan"), dtype=torch.float16, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out)
    torch.cuda.synchronize()
    assert_forward_close(wl, out, oracle_forward(wl))


@pytest.mark.parametrize("intervals", ["short", "long"])
@pytest.mark.parametrize("C", [64, 256])
def test_nvfp4_streaming_regime(bp, C, intervals):
    """A grid whose fp16 output (> 72 MiB) streams past the L2: the NVFP4
    kernel with evict-first stores, fill CTAs after the first wave of compute
    CTAs, every row checked (the few occupied ones and the many zeros)."""
    cells = (72 << 20) // (2 * C) + 1
    NC, D, H, W = 2, 11, 9, 13
    rng = np.random.default_rng(C + 5 + 1000 * (intervals == "long"))
    nf = NC * D * H * W
    cid = rng.integers(0, cells, nf).astype(np.int32)
    hot = rng.random(nf) < (0.3 if intervals == "short" else 0.97)
    cid[hot] = rng.integers(0, 50, int(hot.sum()))      # a dense corner with long intervals
    cid[rng.random(nf) < 0.2] = -1
    wl = workloads._to_nvfp4(workloads.custom(NC, D, H, W, C, cells, cid, seed=C + 9), f"stream_C{C}_nvfp4_{intervals}")
    plan = bp.forward_plan(bp.BEVPOOL_NVFP4, C, *wl.dims(), wl.n_kept, 1, cells)
    assert plan["streaming"] == 1
    cells_d, depth, feat = upload(wl)
    m = bp.build_map(cells_d, *wl.dims(), wl.n_cells)
    out = torch.full((cells, C), float("nan"), dtype=torch.float16, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out)
    torch.cuda.synchronize()
    assert_forward_close(wl, out, oracle_forward(wl))


@pytest.mark.parametrize("name", ["canonical_nvfp4", "wide_c256_nvfp4"])
def test_nvfp4_e4m3_out(bp, name, wl_cache):
    """NVFP4 features with depth and output in FP8, as in the pages' experiment."""
    wl = wl_cache(name)
    s = float(np.abs(oracle_forward(wl)).max()) / 448.0
    cells, depth, feat = upload(wl)
    m = bp.build_map(cells, *wl.dims(), wl.n_cells)
    out = torch.full((wl.n_cells, wl.C), 0x7F, dtype=torch.uint8, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out, out_scale=s)
    torch.cuda.synchronize()
    assert_e4m3_out_matches(wl, out, s)


def test_nvfp4_needs_its_entry_point(bp, wl_cache):
    wl = wl_cache("canonical_nvfp4")
    cells, depth, feat = upload(wl)
    m = bp.build_map(cells, *wl.dims(), wl.n_cells)
    st = bp.bevpool_forward(bp.BEVPOOL_NVFP4, depth.data_ptr(), feat.data_ptr(), *wl.dims(), wl.C, 1.0, 1.0,
                            m.ranks_depth.data_ptr(), m.ranks_feat.data_ptr(), m.ranks_bev.data_ptr(),
                            m.interval_starts.data_ptr(), m.interval_lengths.data_ptr(), m.n_points, m.n_intervals,
                            None, wl.n_cells, feat.data_ptr(), 0)
    assert st == bp.BEVPOOL_ERR_UNSUPPORTED
