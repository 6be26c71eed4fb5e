"""bevpool_build_map_noalloc against bevpool_build_map, through the C ABI.

bevpool_build_map_noalloc exists for callers that may not allocate device
memory when they build a scatter map -- for example an inference-engine
plugin whose enqueue step must not allocate, or real-time code that forbids
allocation after start-up.  It uses scratch compiled into the library
instead of a caller-provided workspace, so it must give exactly the map the
workspace entry point gives, call after call, although every call reuses
(and leaves behind) the same scratch.

This file is collected last on purpose: a run that stops at the first
failure has run every other test before this one.  It also passes on its
own in a fresh process.
"""
import numpy as np
import pytest

from gpu_common import MAP_KEYS

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bp():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from depth_weighted_scatter_gb300 import bevpool

    return bevpool


def _noalloc_map(bp, wl, cells):
    """Map built by bevpool_build_map_noalloc into caller-allocated outputs."""
    m = bp.ScatterMap.allocate(*wl.dims(), wl.n_cells)
    h = np.zeros(3, dtype=np.int32)
    st = bp.bevpool_build_map_noalloc(cells.data_ptr(), *wl.dims(), wl.n_cells, m.ranks_depth.data_ptr(),
                                      m.ranks_feat.data_ptr(), m.ranks_bev.data_ptr(), m.interval_starts.data_ptr(),
                                      m.interval_lengths.data_ptr(), m.d_counts.data_ptr(), h,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == bp.BEVPOOL_OK, bp.bevpool_status_string(st)
    m.n_points, m.n_intervals = int(h[0]), int(h[1])
    return m


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(bp, wl_cache):
    # Consecutive calls with different frusta, then a repeat of the first: each
    # call finds the scratch as the previous one left it.
    for name in ["bevdet", "canonical", "bevdet"]:
        wl = wl_cache(name)
        assert wl.n_frustum <= bp.BEVPOOL_NOALLOC_MAX_FRUSTUM
        cells = torch.from_numpy(wl.cell_ids).cuda()
        ref = bp.build_map(cells, *wl.dims(), wl.n_cells).host()
        got = _noalloc_map(bp, wl, cells).host()
        assert got["n_points"] == ref["n_points"] and got["n_intervals"] == ref["n_intervals"], name
        for k in MAP_KEYS:
            assert np.array_equal(got[k], ref[k]), f"{name}: {k} differs"


def test_noalloc_rejects_frustum_above_its_limit(bp):
    # 2^21 + 8 points: one frustum more than the built-in scratch holds.  The
    # call must refuse before touching the (never dereferenced) pointers.
    fake = 1 << 20
    NC, D, H, W = 1, (1 << 18) + 1, 2, 4
    assert NC * D * H * W > bp.BEVPOOL_NOALLOC_MAX_FRUSTUM
    st = bp.bevpool_build_map_noalloc(fake, NC, D, H, W, 100, fake, fake, fake, fake, fake, fake, None, 0)
    assert st == bp.BEVPOOL_ERR_WORKSPACE
