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


def _noalloc_map(bp, wl, cells, sync=True):
    """Map built by bevpool_build_map_noalloc into caller-allocated outputs;
    with sync=False no host counts are asked for (nothing waits on the GPU)
    and the counts are read from d_counts after a stream synchronize."""
    m = bp.ScatterMap.allocate(*wl.dims(), wl.n_cells)
    h = np.zeros(3, dtype=np.int32) if sync else None
    stream = torch.cuda.current_stream()
    st = bp.bevpool_build_map_noalloc(cells.data_ptr(), *wl.dims(), wl.n_cells, m.ranks_depth.data_ptr(),
                                      m.ranks_feat.data_ptr(), m.ranks_bev.data_ptr(), m.interval_starts.data_ptr(),
                                      m.interval_lengths.data_ptr(), m.d_counts.data_ptr(), h, stream.cuda_stream)
    assert st == bp.BEVPOOL_OK, bp.bevpool_status_string(st)
    if not sync:
        stream.synchronize()
        h = m.d_counts.cpu().numpy()
    m.n_points, m.n_intervals = int(h[0]), int(h[1])
    return m


def _assert_same_map(bp, wl, cells, got):
    ref = bp.build_map(cells, *wl.dims(), wl.n_cells).host()
    assert got["n_points"] == ref["n_points"] and got["n_intervals"] == ref["n_intervals"], wl.name
    for k in MAP_KEYS:
        assert np.array_equal(got[k], ref[k]), f"{wl.name}: {k} differs"


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(bp, wl_cache):
    # Consecutive calls with different frusta, then a repeat of the first: each
    # call finds the scratch as the previous one left it.
    for name in ["bevdet", "canonical", "bevdet"]:
        wl = wl_cache(name)
        assert wl.n_frustum <= bp.BEVPOOL_NOALLOC_MAX_FRUSTUM
        cells = torch.from_numpy(wl.cell_ids).cuda()
        _assert_same_map(bp, wl, cells, _noalloc_map(bp, wl, cells).host())


def _grid_case(n_cells, seed):
    """A small frustum on a grid of n_cells: half the points near the first
    cells, half near the last, 10 % dropped."""
    from depth_weighted_scatter_gb300 import workloads

    NC, D, H, W = 2, 9, 17, 19
    nf = NC * D * H * W
    rng = np.random.default_rng(seed)
    cid = np.where(rng.random(nf) < 0.5, rng.integers(0, 300, nf), rng.integers(n_cells - 300, n_cells, nf))
    cid[rng.random(nf) < 0.1] = -1
    return workloads.custom(NC, D, H, W, 8, n_cells, cid.astype(np.int32), seed=seed, name=f"grid_{n_cells}")


@pytest.mark.parametrize("n_cells", [(1 << 24) + 1, 12_000_000])
def test_noalloc_radix_path_matches_workspace_entry_point(bp, n_cells):
    # Above 2^24 cells the build always takes the radix path; at 12M cells the
    # counting path's per-cell tables (about 96 MB) do not fit in the built-in
    # scratch, so the no-alloc call takes the radix path while the workspace
    # call (given the larger workspace it asks for) takes the counting path.
    # Two calls in a row, the second finding the first one's scratch.
    import oracle

    wl = _grid_case(n_cells, 21)
    cells = torch.from_numpy(wl.cell_ids).cuda()
    ref = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    for _ in range(2):
        got = _noalloc_map(bp, wl, cells).host()
        _assert_same_map(bp, wl, cells, got)
        for k in MAP_KEYS:
            assert np.array_equal(got[k], ref[k]), f"{wl.name}: {k} differs from the oracle"


def test_noalloc_without_host_counts(bp, wl_cache):
    # h_counts = NULL: the call only enqueues work; the counts are read from
    # d_counts once the stream has drained.
    wl = wl_cache("canonical")
    cells = torch.from_numpy(wl.cell_ids).cuda()
    _assert_same_map(bp, wl, cells, _noalloc_map(bp, wl, cells, sync=False).host())


def test_noalloc_rejects_frustum_above_its_limit(bp):
    # 2^21 + 8 points: one frustum more than the built-in scratch holds.  The
    # call must refuse before touching the (never dereferenced) pointers.
    fake = 1 << 20
    NC, D, H, W = 1, (1 << 18) + 1, 2, 4
    assert NC * D * H * W > bp.BEVPOOL_NOALLOC_MAX_FRUSTUM
    st = bp.bevpool_build_map_noalloc(fake, NC, D, H, W, 100, fake, fake, fake, fake, fake, fake, None, 0)
    assert st == bp.BEVPOOL_ERR_WORKSPACE
