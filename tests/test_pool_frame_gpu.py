"""bevpool_pool_frame: map build + forward of one frame without a host
synchronisation.  Bit-identical to the two calls in sequence, within the fp16
tolerance of the oracle, and replayable from a CUDA graph with new geometry
(new cell ids) in the captured buffers."""
import numpy as np
import pytest

from gpu_common import MAP_KEYS, assert_forward_close, dtype_code, oracle_forward, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bp():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from depth_weighted_scatter_gb300 import bevpool

    return bevpool


@pytest.mark.parametrize("name", ["canonical", "bevdet", "canonical_fp8"])
def test_pool_frame_matches_two_calls_and_oracle(bp, name, wl_cache):
    import oracle

    wl = wl_cache(name)
    cells, depth, feat = upload(wl)
    kw = dict(dtype=dtype_code(wl), depth_scale=wl.depth_scale, feat_scale=wl.feat_scale)
    out, m = bp.pool_frame(cells, depth, feat, *wl.dims(), wl.n_cells, wl.C, **kw)
    m2 = bp.build_map(cells, *wl.dims(), wl.n_cells, sync=False)
    nf = wl.n_frustum
    ref2 = bp.forward(m2, depth, feat, wl.C, capacity=(nf, min(nf, wl.n_cells)), **kw)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref2.view(torch.int16))
    assert_forward_close(wl, out, oracle_forward(wl))
    n, ni = (int(v) for v in m.d_counts[:2].cpu())
    ref_map = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    assert (n, ni) == (ref_map["n_points"], ref_map["n_intervals"])
    m.n_points, m.n_intervals = n, ni
    got = m.host()
    for k in MAP_KEYS:
        assert np.array_equal(got[k], ref_map[k])


def test_pool_frame_graph_replay_with_new_geometry(bp):
    """Capture one frame, then replay it for two different sets of cell ids,
    depth and features copied into the captured buffers."""
    from depth_weighted_scatter_gb300 import workloads

    frames = [workloads.canonical(seed=1), workloads.canonical(seed=2)]
    wl0 = frames[0]
    cells, depth, feat = upload(wl0)
    m = bp.ScatterMap.allocate(*wl0.dims(), wl0.n_cells)
    ws = bp.workspace_for(*wl0.dims(), wl0.n_cells)
    out = torch.empty((wl0.n_cells, wl0.C), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        bp.pool_frame(cells, depth, feat, *wl0.dims(), wl0.n_cells, wl0.C, out=out, map_out=m, workspace=ws,
                      stream=s)                        # first call outside the capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            bp.pool_frame(cells, depth, feat, *wl0.dims(), wl0.n_cells, wl0.C, out=out, map_out=m, workspace=ws,
                          stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for wl in frames:
        c, d, f = upload(wl)
        cells.copy_(c)
        depth.copy_(d)
        feat.copy_(f)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_forward_close(wl, out, oracle_forward(wl))
        assert int(m.d_counts[0].item()) == wl.n_kept


def test_frames_on_concurrent_streams_match_sequential(bp):
    """Four frames (two canonical and two BEVDet geometries), each with its own
    buffers and workspace, issued three times over on four streams without a
    synchronisation in between: every output and map is bit-identical to the
    same frame run alone (the library keeps no per-call state of its own)."""
    from depth_weighted_scatter_gb300 import workloads

    frames = [workloads.canonical(seed=1), workloads.canonical(seed=2), workloads.bevdet(seed=3),
              workloads.bevdet(seed=5)]
    setups, refs = [], []
    for wl in frames:
        cells, depth, feat = upload(wl)
        m = bp.ScatterMap.allocate(*wl.dims(), wl.n_cells)
        ws = bp.workspace_for(*wl.dims(), wl.n_cells)
        out = torch.empty((wl.n_cells, wl.C), dtype=torch.float16, device="cuda")
        bp.pool_frame(cells, depth, feat, *wl.dims(), wl.n_cells, wl.C, out=out, map_out=m, workspace=ws)
        torch.cuda.synchronize()
        refs.append((out.clone(), m.d_counts.clone(), m.ranks_bev.clone(), m.ranks_depth.clone()))
        out.fill_(float("nan"))
        setups.append((wl, cells, depth, feat, m, ws, out))
    streams = [torch.cuda.Stream() for _ in frames]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        for s, (wl, cells, depth, feat, m, ws, out) in zip(streams, setups):
            with torch.cuda.stream(s):
                bp.pool_frame(cells, depth, feat, *wl.dims(), wl.n_cells, wl.C, out=out, map_out=m, workspace=ws,
                              stream=s)
    torch.cuda.synchronize()
    for (wl, _, _, _, m, _, out), (r_out, r_counts, r_bev, r_depth) in zip(setups, refs):
        n = int(r_counts[0].item())
        assert torch.equal(m.d_counts, r_counts), wl.name
        assert torch.equal(m.ranks_bev[:n], r_bev[:n]) and torch.equal(m.ranks_depth[:n], r_depth[:n]), wl.name
        assert torch.equal(out.view(torch.int16), r_out.view(torch.int16)), wl.name
