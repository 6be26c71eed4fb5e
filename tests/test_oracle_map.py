"""Pins for the oracle's scatter-map builder.

The map follows "Accelerating BEV Pooling on NVIDIA GPUs for Physical AI
Applications", section "Eliminate redundant scatter traffic" (five INT32
arrays, precomputed explicit indices) and section "Implement interval-owned
scatter-reduce" (one interval per BEV cell that some point reaches).

Pins: a pure-Python per-cell enumeration on the tiny workload, numpy's
library sort / unique on the larger ones, index arithmetic through
numpy's unravel/ravel routines, and partition invariants.
"""
import numpy as np
import pytest

import oracle
from depth_weighted_scatter_gb300 import workloads


def _frustum_coords(p, NC, D, H, W):
    return np.unravel_index(p, (NC, D, H, W))


def _feat_row(p, NC, D, H, W):
    nc, _, h, w = _frustum_coords(p, NC, D, H, W)
    return np.ravel_multi_index((nc, h, w), (NC, H, W)).astype(np.int32)


def _library_map(wl):
    p = np.nonzero(wl.cell_ids >= 0)[0]
    cell = wl.cell_ids[p]
    order = np.lexsort((p, cell))          # primary key cell, ties by p
    p, cell = p[order], cell[order]
    cells, starts, lengths = np.unique(cell, return_index=True, return_counts=True)
    return dict(ranks_bev=cell.astype(np.int32), ranks_depth=p.astype(np.int32),
                ranks_feat=_feat_row(p, *wl.dims()), interval_starts=starts.astype(np.int32),
                interval_lengths=lengths.astype(np.int32))


def check_map_invariants(m, wl):
    """Properties any correct map has; returns the list of violated ones."""
    bad = []
    n, ni = m["n_points"], m["n_intervals"]
    rb, rd, rf = m["ranks_bev"], m["ranks_depth"], m["ranks_feat"]
    st, ln = m["interval_starts"], m["interval_lengths"]
    if len(rb) != n or len(st) != ni:
        bad.append("sizes")
        return bad
    if ni and st[0] != 0:
        bad.append("first start")
    if np.any(ln < 1):
        bad.append("empty interval")
    if ni and np.any(st[1:] != st[:-1] + ln[:-1]):
        bad.append("starts not contiguous")
    if int(ln.sum()) != n:
        bad.append("lengths do not sum to n")
        return bad
    if ni:
        owner = np.repeat(np.arange(ni), ln)
        if np.any(rb != rb[st][owner]):
            bad.append("bev not constant inside an interval")
        if np.any(np.diff(rb[st]) <= 0):
            bad.append("interval cells not strictly increasing")
        # inside an interval, points ascend in frustum order
        same = owner[1:] == owner[:-1]
        if np.any(rd[1:][same] <= rd[:-1][same]):
            bad.append("tie order")
    kept = np.nonzero(wl.cell_ids >= 0)[0]
    if not np.array_equal(np.sort(rd), kept):
        bad.append("ranks_depth is not the kept set")
    elif np.any(wl.cell_ids[rd] != rb):
        bad.append("ranks_bev disagrees with cell_ids")
    if n and np.any(rf != _feat_row(rd, *wl.dims())):
        bad.append("ranks_feat inconsistent with ranks_depth")
    return bad


def test_tiny_matches_per_cell_enumeration():
    wl = workloads.tiny()
    m = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    NC, D, H, W = wl.dims()
    rb, rd, rf, st, ln = [], [], [], [], []
    for cell in range(wl.n_cells):            # cells ascending
        members = [p for p in range(wl.n_frustum) if wl.cell_ids[p] == cell]   # p ascending
        if not members:
            continue
        st.append(len(rb))
        ln.append(len(members))
        for p in members:
            nc = p // (D * H * W)
            h = (p // W) % H
            w = p % W
            rb.append(cell)
            rd.append(p)
            rf.append((nc * H + h) * W + w)
    assert m["n_points"] == len(rb) and m["n_intervals"] == len(st)
    for key, want in [("ranks_bev", rb), ("ranks_depth", rd), ("ranks_feat", rf),
                      ("interval_starts", st), ("interval_lengths", ln)]:
        assert np.array_equal(m[key], np.array(want, dtype=np.int32)), key


@pytest.mark.parametrize("name", ["tiny", "canonical", "bevdet"])
def test_matches_library_sort(name, wl_cache):
    wl = wl_cache(name)
    m = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    lib = _library_map(wl)
    for key, want in lib.items():
        assert np.array_equal(m[key], want), key
    assert check_map_invariants(m, wl) == []


@pytest.mark.slow
def test_dram_batch_invariants(wl_cache):
    wl = wl_cache("dram_batch")
    m = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    assert check_map_invariants(m, wl) == []
    assert m["n_points"] == wl.n_kept


def test_all_dropped_gives_empty_map():
    cells = np.full(2 * 3 * 4 * 5, -1, np.int32)
    m = oracle.build_map(cells, 2, 3, 4, 5, 7)
    assert m["n_points"] == 0 and m["n_intervals"] == 0


def test_single_cell_single_interval():
    NC, D, H, W = 2, 5, 3, 4
    cells = np.full(NC * D * H * W, 3, np.int32)
    m = oracle.build_map(cells, NC, D, H, W, 4)
    assert m["n_intervals"] == 1
    assert m["interval_lengths"][0] == NC * D * H * W
    assert np.array_equal(m["ranks_depth"], np.arange(NC * D * H * W, dtype=np.int32))


@pytest.mark.parametrize("bad", [-2, 7, 1 << 30])
def test_out_of_range_ids_are_rejected(bad):
    cells = np.zeros(1 * 2 * 2 * 2, np.int32)
    cells[5] = bad
    with pytest.raises(oracle.OracleError):
        oracle.build_map(cells, 1, 2, 2, 2, 7)


def test_invariant_checker_catches_planted_mistakes():
    """Mistakes planted in an oracle map (on the CPU) must fail a pin."""
    wl = workloads.tiny()
    good = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    assert check_map_invariants(good, wl) == []
    lib = _library_map(wl)

    def mutated(**changes):
        m = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in good.items()}
        for k, fn in changes.items():
            fn(m[k])
        return m

    i = int(np.argmax(good["interval_lengths"]))       # an interval with >= 2 points
    s = good["interval_starts"][i]

    def swap_tie(a):
        a[s], a[s + 1] = a[s + 1], a[s]

    def bump(a):
        a[0] += 1

    def lengthen(a):
        a[i] += 1

    def shorten(a):
        a[i] -= 1

    def wrong_row(a):
        a[3] ^= 1

    plants = [
        mutated(ranks_depth=swap_tie),             # tie order
        mutated(ranks_depth=bump),                 # wrong point index
        mutated(interval_lengths=lengthen),        # off-by-one length
        mutated(interval_starts=shorten),          # wrong start
        mutated(ranks_feat=wrong_row),             # wrong feature row
    ]
    for m in plants:
        caught = check_map_invariants(m, wl) != [] or any(
            not np.array_equal(m[k], v) for k, v in lib.items())
        assert caught
        assert check_map_invariants(m, wl) != []
