"""The C-ABI library loads, exports every entry point include/bevpool.h
declares, and rejects bad arguments on the host (no GPU needed: these calls
return before any CUDA work)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bevpool.h")


@pytest.fixture(scope="module")
def bp():
    from depth_weighted_scatter_gb300 import _build

    _build.build()
    from depth_weighted_scatter_gb300 import bevpool

    return bevpool


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bevpool_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["bevpool_build_map", "bevpool_forward", "bevpool_build_map_workspace_size",
                 "bevpool_validate_map", "bevpool_status_string"]:
        assert want in names


def test_library_exports_every_declared_symbol(bp):
    lib = ctypes.CDLL(bp.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_library_exports_nothing_else(bp):
    """Internal symbols stay hidden (only the C ABI is visible)."""
    import subprocess

    r = subprocess.run(["nm", "-D", "--defined-only", bp.LIB_PATH], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("nm not available")
    exported = {line.split()[-1] for line in r.stdout.splitlines() if " T " in line}
    assert {n for n in exported if n.startswith("bevpool")} == set(declared_functions())


def test_status_strings(bp):
    assert bp.bevpool_status_string(bp.BEVPOOL_OK) == "ok"
    for s in range(1, 6):
        assert bp.bevpool_status_string(s) not in ("ok", "unknown status")
    assert bp.bevpool_status_string(99) == "unknown status"
    assert bp.bevpool_version() >= 100


def test_supported_channel_counts(bp):
    for dt in (bp.BEVPOOL_F16, bp.BEVPOOL_E4M3):
        for C in (8, 16, 32, 64, 80, 96, 128, 160, 192, 256):
            assert bp.bevpool_forward_supported(dt, C)
        for C in (0, 4, 12, 24, 72, 264, 512):
            assert not bp.bevpool_forward_supported(dt, C)
    assert not bp.bevpool_forward_supported(7, 80)


def test_workspace_size(bp):
    assert bp.bevpool_build_map_workspace_size(0, 10) == 0
    assert bp.bevpool_build_map_workspace_size(10, 0) == 0
    assert bp.bevpool_build_map_workspace_size(1 << 31, 10) == 0
    small = bp.bevpool_build_map_workspace_size(4096, 100)
    big = bp.bevpool_build_map_workspace_size(1_993_728, 129_600)
    assert 0 < small < big
    # counting-sort path: grouped frustum indices + two per-cell tables
    assert big >= 4 * 1_993_728 + 2 * 4 * 129_600
    # grids above 2^24 cells take the radix path: two key/value buffers of int32
    assert bp.bevpool_build_map_workspace_size(1_993_728, (1 << 24) + 1) >= 4 * 4 * 1_993_728


FAKE = 1 << 20   # never dereferenced: every call below fails validation first


def test_build_map_rejects_bad_arguments(bp):
    h = np.zeros(3, np.int32)
    ws = bp.bevpool_build_map_workspace_size(2 * 3 * 4 * 5, 10)
    args = dict(cell_ids=FAKE, NC=2, D=3, H=4, W=5, n_cells=10, ranks_depth=FAKE, ranks_feat=FAKE,
                ranks_bev=FAKE, interval_starts=FAKE, interval_lengths=FAKE, d_counts=FAKE, h_counts=h,
                workspace=FAKE, workspace_bytes=ws, stream=0)
    bad = [dict(NC=0), dict(D=-1), dict(n_cells=0), dict(cell_ids=0), dict(d_counts=0),
           dict(ranks_feat=FAKE + 2), dict(NC=1 << 16, D=1 << 16),
           # products that overflow 64 bits when formed in one expression (2^64 wraps to 0)
           dict(NC=1 << 16, D=1 << 16, H=1 << 16, W=1 << 16), dict(NC=2 ** 31 - 1, D=2 ** 31 - 1, H=2, W=2)]
    for change in bad:
        assert bp.bevpool_build_map(**{**args, **change}) == bp.BEVPOOL_ERR_INVALID_ARG, change
    assert bp.bevpool_build_map(**{**args, "workspace": 0}) == bp.BEVPOOL_ERR_WORKSPACE
    assert bp.bevpool_build_map(**{**args, "workspace_bytes": ws - 1}) == bp.BEVPOOL_ERR_WORKSPACE
    assert bp.bevpool_build_map(**{**args, "workspace": FAKE + 64}) == bp.BEVPOOL_ERR_WORKSPACE


def test_build_map_noalloc_rejects_bad_arguments(bp):
    args = dict(cell_ids=FAKE, NC=2, D=3, H=4, W=5, n_cells=10, ranks_depth=FAKE, ranks_feat=FAKE,
                ranks_bev=FAKE, interval_starts=FAKE, interval_lengths=FAKE, d_counts=FAKE, h_counts=None, stream=0)
    for change in [dict(NC=0), dict(n_cells=0), dict(NC=1 << 16, D=1 << 16, H=1 << 16, W=1 << 16)]:
        assert bp.bevpool_build_map_noalloc(**{**args, **change}) == bp.BEVPOOL_ERR_INVALID_ARG, change
    assert bp.bevpool_build_map_noalloc(**{**args, "D": 1 << 20}) == bp.BEVPOOL_ERR_WORKSPACE


def test_forward_rejects_bad_arguments(bp):
    args = dict(dtype=bp.BEVPOOL_F16, depth=FAKE, feat=FAKE, NC=2, D=3, H=4, W=5, C=80, depth_scale=1.0,
                feat_scale=1.0, ranks_depth=FAKE, ranks_feat=FAKE, ranks_bev=FAKE, interval_starts=FAKE,
                interval_lengths=FAKE, n_points=50, n_intervals=20, d_counts=None, n_cells=30, out=FAKE, stream=0)
    assert bp.bevpool_forward(**{**args, "C": 72}) == bp.BEVPOOL_ERR_UNSUPPORTED
    assert bp.bevpool_forward(**{**args, "dtype": 3}) == bp.BEVPOOL_ERR_UNSUPPORTED
    bad = [dict(NC=0), dict(n_cells=0), dict(n_points=121), dict(n_points=-1), dict(n_intervals=51),
           dict(depth=0), dict(feat=FAKE + 8), dict(out=FAKE + 4), dict(depth=FAKE + 1),
           dict(ranks_bev=0), dict(interval_starts=0), dict(n_cells=1 << 28),
           dict(depth_scale=float("inf")), dict(d_counts=FAKE + 2)]
    for change in bad:
        assert bp.bevpool_forward(**{**args, **change}) == bp.BEVPOOL_ERR_INVALID_ARG, change


def test_validate_map_rejects_bad_arguments(bp):
    args = dict(ranks_depth=FAKE, ranks_feat=FAKE, ranks_bev=FAKE, interval_starts=FAKE, interval_lengths=FAKE,
                n_points=10, n_intervals=3, NC=1, D=2, H=3, W=4, n_cells=9, d_result=FAKE, h_result=None, stream=0)
    for change in [dict(d_result=0), dict(NC=0), dict(n_points=-1), dict(ranks_bev=0), dict(interval_lengths=0)]:
        assert bp.bevpool_validate_map(**{**args, **change}) == bp.BEVPOOL_ERR_INVALID_ARG, change


def test_forward_e4m3_out_rejects_bad_arguments(bp):
    args = dict(dtype=bp.BEVPOOL_F16, depth=FAKE, feat=FAKE, NC=2, D=3, H=4, W=5, C=80, depth_scale=1.0,
                feat_scale=1.0, out_scale=0.5, ranks_depth=FAKE, ranks_feat=FAKE, ranks_bev=FAKE,
                interval_starts=FAKE, interval_lengths=FAKE, n_points=50, n_intervals=20, d_counts=None,
                n_cells=30, out=FAKE, stream=0)
    for change in [dict(C=72), dict(C=8), dict(dtype=3)]:
        assert bp.bevpool_forward_e4m3_out(**{**args, **change}) == bp.BEVPOOL_ERR_UNSUPPORTED, change
    bad = [dict(out_scale=0.0), dict(out_scale=-1.0), dict(out_scale=float("inf")), dict(out_scale=float("nan")),
           dict(out_scale=1e-38, depth_scale=1e30), dict(out=FAKE + 4), dict(NC=0), dict(n_points=121)]
    for change in bad:
        assert bp.bevpool_forward_e4m3_out(**{**args, **change}) == bp.BEVPOOL_ERR_INVALID_ARG, change


def test_pool_frame_rejects_bad_arguments(bp):
    nf = 2 * 3 * 4 * 5
    ws = bp.bevpool_build_map_workspace_size(nf, 30)
    args = dict(cell_ids=FAKE, NC=2, D=3, H=4, W=5, n_cells=30, dtype=bp.BEVPOOL_F16, depth=FAKE, feat=FAKE, C=80,
                depth_scale=1.0, feat_scale=1.0, ranks_depth=FAKE, ranks_feat=FAKE, ranks_bev=FAKE,
                interval_starts=FAKE, interval_lengths=FAKE, d_counts=FAKE, workspace=FAKE, workspace_bytes=ws,
                out=FAKE, stream=0)
    assert bp.bevpool_pool_frame(**{**args, "C": 72}) == bp.BEVPOOL_ERR_UNSUPPORTED
    for change in [dict(NC=0), dict(n_cells=0), dict(feat=FAKE + 8), dict(out=0), dict(cell_ids=0),
                   dict(depth_scale=float("inf"))]:
        assert bp.bevpool_pool_frame(**{**args, **change}) == bp.BEVPOOL_ERR_INVALID_ARG, change
    assert bp.bevpool_pool_frame(**{**args, "workspace_bytes": ws - 1}) == bp.BEVPOOL_ERR_WORKSPACE


def test_forward_nvfp4_rejects_bad_arguments(bp):
    assert bp.bevpool_forward_supported(bp.BEVPOOL_NVFP4, 80)
    assert not bp.bevpool_forward_supported(bp.BEVPOOL_NVFP4, 32)
    args = dict(depth=FAKE, feat=FAKE, feat_block=FAKE, NC=2, D=3, H=4, W=5, C=80, depth_scale=1.0, feat_scale=1.0,
                out_dtype=bp.BEVPOOL_F16, out_scale=0.0, ranks_depth=FAKE, ranks_feat=FAKE, ranks_bev=FAKE,
                interval_starts=FAKE, interval_lengths=FAKE, n_points=50, n_intervals=20, d_counts=None, n_cells=30,
                out=FAKE, stream=0)
    for change in [dict(C=32), dict(C=8), dict(out_dtype=bp.BEVPOOL_NVFP4)]:
        assert bp.bevpool_forward_nvfp4(**{**args, **change}) == bp.BEVPOOL_ERR_UNSUPPORTED, change
    for change in [dict(feat_block=0), dict(feat=FAKE + 8), dict(out_dtype=bp.BEVPOOL_E4M3, out_scale=0.0),
                   dict(NC=0)]:
        assert bp.bevpool_forward_nvfp4(**{**args, **change}) == bp.BEVPOOL_ERR_INVALID_ARG, change


def test_probe_l2_rejects_bad_arguments(bp):
    """Argument checks come before any CUDA call."""
    fake = 1 << 20   # never dereferenced: every call below fails its checks first
    assert bp.bevpool_probe_l2(3, fake, 64, 1, fake, 0) == bp.BEVPOOL_ERR_INVALID_ARG     # no such mode
    assert bp.bevpool_probe_l2(-1, fake, 64, 1, fake, 0) == bp.BEVPOOL_ERR_INVALID_ARG
    assert bp.bevpool_probe_l2(2, fake, 48, 1, 0, 0) == bp.BEVPOOL_ERR_INVALID_ARG        # copy: halves of 16 B
    assert bp.bevpool_probe_l2(0, 0, 64, 1, fake, 0) == bp.BEVPOOL_ERR_INVALID_ARG        # NULL buffer
    assert bp.bevpool_probe_l2(0, fake, 0, 1, fake, 0) == bp.BEVPOOL_ERR_INVALID_ARG      # empty
    assert bp.bevpool_probe_l2(0, fake, 40, 1, fake, 0) == bp.BEVPOOL_ERR_INVALID_ARG     # not 16-byte multiple
    assert bp.bevpool_probe_l2(0, fake + 8, 64, 1, fake, 0) == bp.BEVPOOL_ERR_INVALID_ARG  # misaligned
    assert bp.bevpool_probe_l2(0, fake, 64, 0, fake, 0) == bp.BEVPOOL_ERR_INVALID_ARG     # no pass
    assert bp.bevpool_probe_l2(0, fake, 64, 1, 0, 0) == bp.BEVPOOL_ERR_INVALID_ARG        # read without sink
    assert bp.bevpool_probe_l2(1, fake, (1 << 32) + 16, 1, 0, 0) == bp.BEVPOOL_ERR_INVALID_ARG   # too large


def test_probe_gather_rejects_bad_arguments(bp):
    """Argument checks come before any CUDA call."""
    fake = 1 << 20   # never dereferenced: every call below fails its checks first
    good = dict(feat=fake, n_rows=100, row_bytes=160, rows=fake, n_points=1000, ctas_per_sm=3, d_sink=0, stream=0)
    for change in [dict(feat=0), dict(feat=fake + 8), dict(n_rows=0), dict(row_bytes=8), dict(row_bytes=520),
                   dict(row_bytes=40), dict(n_points=-1), dict(rows=0), dict(rows=fake + 2), dict(ctas_per_sm=0),
                   dict(ctas_per_sm=9)]:
        assert bp.bevpool_probe_gather(**{**good, **change}) == bp.BEVPOOL_ERR_INVALID_ARG, change
