"""Thin ctypes binding of libbevpool (the C ABI in include/bevpool.h).

The functions named like the C entry points (``bevpool_build_map``,
``bevpool_forward``, ...) only marshal arguments: plain ints for device
pointers and streams, numpy arrays for host outputs.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU fallback.
Importing this module raises if ``libbevpool.so`` has not been built.

The tensor-level helpers (``build_map``, ``forward``, ``ScatterMap``) use
PyTorch only to allocate device memory and to name the current stream.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbevpool.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libbevpool.so not found at {LIB_PATH}; build it first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

# status / dtype codes, as in include/bevpool.h
BEVPOOL_OK = 0
BEVPOOL_ERR_INVALID_ARG = 1
BEVPOOL_ERR_OUT_OF_RANGE = 2
BEVPOOL_ERR_UNSUPPORTED = 3
BEVPOOL_ERR_WORKSPACE = 4
BEVPOOL_ERR_CUDA = 5
BEVPOOL_F16 = 0
BEVPOOL_E4M3 = 1
BEVPOOL_NVFP4 = 2
BEVPOOL_NOALLOC_MAX_FRUSTUM = 1 << 21

_i32, _i64, _sz, _vp, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float

_lib.bevpool_status_string.argtypes = [ctypes.c_int]
_lib.bevpool_status_string.restype = ctypes.c_char_p
_lib.bevpool_version.argtypes = []
_lib.bevpool_version.restype = _i32
_lib.bevpool_kernel_launches.argtypes = []
_lib.bevpool_kernel_launches.restype = _i64
_lib.bevpool_forward_supported.argtypes = [ctypes.c_int, _i32]
_lib.bevpool_forward_supported.restype = _i32
_lib.bevpool_forward_plan.argtypes = [ctypes.c_int, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                      _i64, _vp]
_lib.bevpool_forward_plan.restype = ctypes.c_int
_lib.bevpool_build_map_workspace_size.argtypes = [_i64, _i32]
_lib.bevpool_build_map_workspace_size.restype = _sz
_lib.bevpool_build_map.argtypes = [_vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.bevpool_build_map.restype = ctypes.c_int
_lib.bevpool_build_map_noalloc.argtypes = [_vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.bevpool_build_map_noalloc.restype = ctypes.c_int
_lib.bevpool_forward.argtypes = [ctypes.c_int, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _f32,
                                 _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp]
_lib.bevpool_forward.restype = ctypes.c_int
_lib.bevpool_forward_e4m3_out.argtypes = [ctypes.c_int, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _f32, _f32,
                                          _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp]
_lib.bevpool_forward_e4m3_out.restype = ctypes.c_int
_lib.bevpool_forward_nvfp4.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _f32, ctypes.c_int, _f32,
                                       _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp]
_lib.bevpool_forward_nvfp4.restype = ctypes.c_int
_lib.bevpool_pool_frame.argtypes = [_vp, _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _vp, _vp, _i32, _f32, _f32,
                                    _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp]
_lib.bevpool_pool_frame.restype = ctypes.c_int
_lib.bevpool_validate_map.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp]
_lib.bevpool_validate_map.restype = ctypes.c_int
_lib.bevpool_probe_l2.argtypes = [_i32, _vp, _sz, _i32, _vp, _vp]
_lib.bevpool_probe_l2.restype = ctypes.c_int
_lib.bevpool_probe_gather.argtypes = [_vp, _i32, _i32, _vp, _i32, _i32, _vp, _vp]
_lib.bevpool_probe_gather.restype = ctypes.c_int


class BevpoolError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {bevpool_status_string(status)} (status {status})")


def _host_ptr(a: Optional[np.ndarray]) -> Optional[int]:
    return None if a is None else a.ctypes.data


# ---------------------------------------------------------------- raw C entry points

def bevpool_status_string(status: int) -> str:
    return _lib.bevpool_status_string(status).decode()


def bevpool_version() -> int:
    return _lib.bevpool_version()


def bevpool_kernel_launches() -> int:
    return _lib.bevpool_kernel_launches()


def bevpool_forward_supported(dtype: int, C: int) -> bool:
    return bool(_lib.bevpool_forward_supported(dtype, C))


PLAN_FIELDS = ("variant", "ctas_per_sm", "owners", "batch", "round", "n_compute", "fill_cells", "n_fill",
               "streaming")


def bevpool_forward_plan(dtype: int, C: int, e4m3_out: int, NC: int, D: int, H: int, W: int, n_points: int,
                         n_intervals: int, counts_on_device: int, n_cells: int, sm_count: int, l2_bytes: int,
                         plan: np.ndarray) -> int:
    return _lib.bevpool_forward_plan(dtype, C, e4m3_out, NC, D, H, W, n_points, n_intervals, counts_on_device,
                                     n_cells, sm_count, l2_bytes, _host_ptr(plan))


def forward_plan(dtype: int, C: int, NC: int, D: int, H: int, W: int, n_points: int, n_intervals: int,
                 n_cells: int, *, e4m3_out: bool = False, counts_on_device: bool = False, sm_count: int = 0,
                 l2_bytes: int = 0) -> dict:
    """The launch plan of a forward call with these sizes, as a dict of
    PLAN_FIELDS (sm_count and l2_bytes > 0: for that GPU, without one)."""
    plan = np.zeros(len(PLAN_FIELDS), dtype=np.int32)
    st = bevpool_forward_plan(dtype, C, int(e4m3_out), NC, D, H, W, n_points, n_intervals, int(counts_on_device),
                              n_cells, sm_count, l2_bytes, plan)
    if st != BEVPOOL_OK:
        raise BevpoolError(st, "bevpool_forward_plan")
    return dict(zip(PLAN_FIELDS, (int(x) for x in plan)))


def bevpool_build_map_workspace_size(n_frustum: int, n_cells: int) -> int:
    return _lib.bevpool_build_map_workspace_size(n_frustum, n_cells)


def bevpool_build_map(cell_ids: int, NC: int, D: int, H: int, W: int, n_cells: int, ranks_depth: int,
                      ranks_feat: int, ranks_bev: int, interval_starts: int, interval_lengths: int,
                      d_counts: int, h_counts: Optional[np.ndarray], workspace: int, workspace_bytes: int,
                      stream: int) -> int:
    return _lib.bevpool_build_map(cell_ids, NC, D, H, W, n_cells, ranks_depth, ranks_feat, ranks_bev,
                                  interval_starts, interval_lengths, d_counts, _host_ptr(h_counts), workspace,
                                  workspace_bytes, stream)


def bevpool_build_map_noalloc(cell_ids: int, NC: int, D: int, H: int, W: int, n_cells: int, ranks_depth: int,
                              ranks_feat: int, ranks_bev: int, interval_starts: int, interval_lengths: int,
                              d_counts: int, h_counts: Optional[np.ndarray], stream: int) -> int:
    """bevpool_build_map with the library's built-in scratch (no workspace, no allocation)."""
    return _lib.bevpool_build_map_noalloc(cell_ids, NC, D, H, W, n_cells, ranks_depth, ranks_feat, ranks_bev,
                                          interval_starts, interval_lengths, d_counts, _host_ptr(h_counts), stream)


def bevpool_forward(dtype: int, depth: int, feat: int, NC: int, D: int, H: int, W: int, C: int,
                    depth_scale: float, feat_scale: float, ranks_depth: int, ranks_feat: int, ranks_bev: int,
                    interval_starts: int, interval_lengths: int, n_points: int, n_intervals: int,
                    d_counts: Optional[int], n_cells: int, out: int, stream: int) -> int:
    return _lib.bevpool_forward(dtype, depth, feat, NC, D, H, W, C, depth_scale, feat_scale, ranks_depth,
                                ranks_feat, ranks_bev, interval_starts, interval_lengths, n_points, n_intervals,
                                d_counts, n_cells, out, stream)


def bevpool_forward_e4m3_out(dtype: int, depth: int, feat: int, NC: int, D: int, H: int, W: int, C: int,
                             depth_scale: float, feat_scale: float, out_scale: float, ranks_depth: int,
                             ranks_feat: int, ranks_bev: int, interval_starts: int, interval_lengths: int,
                             n_points: int, n_intervals: int, d_counts: Optional[int], n_cells: int, out: int,
                             stream: int) -> int:
    return _lib.bevpool_forward_e4m3_out(dtype, depth, feat, NC, D, H, W, C, depth_scale, feat_scale, out_scale,
                                         ranks_depth, ranks_feat, ranks_bev, interval_starts, interval_lengths,
                                         n_points, n_intervals, d_counts, n_cells, out, stream)


def bevpool_forward_nvfp4(depth: int, feat: int, feat_block: int, NC: int, D: int, H: int, W: int, C: int,
                          depth_scale: float, feat_scale: float, out_dtype: int, out_scale: float,
                          ranks_depth: int, ranks_feat: int, ranks_bev: int, interval_starts: int,
                          interval_lengths: int, n_points: int, n_intervals: int, d_counts: Optional[int],
                          n_cells: int, out: int, stream: int) -> int:
    return _lib.bevpool_forward_nvfp4(depth, feat, feat_block, NC, D, H, W, C, depth_scale, feat_scale, out_dtype,
                                      out_scale, ranks_depth, ranks_feat, ranks_bev, interval_starts,
                                      interval_lengths, n_points, n_intervals, d_counts, n_cells, out, stream)


def bevpool_pool_frame(cell_ids: int, NC: int, D: int, H: int, W: int, n_cells: int, dtype: int, depth: int,
                       feat: int, C: int, depth_scale: float, feat_scale: float, ranks_depth: int, ranks_feat: int,
                       ranks_bev: int, interval_starts: int, interval_lengths: int, d_counts: int, workspace: int,
                       workspace_bytes: int, out: int, stream: int) -> int:
    return _lib.bevpool_pool_frame(cell_ids, NC, D, H, W, n_cells, dtype, depth, feat, C, depth_scale, feat_scale,
                                   ranks_depth, ranks_feat, ranks_bev, interval_starts, interval_lengths, d_counts,
                                   workspace, workspace_bytes, out, stream)


def bevpool_validate_map(ranks_depth: int, ranks_feat: int, ranks_bev: int, interval_starts: int,
                         interval_lengths: int, n_points: int, n_intervals: int, NC: int, D: int, H: int,
                         W: int, n_cells: int, d_result: int, h_result: Optional[np.ndarray], stream: int) -> int:
    return _lib.bevpool_validate_map(ranks_depth, ranks_feat, ranks_bev, interval_starts, interval_lengths,
                                     n_points, n_intervals, NC, D, H, W, n_cells, d_result, _host_ptr(h_result),
                                     stream)


def bevpool_probe_l2(mode: int, buf: int, nbytes: int, passes: int, d_sink: int, stream: int) -> int:
    return _lib.bevpool_probe_l2(mode, buf, nbytes, passes, d_sink, stream)


# ---------------------------------------------------------------- tensor helpers (torch = memory + streams)

def _stream(stream) -> int:
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclasses.dataclass
class ScatterMap:
    """The five-array map (device int32 tensors at full capacity) and its counts."""
    ranks_depth: "object"
    ranks_feat: "object"
    ranks_bev: "object"
    interval_starts: "object"
    interval_lengths: "object"
    d_counts: "object"               # device int32[3]: n_points, n_intervals, n_invalid
    NC: int
    D: int
    H: int
    W: int
    n_cells: int
    n_points: Optional[int] = None   # host copies, when synchronised
    n_intervals: Optional[int] = None

    @classmethod
    def allocate(cls, NC: int, D: int, H: int, W: int, n_cells: int, device="cuda") -> "ScatterMap":
        import torch

        nf = NC * D * H * W
        ni = max(1, min(nf, n_cells))
        e = lambda n: torch.empty(max(n, 1), dtype=torch.int32, device=device)
        return cls(e(nf), e(nf), e(nf), e(ni), e(ni), torch.zeros(3, dtype=torch.int32, device=device),
                   NC, D, H, W, n_cells)

    def host(self) -> dict:
        """Copies of the used part of every array (synchronises)."""
        n, ni = self.n_points, self.n_intervals
        if n is None:
            n, ni = (int(v) for v in self.d_counts[:2].cpu())
        return dict(ranks_depth=self.ranks_depth[:n].cpu().numpy(), ranks_feat=self.ranks_feat[:n].cpu().numpy(),
                    ranks_bev=self.ranks_bev[:n].cpu().numpy(),
                    interval_starts=self.interval_starts[:ni].cpu().numpy(),
                    interval_lengths=self.interval_lengths[:ni].cpu().numpy(), n_points=n, n_intervals=ni)


def workspace_for(NC: int, D: int, H: int, W: int, n_cells: int, device="cuda"):
    import torch

    nbytes = bevpool_build_map_workspace_size(NC * D * H * W, n_cells)
    if nbytes == 0:
        raise BevpoolError(BEVPOOL_ERR_INVALID_ARG, "bevpool_build_map_workspace_size")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def build_map(cell_ids, NC: int, D: int, H: int, W: int, n_cells: int, *, out: Optional[ScatterMap] = None,
              workspace=None, sync: bool = True, stream=None) -> ScatterMap:
    """bevpool_build_map on device tensors.  With sync=True the counts are copied
    to the host (and an out-of-range cell id raises)."""
    m = out if out is not None else ScatterMap.allocate(NC, D, H, W, n_cells, cell_ids.device)
    ws = workspace if workspace is not None else workspace_for(NC, D, H, W, n_cells, cell_ids.device)
    h = np.zeros(3, dtype=np.int32) if sync else None
    st = bevpool_build_map(cell_ids.data_ptr(), NC, D, H, W, n_cells, m.ranks_depth.data_ptr(),
                           m.ranks_feat.data_ptr(), m.ranks_bev.data_ptr(), m.interval_starts.data_ptr(),
                           m.interval_lengths.data_ptr(), m.d_counts.data_ptr(), h, ws.data_ptr(), ws.numel(),
                           _stream(stream))
    if st != BEVPOOL_OK:
        raise BevpoolError(st, "bevpool_build_map")
    if sync:
        m.n_points, m.n_intervals = int(h[0]), int(h[1])
    else:
        m.n_points = m.n_intervals = None
    return m


def forward(m: ScatterMap, depth, feat, C: int, *, dtype: int = BEVPOOL_F16, depth_scale: float = 1.0,
            feat_scale: float = 1.0, out=None, stream=None, capacity: Optional[tuple] = None,
            out_scale: Optional[float] = None, feat_block=None):
    """bevpool_forward over a map.  Returns the [n_cells, C] output tensor:
    fp16, or, when ``out_scale`` is given, uint8 E4M3 codes of value / out_scale
    (bevpool_forward_e4m3_out).  dtype BEVPOOL_NVFP4 takes the packed E2M1
    features in ``feat`` and their E4M3 block scales in ``feat_block``
    (bevpool_forward_nvfp4).

    If the map's host counts are unknown (built with sync=False), the device
    counts are used with ``capacity`` = (max points, max intervals) as bounds."""
    import torch

    if out is None:
        out = torch.empty((m.n_cells, C), dtype=torch.float16 if out_scale is None else torch.uint8,
                          device=feat.device)
    if m.n_points is not None and capacity is None:
        n_pts, n_int, dc = m.n_points, m.n_intervals, None
    else:
        nf = m.NC * m.D * m.H * m.W
        n_pts, n_int = capacity if capacity is not None else (nf, min(nf, m.n_cells))
        dc = m.d_counts.data_ptr()
    maps = (m.ranks_depth.data_ptr(), m.ranks_feat.data_ptr(), m.ranks_bev.data_ptr(), m.interval_starts.data_ptr(),
            m.interval_lengths.data_ptr(), n_pts, n_int, dc, m.n_cells, out.data_ptr(), _stream(stream))
    if dtype == BEVPOOL_NVFP4:
        if feat_block is None:
            raise BevpoolError(BEVPOOL_ERR_INVALID_ARG, "NVFP4 features need feat_block")
        st = bevpool_forward_nvfp4(depth.data_ptr(), feat.data_ptr(), feat_block.data_ptr(), m.NC, m.D, m.H, m.W, C,
                                   depth_scale, feat_scale, BEVPOOL_F16 if out_scale is None else BEVPOOL_E4M3,
                                   0.0 if out_scale is None else out_scale, *maps)
        if st != BEVPOOL_OK:
            raise BevpoolError(st, "bevpool_forward_nvfp4")
    elif out_scale is None:
        st = bevpool_forward(dtype, depth.data_ptr(), feat.data_ptr(), m.NC, m.D, m.H, m.W, C, depth_scale,
                             feat_scale, *maps)
        if st != BEVPOOL_OK:
            raise BevpoolError(st, "bevpool_forward")
    else:
        st = bevpool_forward_e4m3_out(dtype, depth.data_ptr(), feat.data_ptr(), m.NC, m.D, m.H, m.W, C, depth_scale,
                                      feat_scale, out_scale, *maps)
        if st != BEVPOOL_OK:
            raise BevpoolError(st, "bevpool_forward_e4m3_out")
    return out


def validate_map(m: ScatterMap, stream=None) -> int:
    """Violation bit set of a synchronised map (0 = valid); see bevpool_validate_map."""
    import torch

    n, ni = m.n_points, m.n_intervals
    if n is None:
        n, ni = (int(v) for v in m.d_counts[:2].cpu())
    d = torch.zeros(1, dtype=torch.int32, device=m.ranks_bev.device)
    h = np.zeros(1, dtype=np.int32)
    st = bevpool_validate_map(m.ranks_depth.data_ptr(), m.ranks_feat.data_ptr(), m.ranks_bev.data_ptr(),
                              m.interval_starts.data_ptr(), m.interval_lengths.data_ptr(), n, ni, m.NC, m.D, m.H,
                              m.W, m.n_cells, d.data_ptr(), h, _stream(stream))
    if st not in (BEVPOOL_OK, BEVPOOL_ERR_OUT_OF_RANGE):
        raise BevpoolError(st, "bevpool_validate_map")
    return int(h[0])


def pool_frame(cell_ids, depth, feat, NC: int, D: int, H: int, W: int, n_cells: int, C: int, *,
               dtype: int = BEVPOOL_F16, depth_scale: float = 1.0, feat_scale: float = 1.0,
               out=None, map_out: Optional[ScatterMap] = None, workspace=None, stream=None):
    """bevpool_pool_frame: the map build and the forward of one frame, no host sync.
    Returns (out, map); the map's host counts stay unknown (read d_counts)."""
    import torch

    m = map_out if map_out is not None else ScatterMap.allocate(NC, D, H, W, n_cells, cell_ids.device)
    ws = workspace if workspace is not None else workspace_for(NC, D, H, W, n_cells, cell_ids.device)
    if out is None:
        out = torch.empty((n_cells, C), dtype=torch.float16, device=feat.device)
    st = bevpool_pool_frame(cell_ids.data_ptr(), NC, D, H, W, n_cells, dtype, depth.data_ptr(), feat.data_ptr(), C,
                            depth_scale, feat_scale, m.ranks_depth.data_ptr(), m.ranks_feat.data_ptr(),
                            m.ranks_bev.data_ptr(), m.interval_starts.data_ptr(), m.interval_lengths.data_ptr(),
                            m.d_counts.data_ptr(), ws.data_ptr(), ws.numel(), out.data_ptr(), _stream(stream))
    if st != BEVPOOL_OK:
        raise BevpoolError(st, "bevpool_pool_frame")
    m.n_points = m.n_intervals = None
    return out, m


PROBE_READ, PROBE_WRITE, PROBE_COPY = 0, 1, 2


def probe_l2(buf, passes: int, *, mode: int = PROBE_READ, sink=None, stream=None):
    """One launch of the L2 streaming probe over the bytes of ``buf`` (a
    contiguous device tensor); see bevpool_probe_l2.  The read probe adds the
    word sum of every pass to ``sink`` (a device tensor of one 32-bit element
    the caller zeroed; the sum wraps mod 2^32)."""
    nbytes = buf.numel() * buf.element_size()
    st = bevpool_probe_l2(mode, buf.data_ptr(), nbytes, passes, sink.data_ptr() if sink is not None else 0,
                          _stream(stream))
    if st != BEVPOOL_OK:
        raise BevpoolError(st, "bevpool_probe_l2")


def bevpool_probe_gather(feat: int, n_rows: int, row_bytes: int, rows: int, n_points: int, ctas_per_sm: int,
                         d_sink: int, stream: int) -> int:
    return _lib.bevpool_probe_gather(feat, n_rows, row_bytes, rows, n_points, ctas_per_sm, d_sink, stream)


def probe_gather(feat, row_bytes: int, rows, *, ctas_per_sm: int = 3, sink=None, stream=None):
    """One launch of the gather probe over the rows of `feat` (a device
    tensor of n_rows * row_bytes bytes) listed in `rows` (device int32);
    adds the sum of the gathered words to `sink` (device int32, zeroed by the
    caller), or with no sink runs the timing mode."""
    n_rows = feat.numel() * feat.element_size() // row_bytes
    st = bevpool_probe_gather(feat.data_ptr(), n_rows, row_bytes, rows.data_ptr(), rows.numel(), ctas_per_sm,
                              sink.data_ptr() if sink is not None else 0, _stream(stream))
    if st != BEVPOOL_OK:
        raise BevpoolError(st, "bevpool_probe_gather")
    return sink
