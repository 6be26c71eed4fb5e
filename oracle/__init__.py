"""FP64 CPU oracle for BEV pooling -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` may import this package.  The product path
(``depth_weighted_scatter_gb300``) never imports it and has no CPU fallback.

The arithmetic lives in ``bevpool_oracle.c`` (plain single-threaded C,
double precision), compiled here with gcc on first use.  This module only
marshals numpy arrays into it.  See the C file's header for what each
function follows in "Accelerating BEV Pooling on NVIDIA GPUs for Physical AI
Applications" (sections "Eliminate redundant scatter traffic" and
"Implement interval-owned scatter-reduce").

Every function here is pinned by ``tests/test_oracle_*.py`` against things
that are not the oracle: library decoders, a library sort, a dense one-hot
matrix product, a library sparse matrix product, closed forms and
invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bevpool_oracle.c")
_LIB = os.path.join(_HERE, "libbevpool_oracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_RANGE, ERR_NOMEM = 0, 1, 2, 3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libbevpool_oracle.so`` (gcc -O2)."""
    need = force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if need:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i32, i64, vp, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = dbl
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = dbl
            lib.oracle_half_array_to_double.argtypes = [vp, i64, vp]
            lib.oracle_half_array_to_double.restype = None
            lib.oracle_e4m3_array_to_double.argtypes = [vp, i64, vp]
            lib.oracle_double_array_to_e4m3.argtypes = [vp, i64, vp]
            lib.oracle_e2m1_array_to_double.argtypes = [vp, i64, vp]
            lib.oracle_forward_nvfp4.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, dbl, dbl, vp]
            lib.oracle_e4m3_array_to_double.restype = None
            lib.oracle_build_map.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
            lib.oracle_build_map.restype = ctypes.c_int
            lib.oracle_forward.argtypes = [i32, vp, i32, i32, i32, i32, i32, i32, vp, vp, dbl, dbl, vp]
            lib.oracle_forward.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def half_to_double(codes: np.ndarray) -> np.ndarray:
    """Decode binary16 bit patterns (uint16 / float16 array) to float64."""
    src = np.ascontiguousarray(codes).view(np.uint16)
    out = np.empty(src.shape, dtype=np.float64)
    _load().oracle_half_array_to_double(_ptr(src), src.size, _ptr(out))
    return out


def e4m3_to_double(codes: np.ndarray) -> np.ndarray:
    """Decode OCP E4M3 bytes (uint8 array) to float64."""
    src = np.ascontiguousarray(codes).view(np.uint8)
    out = np.empty(src.shape, dtype=np.float64)
    _load().oracle_e4m3_array_to_double(_ptr(src), src.size, _ptr(out))
    return out


def e2m1_to_double(nibbles: np.ndarray) -> np.ndarray:
    """Values of OCP E2M1 codes (the low four bits of each entry)."""
    c = np.ascontiguousarray(nibbles, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e2m1_array_to_double(_ptr(c), c.size, _ptr(out))
    return out


def forward_nvfp4(cell_ids: np.ndarray, NC: int, D: int, H: int, W: int, n_cells: int, C: int,
                  depth: np.ndarray, feat_packed: np.ndarray, feat_block_scales: np.ndarray,
                  depth_scale: float, feat_scale: float) -> np.ndarray:
    """FP64 forward with NVFP4 features: E2M1 nibbles (element 2i in the low
    nibble of byte i of a row of C/2 bytes), one E4M3 scale per 16 elements,
    a per-tensor feat_scale; E4M3 depth times depth_scale."""
    cell_ids = np.ascontiguousarray(cell_ids, dtype=np.int32).reshape(-1)
    nf = NC * D * H * W
    if cell_ids.size != nf or C % 16 != 0:
        raise OracleError("bad shapes for the NVFP4 forward")
    depth = np.ascontiguousarray(depth).view(np.uint8).reshape(-1)
    fp = np.ascontiguousarray(feat_packed).view(np.uint8).reshape(-1)
    fb = np.ascontiguousarray(feat_block_scales).view(np.uint8).reshape(-1)
    if depth.size != nf or fp.size != NC * H * W * C // 2 or fb.size != NC * H * W * C // 16:
        raise OracleError("bad array sizes for the NVFP4 forward")
    out = np.empty((n_cells, C), dtype=np.float64)
    rc = _load().oracle_forward_nvfp4(_ptr(cell_ids), NC, D, H, W, n_cells, C, _ptr(depth), _ptr(fp), _ptr(fb),
                                      float(depth_scale), float(feat_scale), _ptr(out))
    if rc != OK:
        raise OracleError(f"oracle_forward_nvfp4 failed with code {rc}")
    return out


def e4m3_from_double(values: np.ndarray) -> np.ndarray:
    """Nearest OCP E4M3 codes (round half to even, saturating at +-448, sign kept)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_double_array_to_e4m3(_ptr(v), v.size, _ptr(out))
    return out


def build_map(cell_ids: np.ndarray, NC: int, D: int, H: int, W: int, n_cells: int) -> dict:
    """Scatter map of the kept frustum points, as int32 numpy arrays.

    Returns dict(ranks_depth, ranks_feat, ranks_bev, interval_starts,
    interval_lengths, n_points, n_intervals).
    """
    cell_ids = np.ascontiguousarray(cell_ids, dtype=np.int32).reshape(-1)
    nf = NC * D * H * W
    if cell_ids.size != nf:
        raise OracleError(f"cell_ids has {cell_ids.size} entries, expected {nf}")
    arrs = [np.empty(max(nf, 1), dtype=np.int32) for _ in range(5)]
    counts = np.zeros(2, dtype=np.int32)
    rc = _load().oracle_build_map(_ptr(cell_ids), NC, D, H, W, n_cells,
                                  *[_ptr(a) for a in arrs], _ptr(counts))
    if rc != OK:
        raise OracleError(f"oracle_build_map failed with code {rc}")
    n, ni = int(counts[0]), int(counts[1])
    return dict(ranks_depth=arrs[0][:n].copy(), ranks_feat=arrs[1][:n].copy(),
                ranks_bev=arrs[2][:n].copy(), interval_starts=arrs[3][:ni].copy(),
                interval_lengths=arrs[4][:ni].copy(), n_points=n, n_intervals=ni)


def forward(dtype: str, cell_ids: np.ndarray, NC: int, D: int, H: int, W: int, n_cells: int,
            C: int, depth: np.ndarray, feat: np.ndarray, depth_scale: float = 1.0,
            feat_scale: float = 1.0) -> np.ndarray:
    """FP64 BEV pooling straight from the per-frustum-point cell ids.

    ``dtype`` is "f16" (depth/feat hold binary16 codes) or "e4m3" (uint8 OCP
    E4M3 codes scaled by ``depth_scale`` / ``feat_scale``).  Returns a float64
    array of shape [n_cells, C].
    """
    code = {"f16": 0, "e4m3": 1}[dtype]
    cell_ids = np.ascontiguousarray(cell_ids, dtype=np.int32).reshape(-1)
    nf = NC * D * H * W
    if cell_ids.size != nf:
        raise OracleError(f"cell_ids has {cell_ids.size} entries, expected {nf}")
    want = np.uint16 if code == 0 else np.uint8
    depth = np.ascontiguousarray(depth).view(want).reshape(-1)
    feat = np.ascontiguousarray(feat).view(want).reshape(-1)
    if depth.size != nf:
        raise OracleError("depth must have NC*D*H*W entries")
    if feat.size != NC * H * W * C:
        raise OracleError("feat must have NC*H*W*C entries")
    out = np.empty((n_cells, C), dtype=np.float64)
    rc = _load().oracle_forward(code, _ptr(cell_ids), NC, D, H, W, n_cells, C, _ptr(depth),
                                _ptr(feat), float(depth_scale), float(feat_scale), _ptr(out))
    if rc != OK:
        raise OracleError(f"oracle_forward failed with code {rc}")
    return out


def forward_e4m3_out(dtype: str, cell_ids: np.ndarray, NC: int, D: int, H: int, W: int, n_cells: int,
                     C: int, depth: np.ndarray, feat: np.ndarray, depth_scale: float, feat_scale: float,
                     out_scale: float):
    """The forward with an E4M3 output: every output value divided by the
    per-tensor ``out_scale`` and rounded to the nearest E4M3 code.  Returns
    (codes uint8 [n_cells, C], the exact scaled values float64 [n_cells, C])."""
    if not (out_scale > 0.0 and np.isfinite(out_scale)):
        raise OracleError("out_scale must be positive and finite")
    v = forward(dtype, cell_ids, NC, D, H, W, n_cells, C, depth, feat, depth_scale, feat_scale) / out_scale
    return e4m3_from_double(v), v
