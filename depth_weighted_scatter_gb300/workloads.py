"""Seeded synthetic BEV-pooling workloads.

This module only draws inputs: per-frustum-point BEV cell ids (-1 = dropped),
depth probabilities and image features.  It holds none of the pooling
arithmetic (no sort, no map, no scatter-reduce), so both the CUDA path and
the FP64 oracle consume what it produces without sharing any of the method.

The workloads stand in for the configurations of "Accelerating BEV Pooling
on NVIDIA GPUs for Physical AI Applications" (section "Classify the memory
regime": ~209K scatter points, C=80, derived from nuScenes samples; Table 1
lists further sizes).  nuScenes itself is not used: every workload is drawn
from a seeded numpy PCG64 generator.

Layouts (shared by both sides):
  depth  [NC, D, H, W]   (frustum point p = ((nc*D + d)*H + h)*W + w)
  feat   [NC, H, W, C]   (NHWC, one row of C channels per image pixel)
  out    [n_cells, C]
  cell_ids[p] in [0, n_cells) or -1 for a dropped frustum point.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

E4M3_MAX = 448.0


@dataclasses.dataclass
class Workload:
    name: str
    NC: int
    D: int
    H: int
    W: int
    C: int
    n_cells: int
    cell_ids: np.ndarray          # int32 [NC*D*H*W]
    depth: np.ndarray             # float16 [NC,D,H,W]  or uint8 E4M3 codes
    feat: np.ndarray              # float16 [NC,H,W,C], uint8 E4M3 codes, or uint8 [NC,H,W,C/2] E2M1 pairs
    dtype: str = "f16"            # "f16", "e4m3" or "nvfp4" (E2M1 features, E4M3 depth)
    depth_scale: float = 1.0      # E4M3 depth: depth value = code * depth_scale
    feat_scale: float = 1.0       # E4M3 / NVFP4 feat: per-tensor factor of every feature value
    grid: tuple = ()              # (B, Y, X) of the BEV grid, n_cells = B*Y*X
    recipe: str = ""
    feat_block: Optional[np.ndarray] = None   # NVFP4: uint8 [NC,H,W,C/16] E4M3 scale of each 16-element block

    @property
    def n_frustum(self) -> int:
        return self.NC * self.D * self.H * self.W

    @property
    def n_feat_rows(self) -> int:
        return self.NC * self.H * self.W

    @property
    def n_kept(self) -> int:
        return int(np.count_nonzero(self.cell_ids >= 0))

    def dims(self) -> tuple:
        return (self.NC, self.D, self.H, self.W)


def _softmax_depth(rng: np.random.Generator, NC: int, D: int, H: int, W: int, sigma: float) -> np.ndarray:
    logits = rng.normal(0.0, sigma, size=(NC, D, H, W))
    logits -= logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float16)


def _normal_feat(rng: np.random.Generator, NC: int, H: int, W: int, C: int) -> np.ndarray:
    return rng.standard_normal(size=(NC, H, W, C), dtype=np.float32).astype(np.float16)


def quantize_e4m3(x: np.ndarray, scale: float) -> np.ndarray:
    """E4M3 codes of x/scale, rounded to nearest even by torch's CPU cast."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)) / torch.tensor(scale, dtype=torch.float32)
    q = t.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy().copy()


E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])   # magnitudes of the codes 0..7


def quantize_e2m1(x: np.ndarray) -> np.ndarray:
    """E2M1 codes (0..15) of x: the nearest magnitude, ties to the even
    code, saturating at 6; bit 3 is the sign."""
    a = np.minimum(np.abs(x), 6.0)
    dist = np.abs(a[..., None] - E2M1_VALUES)
    best = dist.min(axis=-1, keepdims=True)
    tie_ok = (dist == best) & ((np.arange(8) & 1) == 0)
    plain = dist == best
    pick = np.where(tie_ok.any(axis=-1), np.argmax(tie_ok, axis=-1), np.argmax(plain, axis=-1))
    code = pick.astype(np.uint8)
    return np.where(np.signbit(x) & (code != 0), code | 8, code).astype(np.uint8)


def quantize_nvfp4(feat: np.ndarray):
    """Two-level NVFP4 quantisation of an [..., C] fp32 tensor (C % 16 == 0):
    feat_scale = max|feat| / (6 * 448) per tensor, one E4M3 block scale per 16
    elements (block max / 6 / feat_scale, rounded to nearest even), E2M1
    elements of value / (block scale * feat_scale).  Returns (packed nibbles
    [..., C/2] with element 2i in the low nibble of byte i, block scales
    [..., C/16], feat_scale)."""
    f = np.ascontiguousarray(feat, dtype=np.float32)
    C = f.shape[-1]
    fs = float(np.float32(max(float(np.abs(f).max()), 1e-30) / (6.0 * E4M3_MAX)))
    blocks = f.reshape(f.shape[:-1] + (C // 16, 16))
    bmax = np.abs(blocks).max(axis=-1)
    bcode = quantize_e4m3(bmax / 6.0, fs)
    import torch

    bval = torch.from_numpy(bcode).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    denom = np.where(bval > 0, bval * fs, 1.0)
    q = quantize_e2m1(np.where(bval[..., None] > 0, blocks / denom[..., None], 0.0)).reshape(f.shape)
    packed = (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    return packed, bcode, fs


def tiny(seed: int = 0) -> Workload:
    """1 camera, D=8, 4x8 feature map, C=8, 16x16 grid; uniform cells; 25% dropped.

    Inputs are drawn in fp32 and handed to both sides as fp16."""
    NC, D, H, W, C, Y, X = 1, 8, 4, 8, 8, 16, 16
    rng = np.random.default_rng(seed)
    feat = _normal_feat(rng, NC, H, W, C)
    depth = _softmax_depth(rng, NC, D, H, W, 1.0)
    nf = NC * D * H * W
    dropped = rng.random(nf) < 0.25
    cells = rng.integers(0, Y * X, size=nf, dtype=np.int64).astype(np.int32)
    cells[dropped] = -1
    return Workload("tiny", NC, D, H, W, C, Y * X, cells, depth, feat, grid=(1, Y, X),
                    recipe=f"seed {seed}: feat N(0,1); depth softmax over D of N(0,1) logits; "
                           "cells uniform over 256; Bernoulli(0.25) dropped")


def _ring_cells(rng: np.random.Generator, n: int, centre: float, r_in: float, r_span: float,
                exponent: float, X: int) -> np.ndarray:
    u = rng.random(n)
    theta = rng.random(n) * (2.0 * math.pi)
    r = r_in + r_span * u ** exponent
    y = np.floor(centre + r * np.sin(theta)).astype(np.int64)
    x = np.floor(centre + r * np.cos(theta)).astype(np.int64)
    return (y * X + x).astype(np.int32)


RING_EXPONENT = 1.6


def _ring(name: str, seed: int, keep_p: float, C: int) -> Workload:
    """The canonical frustum (6 cameras, D=118, 32x88 features) into the
    360x360 ring grid, keeping each frustum point with probability keep_p."""
    NC, D, H, W, Y, X = 6, 118, 32, 88, 360, 360
    rng = np.random.default_rng(seed)
    feat = _normal_feat(rng, NC, H, W, C)
    depth = _softmax_depth(rng, NC, D, H, W, 2.0)
    nf = NC * D * H * W
    keep = rng.random(nf) < keep_p
    cells = np.full(nf, -1, dtype=np.int32)
    cells[keep] = _ring_cells(rng, int(keep.sum()), 180.0, 40.0, 110.0, RING_EXPONENT, X)
    return Workload(name, NC, D, H, W, C, Y * X, cells, depth, feat, grid=(1, Y, X),
                    recipe=f"seed {seed}: feat N(0,1) fp16; depth softmax over D of N(0,sigma=2) logits; "
                           f"keep Bernoulli({keep_p}); ring r=40+110*u^{RING_EXPONENT}, theta~U(0,2pi)")


def canonical(seed: int = 1) -> Workload:
    """6 cameras, D=118, 32x88 features, C=80, 360x360 grid (1,993,728 frustum points).

    Each frustum point is kept with probability 0.105 (about 209K kept) and
    lands in a ring of radius 40..150 cells around the grid centre with
    r = 40 + 110*u**1.6, so cells near the inner edge collect more points and
    interval lengths are skewed (1 up to about 60)."""
    return _ring("canonical", seed, 0.105, 80)


def _to_fp8(wl: Workload, name: str) -> Workload:
    """The same workload with feat and depth as E4M3: feat_scale =
    max|feat| / 448 and depth_scale = max(depth), so the depth codes lie in
    [0, 1]; codes are round-to-nearest-even of value/scale."""
    f32 = wl.feat.astype(np.float32)
    d32 = wl.depth.astype(np.float32)
    fs = float(np.float32(np.abs(f32).max() / np.float32(E4M3_MAX)))
    ds = float(np.float32(d32.max()))
    return dataclasses.replace(
        wl, name=name, dtype="e4m3",
        feat=quantize_e4m3(f32, fs).reshape(wl.feat.shape),
        depth=quantize_e4m3(d32, ds).reshape(wl.depth.shape),
        feat_scale=fs, depth_scale=ds,
        recipe=wl.recipe + "; then E4M3 with feat_scale=max|feat|/448, depth_scale=max(depth)")


def _to_nvfp4(wl: Workload, name: str) -> Workload:
    """The same workload with NVFP4 features (quantize_nvfp4) and E4M3 depth
    (depth_scale = max(depth), as in the FP8 workloads)."""
    d32 = wl.depth.astype(np.float32)
    ds = float(np.float32(d32.max()))
    packed, blocks, fs = quantize_nvfp4(wl.feat.astype(np.float32))
    return dataclasses.replace(
        wl, name=name, dtype="nvfp4", feat=packed, feat_block=blocks, feat_scale=fs,
        depth=quantize_e4m3(d32, ds).reshape(wl.depth.shape), depth_scale=ds,
        recipe=wl.recipe + "; then NVFP4 features (E2M1, E4M3 scale per 16, feat_scale=max|feat|/2688) "
                           "and E4M3 depth (depth_scale=max(depth))")


def canonical_fp8(seed: int = 1) -> Workload:
    """The canonical workload (same cell ids) with feat and depth as E4M3."""
    return _to_fp8(canonical(seed), "canonical_fp8")


# The shapes of the pages' Table 1 ("Map the algorithm to hardware"): only C
# is printed, so the point counts are synthetic.  The V2 column's latencies
# (137.8 / 274.0 / 749.9 / 1,675.0 us for small / canonical / large / very
# large) grow with the number of scattered points, so the keep probabilities
# scale the canonical 0.105 by 0.50, 2.74 and 6.11; the wide configs keep the
# canonical points with C = 128 and 256.
TABLE1 = {
    "table1_small": (21, 0.105 * 137.8 / 274.0, 80),
    "table1_large": (22, 0.105 * 749.9 / 274.0, 80),
    "table1_very_large": (23, 0.105 * 1675.0 / 274.0, 80),
    "wide_c128": (24, 0.105, 128),
    "wide_c256": (25, 0.105, 256),
}


def table1(name: str) -> Workload:
    seed, keep_p, C = TABLE1[name]
    return _ring(name, seed, round(keep_p, 4), C)


def bevdet(seed: int = 3) -> Workload:
    """Geometry-derived map: 6 pinhole cameras at the ego origin, yaw k*60 deg.

    fx = fy = 800, image 704x256 with the principal point at its centre,
    16x downsampled to a 16x44 feature map (pixel centre ((w+0.5)*16,
    (h+0.5)*16)), D = 59 depth bins at z = 1..59 m along the optical axis.
    Ego X is forward of camera 0, Y left, Z up.  Cells are 0.8 m over
    +-51.2 m (128x128), cell = iy*128 + ix; points off the grid or with
    Z outside [-5, 3] m are dropped.  C = 64, feat N(0,1), depth softmax of
    N(0,1) logits."""
    NC, D, H, W, C, Y, X = 6, 59, 16, 44, 64, 128, 128
    rng = np.random.default_rng(seed)
    feat = _normal_feat(rng, NC, H, W, C)
    depth = _softmax_depth(rng, NC, D, H, W, 1.0)
    fx = fy = 800.0
    cx, cy = 352.0, 128.0
    z = np.arange(1, D + 1, dtype=np.float64)[:, None, None]            # [D,1,1]
    v = ((np.arange(H, dtype=np.float64) + 0.5) * 16.0)[None, :, None]   # [1,H,1]
    u = ((np.arange(W, dtype=np.float64) + 0.5) * 16.0)[None, None, :]   # [1,1,W]
    x_cam = (u - cx) / fx * z
    y_cam = (v - cy) / fy * z
    cells = np.empty((NC, D, H, W), dtype=np.int32)
    for k in range(NC):
        yaw = math.radians(60.0 * k)
        # forward axis (cos, sin, 0); image-right axis (sin, -cos, 0); image-down axis (0, 0, -1)
        ex = z * math.cos(yaw) + x_cam * math.sin(yaw)
        ey = z * math.sin(yaw) - x_cam * math.cos(yaw)
        ez = -y_cam + 0.0 * ex
        ix = np.floor((ex + 51.2) / 0.8).astype(np.int64)
        iy = np.floor((ey + 51.2) / 0.8).astype(np.int64)
        ok = (ix >= 0) & (ix < X) & (iy >= 0) & (iy < Y) & (ez >= -5.0) & (ez <= 3.0)
        c = np.where(ok, iy * X + ix, -1)
        cells[k] = np.broadcast_to(c, (D, H, W)).astype(np.int32)
    return Workload("bevdet", NC, D, H, W, C, Y * X, cells.reshape(-1), depth, feat, grid=(1, Y, X),
                    recipe=f"seed {seed}: pinhole geometry (fx=fy=800, 704x256 image, /16, yaw k*60deg, "
                           "z=1..59 m), 0.8 m cells over +-51.2 m, Z in [-5,3] m")


def dram_batch(seeds: tuple = (10, 11, 12, 13), keep: float = 0.2759) -> Workload:
    """Four canonical frusta (24 cameras) into a batched [4, 512, 512] grid, C=128.

    Per sample: feat N(0,1) fp16, depth softmax of N(0,2) logits, keep
    Bernoulli(0.2759) (about 2.2M kept in total), cells uniform in the disc
    of radius 250 around (256, 256): r = 250*sqrt(u), theta ~ U(0, 2pi).
    Sample b's cells are offset by b*512*512."""
    D, H, W, C, Y, X = 118, 32, 88, 128, 512, 512
    cams = 6
    feats, depths, cell_parts = [], [], []
    for b, seed in enumerate(seeds):
        rng = np.random.default_rng(seed)
        feats.append(_normal_feat(rng, cams, H, W, C))
        depths.append(_softmax_depth(rng, cams, D, H, W, 2.0))
        nf = cams * D * H * W
        kept = rng.random(nf) < keep
        n = int(kept.sum())
        u = rng.random(n)
        theta = rng.random(n) * (2.0 * math.pi)
        r = 250.0 * np.sqrt(u)
        y = np.floor(256.0 + r * np.sin(theta)).astype(np.int64)
        x = np.floor(256.0 + r * np.cos(theta)).astype(np.int64)
        c = np.full(nf, -1, dtype=np.int32)
        c[kept] = (b * Y * X + y * X + x).astype(np.int32)
        cell_parts.append(c)
    NC = cams * len(seeds)
    return Workload("dram_batch", NC, D, H, W, C, len(seeds) * Y * X, np.concatenate(cell_parts),
                    np.concatenate(depths, axis=0), np.concatenate(feats, axis=0), grid=(len(seeds), Y, X),
                    recipe=f"seeds {list(seeds)}: per sample feat N(0,1), depth softmax N(0,2) logits, "
                           f"keep Bernoulli({keep}), cells uniform in disc r<=250 of a 512x512 grid")


def custom(NC: int, D: int, H: int, W: int, C: int, n_cells: int, cell_ids: np.ndarray,
           seed: int = 0, dtype: str = "f16", name: str = "custom",
           depth: Optional[np.ndarray] = None, feat: Optional[np.ndarray] = None) -> Workload:
    """A workload with caller-chosen cell ids (edge cases); random depth/feat unless given."""
    rng = np.random.default_rng(seed)
    if feat is None:
        feat = _normal_feat(rng, NC, H, W, C)
    if depth is None:
        depth = _softmax_depth(rng, NC, D, H, W, 1.0)
    wl = Workload(name, NC, D, H, W, C, n_cells, np.ascontiguousarray(cell_ids, dtype=np.int32).reshape(-1),
                  np.ascontiguousarray(depth, dtype=np.float16), np.ascontiguousarray(feat, dtype=np.float16),
                  grid=(1, 1, n_cells), recipe=f"custom seed {seed}")
    if dtype == "e4m3":
        f32 = wl.feat.astype(np.float32)
        d32 = wl.depth.astype(np.float32)
        fs = float(np.float32(max(np.abs(f32).max(), 1e-30) / np.float32(E4M3_MAX)))
        ds = float(np.float32(max(d32.max(), 1e-30)))
        wl = dataclasses.replace(wl, dtype="e4m3", feat=quantize_e4m3(f32, fs).reshape(wl.feat.shape),
                                 depth=quantize_e4m3(d32, ds).reshape(wl.depth.shape),
                                 feat_scale=fs, depth_scale=ds)
    return wl


CONFIGS = {
    "tiny": tiny,
    "canonical": canonical,
    "canonical_fp8": canonical_fp8,
    "bevdet": bevdet,
    "dram_batch": dram_batch,
}


def make(name: str) -> Workload:
    """A named workload; '<table-1 shape>_fp8' gives its E4M3 version."""
    if name in CONFIGS:
        return CONFIGS[name]()
    if name in TABLE1:
        return table1(name)
    if name.endswith("_fp8") and name[:-4] in TABLE1:
        return _to_fp8(table1(name[:-4]), name)
    if name == "canonical_nvfp4":
        return _to_nvfp4(canonical(), name)
    if name.endswith("_nvfp4") and name[:-6] in TABLE1:
        return _to_nvfp4(table1(name[:-6]), name)
    raise KeyError(f"unknown workload {name!r}")


ALL_NAMES = (list(CONFIGS) + ["canonical_nvfp4"] + list(TABLE1) + [n + "_fp8" for n in TABLE1] +
             [n + "_nvfp4" for n in TABLE1])
