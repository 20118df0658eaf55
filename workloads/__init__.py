"""Seeded synthetic workloads for multi-scale deformable attention.

This module is shared by the CPU oracle's tests, the CUDA parity tests and the
benchmark.  It only draws random inputs and lays them out; it holds none of the
sampling / interpolation arithmetic of the method itself.

Tensor layouts (one row per tensor):

  value               [B, Nin, M, D]            fp32, or bf16 bits (uint16)
  spatial_shapes      [L, 2] = (H, W)  or  [L, 3] = (Z, H, W)      int64
  level_start_index   [L]   exclusive prefix sum of the level sizes  int64
  sampling_locations  [B, Nq, M, L, P, 2|3]  normalised (x, y[, z])  fp32
  attention_weights   [B, Nq, M, L, P]                               fp32
  grad_out            [B, Nq, M*D]         (backward workloads only)

Component 0 of a location is x (along W), 1 is y (along H), 2 is z (along Z),
the order used by "3D Attention That Knows Where to Look" ("What changes from
2D to 3D": offsets (x, y) become (x, y, z), shapes (H, W) become (D, H, W)).

The five named workloads follow the encoder / decoder / volumetric shapes the
method is used at (Deformable DETR's 4-level pyramid, K = 4 points per level):

  tiny2d      B1  L1 16x16              M2 D8  Nq64     P4  fp32  forward
  encoder2d   B2  L4 100x150..13x19     M8 D32 Nq19947  P4  fp32  forward
  decoder2d   B8  L4 (same pyramid)     M8 D32 Nq300    P4  bf16  forward
  volume3d    B1  L4 64^3,32^3,16^3,8^3 M8 D32 Nq32768  P4  bf16  forward
  encoder2d_bwd  encoder2d shapes, fp32, backward with 10% pushed out of range
  volume3d_bwd   volume3d shapes, bf16 value / grad_out, backward, 10% out of range
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

PYRAMID_2D = [(100, 150), (50, 75), (25, 38), (13, 19)]
PYRAMID_3D = [(64, 64, 64), (32, 32, 32), (16, 16, 16), (8, 8, 8)]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    ndim: int                      # 2 (bilinear) or 3 (trilinear)
    B: int
    shapes: Tuple[Tuple[int, ...], ...]
    Nq: int
    M: int
    D: int
    P: int
    dtype: str                     # "f32" or "bf16" (value / out dtype)
    seed: int
    backward: bool = False
    query_layout: str = "uniform"  # "per_pixel" | "uniform" | "voxel_centres"
    offset_std_px: float = 0.0     # std of the offset in pixels of the sampled level
    oob_fraction: float = 0.0      # fraction of samples pushed out of range

    @property
    def L(self) -> int:
        return len(self.shapes)

    @property
    def Nin(self) -> int:
        return int(sum(int(np.prod(s)) for s in self.shapes))

    @property
    def samples(self) -> int:
        return self.B * self.Nq * self.M * self.L * self.P

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    "tiny2d": Workload("tiny2d", 2, 1, ((16, 16),), 64, 2, 8, 4, "f32", 1000,
                       query_layout="uniform_locations"),
    "encoder2d": Workload("encoder2d", 2, 2, tuple(PYRAMID_2D), 19947, 8, 32, 4,
                          "f32", 1001, query_layout="per_pixel", offset_std_px=2.0),
    "decoder2d": Workload("decoder2d", 2, 8, tuple(PYRAMID_2D), 300, 8, 32, 4,
                          "bf16", 1002, query_layout="uniform", offset_std_px=4.0),
    "volume3d": Workload("volume3d", 3, 1, tuple(PYRAMID_3D), 32768, 8, 32, 4,
                         "bf16", 1003, query_layout="voxel_centres", offset_std_px=2.0),
    "encoder2d_bwd": Workload("encoder2d_bwd", 2, 2, tuple(PYRAMID_2D), 19947, 8, 32,
                              4, "f32", 1004, backward=True, query_layout="per_pixel",
                              offset_std_px=2.0, oob_fraction=0.10),
    "volume3d_bwd": Workload("volume3d_bwd", 3, 1, tuple(PYRAMID_3D), 32768, 8, 32, 4,
                             "bf16", 1005, backward=True, query_layout="voxel_centres",
                             offset_std_px=2.0, oob_fraction=0.10),
}


def level_start_index(shapes: Sequence[Sequence[int]]) -> np.ndarray:
    sizes = [int(np.prod(s)) for s in shapes]
    return np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (round to nearest, ties to even); bits as uint16."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    # finite inputs only: the largest finite pattern plus 0x8000 still fits in 32 bits
    r = (b >> np.uint32(16)) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += b
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _softmax_last(logits: np.ndarray) -> np.ndarray:
    """Normalised weights from logits (input preparation; the core never renormalises)."""
    z = logits.astype(np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def _reference_points(w: Workload, rng: np.random.Generator) -> np.ndarray:
    """Normalised reference point of every query, [B, Nq, ndim] in (x, y[, z]) order."""
    B, Nq, nd = w.B, w.Nq, w.ndim
    if w.query_layout == "per_pixel":
        # one query per pixel of every level, levels in order, row-major inside a level;
        # the reference point is that pixel's centre in normalised coordinates
        pts = []
        for shape in w.shapes:
            if nd == 2:
                H, W = shape
                hh, ww = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
                pts.append(np.stack([(ww.ravel() + 0.5) / W, (hh.ravel() + 0.5) / H], -1))
            else:
                Z, H, W = shape
                zz, hh, ww = np.meshgrid(np.arange(Z), np.arange(H), np.arange(W),
                                         indexing="ij")
                pts.append(np.stack([(ww.ravel() + 0.5) / W, (hh.ravel() + 0.5) / H,
                                     (zz.ravel() + 0.5) / Z], -1))
        ref = np.concatenate(pts, 0)
        assert ref.shape[0] == Nq, (ref.shape, Nq)
        return np.broadcast_to(ref, (B, Nq, nd)).copy()
    if w.query_layout == "voxel_centres":
        # random voxel centres of the second level, drawn with replacement
        Z, H, W = w.shapes[1]
        iz = rng.integers(0, Z, size=(B, Nq))
        ih = rng.integers(0, H, size=(B, Nq))
        iw = rng.integers(0, W, size=(B, Nq))
        return np.stack([(iw + 0.5) / W, (ih + 0.5) / H, (iz + 0.5) / Z], -1)
    return rng.random((B, Nq, nd))


def _extent_xyz(shape: Sequence[int]) -> np.ndarray:
    """Extents in location-component order: (W, H) or (W, H, Z)."""
    return np.array(list(shape)[::-1], dtype=np.float64)


def make_locations(w: Workload, rng: np.random.Generator) -> np.ndarray:
    B, Nq, M, L, P, nd = w.B, w.Nq, w.M, w.L, w.P, w.ndim
    if w.query_layout == "uniform_locations":
        return rng.random((B, Nq, M, L, P, nd)).astype(np.float32)
    ref = _reference_points(w, rng)                                  # [B,Nq,nd]
    off_px = rng.standard_normal((B, Nq, M, L, P, nd)) * w.offset_std_px
    ext = np.stack([_extent_xyz(s) for s in w.shapes], 0)            # [L,nd]
    loc = ref[:, :, None, None, None, :] + off_px / ext[None, None, None, :, None, :]
    if w.oob_fraction > 0:
        loc = _push_out_of_range(loc, w, rng)
    return loc.astype(np.float32)


def _push_out_of_range(loc: np.ndarray, w: Workload, rng: np.random.Generator) -> np.ndarray:
    """Move a seeded fraction of samples out of range along one random axis.

    Half of them straddle an edge (pixel coordinate in (-1, 0) or (E-1, E), so some
    corners fall outside the map), half land fully outside (pixel <= -1 or >= E).
    """
    B, Nq, M, L, P, nd = loc.shape
    flat = loc.reshape(-1, L, P, nd)
    n = flat.shape[0] * L * P
    pick = rng.random(n) < w.oob_fraction
    idx = np.nonzero(pick)[0]
    axis = rng.integers(0, nd, size=idx.size)
    straddle = rng.random(idx.size) < 0.5
    low_side = rng.random(idx.size) < 0.5
    u = rng.random(idx.size)
    lvl = (idx // P) % L
    ext = np.array([_extent_xyz(s) for s in w.shapes])               # [L,nd]
    E = ext[lvl, axis]
    # pixel coordinate = loc*E - 0.5
    pix = np.where(straddle,
                   np.where(low_side, -1.0 + u * 1.0, (E - 1.0) + u * 1.0),
                   np.where(low_side, -1.0 - (0.01 + 3.0 * u), E + (0.01 + 3.0 * u)))
    # keep straddling samples strictly inside the open intervals
    pix = np.where(straddle & low_side, np.clip(pix, -0.999, -0.001), pix)
    pix = np.where(straddle & ~low_side, np.clip(pix, E - 0.999, E - 0.001), pix)
    view = flat.reshape(-1, nd)
    view[idx, axis] = (pix + 0.5) / E
    return flat.reshape(B, Nq, M, L, P, nd)


def make_inputs(w: Workload, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """All inputs of one workload, as numpy arrays in the layouts listed above."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    B, Nin, Nq, M, D, L, P = w.B, w.Nin, w.Nq, w.M, w.D, w.L, w.P
    value32 = rng.standard_normal((B, Nin, M, D), dtype=np.float32)
    out: Dict[str, np.ndarray] = {}
    if w.dtype == "bf16":
        bits = f32_to_bf16_bits(value32)
        out["value_bits"] = bits
        out["value"] = bf16_bits_to_f32(bits)      # the exact values the GPU sees
    else:
        out["value"] = value32
    out["spatial_shapes"] = np.array(w.shapes, dtype=np.int64).reshape(L, w.ndim)
    out["level_start_index"] = level_start_index(w.shapes)
    out["sampling_locations"] = make_locations(w, rng)
    logits = rng.standard_normal((B, Nq, M, L * P))
    out["attention_weights"] = _softmax_last(logits).reshape(B, Nq, M, L, P)
    if w.backward:
        out["grad_out"] = rng.standard_normal((B, Nq, M * D), dtype=np.float32)
        if w.dtype == "bf16":
            out["grad_out_bits"] = f32_to_bf16_bits(out["grad_out"])
            out["grad_out"] = bf16_bits_to_f32(out["grad_out_bits"])
    return out


def make_fused_inputs(w: Workload, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Inputs of the forward with the module's prologue fused in: the value map, per-level
    reference points [B, Nq, L, ndim] (the query's reference point on every level), offsets
    [B, Nq, M, L, P, ndim] in pixels of the sampled level (N(0, offset_std_px), or 1 px for
    a workload that draws its locations directly) and raw logits [B, Nq, M, L, P] ~ N(0,1).
    Seeded like make_inputs (seed + 7919) but drawn independently of it."""
    rng = np.random.default_rng((w.seed if seed is None else seed) + 7919)
    B, Nin, Nq, M, D, L, P, nd = w.B, w.Nin, w.Nq, w.M, w.D, w.L, w.P, w.ndim
    value32 = rng.standard_normal((B, Nin, M, D), dtype=np.float32)
    out: Dict[str, np.ndarray] = {}
    if w.dtype == "bf16":
        out["value_bits"] = f32_to_bf16_bits(value32)
        out["value"] = bf16_bits_to_f32(out["value_bits"])
    else:
        out["value"] = value32
    out["spatial_shapes"] = np.array(w.shapes, dtype=np.int64).reshape(L, nd)
    out["level_start_index"] = level_start_index(w.shapes)
    if w.query_layout == "uniform_locations":
        ref = rng.random((B, Nq, nd))
        std = 1.0
    else:
        ref = _reference_points(w, rng)
        std = w.offset_std_px
    out["reference_points"] = np.repeat(ref[:, :, None, :], L, axis=2).astype(np.float32)
    out["sampling_offsets"] = (rng.standard_normal((B, Nq, M, L, P, nd)) * std).astype(np.float32)
    out["attention_logits"] = rng.standard_normal((B, Nq, M, L, P)).astype(np.float32)
    return out


def out_of_range_fraction(w: Workload, loc: np.ndarray) -> float:
    """Fraction of samples whose location falls outside [0, 1] on some axis."""
    bad = ((loc < 0) | (loc > 1)).any(axis=-1)
    return float(bad.mean())


def shard_range(total: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous [start, stop) share of `total` independent units for one rank."""
    if world < 1 or not (0 <= rank < world):
        raise ValueError(f"bad rank {rank} of {world}")
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def names() -> List[str]:
    return list(WORKLOADS)


def random_problem(ndim: int, shapes: Sequence[Sequence[int]], B: int = 2, Nq: int = 37,
                   M: int = 3, D: int = 8, P: int = 4, dtype: str = "f32", seed: int = 0,
                   margin: float = 1.5, backward: bool = True) -> Dict[str, np.ndarray]:
    """A small random problem in the ``make_inputs`` layout, for parity and edge tests.

    Pixel coordinates are uniform over [-margin, extent - 1 + margin] on every axis, so a
    share of the samples straddles or leaves the level (zero padding is exercised).
    """
    rng = np.random.default_rng(seed)
    shapes = [tuple(int(e) for e in s) for s in shapes]
    L = len(shapes)
    Nin = int(sum(int(np.prod(s)) for s in shapes))
    v32 = rng.standard_normal((B, Nin, M, D), dtype=np.float32)
    out: Dict[str, np.ndarray] = {}
    if dtype == "bf16":
        out["value_bits"] = f32_to_bf16_bits(v32)
        out["value"] = bf16_bits_to_f32(out["value_bits"])
    else:
        out["value"] = v32
    out["spatial_shapes"] = np.array(shapes, dtype=np.int64).reshape(L, ndim)
    out["level_start_index"] = level_start_index(shapes)
    ext = np.stack([_extent_xyz(s) for s in shapes], 0)               # [L, ndim]
    u = rng.random((B, Nq, M, L, P, ndim))
    pix = u * (ext[None, None, None, :, None, :] - 1.0 + 2 * margin) - margin
    out["sampling_locations"] = ((pix + 0.5) / ext[None, None, None, :, None, :]).astype(
        np.float32)
    out["attention_weights"] = _softmax_last(
        rng.standard_normal((B, Nq, M, L * P))).reshape(B, Nq, M, L, P)
    if backward:
        g = rng.standard_normal((B, Nq, M * D), dtype=np.float32)
        if dtype == "bf16":
            out["grad_out_bits"] = f32_to_bf16_bits(g)
            g = bf16_bits_to_f32(out["grad_out_bits"])
        out["grad_out"] = g
    return out
