"""Dense brute-force formulation of the sampling core, used only to pin the oracle.

It shares no logic with the oracle: there is no floor(), no corner enumeration and
no bounds test.  Each sample gets an explicit weight over EVERY pixel of the sampled
level, the separable tent (hat) kernel

    w(pixel) = prod over axes of max(0, 1 - |coord - pixel_index|),

which is what bilinear (2D) and trilinear (3D) interpolation are ("What is Deformable
Attention ...", "(3) Bilinear Interpolation"; "3D Attention That Knows Where to Look",
"What changes from 2D to 3D").  Pixels that do not exist carry no weight, which is
the zero-padding reading.  The sampled value is that weight vector dotted with the
level's value rows, and the output is the attention-weighted sum over all L x P samples
("Deformable Attention Module", DeformAttn equation; multi-scale blending on the 3D page).
Coordinates follow pixel = loc * extent - 0.5 (align_corners = False).

Slow (O(samples x Nin)) and meant for tiny inputs with finite locations.
"""
from __future__ import annotations

import numpy as np


def _tent(coord: float, n: int) -> np.ndarray:
    return np.maximum(0.0, 1.0 - np.abs(coord - np.arange(n, dtype=np.float64)))


def dense_forward(value, shapes, level_start, loc, attn) -> np.ndarray:
    value = np.asarray(value, dtype=np.float64)
    loc = np.asarray(loc, dtype=np.float64)
    attn = np.asarray(attn, dtype=np.float64)
    B, Nin, M, D = value.shape
    _, Nq, _, L, P, nd = loc.shape
    out = np.zeros((B, Nq, M, D))
    for l in range(L):
        shape = [int(s) for s in shapes[l]]
        n = int(np.prod(shape))
        start = int(level_start[l])
        vl = value[:, start:start + n]                      # [B, n, M, D]
        ext = shape[::-1]                                   # (W, H[, Z]) in loc order
        for b in range(B):
            for q in range(Nq):
                for m in range(M):
                    for p in range(P):
                        c = [loc[b, q, m, l, p, k] * ext[k] - 0.5 for k in range(nd)]
                        wx = _tent(c[0], ext[0])
                        wy = _tent(c[1], ext[1])
                        if nd == 2:
                            wmap = np.outer(wy, wx)                       # [H, W]
                        else:
                            wz = _tent(c[2], ext[2])
                            wmap = wz[:, None, None] * np.outer(wy, wx)[None]  # [Z,H,W]
                        s = wmap.reshape(-1) @ vl[b, :, m, :]              # [D]
                        out[b, q, m] += attn[b, q, m, l, p] * s
    return out.reshape(B, Nq, M * D)
