"""Pins for the CPU oracle: checks against facts fixed outside the oracle itself.

Each ``pin_*`` function takes an oracle library handle (``None`` = the built oracle) and
raises ``AssertionError`` when the oracle disagrees with:

* hand-derived worked values (``tests/golden``: the "(7.3, 12.8)" bilinear example of
  "3D Attention That Knows Where to Look", and trilinear cube corners from the same
  page's "What changes from 2D to 3D");
* a dense brute-force tent-kernel formulation with no floor / corner / bounds logic
  (``dense_reference.py``);
* closed forms and invariants: a constant map returns the constant because the weights
  sum to one ("Deformable Attention Module": A in [0, 1], sum over the sampled keys = 1);
  exact gathers at pixel centres; linearity in the attention weights; per-level isolation
  of the multi-scale sum; 3D with a single slice equals 2D;
* the mathematics of the backward pass ("3D Attention That Knows Where to Look": the
  gradients flow back into both the offsets and the weights): central finite differences
  of the forward, exact directional derivatives in the linear arguments, and the adjoint
  identities sum(g*out) = sum(value*grad_value) = sum(A*grad_A).

``tests/test_oracle_mutants.py`` plants plausible mistakes in copies of the oracle and
requires that at least one pin fails for each.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
from dense_reference import dense_forward
from workloads import level_start_index

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _close(a, b, atol, rtol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.abs(a - b)
    bound = atol + rtol * np.abs(b)
    if not np.all(err <= bound):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: max err {err.max():.3e} at {i}: got {a[i]!r} want {b[i]!r}")


def _load_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([float(t) for t in line.split()])
    return np.array(rows)


# --------------------------------------------------------------------------- inputs


def random_case(nd, shapes, B=2, Nq=5, M=2, D=3, P=3, seed=0, margin=1.5):
    """Small random problem whose pixel coordinates cover [-margin, extent-1+margin]."""
    rng = np.random.default_rng(seed)
    shapes = np.array(shapes, dtype=np.int64).reshape(len(shapes), nd)
    L = shapes.shape[0]
    Nin = int(np.prod(shapes, axis=1).sum())
    value = rng.standard_normal((B, Nin, M, D))
    ext = shapes[:, ::-1].astype(np.float64)                        # (W, H[, Z]) per level
    pix = rng.uniform(0, 1, (B, Nq, M, L, P, nd)) * (ext[None, None, None, :, None, :]
                                                     - 1.0 + 2 * margin) - margin
    loc = (pix + 0.5) / ext[None, None, None, :, None, :]
    logits = rng.standard_normal((B, Nq, M, L * P))
    e = np.exp(logits - logits.max(-1, keepdims=True))
    attn = (e / e.sum(-1, keepdims=True)).reshape(B, Nq, M, L, P)
    return dict(value=value, spatial_shapes=shapes, level_start_index=level_start_index(shapes),
                sampling_locations=loc, attention_weights=attn,
                grad_out=rng.standard_normal((B, Nq, M * D)))


SHAPES_2D = [(5, 7), (3, 4)]
SHAPES_3D = [(3, 4, 5), (2, 2, 3)]


def _fwd(nd, c, lib, **over):
    d = dict(c)
    d.update(over)
    return oracle.forward(nd, d["value"], d["spatial_shapes"], d["level_start_index"],
                          d["sampling_locations"], d["attention_weights"], lib=lib)


def _bwd(nd, c, lib):
    return oracle.backward(nd, c["value"], c["spatial_shapes"], c["level_start_index"],
                           c["sampling_locations"], c["attention_weights"], c["grad_out"],
                           lib=lib)


# --------------------------------------------------------------------------- forward pins


def pin_golden_2d(lib=None):
    tab = _load_table("bilinear_worked_2d.txt")
    H = W = 16
    yy, xx = np.meshgrid(np.arange(H, dtype=np.float64), np.arange(W, dtype=np.float64),
                         indexing="ij")
    onehot = lambda x, y: ((xx == x) & (yy == y)).astype(np.float64)
    chans = [xx + 10 * yy, xx * yy, onehot(7, 12), onehot(8, 12), onehot(7, 13),
             onehot(8, 13), xx * xx, yy * yy]
    value = np.stack(chans, -1).reshape(1, H * W, 1, 8)
    n = tab.shape[0]
    loc = ((tab[:, :2] + 0.5) / 16.0).reshape(1, n, 1, 1, 1, 2)
    attn = np.ones((1, n, 1, 1, 1))
    shapes = np.array([[H, W]])
    out = oracle.forward(2, value, shapes, [0], loc, attn, lib=lib)
    _close(out[0], tab[:, 2:], atol=1e-12, rtol=1e-12, what="golden 2d")
    # the same rows blended in ONE query with weights summing to 1 (multi-point sum)
    a = np.array([0.5, 0.25, 0.125, 0.0625, 0.03125, 0.03125])[:n]
    out1 = oracle.forward(2, value, shapes, [0], loc.reshape(1, 1, 1, 1, n, 2),
                          a.reshape(1, 1, 1, 1, n), lib=lib)
    _close(out1[0, 0], a @ tab[:, 2:], atol=1e-12, rtol=1e-12, what="golden 2d blended")


def pin_golden_3d(lib=None):
    tab = _load_table("trilinear_worked_3d.txt")
    S = 8
    zz, yy, xx = np.meshgrid(*(np.arange(S, dtype=np.float64),) * 3, indexing="ij")
    onehot = lambda x, y, z: ((xx == x) & (yy == y) & (zz == z)).astype(np.float64)
    chans = [xx + 10 * yy + 100 * zz, onehot(2, 3, 4), onehot(1, 2, 3), xx * yy * zz]
    value = np.stack(chans, -1).reshape(1, S ** 3, 1, 4)
    n = tab.shape[0]
    loc = ((tab[:, :3] + 0.5) / S).reshape(1, n, 1, 1, 1, 3)
    out = oracle.forward(3, value, np.array([[S, S, S]]), [0], loc, np.ones((1, n, 1, 1, 1)),
                         lib=lib)
    _close(out[0], tab[:, 3:], atol=1e-12, rtol=1e-12, what="golden 3d")


def pin_dense(nd, lib=None):
    shapes = SHAPES_2D if nd == 2 else SHAPES_3D
    for seed in range(3):
        c = random_case(nd, shapes, seed=seed)
        got = _fwd(nd, c, lib)
        want = dense_forward(c["value"], c["spatial_shapes"], c["level_start_index"],
                             c["sampling_locations"], c["attention_weights"])
        _close(got, want, atol=1e-12, what=f"dense {nd}d seed {seed}")


def pin_dense_tiny_workload(lib=None):
    import workloads
    w = workloads.WORKLOADS["tiny2d"]
    inp = workloads.make_inputs(w)
    got = oracle.run_inputs(2, inp, lib=lib)
    want = dense_forward(inp["value"], inp["spatial_shapes"], inp["level_start_index"],
                         inp["sampling_locations"], inp["attention_weights"])
    _close(got, want, atol=1e-12, what="dense tiny2d")


def pin_constant_map(nd, lib=None):
    """value == c everywhere and every corner inside: out = c * sum(A) = c."""
    shapes = SHAPES_2D if nd == 2 else SHAPES_3D
    c = random_case(nd, shapes, seed=7)
    ext = np.array(shapes)[:, ::-1].astype(np.float64)
    rng = np.random.default_rng(8)
    pix = rng.uniform(0, 1, c["sampling_locations"].shape) * (ext[None, None, None, :, None, :] - 1)
    loc = (pix + 0.5) / ext[None, None, None, :, None, :]
    value = np.full_like(c["value"], 2.5)
    out = _fwd(nd, c, lib, value=value, sampling_locations=loc)
    _close(out, np.full_like(out, 2.5), atol=1e-12, what=f"constant map {nd}d")


def pin_exact_gather(lib=None):
    """Pixel-centre locations with a one-hot weight return the value row exactly."""
    rng = np.random.default_rng(3)
    H = W = 16
    value = rng.standard_normal((1, H * W, 2, 8)).astype(np.float32).astype(np.float64)
    ix = rng.integers(0, W, size=(1, 40, 2, 1, 4))
    iy = rng.integers(0, H, size=(1, 40, 2, 1, 4))
    loc = np.stack([(ix + 0.5) / W, (iy + 0.5) / H], -1)
    attn = np.zeros((1, 40, 2, 1, 4))
    attn[..., 2] = 1.0
    out = oracle.forward(2, value, np.array([[H, W]]), [0], loc, attn, lib=lib)
    rows = iy[..., 2] * W + ix[..., 2]                                   # [1,40,2,1]
    want = np.stack([value[0, rows[0, :, m, 0], m] for m in range(2)], 1)  # [40,2,8]
    assert np.array_equal(out[0].reshape(40, 2, 8), want), "exact gather is not bit-exact"


def pin_linearity_and_levels(nd, lib=None):
    shapes = SHAPES_2D if nd == 2 else SHAPES_3D
    c = random_case(nd, shapes, seed=11)
    rng = np.random.default_rng(12)
    A1 = rng.uniform(0, 1, c["attention_weights"].shape)
    A2 = rng.uniform(0, 1, c["attention_weights"].shape)
    o1 = _fwd(nd, c, lib, attention_weights=A1)
    o2 = _fwd(nd, c, lib, attention_weights=A2)
    o12 = _fwd(nd, c, lib, attention_weights=0.75 * A1 - 1.5 * A2)
    _close(o12, 0.75 * o1 - 1.5 * o2, atol=1e-12, what=f"linearity in A {nd}d")
    # per-level isolation: weights only on level l == the single-level op on level l
    ls = c["level_start_index"]
    for l in range(len(shapes)):
        A = np.zeros_like(A1)
        A[..., l, :] = A1[..., l, :]
        full = _fwd(nd, c, lib, attention_weights=A)
        n = int(np.prod(shapes[l]))
        single = oracle.forward(nd, c["value"][:, ls[l]:ls[l] + n],
                                np.array([shapes[l]]), [0],
                                c["sampling_locations"][..., l:l + 1, :, :],
                                A1[..., l:l + 1, :], lib=lib)
        _close(full, single, atol=1e-12, what=f"level isolation {nd}d l={l}")


def pin_3d_single_slice_is_2d(lib=None):
    """Z = 1 and z-location 0.5 (pixel z = 0) reduces trilinear to bilinear exactly."""
    c2 = random_case(2, SHAPES_2D, seed=21)
    shapes3 = np.array([[1, h, w] for h, w in SHAPES_2D])
    loc3 = np.concatenate([c2["sampling_locations"],
                           np.full(c2["sampling_locations"].shape[:-1] + (1,), 0.5)], -1)
    o2 = _fwd(2, c2, lib)
    o3 = oracle.forward(3, c2["value"], shapes3, c2["level_start_index"], loc3,
                        c2["attention_weights"], lib=lib)
    assert np.array_equal(o2, o3), "3D with one slice differs from 2D"
    gv2, gl2, ga2 = _bwd(2, c2, lib)
    gv3, gl3, ga3 = oracle.backward(3, c2["value"], shapes3, c2["level_start_index"], loc3,
                                    c2["attention_weights"], c2["grad_out"], lib=lib)
    assert np.array_equal(gv2, gv3) and np.array_equal(ga2, ga3)
    assert np.array_equal(gl2, gl3[..., :2])


def pin_nonfinite_locations(nd, lib=None):
    shapes = SHAPES_2D if nd == 2 else SHAPES_3D
    c = random_case(nd, shapes, seed=31)
    loc = c["sampling_locations"].copy()
    bad = [np.nan, np.inf, -np.inf, 1e30, -1e30]
    for i, v in enumerate(bad):
        loc[0, i, 0, 0, 0, i % nd] = v
    A = np.zeros_like(c["attention_weights"])
    A[0, :len(bad), 0, 0, 0] = 1.0
    out = _fwd(nd, c, lib, sampling_locations=loc, attention_weights=A)
    assert np.all(out[0, :len(bad), :c["value"].shape[3]] == 0.0), "non-finite sample not zero"
    cc = dict(c, sampling_locations=loc)
    gv, gl, ga = _bwd(nd, cc, lib)
    assert np.all(gl[0, :len(bad), 0, 0, 0] == 0.0) and np.all(ga[0, :len(bad), 0, 0, 0] == 0.0)


# --------------------------------------------------------------------------- backward pins


def _near_kink(pix, tol):
    return np.abs(pix - np.round(pix)) < tol


def pin_backward_finite_differences(nd, lib=None, case=None, h=1e-6, rtol=1e-6):
    shapes = SHAPES_2D if nd == 2 else SHAPES_3D
    c = case if case is not None else random_case(nd, shapes, seed=41)
    shapes = np.asarray(c["spatial_shapes"])
    gv, gl, ga = _bwd(nd, c, lib)
    g = c["grad_out"]
    loc = c["sampling_locations"]
    L, P = loc.shape[3], loc.shape[4]
    ext = shapes[:, ::-1].astype(np.float64)                               # [L, nd]
    B, Nq, M = loc.shape[:3]
    D = c["value"].shape[3]

    def per_head(out):
        return (out * g).reshape(B, Nq, M, D).sum(-1)                      # [B,Nq,M]

    scale_l = max(np.sqrt(np.mean(gl ** 2)), 1e-300)
    for l in range(L):
        for p in range(P):
            for k in range(nd):
                lp = loc.copy(); lm = loc.copy()
                lp[:, :, :, l, p, k] += h
                lm[:, :, :, l, p, k] -= h
                fd = (per_head(_fwd(nd, c, lib, sampling_locations=lp))
                      - per_head(_fwd(nd, c, lib, sampling_locations=lm))) / (2 * h)
                pix = loc[:, :, :, l, p, k] * ext[l, k] - 0.5
                ok = ~_near_kink(pix, 4 * h * ext[l, k])
                an = gl[:, :, :, l, p, k]
                _close(fd[ok], an[ok], atol=rtol * scale_l, rtol=rtol,
                       what=f"d/dloc {nd}d l{l} p{p} k{k}")
    # attention weights: the output is linear in A, so a large step is exact
    A = c["attention_weights"]
    for l in range(L):
        for p in range(P):
            hA = 0.25
            Ap = A.copy(); Am = A.copy()
            Ap[:, :, :, l, p] += hA
            Am[:, :, :, l, p] -= hA
            fd = (per_head(_fwd(nd, c, lib, attention_weights=Ap))
                  - per_head(_fwd(nd, c, lib, attention_weights=Am))) / (2 * hA)
            _close(fd, ga[:, :, :, l, p], atol=1e-10, rtol=1e-10, what=f"d/dA {nd}d")
    # value: linear, so the change along a random direction V is exactly sum(V*grad_value)
    rng = np.random.default_rng(5)
    base = (_fwd(nd, c, lib) * g).sum()
    for _ in range(3):
        V = rng.standard_normal(c["value"].shape)
        moved = (_fwd(nd, c, lib, value=c["value"] + V) * g).sum()
        want = (V * gv).sum()
        _close(moved - base, want, atol=1e-9 * (1 + abs(want)), what=f"d/dvalue {nd}d")


def pin_adjoint_identities(nd, lib=None, case=None):
    shapes = SHAPES_2D if nd == 2 else SHAPES_3D
    c = case if case is not None else random_case(nd, shapes, seed=51, Nq=9)
    out = _fwd(nd, c, lib)
    gv, gl, ga = _bwd(nd, c, lib)
    s_out = float((out * c["grad_out"]).sum())
    s_val = float((c["value"] * gv).sum())
    s_att = float((c["attention_weights"] * ga).sum())
    tol = 1e-9 * max(1.0, abs(s_out))
    assert abs(s_out - s_val) <= tol, ("sum(value*grad_value)", s_out, s_val)
    assert abs(s_out - s_att) <= tol, ("sum(A*grad_A)", s_out, s_att)


def pin_zero_padding_gradients(nd, lib=None):
    shapes = SHAPES_2D if nd == 2 else SHAPES_3D
    c = random_case(nd, shapes, seed=61)
    ext = np.array(shapes)[:, ::-1].astype(np.float64)
    loc = c["sampling_locations"].copy()
    # query 0: every sample fully outside (pixel <= -1 on one axis, or >= extent)
    loc[:, 0, :, :, :, 0] = (-1.25 + 0.5) / ext[None, None, :, None, 0]
    loc[:, 1, :, :, :, nd - 1] = (ext[None, None, :, None, nd - 1] + 0.5) / ext[None, None, :, None, nd - 1]
    cc = dict(c, sampling_locations=loc)
    gv, gl, ga = _bwd(nd, cc, lib)
    assert np.all(gl[:, :2] == 0) and np.all(ga[:, :2] == 0), "fully outside sample has grads"
    # constant map, every corner strictly inside: the location gradient vanishes
    rng = np.random.default_rng(62)
    pix = rng.uniform(0, 1, loc.shape) * (ext[None, None, None, :, None, :] - 1) * 0.999
    loc2 = (pix + 0.5) / ext[None, None, None, :, None, :]
    cc = dict(c, sampling_locations=loc2, value=np.full_like(c["value"], -1.75))
    gv, gl, ga = _bwd(nd, cc, lib)
    _close(gl, np.zeros_like(gl), atol=1e-9, what="constant-map location gradient")


def pin_all(lib=None, quick=False):
    """Run every pin (used by the mutation test)."""
    pin_golden_2d(lib)
    pin_golden_3d(lib)
    for nd in (2, 3):
        pin_dense(nd, lib)
        pin_constant_map(nd, lib)
        pin_linearity_and_levels(nd, lib)
        pin_nonfinite_locations(nd, lib)
        pin_adjoint_identities(nd, lib)
        pin_zero_padding_gradients(nd, lib)
        pin_backward_finite_differences(nd, lib)
    pin_exact_gather(lib)
    pin_3d_single_slice_is_2d(lib)
    if not quick:
        pin_dense_tiny_workload(lib)
