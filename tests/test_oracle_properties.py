"""Property-based pins of the CPU oracle over randomly drawn tiny problems (hypothesis).

The fixed pins in ``test_oracle_pins.py`` check hand-picked shapes.  These draw the shape of
the problem too (2D or 3D, 1-3 levels of 1-5 pixels per axis, any B, Nq, M, D, P up to a
few) and pixel coordinates that sit on the edges the method treats specially: exactly on
pixel centres, on the -1 and extent boundaries where zero padding starts, and in the
half-pixel bands where only some corners exist.  Each property is fixed by the mathematics
of bilinear / trilinear sampling ("What is Deformable Attention ...", "(3) Bilinear
Interpolation"; "3D Attention That Knows Where to Look", "What changes from 2D to 3D") and
of the attention-weighted sum ("Deformable Attention Module", DeformAttn equation), not by
the oracle:

* the forward equals the dense tent-kernel brute force (no floor, corners or bounds test);
* permuting the queries permutes the outputs, and relabelling the levels (moving their
  value rows, starts, locations and weights together) leaves the outputs unchanged;
* the backward satisfies the adjoint identities of the two linear arguments, and its
  location gradient matches a central difference of the forward along a random direction
  wherever no coordinate sits on a kink.

Runs are derandomised, so a failure reproduces.
"""
from __future__ import annotations

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
from dense_reference import dense_forward  # noqa: E402
from workloads import level_start_index  # noqa: E402

SETTINGS = settings(max_examples=60, deadline=None, derandomize=True,
                    suppress_health_check=[HealthCheck.too_slow])


@st.composite
def problems(draw):
    nd = draw(st.sampled_from([2, 3]))
    L = draw(st.integers(1, 3))
    shapes = np.array([[draw(st.integers(1, 5)) for _ in range(nd)] for _ in range(L)],
                      dtype=np.int64)
    B, Nq, M = draw(st.integers(1, 2)), draw(st.integers(1, 3)), draw(st.integers(1, 2))
    D, P = draw(st.integers(1, 3)), draw(st.integers(1, 3))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    Nin = int(np.prod(shapes, axis=1).sum())
    ext = shapes[:, ::-1].astype(np.float64)                  # (W, H[, Z]) per level
    full = ext[None, None, None, :, None, :] * np.ones((B, Nq, M, L, P, nd))
    # pixel coordinates: a mix of free draws over [-1.5, extent + 0.5], pixel centres and
    # the exact zero-padding boundaries -1 and extent
    kind = rng.integers(0, 4, size=full.shape)
    free = rng.uniform(0, 1, size=full.shape) * (full + 2.0) - 1.5
    centre = np.floor(rng.uniform(0, 1, size=full.shape) * full)
    edge = np.where(rng.integers(0, 2, size=full.shape) == 0, -1.0, full)
    half = np.where(rng.integers(0, 2, size=full.shape) == 0,
                    rng.uniform(-1.0, 0.0, size=full.shape),
                    full - 1.0 + rng.uniform(0.0, 1.0, size=full.shape))
    pix = np.choose(kind, [free, centre, edge, half])
    loc = (pix + 0.5) / full
    a = rng.uniform(-1.0, 1.0, (B, Nq, M, L, P))
    return dict(nd=nd, value=rng.standard_normal((B, Nin, M, D)), spatial_shapes=shapes,
                level_start_index=level_start_index(shapes), sampling_locations=loc,
                attention_weights=a, grad_out=rng.standard_normal((B, Nq, M * D)),
                direction=rng.standard_normal(loc.shape), perm=rng.permutation(Nq),
                level_perm=rng.permutation(L))


def _fwd(c, **over):
    d = dict(c, **over)
    return oracle.forward(c["nd"], d["value"], d["spatial_shapes"], d["level_start_index"],
                          d["sampling_locations"], d["attention_weights"])


@SETTINGS
@given(problems())
def test_forward_equals_dense_tent_brute_force(oracle_mod, c):
    got = _fwd(c)
    want = dense_forward(c["value"], c["spatial_shapes"], c["level_start_index"],
                         c["sampling_locations"], c["attention_weights"])
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


@SETTINGS
@given(problems())
def test_query_permutation_and_level_relabelling(oracle_mod, c):
    base = _fwd(c)
    perm = c["perm"]
    got = _fwd(c, sampling_locations=c["sampling_locations"][:, perm],
               attention_weights=c["attention_weights"][:, perm])
    assert np.array_equal(got, base[:, perm])
    # move every level with its value rows, start, locations and weights
    lp = c["level_perm"]
    shapes, starts = c["spatial_shapes"], c["level_start_index"]
    sizes = np.prod(shapes, axis=1)
    rows = np.concatenate([np.arange(starts[l], starts[l] + sizes[l]) for l in lp])
    new_shapes = shapes[lp]
    got = _fwd(c, value=c["value"][:, rows], spatial_shapes=new_shapes,
               level_start_index=level_start_index(new_shapes),
               sampling_locations=c["sampling_locations"][:, :, :, lp],
               attention_weights=c["attention_weights"][:, :, :, lp])
    # the sum over levels runs in another order: equal up to rounding
    np.testing.assert_allclose(got, base, rtol=0, atol=1e-12)


@SETTINGS
@given(problems())
def test_backward_adjoints_and_directional_derivative(oracle_mod, c):
    nd = c["nd"]
    out = _fwd(c)
    gv, gl, ga = oracle.backward(nd, c["value"], c["spatial_shapes"], c["level_start_index"],
                                 c["sampling_locations"], c["attention_weights"],
                                 c["grad_out"])
    g = c["grad_out"]
    inner = float(np.sum(g * out))
    scale = 1.0 + float(np.sum(np.abs(g) * np.abs(out)))
    # the forward is linear in value and in A, so <g, out> is the pairing of either
    # argument with its gradient
    assert abs(float(np.sum(c["value"] * gv)) - inner) <= 1e-12 * scale
    assert abs(float(np.sum(c["attention_weights"] * ga)) - inner) <= 1e-12 * scale
    # directional derivative in the locations, along a direction that leaves every
    # coordinate within 1e-4 px of a kink where it is (an integer pixel coordinate: the
    # corner cell, or the zero padding, changes there and the derivative is one-sided)
    ext = c["spatial_shapes"][:, ::-1].astype(np.float64)[None, None, None, :, None, :]
    pix = c["sampling_locations"] * ext - 0.5
    smooth = np.abs(pix - np.round(pix)) > 1e-4
    h = 1e-7
    dirn = np.where(smooth, c["direction"], 0.0)
    up = _fwd(c, sampling_locations=c["sampling_locations"] + h * dirn)
    dn = _fwd(c, sampling_locations=c["sampling_locations"] - h * dirn)
    fd = float(np.sum(g * (up - dn))) / (2 * h)
    an = float(np.sum(gl * dirn))
    tol = 1e-6 * (1.0 + abs(an)) + 1e-7 * float(np.sum(np.abs(gl) * np.abs(dirn)))
    assert abs(fd - an) <= tol, (fd, an)
