"""Drawn problems: the CUDA path (libmsda through its C ABI) against the CPU oracle.

hypothesis draws the whole problem: 2D or 3D; fp32 or bf16 value; the lanes per value row
(D * sizeof = 16..128 bytes); the compiled (L, P) pairs (4, 4) and (1, 4) or another pair,
which takes the generic kernels; level extents from 1 pixel up; B, Nq and M.  Then about
half of the pixel coordinates are moved onto the places where the sampling rule changes:
pixel centres (a corner weight is exactly 0 or 1), the zero-padding boundaries -1 and
extent (the sample just stops contributing), and the half-pixel bands next to them (only
some corners exist).  Forward and backward must match the oracle within the fp32 / bf16
tolerances of ``gpu_parity``.  Runs are derandomised, so a failure reproduces.
"""
from __future__ import annotations

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import workloads  # noqa: E402
from gpu_parity import check_backward, check_forward  # noqa: E402

pytestmark = pytest.mark.gpu

SETTINGS = settings(max_examples=30, deadline=None, derandomize=True,
                    suppress_health_check=[HealthCheck.too_slow,
                                           HealthCheck.function_scoped_fixture])


@pytest.fixture(scope="module")
def msda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    import scale_deformable_attention_msda3d_b300 as m
    m.load()
    return m


def _edge_coordinates(rng, loc, shapes):
    """Move about half of the pixel coordinates onto pixel centres, the -1 / extent
    boundaries and the half-pixel bands beside them (locations stay fp32)."""
    nd = loc.shape[-1]
    ext = np.array([s[::-1] for s in shapes], dtype=np.float64)        # (W, H[, Z])
    full = ext[None, None, None, :, None, :] * np.ones(loc.shape)
    kind = rng.integers(0, 8, size=loc.shape)                            # 0..3 keep
    centre = np.floor(rng.random(loc.shape) * full)
    edge = np.where(rng.integers(0, 2, size=loc.shape) == 0, -1.0, full)
    half = np.where(rng.integers(0, 2, size=loc.shape) == 0, -rng.random(loc.shape),
                    full - 1.0 + rng.random(loc.shape))
    far = np.where(rng.integers(0, 2, size=loc.shape) == 0, -1.0 - rng.random(loc.shape),
                   full + rng.random(loc.shape))
    pix = np.choose(np.clip(kind - 3, 0, 4), [np.zeros(loc.shape), centre, edge, half, far])
    moved = ((pix + 0.5) / full).astype(np.float32)
    assert moved.shape[-1] == nd
    return np.where(kind >= 4, moved, loc).astype(np.float32)


@st.composite
def problems(draw):
    nd = draw(st.sampled_from([2, 3]))
    dtype = draw(st.sampled_from(["f32", "bf16"]))
    row_bytes = draw(st.sampled_from([16, 32, 64, 128]))
    D = row_bytes // (4 if dtype == "f32" else 2)
    L, P = draw(st.sampled_from([(4, 4), (1, 4), (2, 3), (3, 1), (5, 2)]))
    top = 9 if nd == 2 else 5
    shapes = [tuple(draw(st.integers(1, top)) for _ in range(nd)) for _ in range(L)]
    B = draw(st.integers(1, 2))
    Nq = draw(st.integers(1, 90))
    M = draw(st.integers(1, 4))
    seed = draw(st.integers(0, 2**31 - 1))
    inp = workloads.random_problem(nd, shapes, B=B, Nq=Nq, M=M, D=D, P=P, dtype=dtype,
                                   seed=seed)
    rng = np.random.default_rng(seed + 1)
    inp["sampling_locations"] = _edge_coordinates(rng, inp["sampling_locations"], shapes)
    return nd, dtype, inp


@SETTINGS
@given(problems())
def test_drawn_problems_forward_and_backward(msda, problem):
    nd, dtype, inp = problem
    check_forward(msda, nd, inp, dtype, "drawn fwd")
    check_backward(msda, nd, inp, dtype, "drawn bwd")
