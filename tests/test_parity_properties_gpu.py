"""Drawn problems: the CUDA path (libmsda through its C ABI) against the CPU oracle.

hypothesis draws the whole problem: 2D or 3D; fp32 or bf16 value; the lanes per value row
(D * sizeof = 16..128 bytes); the compiled (L, P) pairs (4, 4) and (1, 4) or another pair,
which takes the generic kernels; level extents from 1 pixel up; B, Nq and M.  Then about
half of the pixel coordinates are moved onto the places where the sampling rule changes:
pixel centres (a corner weight is exactly 0 or 1), the zero-padding boundaries -1 and
extent (the sample just stops contributing), and the half-pixel bands next to them (only
some corners exist).  Forward and backward must match the oracle within the fp32 / bf16
tolerances of ``gpu_parity``.  A second test draws fused-prologue problems (reference
points, offsets, logits) and checks the fused forward and backward against the oracle's
fused composition.  Runs are derandomised, so a failure reproduces.
"""
from __future__ import annotations

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
import workloads  # noqa: E402
from gpu_parity import check, check_backward, check_forward, host  # noqa: E402

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


@st.composite
def fused_problems(draw):
    nd = draw(st.sampled_from([2, 3]))
    dtype = draw(st.sampled_from(["f32", "bf16"]))
    row_bytes = draw(st.sampled_from([16, 32, 64, 128]))
    D = row_bytes // (4 if dtype == "f32" else 2)
    L, P = draw(st.sampled_from([(4, 4), (1, 4), (2, 3), (3, 1)]))
    top = 9 if nd == 2 else 5
    shapes = tuple(tuple(draw(st.integers(1, top)) for _ in range(nd)) for _ in range(L))
    B, Nq, M = draw(st.integers(1, 2)), draw(st.integers(1, 60)), draw(st.integers(1, 4))
    seed = draw(st.integers(0, 2**31 - 1))
    w = workloads.Workload("drawn", nd, B, shapes, Nq, M, D, P, dtype, seed % 100000,
                           query_layout="uniform", offset_std_px=draw(st.sampled_from([0.5, 3.0])))
    f = workloads.make_fused_inputs(w)
    rng = np.random.default_rng(seed)
    # some items with far-apart logits, some references outside [0, 1]
    f["attention_logits"] *= rng.choice([1.0, 6.0], size=f["attention_logits"].shape[:3])[..., None, None]
    f["reference_points"] += rng.choice([0.0, 0.6, -0.6], size=f["reference_points"].shape).astype(np.float32)
    g = rng.standard_normal((B, Nq, M * D), dtype=np.float32)
    bits = None
    if dtype == "bf16":
        bits = workloads.f32_to_bf16_bits(g)
        g = workloads.bf16_bits_to_f32(bits)
    return nd, dtype, f, g, bits


@SETTINGS
@given(fused_problems())
def test_drawn_fused_problems_forward_and_backward(msda, problem):
    """The fused-prologue forward and backward on drawn problems, compiled and generic
    (L, P) pairs, against oracle.forward_fused / oracle.backward_fused."""
    import torch
    nd, dtype, f, g, bits = problem
    dev = torch.device("cuda", 0)
    value = (torch.from_numpy(f["value_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
             if dtype == "bf16" else torch.from_numpy(f["value"]).to(dev))
    ref = torch.from_numpy(f["reference_points"]).to(dev)
    off = torch.from_numpy(f["sampling_offsets"]).to(dev)
    z = torch.from_numpy(f["attention_logits"]).to(dev)
    go = (torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16) if dtype == "bf16"
          else torch.from_numpy(g).to(dev))
    sh, ls = f["spatial_shapes"], f["level_start_index"]
    fwd = msda.msda2d_forward_fused if nd == 2 else msda.msda3d_forward_fused
    bwd = msda.msda2d_backward_fused if nd == 2 else msda.msda3d_backward_fused
    out = fwd(value, sh, ls, ref, off, z)
    gv, goff, gz, gref = bwd(value, sh, ls, ref, off, z, go)
    torch.cuda.synchronize()
    args = (nd, f["value"], sh, ls)
    pro = (f["reference_points"], f["sampling_offsets"], f["attention_logits"])
    check(host(out), oracle.forward_fused(*args, *pro), dtype, "drawn fused fwd")
    rgv, rgoff, rgz, rgref = oracle.backward_fused(*args, *pro, g)
    loc = oracle.fused_locations(sh, f["reference_points"], f["sampling_offsets"])
    a = oracle.softmax_weights(f["attention_logits"])
    mag_v, _, _ = oracle.backward(*args, loc, a, np.abs(g))
    _, gl, _ = oracle.backward(*args, loc, a, g)
    # the gradients are fp32 results, whatever the value dtype
    check(host(gv), rgv, "f32", "drawn fused grad_value", mag_v)
    check(host(goff), rgoff, "f32", "drawn fused grad_offsets")
    check(host(gz), rgz, "f32", "drawn fused grad_logits")
    check(host(gref), rgref, "f32", "drawn fused grad_ref", np.abs(gl).sum(axis=(2, 4)))
