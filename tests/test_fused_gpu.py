"""Forward with the module's prologue fused in (msda{2,3}d_forward_fused) against the
oracle composition: fp32 locations from reference points and pixel offsets, a softmax of
the logits over each query-head's L x P samples, then the core.

The GPU's softmax uses expf in fp32 (error a few ulp per weight, relative ~1e-6 after the
sum and division), which stays well inside the forward tolerance (1e-5 relative for an fp32
result, plus half a bf16 ulp for a result stored in bf16).  The locations are formed with the same two IEEE fp32
operations on both sides.
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads
from gpu_parity import check, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    import scale_deformable_attention_msda3d_b300 as m
    m.load()
    return m


def _device(f, dtype):
    import torch
    dev = torch.device("cuda", 0)
    if dtype == "bf16":
        value = torch.from_numpy(f["value_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        value = torch.from_numpy(np.ascontiguousarray(f["value"])).to(dev)
    return dict(value=value,
                ref=torch.from_numpy(f["reference_points"]).to(dev),
                off=torch.from_numpy(f["sampling_offsets"]).to(dev),
                logits=torch.from_numpy(f["attention_logits"]).to(dev))


def _run(msda, nd, f, dtype):
    import torch
    d = _device(f, dtype)
    fn = msda.msda2d_forward_fused if nd == 2 else msda.msda3d_forward_fused
    out = fn(d["value"], f["spatial_shapes"], f["level_start_index"], d["ref"], d["off"],
             d["logits"])
    torch.cuda.synchronize()
    return host(out)


def _want(nd, f):
    return oracle.forward_fused(nd, f["value"], f["spatial_shapes"], f["level_start_index"],
                                f["reference_points"], f["sampling_offsets"],
                                f["attention_logits"])


@pytest.mark.parametrize("name", ["encoder2d", "decoder2d", "volume3d", "tiny2d"])
def test_fused_named_workloads_full_size(msda, name):
    w = workloads.WORKLOADS[name]
    f = workloads.make_fused_inputs(w)
    check(_run(msda, w.ndim, f, w.dtype), _want(w.ndim, f), w.dtype, f"fused {name}")


CASES = [
    # nd, dtype, D, shapes, P, B, Nq, M
    (2, "f32", 32, [(13, 17), (7, 5), (3, 4), (1, 2)], 4, 2, 129, 8),   # compiled, G=8
    (2, "f32", 8, [(13, 17)], 4, 1, 257, 2),                            # compiled (1, 4), G=2
    (2, "bf16", 32, [(13, 17), (7, 5), (3, 4), (1, 2)], 4, 1, 40, 8),   # few items: SPLIT
    (2, "f32", 16, [(13, 17), (7, 5), (3, 4)], 5, 2, 77, 3),            # generic (3, 5)
    (3, "bf16", 32, [(5, 6, 7), (3, 2, 4), (1, 3, 2), (2, 2, 2)], 4, 1, 300, 8),
    (3, "f32", 32, [(5, 6, 7), (3, 2, 4), (1, 3, 2), (2, 2, 2)], 4, 2, 65, 4),
    (3, "f32", 8, [(5, 6, 7), (3, 2, 4)], 3, 1, 90, 2),                 # generic 3D
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}d-{c[1]}-D{c[2]}-L{len(c[3])}-P{c[4]}"
                                             for c in CASES])
def test_fused_shapes(msda, case):
    nd, dtype, D, shapes, P, B, Nq, M = case
    w = workloads.Workload("case", nd, B, tuple(tuple(s) for s in shapes), Nq, M, D, P, dtype,
                           zlib.crc32(repr(case).encode()) % 100000,
                           query_layout="uniform", offset_std_px=2.0)
    f = workloads.make_fused_inputs(w)
    # a few logits far apart and a few references outside [0, 1]
    f["attention_logits"][0, :3] *= 8.0
    f["reference_points"][0, 3:6] += 0.7
    check(_run(msda, nd, f, dtype), _want(nd, f), dtype, f"fused {case}")


# ------------------------------------------------------------------ fused backward
#
# msda{2,3}d_backward_fused against oracle.backward_fused (the core's double backward at
# the fused locations and weights, chained through location = ref + offset / extent and
# the softmax).  grad_value and grad_reference_points are sums of many terms: their fp32
# bound is taken against the magnitude sum of those terms, as for the core backward.


def _grad_out(w, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((w.B, w.Nq, w.M * w.D), dtype=np.float32)
    if w.dtype == "bf16":
        bits = workloads.f32_to_bf16_bits(g)
        return workloads.bf16_bits_to_f32(bits), bits
    return g, None


def _run_bwd(msda, nd, f, g, g_bits, dtype, need_ref=True):
    import torch
    d = _device(f, dtype)
    dev = d["value"].device
    go = (torch.from_numpy(g_bits.view(np.int16)).to(dev).view(torch.bfloat16)
          if dtype == "bf16" else torch.from_numpy(g).to(dev))
    fn = msda.msda2d_backward_fused if nd == 2 else msda.msda3d_backward_fused
    res = fn(d["value"], f["spatial_shapes"], f["level_start_index"], d["ref"], d["off"],
             d["logits"], go, need_reference_grad=need_ref)
    torch.cuda.synchronize()
    return [None if r is None else host(r) for r in res]


def _check_bwd(msda, nd, f, w, what):
    g, g_bits = _grad_out(w, w.seed + 17)
    gv, goff, gz, gref = _run_bwd(msda, nd, f, g, g_bits, w.dtype)
    args = (nd, f["value"], f["spatial_shapes"], f["level_start_index"])
    rgv, rgoff, rgz, rgref = oracle.backward_fused(*args, f["reference_points"],
                                                   f["sampling_offsets"],
                                                   f["attention_logits"], g)
    loc = oracle.fused_locations(f["spatial_shapes"], f["reference_points"],
                                 f["sampling_offsets"])
    a = oracle.softmax_weights(f["attention_logits"])
    mag_v, _, _ = oracle.backward(*args, loc, a, np.abs(g))
    _, gl_abs, _ = oracle.backward(*args, loc, a, g)
    # all four gradients are fp32 results, whatever the value dtype
    check(gv, rgv, "f32", what + " grad_value", mag_v)
    check(goff, rgoff, "f32", what + " grad_sampling_offsets")
    check(gz, rgz, "f32", what + " grad_attention_logits")
    check(gref, rgref, "f32", what + " grad_reference_points",
          np.abs(gl_abs).sum(axis=(2, 4)))
    # the logit gradients of every (query, head) sum to zero (softmax shift invariance)
    s = gz.reshape(gz.shape[:3] + (-1,)).sum(-1)
    assert np.abs(s).max() <= 1e-4 * (1.0 + np.abs(gz).max())


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}d-{c[1]}-D{c[2]}-L{len(c[3])}-P{c[4]}"
                                             for c in CASES])
def test_fused_backward_shapes(msda, case):
    nd, dtype, D, shapes, P, B, Nq, M = case
    w = workloads.Workload("case", nd, B, tuple(tuple(s) for s in shapes), Nq, M, D, P, dtype,
                           zlib.crc32(repr(case).encode()) % 100000,
                           query_layout="uniform", offset_std_px=2.0)
    f = workloads.make_fused_inputs(w)
    f["attention_logits"][0, :3] *= 8.0
    f["reference_points"][0, 3:6] += 0.7
    _check_bwd(msda, nd, f, w, f"fused bwd {case}")


@pytest.mark.parametrize("name", ["encoder2d", "volume3d"])
def test_fused_backward_full_size(msda, name):
    w = workloads.WORKLOADS[name]
    f = workloads.make_fused_inputs(w)
    _check_bwd(msda, w.ndim, f, w, f"fused bwd {name}")


def test_fused_backward_without_reference_gradient(msda):
    """grad_reference_points = NULL skips that output; the others are unchanged."""
    case = CASES[0]
    nd, dtype, D, shapes, P, B, Nq, M = case
    w = workloads.Workload("case", nd, B, tuple(tuple(s) for s in shapes), Nq, M, D, P, dtype,
                           123, query_layout="uniform", offset_std_px=2.0)
    f = workloads.make_fused_inputs(w)
    g, g_bits = _grad_out(w, 5)
    with_ref = _run_bwd(msda, nd, f, g, g_bits, dtype, need_ref=True)
    without = _run_bwd(msda, nd, f, g, g_bits, dtype, need_ref=False)
    assert without[3] is None
    # offsets and logits are written without atomics: identical; grad_value up to the
    # order of its atomic additions
    assert np.array_equal(with_ref[1], without[1]) and np.array_equal(with_ref[2], without[2])
    check(without[0], with_ref[0], "f32", "grad_value with / without the reference gradient")


def test_fused_autograd_wrapper(msda):
    """ms_deform_attn_fused: forward equals the fused call, and its gradients are the fused
    backward's (value, reference points, offsets, logits)."""
    import torch
    case = CASES[4]                                            # 3D bf16, compiled (4, 4)
    nd, dtype, D, shapes, P, B, Nq, M = case
    w = workloads.Workload("case", nd, B, tuple(tuple(s) for s in shapes), Nq, M, D, P, dtype,
                           321, query_layout="uniform", offset_std_px=2.0)
    f = workloads.make_fused_inputs(w)
    d = _device(f, dtype)
    for k in ("value", "ref", "off", "logits"):
        d[k].requires_grad_(True)
    out = msda.ms_deform_attn_fused(d["value"], f["spatial_shapes"], f["level_start_index"],
                                    d["ref"], d["off"], d["logits"])
    g, g_bits = _grad_out(w, 9)
    go = torch.from_numpy(g_bits.view(np.int16)).to(out.device).view(torch.bfloat16)
    out.backward(go)
    torch.cuda.synchronize()
    check(host(out), _want(nd, f), dtype, "autograd fused forward")
    rgv, rgoff, rgz, rgref = oracle.backward_fused(nd, f["value"], f["spatial_shapes"],
                                                   f["level_start_index"],
                                                   f["reference_points"],
                                                   f["sampling_offsets"],
                                                   f["attention_logits"], g)
    loc = oracle.fused_locations(f["spatial_shapes"], f["reference_points"],
                                 f["sampling_offsets"])
    a = oracle.softmax_weights(f["attention_logits"])
    args = (nd, f["value"], f["spatial_shapes"], f["level_start_index"])
    mag_v, _, _ = oracle.backward(*args, loc, a, np.abs(g))
    _, gl, _ = oracle.backward(*args, loc, a, g)
    # value's gradient comes back in value's dtype (bf16: the fp32 sum rounded once); the
    # others are fp32
    assert d["value"].grad.dtype == torch.bfloat16
    check(host(d["value"].grad), rgv, "bf16", "autograd fused grad_value", mag_v)
    check(host(d["off"].grad), rgoff, "f32", "autograd fused grad_offsets")
    check(host(d["logits"].grad), rgz, "f32", "autograd fused grad_logits")
    check(host(d["ref"].grad), rgref, "f32", "autograd fused grad_ref",
          np.abs(gl).sum(axis=(2, 4)))
