"""Locality-aware query order (msda_query_order, msda{2,3}d_forward_ordered,
msda{2,3}d_backward_ordered) on the GPU.

The order is a schedule, not part of the method's arithmetic: the ordered forward must
give exactly the unordered forward's result (bit for bit, every item's arithmetic is the
same), the order must be a permutation of each batch's queries, and it must actually
bring queries with nearby samples together.  The ordered backward gives the plain
backward's location and weight gradients bit for bit (each query's lane group does the
same arithmetic) and its grad_value up to the order of the fp32 reductions.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_parity import (check, device_inputs, grad_value_magnitude, host, run_backward,
                         run_forward)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    import scale_deformable_attention_msda3d_b300 as m
    m.load()
    return m


def _order(msda, dev_inp):
    import torch
    order = msda.msda_query_order(dev_inp["sampling_locations"])
    torch.cuda.synchronize()
    return order


def _forward_ordered(msda, nd, d, order):
    import torch
    fn = msda.msda2d_forward_ordered if nd == 2 else msda.msda3d_forward_ordered
    out = fn(d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
             d["attention_weights"], order)
    torch.cuda.synchronize()
    return out


def _mean_locations(loc):
    """Mean finite sampling location of every query, [B, Nq, ndim] (host, float64)."""
    l64 = loc.astype(np.float64)
    B, Nq = l64.shape[:2]
    flat = l64.reshape(B, Nq, -1, l64.shape[-1])
    fin = np.isfinite(flat).all(-1, keepdims=True)
    s = np.where(fin, flat, 0).sum(2)
    n = fin.sum(2)
    return s / np.maximum(n, 1)


def _is_permutation(order, Nq):
    return all(np.array_equal(np.sort(o), np.arange(Nq)) for o in order)


@pytest.mark.parametrize("name", ["decoder2d", "volume3d", "encoder2d"])
def test_order_is_a_local_permutation_and_keeps_the_result(msda, name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w)
    d = device_inputs(inp, w.dtype)
    order = _order(msda, d)
    o = order.cpu().numpy()
    assert o.shape == (w.B, w.Nq) and o.dtype == np.int32
    assert _is_permutation(o, w.Nq)
    # nearby queries end up next to each other: the mean step between consecutive queries'
    # mean locations shrinks against the given order (random queries) or stays small
    # (queries that already come in raster order)
    mean = _mean_locations(inp["sampling_locations"])
    step_given = np.linalg.norm(np.diff(mean, axis=1), axis=-1).mean()
    reordered = np.take_along_axis(mean, o[..., None].astype(np.int64), axis=1)
    step_ordered = np.linalg.norm(np.diff(reordered, axis=1), axis=-1).mean()
    if w.query_layout == "per_pixel":
        assert step_ordered < 4 * step_given
    else:
        assert step_ordered < 0.25 * step_given, (step_ordered, step_given)
    # the ordered forward is the unordered forward, bit for bit
    plain = host(run_forward(msda, w.ndim, d))
    ordered = host(_forward_ordered(msda, w.ndim, d, order))
    assert np.array_equal(plain, ordered)


@pytest.mark.parametrize("nd,shapes,dtype,D", [
    (2, [(13, 17), (7, 5), (3, 4)], "f32", 32),     # generic (L, P) = (3, 5) path below
    (2, [(13, 17), (7, 5), (3, 4), (1, 2)], "bf16", 32),
    (3, [(5, 6, 7), (3, 2, 4), (1, 3, 2), (2, 2, 2)], "bf16", 32),
    (3, [(5, 6, 7)], "f32", 16),
])
def test_ordered_forward_matches_oracle(msda, nd, shapes, dtype, D):
    P = 5 if len(shapes) == 3 else 4
    inp = workloads.random_problem(nd, shapes, B=3, Nq=211, M=4, D=D, P=P, dtype=dtype,
                                   seed=len(shapes) * 10 + nd, backward=False)
    d = device_inputs(inp, dtype)
    order = _order(msda, d)
    assert _is_permutation(order.cpu().numpy(), 211)
    out = host(_forward_ordered(msda, nd, d, order))
    check(out, oracle.run_inputs(nd, inp), dtype, f"ordered {nd}d {dtype}")


def test_reversed_order_and_non_finite_locations(msda):
    import torch
    inp = workloads.random_problem(2, [(9, 11), (4, 6)], B=2, Nq=77, M=2, D=8, P=4, seed=31,
                                   backward=False)
    inp["sampling_locations"][0, :5] = np.nan            # queries with no finite sample
    d = device_inputs(inp, "f32")
    order = _order(msda, d)
    assert _is_permutation(order.cpu().numpy(), 77)
    # the last bucket takes the queries without a finite sample
    assert set(order.cpu().numpy()[0, -5:].tolist()) == set(range(5))
    rev = torch.arange(76, -1, -1, dtype=torch.int32, device="cuda").repeat(2, 1).contiguous()
    out = host(_forward_ordered(msda, 2, d, rev))
    check(out, oracle.run_inputs(2, inp), "f32", "reversed order")


def test_out_of_range_order_entries_are_clamped(msda):
    import torch
    inp = workloads.random_problem(2, [(9, 11)], B=2, Nq=40, M=2, D=8, P=4, seed=32,
                                   backward=False)
    d = device_inputs(inp, "f32")
    bad = torch.full((2, 40), 1000, dtype=torch.int32, device="cuda")   # clamps to Nq - 1
    bad[:, :20] = -7                                                     # clamps to 0
    out = torch.full((2, 40, 16), 123.0, device="cuda")
    msda.msda2d_forward_ordered(d["value"], d["spatial_shapes"], d["level_start_index"],
                                d["sampling_locations"], d["attention_weights"], bad, out=out)
    torch.cuda.synchronize()
    ref = oracle.run_inputs(2, inp)
    got = host(out)
    # only queries 0 and Nq-1 were computed; every other row is untouched
    check(got[:, [0, 39]], ref[:, [0, 39]], "f32", "clamped order")
    assert np.all(got[:, 1:39] == 123.0)


# ------------------------------------------------------------------ ordered backward


def _backward_ordered(msda, nd, d, order):
    import torch
    fn = msda.msda2d_backward_ordered if nd == 2 else msda.msda3d_backward_ordered
    res = fn(d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
             d["attention_weights"], order, d["grad_out"])
    torch.cuda.synchronize()
    return res


def _check_ordered_backward(msda, nd, inp, dtype, what, order=None):
    d = device_inputs(inp, dtype)
    if order is None:
        order = _order(msda, d)
    gv, gl, ga = _backward_ordered(msda, nd, d, order)
    _, pgl, pga = run_backward(msda, nd, d)
    assert np.array_equal(host(gl), host(pgl)), what
    assert np.array_equal(host(ga), host(pga)), what
    rgv, rgl, rga = oracle.run_inputs(nd, inp, backward_pass=True)
    check(host(gv), rgv, "f32", what + " grad_value", grad_value_magnitude(nd, inp))
    check(host(gl), rgl, "f32", what + " grad_sampling_locations")
    check(host(ga), rga, "f32", what + " grad_attention_weights")


@pytest.mark.parametrize("nd,shapes,dtype,D,P", [
    (2, [(13, 17), (7, 5), (3, 4), (1, 2)], "f32", 32, 4),              # tiled (4, 4)
    (2, [(13, 17), (7, 5), (3, 4)], "bf16", 16, 5),                     # generic (3, 5)
    (3, [(5, 6, 7), (3, 2, 4), (1, 3, 2), (2, 2, 2)], "bf16", 32, 4),   # tiled, 3D
    (3, [(5, 6, 7)], "f32", 16, 4),                                     # tiled (1, 4), 3D
    (3, [(5, 6, 7), (3, 2, 4)], "f32", 8, 3),                           # generic 3D
])
def test_ordered_backward_matches_plain_and_oracle(msda, nd, shapes, dtype, D, P):
    inp = workloads.random_problem(nd, shapes, B=3, Nq=211, M=4, D=D, P=P, dtype=dtype,
                                   seed=100 + len(shapes) * 10 + nd * 3 + P)
    _check_ordered_backward(msda, nd, inp, dtype, f"ordered backward {nd}d {dtype} L{len(shapes)}")


def test_ordered_backward_reversed_order(msda):
    import torch
    inp = workloads.random_problem(2, [(9, 11), (4, 6), (2, 3), (1, 2)], B=2, Nq=77, M=2,
                                   D=32, P=4, seed=33)
    rev = torch.arange(76, -1, -1, dtype=torch.int32, device="cuda").repeat(2, 1).contiguous()
    _check_ordered_backward(msda, 2, inp, "f32", "ordered backward, reversed order", rev)


def test_ordered_backward_volume_full_size(msda):
    """The volume backward (bf16 value, 10 % of the samples out of range) with its queries
    in the locality order: the configuration this entry point is for."""
    w = workloads.WORKLOADS["volume3d_bwd"]
    inp = workloads.make_inputs(w)
    _check_ordered_backward(msda, 3, inp, w.dtype, "ordered volume3d_bwd")


def test_autograd_wrapper_with_a_query_order(msda):
    """ms_deform_attn(..., query_order=...) runs the ordered forward and backward: the same
    output bit for bit, the same location and weight gradients bit for bit, grad_value up
    to the order of its fp32 sums."""
    import torch
    inp = workloads.random_problem(3, [(5, 6, 7), (3, 2, 4), (1, 3, 2), (2, 2, 2)], B=2,
                                   Nq=150, M=8, D=32, P=4, dtype="bf16", seed=41)
    d = device_inputs(inp, "bf16")
    order = _order(msda, d)
    res = []
    for qo in (None, order):
        v = d["value"].detach().clone().requires_grad_(True)
        loc = d["sampling_locations"].detach().clone().requires_grad_(True)
        a = d["attention_weights"].detach().clone().requires_grad_(True)
        out = msda.ms_deform_attn(v, d["spatial_shapes"], d["level_start_index"], loc, a,
                                  query_order=qo)
        out.backward(d["grad_out"])
        torch.cuda.synchronize()
        res.append((host(out), host(v.grad), host(loc.grad), host(a.grad)))
    (o0, gv0, gl0, ga0), (o1, gv1, gl1, ga1) = res
    assert np.array_equal(o0, o1)
    assert np.array_equal(gl0, gl1) and np.array_equal(ga0, ga1)
    rgv, _, _ = oracle.run_inputs(3, inp, backward_pass=True)
    # value's gradient comes back in value's dtype (bf16: the fp32 sum rounded once)
    check(gv1, rgv, "bf16", "autograd ordered grad_value", grad_value_magnitude(3, inp))
