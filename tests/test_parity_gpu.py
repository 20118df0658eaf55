"""CUDA path (libmsda through its C ABI) against the CPU oracle, element by element.

Full-size runs of the five named workloads use the same binding call, kernels and launch
configuration as bench.py.  Smaller cases cover every lane-group width (G = 1..32 lanes per
row), the compiled (L, P) = (4, 4) / (1, 4) paths and the generic path, ragged tails
(item counts that are not multiples of the warp / block tile), the largest L and P, and
the edge cases: empty calls, a single query, exact gathers, non-finite and out-of-range
locations, a non-default stream and the autograd wrapper.
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads
from gpu_parity import (check, check_backward, check_forward, device_inputs,
                        grad_value_magnitude, host, run_backward, run_forward)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    import scale_deformable_attention_msda3d_b300 as m
    m.load()
    return m


def _named(name):
    w = workloads.WORKLOADS[name]
    return w, workloads.make_inputs(w)


# ------------------------------------------------------------------ the named workloads


def test_tiny2d_forward(msda):
    w, inp = _named("tiny2d")
    check_forward(msda, 2, inp, w.dtype, "tiny2d")


def test_encoder2d_forward_full_size(msda):
    w, inp = _named("encoder2d")
    check_forward(msda, 2, inp, w.dtype, "encoder2d")


def test_decoder2d_forward_bf16_full_size(msda):
    w, inp = _named("decoder2d")
    check_forward(msda, 2, inp, w.dtype, "decoder2d")


def test_volume3d_forward_bf16_full_size(msda):
    w, inp = _named("volume3d")
    check_forward(msda, 3, inp, w.dtype, "volume3d")


def test_encoder2d_backward_full_size(msda):
    w, inp = _named("encoder2d_bwd")
    check_backward(msda, 2, inp, w.dtype, "encoder2d_bwd")


def test_encoder2d_backward_adjoint_identities(msda):
    """sum(g * out) = sum(value * grad_value) = sum(A * grad_A), all from the GPU."""
    w, inp = _named("encoder2d_bwd")
    dev = device_inputs(inp, w.dtype)
    out = host(run_forward(msda, 2, dev))
    gv, gl, ga = (host(t) for t in run_backward(msda, 2, dev))
    s_out = float((out * inp["grad_out"]).sum())
    s_val = float((inp["value"].astype(np.float64) * gv).sum())
    s_att = float((inp["attention_weights"].astype(np.float64) * ga).sum())
    scale = float(np.abs(out * inp["grad_out"]).sum())
    assert abs(s_out - s_val) <= 1e-5 * scale and abs(s_out - s_att) <= 1e-5 * scale


def test_volume3d_backward_bf16_full_size(msda):
    w, inp = _named("volume3d")
    w = w.with_(backward=True)
    inp = workloads.make_inputs(w)
    check_backward(msda, 3, inp, w.dtype, "volume3d_bwd")


# ------------------------------------------------------------------ coverage of shapes

SHAPES2 = [(13, 17), (7, 5), (3, 4), (1, 2)]
SHAPES3 = [(5, 6, 7), (3, 2, 4), (1, 3, 2)]

CASES = [
    # nd, dtype, D, L, P, B, Nq, M          (G = D * sizeof / 16)
    (2, "f32", 4, 3, 5, 2, 1001, 3),        # G=1, generic (L, P)
    (2, "f32", 8, 1, 4, 1, 257, 2),         # G=2, compiled (1, 4)
    (2, "f32", 16, 4, 4, 2, 129, 5),        # G=4, compiled (4, 4)
    (2, "f32", 32, 4, 4, 1, 77, 8),         # G=8, compiled (4, 4), ragged
    (2, "f32", 64, 2, 3, 1, 45, 3),         # G=16
    (2, "f32", 128, 1, 4, 2, 19, 2),        # G=32
    (2, "bf16", 8, 4, 4, 2, 301, 3),        # G=1
    (2, "bf16", 16, 2, 2, 1, 99, 4),        # G=2
    (2, "bf16", 32, 4, 4, 3, 50, 8),        # G=4
    (2, "bf16", 64, 1, 4, 1, 33, 2),        # G=8
    (2, "bf16", 256, 2, 1, 1, 21, 1),       # G=32
    (3, "f32", 16, 3, 3, 2, 201, 3),        # G=4, generic
    (3, "f32", 32, 4, 4, 1, 65, 4),         # G=8, compiled (4, 4) -- 3D uses 4 levels
    (3, "bf16", 32, 4, 4, 2, 130, 8),       # G=4
    (3, "bf16", 8, 1, 4, 1, 97, 2),         # G=1, compiled (1, 4)
    (3, "f32", 128, 2, 2, 1, 9, 1),         # G=32
]


def _shapes_for(nd, L):
    base = SHAPES2 if nd == 2 else SHAPES3
    return [base[i % len(base)] for i in range(L)]


@pytest.mark.parametrize("case", CASES, ids=[
    f"{c[0]}d-{c[1]}-D{c[2]}-L{c[3]}-P{c[4]}-B{c[5]}-Nq{c[6]}-M{c[7]}" for c in CASES])
def test_forward_and_backward_shapes(msda, case):
    nd, dtype, D, L, P, B, Nq, M = case
    inp = workloads.random_problem(nd, _shapes_for(nd, L), B=B, Nq=Nq, M=M, D=D, P=P,
                                   dtype=dtype, seed=zlib.crc32(repr(case).encode()))
    check_forward(msda, nd, inp, dtype, f"fwd {case}")
    check_backward(msda, nd, inp, dtype, f"bwd {case}")


def test_maximum_levels_and_points(msda):
    shapes = [(3 + (l % 4), 2 + (l % 3)) for l in range(16)]
    inp = workloads.random_problem(2, shapes, B=1, Nq=33, M=2, D=8, P=32, seed=5)
    check_forward(msda, 2, inp, "f32", "L16 P32 fwd")
    check_backward(msda, 2, inp, "f32", "L16 P32 bwd")


def test_maximum_channels(msda):
    inp = workloads.random_problem(2, [(9, 11)], B=1, Nq=40, M=1, D=256, P=4, dtype="bf16",
                                   seed=6)
    check_forward(msda, 2, inp, "bf16", "bf16 D=256")
    inp = workloads.random_problem(3, [(3, 4, 5)], B=1, Nq=40, M=2, D=128, P=4, seed=7)
    check_forward(msda, 3, inp, "f32", "3d f32 D=128")


@pytest.mark.parametrize("nd,shape", [(2, (1, (1 << 23) - 1)), (3, ((1 << 23) - 1, 1, 2))],
                         ids=["2d-W=2^23-1", "3d-Z=2^23-1"])
def test_maximum_extents(msda, nd, shape):
    """The largest extent the ABI accepts along one axis, 2^23 - 1 (2D: an 8.4 M-pixel row;
    3D: as many slices): fp32 locations then resolve about half a pixel, and the cell is
    still decided from the exact coordinate loc * extent - 0.5 on both sides.  Row indices
    reach 2^23 and more, and the samples spread over the whole long axis."""
    inp = workloads.random_problem(nd, [shape], B=1, Nq=48, M=1, D=4, P=4, seed=8,
                                   margin=0.0)
    check_forward(msda, nd, inp, "f32", f"max extent {shape} fwd")
    check_backward(msda, nd, inp, "f32", f"max extent {shape} bwd")


def test_value_tensor_beyond_2gb(msda):
    """A value tensor past 2^31 bytes (one 11600 x 11600 level, 16-byte rows: 2.15 GB) with
    samples spread over all of it, so that about half of the corner rows sit beyond byte
    offset 2^31: the 64-bit address arithmetic of the forward and backward."""
    inp = workloads.random_problem(2, [(11600, 11600)], B=1, Nq=48, M=1, D=4, P=4, seed=9,
                                   margin=0.0)
    assert inp["value"].nbytes > 2 ** 31
    check_forward(msda, 2, inp, "f32", "2.15 GB value fwd")
    check_backward(msda, 2, inp, "f32", "2.15 GB value bwd")


# ------------------------------------------------------------------ edge cases


def test_exact_gather_is_bit_exact(msda):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    H = W = 16
    B, Nq, M, D, P = 1, 300, 4, 32, 4
    value = rng.standard_normal((B, H * W, M, D), dtype=np.float32)
    ix = rng.integers(0, W, size=(B, Nq, M, 1, P))
    iy = rng.integers(0, H, size=(B, Nq, M, 1, P))
    loc = np.stack([(ix + 0.5) / W, (iy + 0.5) / H], -1).astype(np.float32)
    attn = np.zeros((B, Nq, M, 1, P), dtype=np.float32)
    attn[..., 1] = 1.0
    inp = dict(value=value, spatial_shapes=np.array([[H, W]]), level_start_index=np.array([0]),
               sampling_locations=loc, attention_weights=attn)
    out = host(run_forward(msda, 2, device_inputs(inp, "f32"))).reshape(Nq, M, D)
    rows = (iy[0, :, :, 0, 1] * W + ix[0, :, :, 0, 1])
    want = np.stack([value[0, rows[:, m], m] for m in range(M)], 1)
    assert np.array_equal(out, want.astype(np.float64))


@pytest.mark.parametrize("nd", [2, 3])
def test_non_finite_and_out_of_range_locations(msda, nd):
    shapes = _shapes_for(nd, 2)
    inp = workloads.random_problem(nd, shapes, B=1, Nq=64, M=2, D=8, P=4, seed=12)
    loc = inp["sampling_locations"]
    specials = [np.nan, np.inf, -np.inf, 3.0e38, -3.0e38, -0.75, 1.75, 0.0, 1.0]
    for i, v in enumerate(specials):
        loc[0, i, :, :, :, i % nd] = v
    check_forward(msda, nd, inp, "f32", f"{nd}d specials fwd")
    check_backward(msda, nd, inp, "f32", f"{nd}d specials bwd")
    ref = oracle.run_inputs(nd, inp)
    assert np.all(ref[0, 0:3] == 0.0)


def test_empty_calls(msda):
    torch = pytest.importorskip("torch")
    inp = workloads.random_problem(2, SHAPES2[:2], B=2, Nq=0, M=2, D=8, P=4, seed=13)
    dev = device_inputs(inp, "f32")
    out = run_forward(msda, 2, dev)
    assert tuple(out.shape) == (2, 0, 16)
    gv = torch.full(tuple(dev["value"].shape), 7.0, device="cuda")
    gv, gl, ga = msda.msda2d_backward(dev["value"], inp["spatial_shapes"],
                                      inp["level_start_index"], dev["sampling_locations"],
                                      dev["attention_weights"], dev["grad_out"], grad_value=gv)
    torch.cuda.synchronize()
    assert float(gv.abs().max()) == 0.0          # no queries: the value gradient is zero


def test_single_query_single_head(msda):
    inp = workloads.random_problem(2, SHAPES2, B=1, Nq=1, M=1, D=32, P=4, seed=14)
    check_forward(msda, 2, inp, "f32", "1 query")
    check_backward(msda, 2, inp, "f32", "1 query")


def test_non_default_stream(msda):
    torch = pytest.importorskip("torch")
    inp = workloads.random_problem(2, SHAPES2, B=2, Nq=500, M=4, D=32, P=4, seed=15)
    dev = device_inputs(inp, "f32")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = msda.msda2d_forward(dev["value"], inp["spatial_shapes"],
                                  inp["level_start_index"], dev["sampling_locations"],
                                  dev["attention_weights"])
    s.synchronize()
    check(host(out), oracle.run_inputs(2, inp), "f32", "side stream")


def test_cuda_graph_capture_and_replay(msda):
    """The calls enqueue plain kernel launches on the given stream and allocate nothing, so
    a CUDA graph can capture them: replaying a captured forward + backward on new inputs
    (copied into the captured buffers) matches the oracle on those inputs."""
    torch = pytest.importorskip("torch")
    first = workloads.random_problem(3, SHAPES3, B=1, Nq=90, M=4, D=32, P=4, seed=21)
    second = workloads.random_problem(3, SHAPES3, B=1, Nq=90, M=4, D=32, P=4, seed=22)
    dev = device_inputs(first, "f32")
    out = torch.empty((1, 90, 4 * 32), dtype=torch.float32, device=dev["value"].device)
    gv = torch.empty_like(dev["value"])
    gl = torch.empty_like(dev["sampling_locations"])
    ga = torch.empty_like(dev["attention_weights"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    args = (dev["value"], first["spatial_shapes"], first["level_start_index"],
            dev["sampling_locations"], dev["attention_weights"])
    with torch.cuda.stream(s):                       # warm-up outside the capture
        msda.msda3d_forward(*args, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        msda.msda3d_forward(*args, out=out, stream=s)
        msda.msda3d_backward(*args, dev["grad_out"], grad_value=gv, grad_sampling_locations=gl,
                             grad_attention_weights=ga, stream=s)
        g.capture_end()
    new = device_inputs(second, "f32")
    for k in ("value", "sampling_locations", "attention_weights", "grad_out"):
        dev[k].copy_(new[k])
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    check(host(out), oracle.run_inputs(3, second), "f32", "graph replay forward")
    rgv, rgl, rga = oracle.run_inputs(3, second, backward_pass=True)
    check(host(gv), rgv, "f32", "graph replay grad_value", grad_value_magnitude(3, second))
    check(host(gl), rgl, "f32", "graph replay grad_loc")
    check(host(ga), rga, "f32", "graph replay grad_attn")


def test_concurrent_streams(msda):
    """Independent calls on four streams at once (different problems, 2D and 3D, both
    dtypes) each match the oracle: the calls share no state on the device."""
    torch = pytest.importorskip("torch")
    cases = [(2, "f32", 31), (3, "bf16", 32), (2, "bf16", 33), (3, "f32", 34)]
    streams = [torch.cuda.Stream() for _ in cases]
    runs = []
    for (nd, dtype, seed), st in zip(cases, streams):
        inp = workloads.random_problem(nd, SHAPES2 if nd == 2 else SHAPES3, B=2, Nq=300, M=8,
                                       D=32, P=4, dtype=dtype, seed=seed)
        dev = device_inputs(inp, dtype)
        st.wait_stream(torch.cuda.current_stream())
        fwd = msda.msda2d_forward if nd == 2 else msda.msda3d_forward
        bwd = msda.msda2d_backward if nd == 2 else msda.msda3d_backward
        a = (dev["value"], inp["spatial_shapes"], inp["level_start_index"],
             dev["sampling_locations"], dev["attention_weights"])
        with torch.cuda.stream(st):
            out = fwd(*a, stream=st)
            grads = bwd(*a, dev["grad_out"], stream=st)
        runs.append((nd, dtype, inp, out, grads))
    torch.cuda.synchronize()
    for nd, dtype, inp, out, (gv, gl, ga) in runs:
        check(host(out), oracle.run_inputs(nd, inp), dtype, f"stream fwd {nd}d {dtype}")
        rgv, rgl, rga = oracle.run_inputs(nd, inp, backward_pass=True)
        check(host(gv), rgv, "f32", f"stream grad_value {nd}d", grad_value_magnitude(nd, inp))
        check(host(gl), rgl, "f32", f"stream grad_loc {nd}d {dtype}")
        check(host(ga), rga, "f32", f"stream grad_attn {nd}d {dtype}")


def test_autograd_wrapper_matches_backward_call(msda):
    torch = pytest.importorskip("torch")
    inp = workloads.random_problem(2, SHAPES2, B=1, Nq=40, M=2, D=16, P=4, seed=16)
    dev = device_inputs(inp, "f32")
    v = dev["value"].clone().requires_grad_(True)
    loc = dev["sampling_locations"].clone().requires_grad_(True)
    a = dev["attention_weights"].clone().requires_grad_(True)
    out = msda.ms_deform_attn(v, inp["spatial_shapes"], inp["level_start_index"], loc, a)
    (out * dev["grad_out"]).sum().backward()
    rgv, rgl, rga = oracle.run_inputs(2, inp, backward_pass=True)
    check(host(v.grad), rgv, "f32", "autograd grad_value", mag=grad_value_magnitude(2, inp))
    check(host(loc.grad), rgl, "f32", "autograd grad_loc")
    check(host(a.grad), rga, "f32", "autograd grad_attn")


def test_autograd_wrapper_3d_bf16(msda):
    torch = pytest.importorskip("torch")
    inp = workloads.random_problem(3, SHAPES3, B=1, Nq=30, M=2, D=16, P=4, dtype="bf16",
                                   seed=18)
    dev = device_inputs(inp, "bf16")
    v = dev["value"].clone().requires_grad_(True)
    loc = dev["sampling_locations"].clone().requires_grad_(True)
    a = dev["attention_weights"].clone().requires_grad_(True)
    out = msda.ms_deform_attn(v, inp["spatial_shapes"], inp["level_start_index"], loc, a)
    check(host(out), oracle.run_inputs(3, inp), "bf16", "autograd 3d forward")
    (out.float() * dev["grad_out"].float()).sum().backward()
    rgv, rgl, rga = oracle.run_inputs(3, inp, backward_pass=True)
    assert v.grad.dtype == torch.bfloat16          # the gradient comes back in value's dtype
    # value's gradient is the fp32 sum rounded once to bf16; the others are fp32
    check(host(v.grad), rgv, "bf16", "autograd 3d grad_value", grad_value_magnitude(3, inp))
    check(host(loc.grad), rgl, "f32", "autograd 3d grad_loc")
    check(host(a.grad), rga, "f32", "autograd 3d grad_attn")


# ------------------------------------------------------------------ runtime (L, P) path

# (L, P) pairs outside the compiled (4, 4) / (1, 4) with L * P <= 32 take the runtime-(L, P)
# form of the tiled forward (rows of 2 to 16 sixteen-byte lanes): every sample count from 2
# to 32 that the pairs below give, narrow and wide rows, a ragged item count, 2D and 3D.
RT_CASES = [
    # nd, dtype, D, L, P
    (2, "f32", 32, 2, 3), (2, "f32", 32, 3, 5), (2, "f32", 32, 5, 4), (2, "f32", 32, 4, 8),
    (2, "f32", 32, 8, 4), (2, "f32", 32, 2, 16), (2, "f32", 32, 16, 2), (2, "f32", 32, 3, 1),
    (2, "f32", 16, 4, 2), (2, "f32", 8, 1, 8), (2, "f32", 64, 7, 3),
    (2, "bf16", 32, 4, 8), (2, "bf16", 32, 3, 4), (2, "bf16", 64, 2, 5), (2, "bf16", 16, 5, 6),
    (3, "bf16", 32, 4, 8), (3, "bf16", 32, 3, 3), (3, "f32", 16, 2, 4), (3, "f32", 32, 5, 2),
]


@pytest.mark.parametrize("case", RT_CASES, ids=[f"{c[0]}d-{c[1]}-D{c[2]}-L{c[3]}-P{c[4]}"
                                                for c in RT_CASES])
def test_runtime_level_point_forward(msda, case):
    nd, dtype, D, L, P = case
    inp = workloads.random_problem(nd, _shapes_for(nd, L), B=2, Nq=203, M=3, D=D, P=P,
                                   dtype=dtype, seed=zlib.crc32(repr(case).encode()),
                                   backward=False)
    check_forward(msda, nd, inp, dtype, f"runtime (L, P) fwd {case}")


def test_runtime_level_point_forward_modes(msda):
    """The runtime-(L, P) form under pruning, a query order and a non-default stream: the
    same results as the pruning oracle, bit-identical ordered and unordered outputs."""
    torch = pytest.importorskip("torch")
    for nd, dtype, L, P in ((2, "f32", 4, 8), (3, "bf16", 3, 3)):
        inp = workloads.random_problem(nd, _shapes_for(nd, L), B=2, Nq=150, M=4, D=32, P=P,
                                       dtype=dtype, seed=90 + nd, backward=False)
        d = device_inputs(inp, dtype)
        a = (d["value"], inp["spatial_shapes"], inp["level_start_index"],
             d["sampling_locations"], d["attention_weights"])
        fwd = msda.msda2d_forward if nd == 2 else msda.msda3d_forward
        fwd_p = msda.msda2d_forward_pruned if nd == 2 else msda.msda3d_forward_pruned
        fwd_o = msda.msda2d_forward_ordered if nd == 2 else msda.msda3d_forward_ordered
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            plain = fwd(*a, stream=st)
            pruned = fwd_p(*a, 0.05, stream=st)
            order = msda.msda_query_order(d["sampling_locations"], stream=st)
            ordered = fwd_o(*a, order, stream=st)
        torch.cuda.synchronize()
        args = (nd, inp["value"], inp["spatial_shapes"], inp["level_start_index"],
                inp["sampling_locations"], inp["attention_weights"])
        check(host(plain), oracle.forward(*args), dtype, f"runtime (L, P) {nd}d")
        check(host(pruned), oracle.forward_pruned(*args, 0.05), dtype, f"runtime pruned {nd}d")
        assert torch.equal(plain, ordered), f"runtime ordered {nd}d differs from unordered"
