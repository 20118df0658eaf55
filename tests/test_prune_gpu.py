"""Probability-aware pruning (msda{2,3}d_forward_pruned) on the GPU against the oracle.

threshold = 0 must reproduce the exact forward bit for bit; a positive threshold must
match the oracle that drops the same samples (forward_pruned), and stay within the stated
bound of the exact result; a threshold above every weight gives an all-zero output.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_parity import check, device_inputs, host, run_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    import scale_deformable_attention_msda3d_b300 as m
    m.load()
    return m


def _pruned(msda, nd, d, tau):
    import torch
    fn = msda.msda2d_forward_pruned if nd == 2 else msda.msda3d_forward_pruned
    out = fn(d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
             d["attention_weights"], tau)
    torch.cuda.synchronize()
    return host(out)


def _args(nd, inp):
    return (nd, inp["value"], inp["spatial_shapes"], inp["level_start_index"],
            inp["sampling_locations"], inp["attention_weights"])


@pytest.mark.parametrize("nd,shapes,dtype,D,P", [
    (2, [(13, 17), (7, 5), (3, 4), (1, 2)], "f32", 32, 4),   # compiled (4, 4)
    (2, [(13, 17), (7, 5), (3, 4)], "bf16", 16, 5),          # generic (3, 5)
    (3, [(5, 6, 7), (3, 2, 4), (1, 3, 2), (2, 2, 2)], "bf16", 32, 4),
    (3, [(5, 6, 7), (3, 2, 4)], "f32", 8, 3),                # generic 3D
])
def test_pruned_forward_matches_oracle_and_bound(msda, nd, shapes, dtype, D, P):
    inp = workloads.random_problem(nd, shapes, B=2, Nq=97, M=4, D=D, P=P, dtype=dtype,
                                   seed=17 + nd + P, backward=False)
    d = device_inputs(inp, dtype)
    exact = host(run_forward(msda, nd, d))
    assert np.array_equal(_pruned(msda, nd, d, 0.0), exact)
    a = _args(nd, inp)
    for tau in (0.02, 0.06):
        got = _pruned(msda, nd, d, tau)
        check(got, oracle.forward_pruned(*a, tau), dtype, f"pruned tau={tau}")
        bound = oracle.pruning_bound(*a, tau)
        # rounding of the GPU result: the fp32 bound, plus half a bf16 ulp when stored in bf16
        slack = 1e-5 * max(1.0, float(np.abs(exact).max()))
        if dtype == "bf16":
            slack = slack + 2.0 ** -8 * np.abs(got)
        assert np.all(np.abs(got - oracle.forward(*a)) <= bound + slack)
    big = 2 * float(np.abs(inp["attention_weights"]).max())
    assert np.all(_pruned(msda, nd, d, big) == 0.0)


def test_pruned_encoder_full_size(msda):
    w = workloads.WORKLOADS["encoder2d"]
    inp = workloads.make_inputs(w)
    d = device_inputs(inp, w.dtype)
    got = _pruned(msda, 2, d, 0.02)
    check(got, oracle.forward_pruned(*_args(2, inp), 0.02), "f32", "encoder2d pruned 0.02")
