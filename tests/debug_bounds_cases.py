"""Cases run against the bounds-checking build (libmsda_debug.so) in a child process that
selects it with MSDA_LIBRARY (see tests/test_debug_bounds_gpu.py).  Every call must give
the oracle's result within the usual tolerances and leave the bounds-check record empty;
the self-test must come back as MSDA_ERR_INTERNAL naming its made-up offender."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
import workloads  # noqa: E402
from gpu_parity import check, check_backward, check_forward, device_inputs, host  # noqa: E402


def main():
    import torch
    import scale_deformable_attention_msda3d_b300 as msda
    lib = msda.load()
    assert os.environ["MSDA_LIBRARY"].endswith("libmsda_debug.so")
    assert msda.msda_build_flags() == msda.MSDA_BUILD_DEBUG_BOUNDS
    assert msda.msda_debug_bounds_status() == msda.MSDA_OK, msda.msda_last_error()

    def clean(what):
        st = msda.msda_debug_bounds_status()
        assert st == msda.MSDA_OK, (what, msda.msda_last_error())

    shapes2 = [(9, 11), (5, 6), (3, 3), (1, 2)]
    shapes3 = [(4, 5, 6), (2, 3, 3), (1, 2, 2), (1, 1, 1)]
    n = 0
    for nd, shapes in ((2, shapes2), (3, shapes3)):
        for dtype, D in (("f32", 32), ("bf16", 32), ("f32", 8)):
            for L, P in ((4, 4), (1, 4), (3, 5)):
                inp = workloads.random_problem(nd, shapes[:L], B=2, Nq=37, M=3, D=D, P=P,
                                               dtype=dtype, seed=400 + n)
                check_forward(msda, nd, inp, dtype, f"debug fwd {nd}d {dtype} L{L} P{P}")
                clean("forward")
                check_backward(msda, nd, inp, dtype, f"debug bwd {nd}d {dtype} L{L} P{P}")
                clean("backward")
                n += 1
    # pruned, ordered and fused forms go through the same checks
    w = workloads.WORKLOADS["tiny2d"]
    inp = workloads.make_inputs(w)
    d = device_inputs(inp, "f32")
    a = (d["value"], inp["spatial_shapes"], inp["level_start_index"], d["sampling_locations"],
         d["attention_weights"])
    out = msda.msda2d_forward_pruned(*a, 0.05)
    torch.cuda.synchronize()
    args = (2, inp["value"], inp["spatial_shapes"], inp["level_start_index"],
            inp["sampling_locations"], inp["attention_weights"])
    check(host(out), oracle.forward_pruned(*args, 0.05), "f32", "debug pruned")
    clean("pruned")
    order = msda.msda_query_order(d["sampling_locations"])
    out = msda.msda2d_forward_ordered(*a, order)
    torch.cuda.synchronize()
    check(host(out), oracle.forward(*args), "f32", "debug ordered")
    clean("ordered")
    wf = workloads.Workload("case", 3, 1, tuple(shapes3), 29, 2, 16, 4, "bf16", 77,
                            query_layout="uniform", offset_std_px=2.0)
    f = workloads.make_fused_inputs(wf)
    dev = torch.device("cuda", 0)
    value = torch.from_numpy(f["value_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    ref = torch.from_numpy(f["reference_points"]).to(dev)
    off = torch.from_numpy(f["sampling_offsets"]).to(dev)
    z = torch.from_numpy(f["attention_logits"]).to(dev)
    out = msda.msda3d_forward_fused(value, f["spatial_shapes"], f["level_start_index"], ref, off, z)
    g = torch.ones_like(out)
    res = msda.msda3d_backward_fused(value, f["spatial_shapes"], f["level_start_index"], ref, off,
                                     z, g)
    torch.cuda.synchronize()
    fa = (3, f["value"], f["spatial_shapes"], f["level_start_index"])
    pro = (f["reference_points"], f["sampling_offsets"], f["attention_logits"])
    check(host(out), oracle.forward_fused(*fa, *pro), "bf16", "debug fused fwd")
    rgv = oracle.backward_fused(*fa, *pro, np.ones((1, 29, 32)))[0]
    loc = oracle.fused_locations(f["spatial_shapes"], *pro[:2])
    mag = oracle.backward(*fa, loc, oracle.softmax_weights(pro[2]), np.ones((1, 29, 32)))[0]
    check(host(res[0]), rgv, "f32", "debug fused grad_value", mag)
    clean("fused")

    # the reporting path, on a made-up offender recorded by the kernels' own check
    assert msda.msda_debug_bounds_selftest(0) == msda.MSDA_OK, msda.msda_last_error()
    st = msda.msda_debug_bounds_status()
    msg = msda.msda_last_error()
    assert st == msda.MSDA_ERR_INTERNAL, (st, msg)
    assert "row -5 outside [0, 10)" in msg and "batch 1, query 2, head 1, level 1, point 1" in msg, msg
    clean("after the self-test report")     # the status call cleared the record
    print(f"debug bounds: {n} core cases + pruned, ordered, fused; self-test reported")


if __name__ == "__main__":
    main()
