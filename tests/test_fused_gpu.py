"""Forward with the module's prologue fused in (msda{2,3}d_forward_fused) against the
oracle composition: fp32 locations from reference points and pixel offsets, a softmax of
the logits over each query-head's L x P samples, then the core.

The GPU's softmax uses expf in fp32 (error a few ulp per weight, relative ~1e-6 after the
sum and division), which stays well inside the forward tolerance (1e-5 relative for fp32
values, 2e-2 absolute for bf16).  The locations are formed with the same two IEEE fp32
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
