"""Helpers for the GPU parity tests: move seeded inputs to the device, call libmsda
through its binding (the C ABI), run the oracle on the same values, compare.

Tolerances (written here, used by every GPU test).  They depend on how a result is
STORED, not on the dtype of the problem's value tensor: both sides see the same inputs
(bf16 values are widened exactly), so every result is an fp32 computation, and a bf16
result is that fp32 result rounded to nearest even once.

  fp32 results (every gradient, and the forward output of an fp32 problem):
      |gpu - ref| <= e32 = 1e-5 * max(|ref|, rms(ref), mag) per element, where mag is the
      magnitude sum of the terms that make up an accumulated gradient entry (the standard
      forward-error scale of a floating-point sum of those terms).
  bf16 results (the forward output of a bf16 problem, a gradient returned in bf16):
      |gpu - ref| <= 2^-8 * (|ref| + e32) + e32: the fp32 bound plus half a bf16 ulp of
      the fp32 result (half an ulp of x is at most 2^-8 |x| with 8 significant bits).
      This is far tighter than the 2e-2 absolute bar stated for unit-scale bf16 outputs,
      which it implies for |ref| <= 5.
"""
from __future__ import annotations

import numpy as np

import oracle

REL_F32 = 1e-5
HALF_ULP_BF16 = 2.0 ** -8


def torch_mod():
    import torch
    return torch


def device_inputs(inp, dtype):
    torch = torch_mod()
    dev = torch.device("cuda", 0)
    if dtype == "bf16":
        value = torch.from_numpy(inp["value_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        value = torch.from_numpy(np.ascontiguousarray(inp["value"])).to(dev)
    d = dict(value=value,
             spatial_shapes=inp["spatial_shapes"], level_start_index=inp["level_start_index"],
             sampling_locations=torch.from_numpy(inp["sampling_locations"]).to(dev),
             attention_weights=torch.from_numpy(inp["attention_weights"]).to(dev))
    if "grad_out" in inp:
        if dtype == "bf16":
            d["grad_out"] = torch.from_numpy(inp["grad_out_bits"].view(np.int16)).to(dev).view(
                torch.bfloat16)
        else:
            d["grad_out"] = torch.from_numpy(inp["grad_out"]).to(dev)
    return d


def host(t) -> np.ndarray:
    torch = torch_mod()
    if t.dtype == torch.bfloat16:
        return (t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32)
                << 16).view(np.float32).astype(np.float64)
    return t.detach().cpu().numpy().astype(np.float64)


def check(gpu, ref, stored, what, mag=None):
    """Element-wise comparison; `stored` is the dtype the result is stored in ("f32" or
    "bf16")."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu) == np.isfinite(ref)), f"{what}: non-finite mismatch"
    fin = np.isfinite(ref)
    err = np.abs(gpu - ref)
    err[~fin] = 0.0
    assert stored in ("f32", "bf16"), stored
    rms = float(np.sqrt(np.mean(ref[fin] ** 2))) if fin.any() else 0.0
    scale = np.maximum(np.abs(ref), rms)
    if mag is not None:
        scale = np.maximum(scale, mag)
    bound = REL_F32 * scale
    if stored == "bf16":
        bound = HALF_ULP_BF16 * (np.abs(ref) + bound) + bound
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} outside tolerance; worst "
                             f"at {i}: gpu {gpu[i]!r} ref {ref[i]!r} bound {bound[i]:.3e}")
    return float(err.max()) if err.size else 0.0


def run_forward(msda, nd, dev_inp):
    fn = msda.msda2d_forward if nd == 2 else msda.msda3d_forward
    out = fn(dev_inp["value"], dev_inp["spatial_shapes"], dev_inp["level_start_index"],
             dev_inp["sampling_locations"], dev_inp["attention_weights"])
    torch_mod().cuda.synchronize()
    return out


def run_backward(msda, nd, dev_inp):
    fn = msda.msda2d_backward if nd == 2 else msda.msda3d_backward
    res = fn(dev_inp["value"], dev_inp["spatial_shapes"], dev_inp["level_start_index"],
             dev_inp["sampling_locations"], dev_inp["attention_weights"], dev_inp["grad_out"])
    torch_mod().cuda.synchronize()
    return res


def grad_value_magnitude(nd, inp):
    """Per-entry sum of |a * w_c * g| over every contribution to grad_value (oracle)."""
    gv_abs, _, _ = oracle.backward(nd, inp["value"], inp["spatial_shapes"],
                                   inp["level_start_index"], inp["sampling_locations"],
                                   np.abs(inp["attention_weights"]), np.abs(inp["grad_out"]))
    return gv_abs


def check_forward(msda, nd, inp, dtype, what):
    dev = device_inputs(inp, dtype)
    out = run_forward(msda, nd, dev)
    ref = oracle.run_inputs(nd, inp)
    return check(host(out), ref, dtype, what)


def check_backward(msda, nd, inp, dtype, what):
    dev = device_inputs(inp, dtype)
    gv, gl, ga = run_backward(msda, nd, dev)
    rgv, rgl, rga = oracle.run_inputs(nd, inp, backward_pass=True)
    mag = grad_value_magnitude(nd, inp)
    # every gradient is an fp32 result, whatever the value dtype
    e1 = check(host(gv), rgv, "f32", what + " grad_value", mag)
    e2 = check(host(gl), rgl, "f32", what + " grad_sampling_locations")
    e3 = check(host(ga), rga, "f32", what + " grad_attention_weights")
    return e1, e2, e3
