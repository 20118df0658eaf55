"""CPU oracle for the multi-scale deformable attention core -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The shipped library never does, and this
package imports nothing from it: the oracle is plain C (``msda_oracle.c``) evaluated
in double precision, loaded here through ctypes.

Every function takes numpy arrays in the layouts of ``workloads`` and returns float64
arrays.  Inputs are widened to float64 exactly (fp32 and bf16 values are exact in
double), so the oracle and the CUDA path see the same input values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmsda_oracle.so")
_lib = None

_I64 = ctypes.c_int64
_DP = ctypes.POINTER(ctypes.c_double)
_LP = ctypes.POINTER(ctypes.c_int64)


def compile_source(src: str, out_path: str) -> str:
    """Compile an oracle source file with gcc (IEEE double, no FMA contraction)."""
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                    "-fopenmp", "-shared", "-fPIC", "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile ``msda_oracle.c`` into ``_build/libmsda_oracle.so`` when stale."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        os.makedirs(_BUILD_DIR, exist_ok=True)
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Bind another build of the oracle source (used by the mutation tests)."""
    return _bind(path)


def _bind(path: str):
    lib = ctypes.CDLL(path)
    fwd_args = [_I64] * 7 + [_LP, _LP, _DP, _DP, _DP, _DP]
    bwd_args = [_I64] * 7 + [_LP, _LP, _DP, _DP, _DP, _DP, _DP, _DP, _DP]
    for name in ("oracle_msda2d_forward", "oracle_msda3d_forward"):
        getattr(lib, name).argtypes = fwd_args
        getattr(lib, name).restype = ctypes.c_int
    for name in ("oracle_msda2d_backward", "oracle_msda3d_backward"):
        getattr(lib, name).argtypes = bwd_args
        getattr(lib, name).restype = ctypes.c_int
    if hasattr(lib, "oracle_msda2d_forward_threads"):
        for name in ("oracle_msda2d_forward_threads", "oracle_msda3d_forward_threads"):
            getattr(lib, name).argtypes = fwd_args + [ctypes.c_int]
            getattr(lib, name).restype = ctypes.c_int
        lib.oracle_default_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _d(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int64)


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def _dims(value: np.ndarray, loc: np.ndarray, shapes: np.ndarray, nd: int):
    B, Nin, M, D = value.shape
    if loc.ndim != 6 or loc.shape[-1] != nd:
        raise ValueError(f"sampling_locations must be [B,Nq,M,L,P,{nd}], got {loc.shape}")
    _, Nq, M2, L, P, _ = loc.shape
    if M2 != M or loc.shape[0] != B or shapes.shape != (L, nd):
        raise ValueError("inconsistent shapes")
    return B, Nin, Nq, M, D, L, P


def default_threads() -> int:
    """Threads the oracle's multi-core forward uses by default (OpenMP's count)."""
    return int(_load().oracle_default_threads())


def forward(nd: int, value, spatial_shapes, level_start_index, sampling_locations,
            attention_weights, lib=None, threads: int = 1) -> np.ndarray:
    """out[B, Nq, M*D] in float64.  ``lib`` selects another build of the oracle.
    ``threads`` != 1 runs the same serial forward on blocks of queries over that many
    host threads (0: OpenMP's default); every output is computed identically."""
    v, loc, a = _d(value), _d(sampling_locations), _d(attention_weights)
    sh, ls = _i(spatial_shapes), _i(level_start_index)
    B, Nin, Nq, M, D, L, P = _dims(v, loc, sh, nd)
    out = np.zeros((B, Nq, M * D), dtype=np.float64)
    lib = lib or _load()
    args = (B, Nin, Nq, M, D, L, P, _ptr(sh, _LP), _ptr(ls, _LP), _ptr(v, _DP),
            _ptr(loc, _DP), _ptr(a, _DP), _ptr(out, _DP))
    if threads != 1:
        fn = lib.oracle_msda2d_forward_threads if nd == 2 else lib.oracle_msda3d_forward_threads
        rc = fn(*args, int(threads))
    else:
        fn = lib.oracle_msda2d_forward if nd == 2 else lib.oracle_msda3d_forward
        rc = fn(*args)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def backward(nd: int, value, spatial_shapes, level_start_index, sampling_locations,
             attention_weights, grad_out, lib=None) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(grad_value, grad_sampling_locations, grad_attention_weights) in float64."""
    v, loc, a = _d(value), _d(sampling_locations), _d(attention_weights)
    g = _d(grad_out)
    sh, ls = _i(spatial_shapes), _i(level_start_index)
    B, Nin, Nq, M, D, L, P = _dims(v, loc, sh, nd)
    gv = np.zeros_like(v)
    gl = np.zeros_like(loc)
    ga = np.zeros_like(a)
    lib = lib or _load()
    fn = lib.oracle_msda2d_backward if nd == 2 else lib.oracle_msda3d_backward
    rc = fn(B, Nin, Nq, M, D, L, P, _ptr(sh, _LP), _ptr(ls, _LP), _ptr(v, _DP),
            _ptr(loc, _DP), _ptr(a, _DP), _ptr(g, _DP), _ptr(gv, _DP), _ptr(gl, _DP),
            _ptr(ga, _DP))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return gv, gl, ga


def msda2d_forward(value, spatial_shapes, level_start_index, sampling_locations,
                   attention_weights):
    return forward(2, value, spatial_shapes, level_start_index, sampling_locations,
                   attention_weights)


def msda3d_forward(value, spatial_shapes, level_start_index, sampling_locations,
                   attention_weights):
    return forward(3, value, spatial_shapes, level_start_index, sampling_locations,
                   attention_weights)


def msda2d_backward(value, spatial_shapes, level_start_index, sampling_locations,
                    attention_weights, grad_out):
    return backward(2, value, spatial_shapes, level_start_index, sampling_locations,
                    attention_weights, grad_out)


def msda3d_backward(value, spatial_shapes, level_start_index, sampling_locations,
                    attention_weights, grad_out):
    return backward(3, value, spatial_shapes, level_start_index, sampling_locations,
                    attention_weights, grad_out)


def fused_locations(spatial_shapes, reference_points, sampling_offsets) -> np.ndarray:
    """Sampling locations of the module's prologue ("3D Attention That Knows Where to
    Look": reference point plus predicted offsets), in fp32 as an fp32 module forms them:
    loc[b,q,m,l,p,k] = ref[b,q,l,k] + offset[b,q,m,l,p,k] / E_lk, E_l = (W_l, H_l[, Z_l]),
    one IEEE division then one IEEE addition."""
    sh = np.asarray(spatial_shapes, dtype=np.int64)
    ext = sh[:, ::-1].astype(np.float32)                             # [L, nd] = (W, H[, Z])
    ref = np.asarray(reference_points, dtype=np.float32)             # [B, Nq, L, nd]
    off = np.asarray(sampling_offsets, dtype=np.float32)             # [B, Nq, M, L, P, nd]
    q = off / ext[None, None, None, :, None, :]
    return ref[:, :, None, :, None, :] + q


def softmax_weights(attention_logits) -> np.ndarray:
    """Attention weights from the logits ("Deformable Attention Module": a softmax over the
    sampled keys; "3D Attention That Knows Where to Look": one weighted sum over all L x P
    samples), in double: softmax over the last two axes (L, P) of [B, Nq, M, L, P]."""
    z = np.asarray(attention_logits, dtype=np.float64)
    shape = z.shape
    z = z.reshape(shape[:3] + (-1,))
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return (e / e.sum(axis=-1, keepdims=True)).reshape(shape)


def forward_fused(nd: int, value, spatial_shapes, level_start_index, reference_points,
                  sampling_offsets, attention_logits, lib=None, threads: int = 1) -> np.ndarray:
    """The core fed by the module's prologue: locations from reference points and offsets
    (fp32, as above), weights from a double-precision softmax of the logits."""
    loc = fused_locations(spatial_shapes, reference_points, sampling_offsets)
    return forward(nd, value, spatial_shapes, level_start_index, loc,
                   softmax_weights(attention_logits), lib=lib, threads=threads)


def backward_fused(nd: int, value, spatial_shapes, level_start_index, reference_points,
                   sampling_offsets, attention_logits, grad_out, lib=None):
    """Gradients of ``forward_fused`` ("3D Attention That Knows Where to Look": gradients
    flow back into both the offsets and the weights; "Deformable Attention Module": the
    weights are a softmax of the predicted logits), by the chain rule through the prologue,
    in double:

      grad_offset[b,q,m,l,p,k] = grad_location[b,q,m,l,p,k] / E_lk  (location = ref + offset / E)
      grad_logit[b,q,m,s]      = A_s * (grad_A_s - sum_t A_t * grad_A_t)  over the item's L x P
      grad_ref[b,q,l,k]        = sum over m and p of grad_location[b,q,m,l,p,k]

    where grad_value, grad_location and grad_A are the core's backward at the fused
    locations and weights.  Returns (grad_value, grad_offsets, grad_logits, grad_ref)."""
    sh = np.asarray(spatial_shapes, dtype=np.int64)
    loc = fused_locations(sh, reference_points, sampling_offsets)
    a = softmax_weights(attention_logits)
    gv, gl, ga = backward(nd, value, sh, level_start_index, loc, a, grad_out, lib=lib)
    ext = sh[:, ::-1].astype(np.float64)                              # [L, nd] = (W, H[, Z])
    g_off = gl / ext[None, None, None, :, None, :]
    B, Nq, M, L, P = a.shape
    a2 = a.reshape(B, Nq, M, L * P)
    g2 = ga.reshape(B, Nq, M, L * P)
    g_logit = (a2 * (g2 - (a2 * g2).sum(axis=-1, keepdims=True))).reshape(a.shape)
    g_ref = gl.sum(axis=(2, 4))                                       # [B, Nq, L, nd]
    return gv, g_off, g_logit, g_ref


def forward_pruned(nd: int, value, spatial_shapes, level_start_index, sampling_locations,
                   attention_weights, threshold: float, lib=None, threads: int = 1) -> np.ndarray:
    """The core with probability-aware pruning of sampling points ("DEFA: Efficient
    Deformable Attention Acceleration via Pruning-Assisted Grid-Sampling and Multi-Scale
    Parallel Processing", abstract): a sample whose weight has |A| < threshold is dropped
    from the weighted sum.  A dropped sample contributes exactly nothing, which is what a
    zero weight contributes to the plain definition (finite values), so the rule is applied
    to the weights and the plain oracle does the rest."""
    a = np.asarray(attention_weights, dtype=np.float64)
    a = np.where(np.abs(a) < threshold, 0.0, a)
    return forward(nd, value, spatial_shapes, level_start_index, sampling_locations, a,
                   lib=lib, threads=threads)


def pruning_bound(nd: int, value, spatial_shapes, level_start_index, sampling_locations,
                  attention_weights, threshold: float, lib=None) -> np.ndarray:
    """Per output channel, the sum over the dropped samples of |A| * max_c |v_c|, v_c the
    sample's in-level corner values in that channel: an upper bound on |pruned - unpruned|
    because a sample's corner weights are non-negative and sum to at most 1.  Brute force
    over every sample and corner (test infrastructure)."""
    a = np.abs(np.asarray(attention_weights, dtype=np.float64))
    dropped = np.where(a < threshold, a, 0.0)
    v = np.abs(np.asarray(value, dtype=np.float64))
    loc = np.asarray(sampling_locations, dtype=np.float64)
    shapes = np.asarray(spatial_shapes, dtype=np.int64)
    starts = np.asarray(level_start_index, dtype=np.int64)
    B, Nq, M, L, P, _ = loc.shape
    D = v.shape[-1]
    bound = np.zeros((B, Nq, M, D))
    for l in range(L):
        ext = shapes[l][::-1]                                          # (W, H[, Z])
        pix = loc[:, :, :, l] * ext - 0.5                              # [B,Nq,M,P,nd]
        fin = np.all(np.isfinite(pix), axis=-1)
        i0 = np.floor(np.where(np.isfinite(pix), pix, -5)).astype(np.int64)
        vmax = np.zeros((B, Nq, M, P, D))
        for c in range(2 ** nd):
            idx = i0 + np.array([(c >> k) & 1 for k in range(nd)])
            inside = fin & np.all((idx >= 0) & (idx < ext), axis=-1)
            if nd == 2:
                row = idx[..., 1] * ext[0] + idx[..., 0]
            else:
                row = (idx[..., 2] * ext[1] + idx[..., 1]) * ext[0] + idx[..., 0]
            row = np.where(inside, starts[l] + row, 0)
            bb = np.arange(B)[:, None, None, None]
            mm = np.arange(M)[None, None, :, None]
            vc = v[bb, row, mm]                                        # [B,Nq,M,P,D]
            vmax = np.maximum(vmax, np.where(inside[..., None], vc, 0.0))
        bound += (dropped[:, :, :, l, :, None] * vmax).sum(3)
    return bound.reshape(B, Nq, M * D)


def run_inputs(nd: int, inp: Dict[str, np.ndarray], backward_pass: bool = False, lib=None):
    """Convenience: run the oracle on a dict from ``workloads.make_inputs``."""
    args = (inp["value"], inp["spatial_shapes"], inp["level_start_index"],
            inp["sampling_locations"], inp["attention_weights"])
    if backward_pass:
        return backward(nd, *args, inp["grad_out"], lib=lib)
    return forward(nd, *args, lib=lib)
