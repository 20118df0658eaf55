"""ctypes binding of libmsda (include/msda.h): argument marshalling only.

Every computation runs in the CUDA kernels of libmsda.so; this module only turns torch
tensors into pointers, sizes and a stream handle, calls the C ABI and raises on a non-OK
status.  There is no CPU fallback: if the library cannot be built or loaded, the first
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple, Union

import numpy as np

MSDA_OK, MSDA_ERR_INVALID_ARG, MSDA_ERR_UNSUPPORTED, MSDA_ERR_CUDA, MSDA_ERR_INTERNAL = range(5)
MSDA_F32, MSDA_BF16 = 0, 1
MSDA_MAX_LEVELS = 16
MSDA_MAX_POINTS = 32

STATUS_NAMES = {0: "MSDA_OK", 1: "MSDA_ERR_INVALID_ARG", 2: "MSDA_ERR_UNSUPPORTED",
                3: "MSDA_ERR_CUDA", 4: "MSDA_ERR_INTERNAL"}

# Every symbol include/msda.h declares.
EXPORTS = ("msda2d_forward", "msda2d_backward", "msda3d_forward", "msda3d_backward",
           "msda_last_error", "msda_abi_version", "msda_query_order",
           "msda_query_order_workspace_size", "msda2d_forward_ordered", "msda3d_forward_ordered",
           "msda_query_order_static", "msda2d_forward_pruned", "msda3d_forward_pruned",
           "msda2d_forward_fused", "msda3d_forward_fused", "msda2d_backward_fused",
           "msda3d_backward_fused", "msda_build_flags", "msda_debug_bounds_status",
           "msda_debug_bounds_selftest", "msda2d_backward_ordered", "msda3d_backward_ordered")
MSDA_BUILD_DEBUG_BOUNDS = 1


class MsdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class msda_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("Nin", ctypes.c_int64), ("Nq", ctypes.c_int64),
                ("M", ctypes.c_int32), ("D", ctypes.c_int32), ("L", ctypes.c_int32),
                ("P", ctypes.c_int32), ("value_dtype", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()
_VP = ctypes.c_void_p
_I64P = ctypes.POINTER(ctypes.c_int64)
_DIMS_P = ctypes.POINTER(msda_dims)


def _builder():
    from . import build
    return build


def library_path() -> str:
    return _builder().LIB


def load(path: Optional[str] = None):
    """Load libmsda.so (building it in-tree first when missing or stale).  The environment
    variable MSDA_LIBRARY, when set, names the library the module functions use instead
    (for example the bounds-checking build, libmsda_debug.so)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        default = path is None
        if path is None:
            path = os.environ.get("MSDA_LIBRARY") or _builder().build()
        if not os.path.exists(path):
            raise RuntimeError(f"libmsda not found at {path}")
        lib = ctypes.CDLL(path)
        fwd = [_DIMS_P, _VP, _I64P, _I64P, _VP, _VP, _VP, _VP]
        bwd = [_DIMS_P, _VP, _I64P, _I64P, _VP, _VP, _VP, _VP, _VP, _VP, _VP]
        for name in ("msda2d_forward", "msda3d_forward"):
            getattr(lib, name).argtypes = fwd
            getattr(lib, name).restype = ctypes.c_int
        for name in ("msda2d_backward", "msda3d_backward"):
            getattr(lib, name).argtypes = bwd
            getattr(lib, name).restype = ctypes.c_int
        fwd_o = [_DIMS_P, _VP, _I64P, _I64P, _VP, _VP, _VP, _VP, _VP]
        for name in ("msda2d_forward_ordered", "msda3d_forward_ordered"):
            getattr(lib, name).argtypes = fwd_o
            getattr(lib, name).restype = ctypes.c_int
        bwd_o = [_DIMS_P, _VP, _I64P, _I64P, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]
        for name in ("msda2d_backward_ordered", "msda3d_backward_ordered"):
            getattr(lib, name).argtypes = bwd_o
            getattr(lib, name).restype = ctypes.c_int
        lib.msda_query_order_workspace_size.argtypes = [_DIMS_P, ctypes.c_int32,
                                                        ctypes.POINTER(ctypes.c_size_t)]
        lib.msda_query_order_workspace_size.restype = ctypes.c_int
        lib.msda_query_order.argtypes = [_DIMS_P, ctypes.c_int32, _VP, _VP, _VP, ctypes.c_size_t,
                                         _VP]
        lib.msda_query_order.restype = ctypes.c_int
        for name in ("msda2d_forward_fused", "msda3d_forward_fused"):
            getattr(lib, name).argtypes = [_DIMS_P, _VP, _I64P, _I64P, _VP, _VP, _VP, _VP, _VP]
            getattr(lib, name).restype = ctypes.c_int
        for name in ("msda2d_backward_fused", "msda3d_backward_fused"):
            getattr(lib, name).argtypes = [_DIMS_P, _VP, _I64P, _I64P, _VP, _VP, _VP, _VP, _VP,
                                           _VP, _VP, _VP, _VP]
            getattr(lib, name).restype = ctypes.c_int
        fwd_p = [_DIMS_P, _VP, _I64P, _I64P, _VP, _VP, ctypes.c_float, _VP, _VP]
        for name in ("msda2d_forward_pruned", "msda3d_forward_pruned"):
            getattr(lib, name).argtypes = fwd_p
            getattr(lib, name).restype = ctypes.c_int
        lib.msda_query_order_static.argtypes = [_DIMS_P, ctypes.c_int32, _VP, _VP, _VP]
        lib.msda_query_order_static.restype = ctypes.c_int
        lib.msda_last_error.argtypes = []
        lib.msda_last_error.restype = ctypes.c_char_p
        lib.msda_abi_version.argtypes = []
        lib.msda_abi_version.restype = ctypes.c_int32
        lib.msda_build_flags.argtypes = []
        lib.msda_build_flags.restype = ctypes.c_int32
        lib.msda_debug_bounds_status.argtypes = []
        lib.msda_debug_bounds_status.restype = ctypes.c_int
        lib.msda_debug_bounds_selftest.argtypes = [_VP]
        lib.msda_debug_bounds_selftest.restype = ctypes.c_int
        if default or path == _builder().LIB:
            _lib = lib
        return lib


def _check(lib, status: int) -> None:
    if status != MSDA_OK:
        raise MsdaError(status, lib.msda_last_error().decode(errors="replace"))


# ----------------------------------------------------------------------------- raw layer
# Plain pointers (ints), host metadata arrays and a cudaStream_t (int), as in the header.


def _host_i64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor
        if a.is_cuda:
            raise ValueError("spatial_shapes / level_start_index are host arrays; pass CPU "
                             "tensors or numpy arrays")
        a = a.detach().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def make_dims(B, Nin, Nq, M, D, L, P, value_dtype) -> msda_dims:
    return msda_dims(int(B), int(Nin), int(Nq), int(M), int(D), int(L), int(P),
                     int(value_dtype))


def forward_raw(ndim: int, dims: msda_dims, value: int, spatial_shapes, level_start_index,
                sampling_locations: int, attention_weights: int, out: int, stream: int = 0,
                lib=None) -> int:
    """Call msda{2,3}d_forward with raw device pointers; returns the status (no raise)."""
    lib = lib or load()
    sh, ls = _host_i64(spatial_shapes), _host_i64(level_start_index)
    fn = lib.msda2d_forward if ndim == 2 else lib.msda3d_forward
    return fn(ctypes.byref(dims), _VP(value), sh.ctypes.data_as(_I64P),
              ls.ctypes.data_as(_I64P), _VP(sampling_locations), _VP(attention_weights),
              _VP(out), _VP(stream))


def forward_fused_raw(ndim: int, dims: msda_dims, value: int, spatial_shapes,
                      level_start_index, reference_points: int, sampling_offsets: int,
                      attention_logits: int, out: int, stream: int = 0, lib=None) -> int:
    """Call msda{2,3}d_forward_fused with raw device pointers; returns the status."""
    lib = lib or load()
    sh, ls = _host_i64(spatial_shapes), _host_i64(level_start_index)
    fn = lib.msda2d_forward_fused if ndim == 2 else lib.msda3d_forward_fused
    return fn(ctypes.byref(dims), _VP(value), sh.ctypes.data_as(_I64P),
              ls.ctypes.data_as(_I64P), _VP(reference_points), _VP(sampling_offsets),
              _VP(attention_logits), _VP(out), _VP(stream))


def forward_pruned_raw(ndim: int, dims: msda_dims, value: int, spatial_shapes,
                       level_start_index, sampling_locations: int, attention_weights: int,
                       threshold: float, out: int, stream: int = 0, lib=None) -> int:
    """Call msda{2,3}d_forward_pruned with raw device pointers; returns the status."""
    lib = lib or load()
    sh, ls = _host_i64(spatial_shapes), _host_i64(level_start_index)
    fn = lib.msda2d_forward_pruned if ndim == 2 else lib.msda3d_forward_pruned
    return fn(ctypes.byref(dims), _VP(value), sh.ctypes.data_as(_I64P),
              ls.ctypes.data_as(_I64P), _VP(sampling_locations), _VP(attention_weights),
              ctypes.c_float(threshold), _VP(out), _VP(stream))


def forward_ordered_raw(ndim: int, dims: msda_dims, value: int, spatial_shapes,
                        level_start_index, sampling_locations: int, attention_weights: int,
                        query_order: int, out: int, stream: int = 0, lib=None) -> int:
    """Call msda{2,3}d_forward_ordered with raw device pointers; returns the status."""
    lib = lib or load()
    sh, ls = _host_i64(spatial_shapes), _host_i64(level_start_index)
    fn = lib.msda2d_forward_ordered if ndim == 2 else lib.msda3d_forward_ordered
    return fn(ctypes.byref(dims), _VP(value), sh.ctypes.data_as(_I64P),
              ls.ctypes.data_as(_I64P), _VP(sampling_locations), _VP(attention_weights),
              _VP(query_order), _VP(out), _VP(stream))


def query_order_workspace_raw(ndim: int, dims: msda_dims, lib=None) -> Tuple[int, int]:
    """(status, bytes) of msda_query_order_workspace_size."""
    lib = lib or load()
    n = ctypes.c_size_t(0)
    st = lib.msda_query_order_workspace_size(ctypes.byref(dims), int(ndim), ctypes.byref(n))
    return st, int(n.value)


def query_order_raw(ndim: int, dims: msda_dims, sampling_locations: int, query_order: int,
                    workspace: int, workspace_bytes: int, stream: int = 0, lib=None) -> int:
    lib = lib or load()
    return lib.msda_query_order(ctypes.byref(dims), int(ndim), _VP(sampling_locations),
                                _VP(query_order), _VP(workspace), int(workspace_bytes),
                                _VP(stream))


def query_order_static_raw(ndim: int, dims: msda_dims, sampling_locations: int,
                           query_order: int, stream: int = 0, lib=None) -> int:
    """msda_query_order_static: the query order with the library's fixed scratch (no
    workspace, no allocation); returns the status."""
    lib = lib or load()
    return lib.msda_query_order_static(ctypes.byref(dims), int(ndim), _VP(sampling_locations),
                                       _VP(query_order), _VP(stream))


def backward_raw(ndim: int, dims: msda_dims, value: int, spatial_shapes, level_start_index,
                 sampling_locations: int, attention_weights: int, grad_out: int,
                 grad_value: int, grad_sampling_locations: int, grad_attention_weights: int,
                 stream: int = 0, lib=None) -> int:
    lib = lib or load()
    sh, ls = _host_i64(spatial_shapes), _host_i64(level_start_index)
    fn = lib.msda2d_backward if ndim == 2 else lib.msda3d_backward
    return fn(ctypes.byref(dims), _VP(value), sh.ctypes.data_as(_I64P),
              ls.ctypes.data_as(_I64P), _VP(sampling_locations), _VP(attention_weights),
              _VP(grad_out), _VP(grad_value), _VP(grad_sampling_locations),
              _VP(grad_attention_weights), _VP(stream))


def backward_ordered_raw(ndim: int, dims: msda_dims, value: int, spatial_shapes,
                         level_start_index, sampling_locations: int, attention_weights: int,
                         query_order: int, grad_out: int, grad_value: int,
                         grad_sampling_locations: int, grad_attention_weights: int,
                         stream: int = 0, lib=None) -> int:
    """Call msda{2,3}d_backward_ordered with raw device pointers; returns the status."""
    lib = lib or load()
    sh, ls = _host_i64(spatial_shapes), _host_i64(level_start_index)
    fn = lib.msda2d_backward_ordered if ndim == 2 else lib.msda3d_backward_ordered
    return fn(ctypes.byref(dims), _VP(value), sh.ctypes.data_as(_I64P),
              ls.ctypes.data_as(_I64P), _VP(sampling_locations), _VP(attention_weights),
              _VP(query_order), _VP(grad_out), _VP(grad_value), _VP(grad_sampling_locations),
              _VP(grad_attention_weights), _VP(stream))


def backward_fused_raw(ndim: int, dims: msda_dims, value: int, spatial_shapes,
                       level_start_index, reference_points: int, sampling_offsets: int,
                       attention_logits: int, grad_out: int, grad_value: int,
                       grad_sampling_offsets: int, grad_attention_logits: int,
                       grad_reference_points: int = 0, stream: int = 0, lib=None) -> int:
    """Call msda{2,3}d_backward_fused with raw device pointers (grad_reference_points 0 =
    not wanted); returns the status (no raise)."""
    lib = lib or load()
    sh, ls = _host_i64(spatial_shapes), _host_i64(level_start_index)
    fn = lib.msda2d_backward_fused if ndim == 2 else lib.msda3d_backward_fused
    return fn(ctypes.byref(dims), _VP(value), sh.ctypes.data_as(_I64P),
              ls.ctypes.data_as(_I64P), _VP(reference_points), _VP(sampling_offsets),
              _VP(attention_logits), _VP(grad_out), _VP(grad_value),
              _VP(grad_sampling_offsets), _VP(grad_attention_logits),
              _VP(grad_reference_points or None), _VP(stream))


# ----------------------------------------------------------------------------- torch layer


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return MSDA_F32
    if t.dtype == torch.bfloat16:
        return MSDA_BF16
    raise MsdaError(MSDA_ERR_UNSUPPORTED, f"value dtype {t.dtype} (supported: float32, bfloat16)")


def _require(t, name: str, dtype=None):
    if not t.is_cuda:
        raise MsdaError(MSDA_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise MsdaError(MSDA_ERR_INVALID_ARG, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise MsdaError(MSDA_ERR_INVALID_ARG, f"{name} must be {dtype}, got {t.dtype}")


def _stream_handle(stream, device) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dims_from(value, sampling_locations, ndim: int) -> msda_dims:
    if value.dim() != 4:
        raise MsdaError(MSDA_ERR_INVALID_ARG, "value must be [B, Nin, M, D]")
    if sampling_locations.dim() != 6 or sampling_locations.shape[-1] != ndim:
        raise MsdaError(MSDA_ERR_INVALID_ARG,
                        f"sampling_locations must be [B, Nq, M, L, P, {ndim}]")
    B, Nin, M, D = value.shape
    B2, Nq, M2, L, P, _ = sampling_locations.shape
    if B2 != B or M2 != M:
        raise MsdaError(MSDA_ERR_INVALID_ARG, "value and sampling_locations disagree on B or M")
    return make_dims(B, Nin, Nq, M, D, L, P, _dtype_code(value))


def _prepare_forward(ndim, value, sampling_locations, attention_weights, out,
                     loc_name="sampling_locations", attn_name="attention_weights"):
    """Checks shared by every forward call; returns (dims, out), allocating out if None."""
    torch = _torch()
    dims = _dims_from(value, sampling_locations, ndim)
    _require(value, "value")
    _require(sampling_locations, loc_name, torch.float32)
    _require(attention_weights, attn_name, torch.float32)
    if tuple(attention_weights.shape) != tuple(sampling_locations.shape[:-1]):
        raise MsdaError(MSDA_ERR_INVALID_ARG, f"{attn_name} must be [B, Nq, M, L, P]")
    if out is None:
        out = torch.empty((dims.B, dims.Nq, dims.M * dims.D), dtype=value.dtype,
                          device=value.device)
    _require(out, "out", value.dtype)
    if tuple(out.shape) != (dims.B, dims.Nq, dims.M * dims.D):
        raise MsdaError(MSDA_ERR_INVALID_ARG, "out must be [B, Nq, M*D]")
    return dims, out


def _forward(ndim, value, spatial_shapes, level_start_index, sampling_locations,
             attention_weights, out=None, stream=None):
    dims, out = _prepare_forward(ndim, value, sampling_locations, attention_weights, out)
    lib = load()
    st = forward_raw(ndim, dims, value.data_ptr(), spatial_shapes, level_start_index,
                     sampling_locations.data_ptr(), attention_weights.data_ptr(),
                     out.data_ptr(), _stream_handle(stream, value.device), lib=lib)
    _check(lib, st)
    return out


def _backward(ndim, value, spatial_shapes, level_start_index, sampling_locations,
              attention_weights, grad_out, grad_value=None, grad_sampling_locations=None,
              grad_attention_weights=None, stream=None, query_order=None):
    torch = _torch()
    dims = _dims_from(value, sampling_locations, ndim)
    _require(value, "value")
    _require(sampling_locations, "sampling_locations", torch.float32)
    _require(attention_weights, "attention_weights", torch.float32)
    _require(grad_out, "grad_out", value.dtype)
    if tuple(grad_out.shape) != (dims.B, dims.Nq, dims.M * dims.D):
        raise MsdaError(MSDA_ERR_INVALID_ARG, "grad_out must be [B, Nq, M*D]")
    dev = value.device
    if grad_value is None:
        grad_value = torch.empty(value.shape, dtype=torch.float32, device=dev)
    if grad_sampling_locations is None:
        grad_sampling_locations = torch.empty_like(sampling_locations)
    if grad_attention_weights is None:
        grad_attention_weights = torch.empty_like(attention_weights)
    _require(grad_value, "grad_value", torch.float32)
    _require(grad_sampling_locations, "grad_sampling_locations", torch.float32)
    _require(grad_attention_weights, "grad_attention_weights", torch.float32)
    lib = load()
    if query_order is None:
        st = backward_raw(ndim, dims, value.data_ptr(), spatial_shapes, level_start_index,
                          sampling_locations.data_ptr(), attention_weights.data_ptr(),
                          grad_out.data_ptr(), grad_value.data_ptr(),
                          grad_sampling_locations.data_ptr(), grad_attention_weights.data_ptr(),
                          _stream_handle(stream, dev), lib=lib)
    else:
        _require(query_order, "query_order", torch.int32)
        if tuple(query_order.shape) != (dims.B, dims.Nq):
            raise MsdaError(MSDA_ERR_INVALID_ARG, "query_order must be [B, Nq]")
        st = backward_ordered_raw(ndim, dims, value.data_ptr(), spatial_shapes,
                                  level_start_index, sampling_locations.data_ptr(),
                                  attention_weights.data_ptr(), query_order.data_ptr(),
                                  grad_out.data_ptr(), grad_value.data_ptr(),
                                  grad_sampling_locations.data_ptr(),
                                  grad_attention_weights.data_ptr(),
                                  _stream_handle(stream, dev), lib=lib)
    _check(lib, st)
    return grad_value, grad_sampling_locations, grad_attention_weights


def msda2d_forward(value, spatial_shapes, level_start_index, sampling_locations,
                   attention_weights, out=None, stream=None):
    """2D forward (bilinear).  value [B,Nin,M,D] fp32/bf16 CUDA; spatial_shapes [L,2] and
    level_start_index [L] on the HOST; sampling_locations [B,Nq,M,L,P,2] and
    attention_weights [B,Nq,M,L,P] fp32 CUDA.  Returns out [B,Nq,M*D] (value dtype),
    enqueued on ``stream`` (default: torch's current stream)."""
    return _forward(2, value, spatial_shapes, level_start_index, sampling_locations,
                    attention_weights, out, stream)


def msda3d_forward(value, spatial_shapes, level_start_index, sampling_locations,
                   attention_weights, out=None, stream=None):
    """3D forward (trilinear); spatial_shapes [L,3] = (Z,H,W), locations (x,y,z)."""
    return _forward(3, value, spatial_shapes, level_start_index, sampling_locations,
                    attention_weights, out, stream)


def msda2d_backward(value, spatial_shapes, level_start_index, sampling_locations,
                    attention_weights, grad_out, grad_value=None, grad_sampling_locations=None,
                    grad_attention_weights=None, stream=None):
    """2D backward.  Returns (grad_value fp32, grad_sampling_locations, grad_attention_weights)."""
    return _backward(2, value, spatial_shapes, level_start_index, sampling_locations,
                     attention_weights, grad_out, grad_value, grad_sampling_locations,
                     grad_attention_weights, stream)


def msda3d_backward(value, spatial_shapes, level_start_index, sampling_locations,
                    attention_weights, grad_out, grad_value=None, grad_sampling_locations=None,
                    grad_attention_weights=None, stream=None):
    """3D backward (trilinear)."""
    return _backward(3, value, spatial_shapes, level_start_index, sampling_locations,
                     attention_weights, grad_out, grad_value, grad_sampling_locations,
                     grad_attention_weights, stream)


def msda2d_backward_ordered(value, spatial_shapes, level_start_index, sampling_locations,
                            attention_weights, query_order, grad_out, grad_value=None,
                            grad_sampling_locations=None, grad_attention_weights=None,
                            stream=None):
    """msda2d_backward walking each batch's queries in ``query_order`` (int32 [B, Nq])."""
    return _backward(2, value, spatial_shapes, level_start_index, sampling_locations,
                     attention_weights, grad_out, grad_value, grad_sampling_locations,
                     grad_attention_weights, stream, query_order)


def msda3d_backward_ordered(value, spatial_shapes, level_start_index, sampling_locations,
                            attention_weights, query_order, grad_out, grad_value=None,
                            grad_sampling_locations=None, grad_attention_weights=None,
                            stream=None):
    """msda3d_backward walking each batch's queries in ``query_order`` (int32 [B, Nq])."""
    return _backward(3, value, spatial_shapes, level_start_index, sampling_locations,
                     attention_weights, grad_out, grad_value, grad_sampling_locations,
                     grad_attention_weights, stream, query_order)


def msda_query_order(sampling_locations, query_order=None, workspace=None, stream=None):
    """Locality-aware query order: int32 [B, Nq] (device), per batch a permutation of the
    queries sorted by the Morton code of their mean sampling location.  ``workspace`` (a
    CUDA uint8 tensor of at least ``query_order_workspace_bytes`` bytes) is allocated when
    not given."""
    torch = _torch()
    loc = sampling_locations
    _require(loc, "sampling_locations", torch.float32)
    if loc.dim() != 6 or loc.shape[-1] not in (2, 3):
        raise MsdaError(MSDA_ERR_INVALID_ARG, "sampling_locations must be [B, Nq, M, L, P, 2|3]")
    ndim = int(loc.shape[-1])
    B, Nq, M, L, P, _ = loc.shape
    dims = make_dims(B, 1, Nq, M, 4, L, P, MSDA_F32)
    lib = load()
    st, nbytes = query_order_workspace_raw(ndim, dims, lib=lib)
    _check(lib, st)
    if query_order is None:
        query_order = torch.empty((B, Nq), dtype=torch.int32, device=loc.device)
    _require(query_order, "query_order", torch.int32)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=loc.device)
    _require(workspace, "workspace")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = query_order_raw(ndim, dims, loc.data_ptr(), query_order.data_ptr(),
                         workspace.data_ptr(), ws_bytes, _stream_handle(stream, loc.device),
                         lib=lib)
    _check(lib, st)
    return query_order


def query_order_workspace_bytes(B, Nq, M, L, P, ndim) -> int:
    lib = load()
    st, nbytes = query_order_workspace_raw(ndim, make_dims(B, 1, Nq, M, 4, L, P, MSDA_F32), lib=lib)
    _check(lib, st)
    return nbytes


def _forward_ordered(ndim, value, spatial_shapes, level_start_index, sampling_locations,
                     attention_weights, query_order, out=None, stream=None):
    torch = _torch()
    dims, out = _prepare_forward(ndim, value, sampling_locations, attention_weights, out)
    _require(query_order, "query_order", torch.int32)
    if tuple(query_order.shape) != (dims.B, dims.Nq):
        raise MsdaError(MSDA_ERR_INVALID_ARG, "query_order must be [B, Nq]")
    lib = load()
    st = forward_ordered_raw(ndim, dims, value.data_ptr(), spatial_shapes, level_start_index,
                             sampling_locations.data_ptr(), attention_weights.data_ptr(),
                             query_order.data_ptr(), out.data_ptr(),
                             _stream_handle(stream, value.device), lib=lib)
    _check(lib, st)
    return out


def msda2d_forward_ordered(value, spatial_shapes, level_start_index, sampling_locations,
                           attention_weights, query_order, out=None, stream=None):
    """msda2d_forward walking each batch's queries in ``query_order`` (same result)."""
    return _forward_ordered(2, value, spatial_shapes, level_start_index, sampling_locations,
                            attention_weights, query_order, out, stream)


def msda3d_forward_ordered(value, spatial_shapes, level_start_index, sampling_locations,
                           attention_weights, query_order, out=None, stream=None):
    """msda3d_forward walking each batch's queries in ``query_order`` (same result)."""
    return _forward_ordered(3, value, spatial_shapes, level_start_index, sampling_locations,
                            attention_weights, query_order, out, stream)


def _forward_pruned(ndim, value, spatial_shapes, level_start_index, sampling_locations,
                    attention_weights, threshold, out=None, stream=None):
    dims, out = _prepare_forward(ndim, value, sampling_locations, attention_weights, out)
    lib = load()
    st = forward_pruned_raw(ndim, dims, value.data_ptr(), spatial_shapes, level_start_index,
                            sampling_locations.data_ptr(), attention_weights.data_ptr(),
                            float(threshold), out.data_ptr(),
                            _stream_handle(stream, value.device), lib=lib)
    _check(lib, st)
    return out


def _forward_fused(ndim, value, spatial_shapes, level_start_index, reference_points,
                   sampling_offsets, attention_logits, out=None, stream=None):
    torch = _torch()
    dims, out = _prepare_forward(ndim, value, sampling_offsets, attention_logits, out,
                                 "sampling_offsets", "attention_logits")
    _require(reference_points, "reference_points", torch.float32)
    if tuple(reference_points.shape) != (dims.B, dims.Nq, dims.L, ndim):
        raise MsdaError(MSDA_ERR_INVALID_ARG, f"reference_points must be [B, Nq, L, {ndim}]")
    lib = load()
    st = forward_fused_raw(ndim, dims, value.data_ptr(), spatial_shapes, level_start_index,
                           reference_points.data_ptr(), sampling_offsets.data_ptr(),
                           attention_logits.data_ptr(), out.data_ptr(),
                           _stream_handle(stream, value.device), lib=lib)
    _check(lib, st)
    return out


def msda2d_forward_fused(value, spatial_shapes, level_start_index, reference_points,
                         sampling_offsets, attention_logits, out=None, stream=None):
    """Forward with the prologue fused: location = reference + offset / (W_l, H_l),
    weights = softmax of the logits over the L*P samples of each query and head."""
    return _forward_fused(2, value, spatial_shapes, level_start_index, reference_points,
                          sampling_offsets, attention_logits, out, stream)


def msda3d_forward_fused(value, spatial_shapes, level_start_index, reference_points,
                         sampling_offsets, attention_logits, out=None, stream=None):
    """3D forward with the prologue fused (offsets in voxels of the sampled level)."""
    return _forward_fused(3, value, spatial_shapes, level_start_index, reference_points,
                          sampling_offsets, attention_logits, out, stream)


def _backward_fused(ndim, value, spatial_shapes, level_start_index, reference_points,
                    sampling_offsets, attention_logits, grad_out, need_reference_grad=True,
                    stream=None, grad_value=None, grad_sampling_offsets=None,
                    grad_attention_logits=None, grad_reference_points=None):
    torch = _torch()
    dims = _dims_from(value, sampling_offsets, ndim)
    _require(value, "value")
    _require(reference_points, "reference_points", torch.float32)
    _require(sampling_offsets, "sampling_offsets", torch.float32)
    _require(attention_logits, "attention_logits", torch.float32)
    _require(grad_out, "grad_out", value.dtype)
    if tuple(reference_points.shape) != (dims.B, dims.Nq, dims.L, ndim):
        raise MsdaError(MSDA_ERR_INVALID_ARG, f"reference_points must be [B, Nq, L, {ndim}]")
    if tuple(attention_logits.shape) != tuple(sampling_offsets.shape[:-1]):
        raise MsdaError(MSDA_ERR_INVALID_ARG, "attention_logits must be [B, Nq, M, L, P]")
    if tuple(grad_out.shape) != (dims.B, dims.Nq, dims.M * dims.D):
        raise MsdaError(MSDA_ERR_INVALID_ARG, "grad_out must be [B, Nq, M*D]")
    dev = value.device
    if grad_value is None:
        grad_value = torch.empty(value.shape, dtype=torch.float32, device=dev)
    grad_off = (torch.empty_like(sampling_offsets) if grad_sampling_offsets is None
                else grad_sampling_offsets)
    grad_logits = (torch.empty_like(attention_logits) if grad_attention_logits is None
                   else grad_attention_logits)
    grad_ref = None
    if need_reference_grad:
        grad_ref = (torch.empty_like(reference_points) if grad_reference_points is None
                    else grad_reference_points)
        _require(grad_ref, "grad_reference_points", torch.float32)
    _require(grad_value, "grad_value", torch.float32)
    _require(grad_off, "grad_sampling_offsets", torch.float32)
    _require(grad_logits, "grad_attention_logits", torch.float32)
    lib = load()
    st = backward_fused_raw(ndim, dims, value.data_ptr(), spatial_shapes, level_start_index,
                            reference_points.data_ptr(), sampling_offsets.data_ptr(),
                            attention_logits.data_ptr(), grad_out.data_ptr(),
                            grad_value.data_ptr(), grad_off.data_ptr(), grad_logits.data_ptr(),
                            grad_ref.data_ptr() if grad_ref is not None else 0,
                            _stream_handle(stream, dev), lib=lib)
    _check(lib, st)
    return grad_value, grad_off, grad_logits, grad_ref


def msda2d_backward_fused(value, spatial_shapes, level_start_index, reference_points,
                          sampling_offsets, attention_logits, grad_out, need_reference_grad=True,
                          stream=None, **outs):
    """Backward of msda2d_forward_fused.  Returns (grad_value fp32, grad_sampling_offsets,
    grad_attention_logits, grad_reference_points or None when need_reference_grad is
    False).  Output tensors may be passed in as grad_value=, grad_sampling_offsets=,
    grad_attention_logits=, grad_reference_points=."""
    return _backward_fused(2, value, spatial_shapes, level_start_index, reference_points,
                           sampling_offsets, attention_logits, grad_out, need_reference_grad,
                           stream, **outs)


def msda3d_backward_fused(value, spatial_shapes, level_start_index, reference_points,
                          sampling_offsets, attention_logits, grad_out, need_reference_grad=True,
                          stream=None, **outs):
    """Backward of msda3d_forward_fused (see msda2d_backward_fused)."""
    return _backward_fused(3, value, spatial_shapes, level_start_index, reference_points,
                           sampling_offsets, attention_logits, grad_out, need_reference_grad,
                           stream, **outs)


def msda2d_forward_pruned(value, spatial_shapes, level_start_index, sampling_locations,
                          attention_weights, threshold, out=None, stream=None):
    """msda2d_forward skipping samples with |A| < threshold (opt-in approximation)."""
    return _forward_pruned(2, value, spatial_shapes, level_start_index, sampling_locations,
                           attention_weights, threshold, out, stream)


def msda3d_forward_pruned(value, spatial_shapes, level_start_index, sampling_locations,
                          attention_weights, threshold, out=None, stream=None):
    """msda3d_forward skipping samples with |A| < threshold (opt-in approximation)."""
    return _forward_pruned(3, value, spatial_shapes, level_start_index, sampling_locations,
                           attention_weights, threshold, out, stream)


def msda_last_error() -> str:
    lib = load()
    return lib.msda_last_error().decode(errors="replace")


def msda_build_flags() -> int:
    return int(load().msda_build_flags())


def msda_debug_bounds_status() -> int:
    """Status of the bounds-check record (see include/msda.h); returns the status code."""
    return int(load().msda_debug_bounds_status())


def msda_debug_bounds_selftest(stream: int = 0) -> int:
    return int(load().msda_debug_bounds_selftest(_VP(stream)))


def msda_abi_version() -> int:
    return int(load().msda_abi_version())
