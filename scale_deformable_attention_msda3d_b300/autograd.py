"""torch.autograd wrapper around the libmsda forward / backward calls (marshalling only)."""
from __future__ import annotations

import numpy as np

from . import _binding


def _import_torch():
    import torch
    return torch


class _Fn:
    """Lazily built autograd.Function so that importing the package does not need torch."""
    cls = None

    @classmethod
    def get(cls):
        if cls.cls is None:
            torch = _import_torch()

            class MSDeformAttn(torch.autograd.Function):
                @staticmethod
                def forward(ctx, value, spatial_shapes, level_start_index,
                            sampling_locations, attention_weights, query_order=None):
                    ndim = sampling_locations.shape[-1]
                    shapes = np.asarray(spatial_shapes, dtype=np.int64)
                    starts = np.asarray(level_start_index, dtype=np.int64)
                    if query_order is None:
                        fwd = _binding.msda2d_forward if ndim == 2 else _binding.msda3d_forward
                        out = fwd(value, shapes, starts, sampling_locations, attention_weights)
                    else:
                        fwd = (_binding.msda2d_forward_ordered if ndim == 2
                               else _binding.msda3d_forward_ordered)
                        out = fwd(value, shapes, starts, sampling_locations, attention_weights,
                                  query_order)
                    ctx.save_for_backward(value, sampling_locations, attention_weights)
                    ctx.meta = (ndim, shapes, starts)
                    ctx.query_order = query_order
                    return out

                @staticmethod
                def backward(ctx, grad_out):
                    value, loc, attn = ctx.saved_tensors
                    ndim, shapes, starts = ctx.meta
                    order = ctx.query_order
                    if order is None:
                        bwd = _binding.msda2d_backward if ndim == 2 else _binding.msda3d_backward
                        gv, gl, ga = bwd(value, shapes, starts, loc, attn, grad_out.contiguous())
                    else:
                        bwd = (_binding.msda2d_backward_ordered if ndim == 2
                               else _binding.msda3d_backward_ordered)
                        gv, gl, ga = bwd(value, shapes, starts, loc, attn, order,
                                         grad_out.contiguous())
                    return gv.to(value.dtype), None, None, gl, ga, None

            cls.cls = MSDeformAttn
        return cls.cls


class MSDeformAttnFunction:
    """``MSDeformAttnFunction.apply(value, spatial_shapes, level_start_index, loc, attn
    [, query_order])``."""

    @staticmethod
    def apply(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
              query_order=None):
        return _Fn.get().apply(value, spatial_shapes, level_start_index, sampling_locations,
                               attention_weights, query_order)


def ms_deform_attn(value, spatial_shapes, level_start_index, sampling_locations,
                   attention_weights, query_order=None):
    """Differentiable multi-scale deformable attention core (2D or 3D by the last dim of
    ``sampling_locations``).  ``spatial_shapes`` / ``level_start_index`` are host arrays.
    ``query_order`` (int32 [B, Nq] on the device, e.g. from ``msda_query_order``) runs the
    ordered forward and backward: the same results (the backward's grad_value up to the
    order of its fp32 sums), for inputs whose queries come in no local order."""
    return MSDeformAttnFunction.apply(value, spatial_shapes, level_start_index,
                                      sampling_locations, attention_weights, query_order)


class _FusedFn:
    """Lazily built autograd.Function for the fused-prologue call."""
    cls = None

    @classmethod
    def get(cls):
        if cls.cls is None:
            torch = _import_torch()

            class MSDeformAttnFused(torch.autograd.Function):
                @staticmethod
                def forward(ctx, value, spatial_shapes, level_start_index, reference_points,
                            sampling_offsets, attention_logits):
                    ndim = sampling_offsets.shape[-1]
                    shapes = np.asarray(spatial_shapes, dtype=np.int64)
                    starts = np.asarray(level_start_index, dtype=np.int64)
                    fwd = (_binding.msda2d_forward_fused if ndim == 2
                           else _binding.msda3d_forward_fused)
                    out = fwd(value, shapes, starts, reference_points, sampling_offsets,
                              attention_logits)
                    ctx.save_for_backward(value, reference_points, sampling_offsets,
                                          attention_logits)
                    ctx.meta = (ndim, shapes, starts)
                    return out

                @staticmethod
                def backward(ctx, grad_out):
                    value, ref, off, logits = ctx.saved_tensors
                    ndim, shapes, starts = ctx.meta
                    bwd = (_binding.msda2d_backward_fused if ndim == 2
                           else _binding.msda3d_backward_fused)
                    gv, goff, gz, gref = bwd(value, shapes, starts, ref, off, logits,
                                             grad_out.contiguous(),
                                             need_reference_grad=ctx.needs_input_grad[3])
                    return gv.to(value.dtype), None, None, gref, goff, gz

            cls.cls = MSDeformAttnFused
        return cls.cls


def ms_deform_attn_fused(value, spatial_shapes, level_start_index, reference_points,
                         sampling_offsets, attention_logits):
    """Differentiable core with the module's prologue fused in: location = reference point
    + offset / extent (offsets in pixels of the sampled level), weights = softmax of the
    logits over each query and head's L x P samples.  Gradients flow to value, the
    reference points, the offsets and the logits."""
    return _FusedFn.get().apply(value, spatial_shapes, level_start_index, reference_points,
                                sampling_offsets, attention_logits)
