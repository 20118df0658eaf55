// Internal interface between the C-ABI layer (msda_abi.cpp) and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace msda {

constexpr int kF32 = 0;
constexpr int kBF16 = 1;
constexpr int kMaxLevels = 16;
constexpr int kMaxPoints = 32;

// First out-of-range corner row seen by a kernel of a build with MSDA_DEBUG_BOUNDS (the
// debug build checks every corner row index against [0, N_in) before its access, records
// the first offender here and skips the access).  flag: 0 none, 1 being written, 2 set.
struct DebugRecord {
    unsigned flag;
    int sample;        // l * P + p
    long long row;     // the offending row index within its batch
    long long item;    // (b * Nq + q) * M + m
    long long nin;     // N_in, Nq, M and P of the call, to decode item and sample
    long long nq;
    int m_count, p_count;
};

// Everything a kernel needs, passed by value as a __grid_constant__ parameter.
// All level geometry is validated on the host before it gets here.
struct Params {
    // tensors
    const void *value;          // [B, Nin, M, D]
    const float *loc;           // [B, Nq, M, L, P, NDIM]
    const float *attn;          // [B, Nq, M, L, P]
    void *out;                  // [B, Nq, M*D]           (forward)
    const void *grad_out;       // [B, Nq, M*D]           (backward)
    float *grad_value;          // [B, Nin, M, D]         (backward)
    float *grad_loc;            // like loc               (backward)
    float *grad_attn;           // like attn              (backward)
    const int *order;           // [B, Nq] query order, or null (forward and backward)
    float prune;                // forward: samples with |A| < prune are skipped (0: exact)
    // fused prologue (forward): when set, `loc` holds sampling offsets in pixels of the
    // sampled level and `attn` the attention logits; the location is ref[b, q, l] + offset /
    // extent and the weights are the softmax of the logits over the item's L * P samples
    const float *ref;           // [B, Nq, L, NDIM] reference points, or null
    float *grad_ref;            // [B, Nq, L, NDIM] fused backward: reference-point gradient,
                                // or null (not wanted)
    // sizes
    long long B, Nin, Nq;
    long long n_items;          // B * Nq * M work items (b, q, m)
    int M, D, L, P;
    long long row_bytes;        // M * D * sizeof(value dtype): stride between value rows
    int rb32;                   // row_bytes as a 32-bit int (validated to fit)
    int pinv;                   // ceil(2^16 / P): level of sample j < 512 is (j * pinv) >> 16
    int pack_taps;              // forward tap records may carry the validity bits under the
                                // row (N_in < 2^27 in 2D, < 2^22 in 3D)
    // level geometry (entries >= L unused)
    int W[kMaxLevels], H[kMaxLevels], Z[kMaxLevels], start[kMaxLevels];
    float fW[kMaxLevels], fH[kMaxLevels], fZ[kMaxLevels];
    long long sy[kMaxLevels];   // bytes between value rows one image row apart (W * row_bytes)
    long long sz[kMaxLevels];   // bytes between value rows one slice apart (H * W * row_bytes)
    DebugRecord *dbg;           // debug build: where a kernel records an out-of-range row
    // backward work split: CTA c handles batch b = c / (M * nchunk), head m = (c / nchunk) % M,
    // and queries [chunk * qchunk, (chunk + 1) * qchunk) with chunk = c % nchunk
    int nchunk, qchunk;
};

// (L, P) pairs with a compiled backward (bwd_tiled); others take the generic kernels.
inline bool backward_is_tiled(const Params &p) { return p.P == 4 && (p.L == 4 || p.L == 1); }

// Launchers: enqueue on `stream`, return the launch status.  dtype is kF32 / kBF16,
// G = D * sizeof(dtype) / 16 lanes per work item.
cudaError_t launch_forward(int ndim, int dtype, int G, const Params &p, cudaStream_t stream);
// launch_backward: with p.ref set, the backward of the fused forward (loc = offsets,
// attn = logits; grad_loc / grad_attn receive the offset and logit gradients, and
// p.grad_ref, when set, the reference-point gradient).
cudaError_t launch_backward(int ndim, int dtype, int G, const Params &p, cudaStream_t stream);
cudaError_t launch_zero_fill(float *ptr, long long n_floats, cudaStream_t stream);

// Per-(dtype, ndim) instantiations behind launch_forward / launch_backward.
cudaError_t launch_forward_f32_2d(int G, const Params &p, cudaStream_t stream);
cudaError_t launch_forward_f32_3d(int G, const Params &p, cudaStream_t stream);
cudaError_t launch_forward_bf16_2d(int G, const Params &p, cudaStream_t stream);
cudaError_t launch_forward_bf16_3d(int G, const Params &p, cudaStream_t stream);
// Runtime-(L, P) form of the tiled forward (msda_forward_rt_*.cu): L * P <= 32, G (lanes
// per row at 16 bytes per lane) in {2, 4, 8, 16}.
cudaError_t launch_forward_rt_f32_2d(int G, const Params &p, cudaStream_t stream);
cudaError_t launch_forward_rt_f32_3d(int G, const Params &p, cudaStream_t stream);
cudaError_t launch_forward_rt_bf16_2d(int G, const Params &p, cudaStream_t stream);
cudaError_t launch_forward_rt_bf16_3d(int G, const Params &p, cudaStream_t stream);
cudaError_t launch_backward_2d(int dtype, int G, const Params &p, cudaStream_t stream);
cudaError_t launch_backward_3d(int dtype, int G, const Params &p, cudaStream_t stream);
cudaError_t launch_backward_fused_2d(int dtype, int G, const Params &p, cudaStream_t stream);
cudaError_t launch_backward_fused_3d(int dtype, int G, const Params &p, cudaStream_t stream);

// Query order (msda_order.cu): sorts each batch's queries by the Morton code of the mean
// of their sampling locations.  `hist` holds B * kOrderBuckets ints, `keys` B * Nq ints.
constexpr int kOrderBits2d = 6;    // bits per axis of the 2D key (64 x 64 cells)
constexpr int kOrderBits3d = 4;    // bits per axis of the 3D key (16 x 16 x 16 cells)
constexpr int kOrderBuckets = 1 << 12;
cudaError_t launch_query_order(int ndim, const Params &p, int *order, int *hist, int *keys,
                               cudaStream_t stream);

// The same order with its scratch in a fixed device array of the library
// (msda_order_static.cu); static_order_fits tells whether (B, Nq) fits that array.
bool static_order_fits(long long B, long long Nq);

// Debug build (MSDA_DEBUG_BOUNDS, msda_debug.cu): the device address of this device's
// DebugRecord (looked up once per device), reading and clearing it, and a kernel that
// records a made-up offender so that the reporting path can be tested without any
// out-of-range access.  Without MSDA_DEBUG_BOUNDS these return cudaErrorNotSupported.
cudaError_t debug_record(DebugRecord **ptr);
cudaError_t debug_record_take(DebugRecord *out);
cudaError_t launch_debug_selftest(const Params &p, long long row, long long item, int sample,
                                  cudaStream_t stream);
cudaError_t launch_query_order_static(int ndim, const Params &p, int *order, cudaStream_t stream);

}  // namespace msda
