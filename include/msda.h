/*
 * libmsda -- multi-scale deformable attention core for NVIDIA B300 (sm_103a).
 *
 * The operation ("Deformable Attention Module", Code with Papers: the DeformAttn equation
 * and the paragraph under it; "3D Attention That Knows Where to Look": the per-query
 * recipe, the multi-scale paragraph and "What changes from 2D to 3D"):
 *
 *   out[b, q, m*D + d] = sum_{l < L} sum_{p < P}  A[b,q,m,l,p] * x_l(loc[b,q,m,l,p])[m, d]
 *
 * where x_l(.) samples level l of the per-head value map bilinearly (2D: the 4 pixels
 * around the location) or trilinearly (3D: the 8 corners of the surrounding voxel cell).
 * The attention weights A are used as given (callers normalise them over the L x P
 * samples of each query and head; the library never renormalises).  The projections
 * W_m / W'_m of the full module are not part of this core.
 *
 * Sampling convention (the pages do not fix one; this is the library's definition):
 *   pixel coordinate  x = loc_x * W_l - 0.5,  y = loc_y * H_l - 0.5  [, z = loc_z * Z_l - 0.5]
 *   (grid_sample with align_corners = false).  Corners outside level l contribute zero
 *   and receive no gradient (zero padding); a sample with a non-finite coordinate
 *   contributes zero and gets zero gradients.  At an integer coordinate the cell chosen
 *   by floor() defines the (right-hand) location gradient.
 *
 * Layouts (row-major, last index fastest; all device memory unless marked host):
 *   value                [B, Nin, M, D]          value dtype (fp32 or bf16)
 *   spatial_shapes       host int64 [L][2] = (H, W)   or  [L][3] = (Z, H, W)
 *   level_start_index    host int64 [L], must equal the exclusive prefix sum of the
 *                        level sizes; the sizes must add up to Nin.  Pixel (h, w) of
 *                        level l is value row level_start_index[l] + h*W + w; voxel
 *                        (z, h, w) is row level_start_index[l] + (z*H + h)*W + w.
 *   sampling_locations   [B, Nq, M, L, P, 2|3]   fp32, normalised (x, y[, z]):
 *                        component 0 runs along W, 1 along H, 2 along Z.
 *   attention_weights    [B, Nq, M, L, P]        fp32
 *   out / grad_out       [B, Nq, M*D]            value dtype
 *   grad_value           [B, Nin, M, D]          fp32 (always)
 *   grad_sampling_locations   like sampling_locations, fp32
 *   grad_attention_weights    like attention_weights,  fp32
 *
 * Ownership and execution: the caller owns every buffer; these calls allocate no memory
 * (no cudaMalloc / cudaFree).  Work is enqueued on `stream` (0 = legacy default stream)
 * and the call returns without synchronising.  Outputs are overwritten, never
 * accumulated into.  The backward zero-fills grad_value itself, on `stream`.
 *
 * Errors: arguments are validated on the host BEFORE anything is enqueued; a failed
 * check returns MSDA_ERR_INVALID_ARG or MSDA_ERR_UNSUPPORTED with nothing enqueued.  A
 * launch failure returns MSDA_ERR_CUDA.  Faults during execution surface at the caller's
 * next synchronisation, as for any CUDA work.  msda_last_error() gives a message for the
 * last non-OK status returned on the calling thread.
 *
 * Limits: 1 <= L <= MSDA_MAX_LEVELS, 1 <= P <= MSDA_MAX_POINTS, Nin <= 2^30, every level
 * extent in [1, 2^23) (an extent of 2^23 or more returns MSDA_ERR_UNSUPPORTED: the pixel
 * coordinate loc * extent - 0.5 is formed exactly in fp32, which needs the product below
 * 2^23) and every level at most 2^30 pixels, M * D * sizeof(value dtype)
 * below 2^31 bytes; D * sizeof(value dtype) must be 16, 32, 64, 128, 256 or 512 bytes
 * (fp32: D in {4, 8, 16, 32, 64, 128}; bf16: D in {8, 16, 32, 64, 128, 256}); every
 * pointer must be 16-byte aligned.  B == 0 or Nq == 0 is a valid empty call (the
 * backward then still zero-fills grad_value).
 */
#ifndef MSDA_H_
#define MSDA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t, without including CUDA headers. */
typedef struct CUstream_st *msda_stream_t;

#define MSDA_MAX_LEVELS 16
#define MSDA_MAX_POINTS 32

typedef enum {
    MSDA_OK = 0,
    MSDA_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent shapes, misalignment */
    MSDA_ERR_UNSUPPORTED = 2, /* valid but outside what the library handles: D or dtype,
                                 L / P above their maxima, extents of 2^23 or more, and
                                 the fixed-scratch order's size limits                  */
    MSDA_ERR_CUDA = 3,        /* a CUDA call or kernel launch failed                      */
    MSDA_ERR_INTERNAL = 4
} msda_status;

typedef enum { MSDA_F32 = 0, MSDA_BF16 = 1 } msda_dtype;

typedef struct {
    int64_t B;        /* batch                                   */
    int64_t Nin;      /* value rows per batch (all levels)        */
    int64_t Nq;       /* queries per batch                        */
    int32_t M;        /* heads                                    */
    int32_t D;        /* channels per head                        */
    int32_t L;        /* pyramid levels                           */
    int32_t P;        /* sampling points per level                */
    int32_t value_dtype; /* msda_dtype of value, out and grad_out */
} msda_dims;

/*
 * 2D forward: out = sum over levels and points of A times the bilinear sample.
 * Defined by the DeformAttn equation ("Deformable Attention Module") with the
 * multi-scale sum of "3D Attention That Knows Where to Look".
 */
msda_status msda2d_forward(const msda_dims *dims, const void *value,
                           const int64_t *spatial_shapes, const int64_t *level_start_index,
                           const float *sampling_locations, const float *attention_weights,
                           void *out, msda_stream_t stream);

/*
 * 2D backward: given grad_out = dLoss/dout, writes dLoss/dvalue (fp32), dLoss/dlocations
 * and dLoss/dweights ("3D Attention That Knows Where to Look": gradients flow back into
 * both the offsets and the weights; the value gradient is the transpose of the gather).
 * grad_value is zero-filled on `stream` first, then accumulated with atomics, so its
 * summation order (and last bits) may vary between runs.
 */
msda_status msda2d_backward(const msda_dims *dims, const void *value,
                            const int64_t *spatial_shapes, const int64_t *level_start_index,
                            const float *sampling_locations, const float *attention_weights,
                            const void *grad_out, float *grad_value,
                            float *grad_sampling_locations, float *grad_attention_weights,
                            msda_stream_t stream);

/*
 * 3D forward: as msda2d_forward with trilinear sampling over the 8 corners of the voxel
 * cell ("3D Attention That Knows Where to Look", "What changes from 2D to 3D"):
 * spatial_shapes is [L][3] = (Z, H, W) and locations are (x, y, z).
 */
msda_status msda3d_forward(const msda_dims *dims, const void *value,
                           const int64_t *spatial_shapes, const int64_t *level_start_index,
                           const float *sampling_locations, const float *attention_weights,
                           void *out, msda_stream_t stream);

/* 3D backward: as msda2d_backward, trilinear, three location components. */
msda_status msda3d_backward(const msda_dims *dims, const void *value,
                            const int64_t *spatial_shapes, const int64_t *level_start_index,
                            const float *sampling_locations, const float *attention_weights,
                            const void *grad_out, float *grad_value,
                            float *grad_sampling_locations, float *grad_attention_weights,
                            msda_stream_t stream);

/*
 * Forward with the module's prologue fused in.  The module predicts, per query, sampling
 * offsets around a reference point and attention logits, and normalises the logits with
 * a softmax ("Deformable Attention Module": a linear layer gives 3MK channels, 2MK of
 * offsets and MK logits that a softmax turns into weights; "3D Attention That Knows Where
 * to Look": reference point plus offsets give the sampling locations; the weights are
 * blended over all L x P samples).  These calls take those raw pieces and compute
 *   location[b,q,m,l,p,k] = reference_points[b,q,l,k] + sampling_offsets[b,q,m,l,p,k] / E_lk
 *   A[b,q,m,:]            = softmax(attention_logits[b,q,m,:]) over the L x P samples
 * with E_l = (W_l, H_l[, Z_l]) (component k of an offset is in pixels of level l along
 * W, H, Z), then the core on them, without writing locations or weights to memory.
 *   reference_points  [B, Nq, L, 2|3]       fp32, normalised (x, y[, z]) per level
 *   sampling_offsets  [B, Nq, M, L, P, 2|3] fp32, pixels of the sampled level
 *   attention_logits  [B, Nq, M, L, P]      fp32
 * The location is formed in fp32 as written (IEEE division, then addition, both
 * round-to-nearest); the softmax uses the CUDA math library's expf in fp32.  All other
 * arguments, limits and errors are those of msda2d_forward / msda3d_forward;
 * reference_points must be non-null and 16-byte aligned.
 */
msda_status msda2d_forward_fused(const msda_dims *dims, const void *value,
                                 const int64_t *spatial_shapes, const int64_t *level_start_index,
                                 const float *reference_points, const float *sampling_offsets,
                                 const float *attention_logits, void *out, msda_stream_t stream);

msda_status msda3d_forward_fused(const msda_dims *dims, const void *value,
                                 const int64_t *spatial_shapes, const int64_t *level_start_index,
                                 const float *reference_points, const float *sampling_offsets,
                                 const float *attention_logits, void *out, msda_stream_t stream);

/*
 * Backward of msda2d_forward_fused / msda3d_forward_fused: the gradients of
 * sum(grad_out * out) with respect to value, the sampling offsets, the attention logits
 * and (optionally) the reference points ("3D Attention That Knows Where to Look": gradients
 * flow back into both the offsets and the weights; "Deformable Attention Module": the
 * weights are a softmax of predicted logits).  With grad_location and grad_A the core's
 * gradients at the fused locations and weights (as msda2d_backward defines them):
 *   grad_sampling_offsets[b,q,m,l,p,k] = grad_location[b,q,m,l,p,k] / E_lk
 *   grad_attention_logits[b,q,m,s]     = A_s * (grad_A_s - sum_t A_t * grad_A_t)
 *                                        (s, t over the item's L x P samples)
 *   grad_reference_points[b,q,l,k]     = sum over m and p of grad_location[b,q,m,l,p,k]
 *   grad_sampling_offsets  [B, Nq, M, L, P, 2|3] fp32, overwritten
 *   grad_attention_logits  [B, Nq, M, L, P]      fp32, overwritten
 *   grad_reference_points  [B, Nq, L, 2|3]       fp32, overwritten; may be NULL when the
 *                                                reference points need no gradient
 * grad_value is zero-filled by the call and accumulated with fp32 atomics, as in
 * msda2d_backward.  The locations and weights are formed exactly as the fused forward
 * forms them.  The backward kernel forms the logit gradients itself for the compiled
 * (L, P) pairs, and a second small kernel on the same stream forms them for the others;
 * the reference-point gradients (a sum in the order m, p) come from one more.  All
 * other arguments, limits and errors are those of msda2d_backward / msda3d_backward and
 * msda2d_forward_fused.
 */
msda_status msda2d_backward_fused(const msda_dims *dims, const void *value,
                                  const int64_t *spatial_shapes, const int64_t *level_start_index,
                                  const float *reference_points, const float *sampling_offsets,
                                  const float *attention_logits, const void *grad_out,
                                  float *grad_value, float *grad_sampling_offsets,
                                  float *grad_attention_logits, float *grad_reference_points,
                                  msda_stream_t stream);

msda_status msda3d_backward_fused(const msda_dims *dims, const void *value,
                                  const int64_t *spatial_shapes, const int64_t *level_start_index,
                                  const float *reference_points, const float *sampling_offsets,
                                  const float *attention_logits, const void *grad_out,
                                  float *grad_value, float *grad_sampling_offsets,
                                  float *grad_attention_logits, float *grad_reference_points,
                                  msda_stream_t stream);

/*
 * Probability-aware pruning of sampling points (an opt-in approximation; "DEFA: Efficient
 * Deformable Attention Acceleration via Pruning-Assisted Grid-Sampling and Multi-Scale
 * Parallel Processing", abstract: pruning of sampling points by their probability).
 * As msda2d_forward / msda3d_forward, except that every sample whose attention weight
 * has |A| < threshold is skipped: it contributes zero and its corner rows are not read.
 * threshold = 0 gives exactly the unpruned result.  For every output channel,
 *   |out_pruned - out| <= sum over skipped samples s of |A_s| * max_c |v_c|
 * where v_c runs over the in-level corner values of s in that channel (the corner weights
 * of a sample sum to at most 1).  threshold must be finite and >= 0 (else
 * MSDA_ERR_INVALID_ARG); all other arguments and errors are those of the forward.
 */
msda_status msda2d_forward_pruned(const msda_dims *dims, const void *value,
                                  const int64_t *spatial_shapes, const int64_t *level_start_index,
                                  const float *sampling_locations, const float *attention_weights,
                                  float threshold, void *out, msda_stream_t stream);

msda_status msda3d_forward_pruned(const msda_dims *dims, const void *value,
                                  const int64_t *spatial_shapes, const int64_t *level_start_index,
                                  const float *sampling_locations, const float *attention_weights,
                                  float threshold, void *out, msda_stream_t stream);

/*
 * Locality-aware query order.  The core's result does not depend on the order in which
 * queries are processed, but the speed of its gather does: queries whose samples land
 * close together reuse the same value rows when they run side by side.  This is the
 * feature-map reuse that "DEFA: Efficient Deformable Attention Acceleration via
 * Pruning-Assisted Grid-Sampling and Multi-Scale Parallel Processing" (abstract) names
 * among its memory-access savings, recast as a schedule for a GPU.
 *
 * msda_query_order writes query_order[B][Nq] (int32, device memory): for every batch b,
 * a permutation of 0 .. Nq-1 that sorts the queries by the Morton (Z-order) code of the
 * mean of their finite sampling locations (all heads, levels and points) on a 64 x 64
 * (2D) or 16 x 16 x 16 (3D) grid over the normalised square / cube.  Queries with equal
 * codes come in arbitrary order, which may differ between runs.  Only dims->B, Nq, M, L,
 * P are used (value_dtype, Nin and D are ignored); ndim is 2 or 3 and
 * sampling_locations is [B, Nq, M, L, P, ndim] fp32 as for the core.  It needs a
 * caller-owned device workspace of at least the size msda_query_order_workspace_size
 * reports (4 * B * (4096 + Nq) bytes plus alignment), 16-byte aligned; its contents on
 * entry are ignored and on return are unspecified.  Work is enqueued on `stream`.
 * Nq must be below 2^31.
 *
 * msda2d_forward_ordered / msda3d_forward_ordered compute exactly what msda2d_forward /
 * msda3d_forward compute (bit for bit: every item's arithmetic is unchanged), walking the
 * queries of batch b in the order query_order[b][0 .. Nq-1].  query_order must be a
 * permutation of 0 .. Nq-1 per batch (for example from msda_query_order; 4-byte
 * aligned, device memory).  Entries outside [0, Nq) are clamped into range, which gives
 * wrong results for the affected queries but never an out-of-range access; a query that
 * appears twice is computed twice and one that is missing is not written.
 *
 * msda2d_backward_ordered / msda3d_backward_ordered compute what msda2d_backward /
 * msda3d_backward compute, walking the queries of batch b in the order
 * query_order[b][0 .. Nq-1] (same requirements as for the ordered forward).  The location
 * and weight gradients of every sample are bit for bit those of the plain call; grad_value
 * equals it up to the order of the fp32 reductions, which is unspecified in both.  With
 * a locality order the work in flight covers a compact region of the maps for all heads
 * at once, so the value lines that neighbouring heads share are fetched once: on a B300
 * the volume backward (randomly placed queries) took 694 us per step against 725 us for
 * the plain call.
 * Queries that already come in a local order (raster order, as in an encoder) do better
 * with the plain call (397 us against 429 us on the encoder backward).  A query that appears
 * twice adds its grad_value contribution twice; one that is missing gets no location or
 * weight gradient written and adds nothing.
 */
msda_status msda_query_order_workspace_size(const msda_dims *dims, int32_t ndim, size_t *bytes);

msda_status msda_query_order(const msda_dims *dims, int32_t ndim, const float *sampling_locations,
                             int32_t *query_order, void *workspace, size_t workspace_bytes,
                             msda_stream_t stream);

/*
 * msda_query_order without a workspace and without any allocation.  The pages have no
 * counterpart: this is a service for callers that may not allocate device memory on
 * their path (a loop that forbids allocation once running, a plugin whose host owns all
 * device memory, a caller with nowhere to keep a workspace between calls).  The scratch
 * (per-batch histograms and per-query keys) is a fixed array of about 5 MB inside the
 * library's device image, present on every GPU that loads the library until the process
 * exits.  Limits: B <= 64 and B * Nq <= 1048576; larger problems return
 * MSDA_ERR_UNSUPPORTED (use msda_query_order with a workspace).  The output, arguments
 * and other errors are those of msda_query_order; no memory is allocated or freed.
 * The first call on each device looks up that device's copy of the array (make it with
 * the device current, before capturing any stream on that device).  All calls share the
 * array: each clears what it needs, but calls whose GPU work overlaps (other streams or
 * host threads) race on it and may return wrong orders; serialise them.
 */
msda_status msda_query_order_static(const msda_dims *dims, int32_t ndim,
                                    const float *sampling_locations, int32_t *query_order,
                                    msda_stream_t stream);

msda_status msda2d_forward_ordered(const msda_dims *dims, const void *value,
                                   const int64_t *spatial_shapes, const int64_t *level_start_index,
                                   const float *sampling_locations, const float *attention_weights,
                                   const int32_t *query_order, void *out, msda_stream_t stream);

msda_status msda3d_forward_ordered(const msda_dims *dims, const void *value,
                                   const int64_t *spatial_shapes, const int64_t *level_start_index,
                                   const float *sampling_locations, const float *attention_weights,
                                   const int32_t *query_order, void *out, msda_stream_t stream);

msda_status msda2d_backward_ordered(const msda_dims *dims, const void *value,
                                    const int64_t *spatial_shapes,
                                    const int64_t *level_start_index,
                                    const float *sampling_locations,
                                    const float *attention_weights, const int32_t *query_order,
                                    const void *grad_out, float *grad_value,
                                    float *grad_sampling_locations,
                                    float *grad_attention_weights, msda_stream_t stream);

msda_status msda3d_backward_ordered(const msda_dims *dims, const void *value,
                                    const int64_t *spatial_shapes,
                                    const int64_t *level_start_index,
                                    const float *sampling_locations,
                                    const float *attention_weights, const int32_t *query_order,
                                    const void *grad_out, float *grad_value,
                                    float *grad_sampling_locations,
                                    float *grad_attention_weights, msda_stream_t stream);

/* Message for the last non-OK status returned on this thread ("" if none).  The string
 * is owned by the library and stays valid until the next call on the same thread. */
const char *msda_last_error(void);

/* Version of this interface (major * 10000 + minor * 100 + patch). */
int32_t msda_abi_version(void);

/*
 * Bounds-checking build.  The pages fix no such facility; it is a debugging aid of this
 * library.  The same sources compiled with MSDA_DEBUG_BOUNDS give libmsda_debug.so, with
 * the same entry points: before every value-row access (loads in the forward and
 * backward, grad_value reductions in the backward) a kernel checks the corner's row index
 * against [0, Nin); a row outside that range is skipped, and the first one met on the
 * device is recorded (with its batch, query, head, level and point; no trap, no wait).
 * With correct index arithmetic and valid arguments nothing is ever recorded.
 *
 * msda_build_flags: MSDA_BUILD_DEBUG_BOUNDS when this library checks, else 0.
 * msda_debug_bounds_status: debug build: synchronises the current device, reads and
 *   clears its record, and returns MSDA_ERR_INTERNAL with the offender in
 *   msda_last_error() when one was recorded since the last call, else MSDA_OK.  Normal
 *   build: MSDA_OK (nothing is checked); no CUDA call.
 * msda_debug_bounds_selftest: debug build: enqueues on `stream` one thread that runs the
 *   kernels' check on a made-up offender (Nin = 10, row -5, batch 1, query 2, head 1,
 *   level 1, point 1 of Nq = 7, M = 3, P = 2), which the next status call reports; it
 *   touches no memory but the record.  Normal build: MSDA_ERR_UNSUPPORTED.
 * Records are per device; calls whose work overlaps on the GPU share the record.
 */
#define MSDA_BUILD_DEBUG_BOUNDS 1
int32_t msda_build_flags(void);
msda_status msda_debug_bounds_status(void);
msda_status msda_debug_bounds_selftest(msda_stream_t stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* MSDA_H_ */
