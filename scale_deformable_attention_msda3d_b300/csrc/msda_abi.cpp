// C ABI of libmsda: host-side validation, parameter packing and dispatch.
// Nothing is enqueued unless every check passes; no memory is allocated.
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/msda.h"
#include "msda_internal.h"

namespace {

thread_local char g_err[512] = "";

msda_status fail(msda_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

bool mul_ok(int64_t a, int64_t b, int64_t *r) { return !__builtin_mul_overflow(a, b, r); }

bool misaligned(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; }

// Validates sizes and level metadata and fills the kernel parameters; *G receives the
// lanes per value row at 16 bytes per lane.
msda_status build_params(const msda_dims *d, int ndim, const int64_t *shapes,
                         const int64_t *level_start, msda::Params *p, int *G) {
    if (!d) return fail(MSDA_ERR_INVALID_ARG, "dims is NULL");
    if (d->value_dtype != MSDA_F32 && d->value_dtype != MSDA_BF16)
        return fail(MSDA_ERR_INVALID_ARG, "value_dtype %d is not MSDA_F32 or MSDA_BF16",
                    d->value_dtype);
    if (d->B < 0 || d->Nq < 0)
        return fail(MSDA_ERR_INVALID_ARG, "B (%lld) and Nq (%lld) must be >= 0",
                    (long long)d->B, (long long)d->Nq);
    if (d->Nin < 1 || d->M < 1 || d->D < 1 || d->L < 1 || d->P < 1)
        return fail(MSDA_ERR_INVALID_ARG, "Nin, M, D, L, P must be >= 1 (got %lld %d %d %d %d)",
                    (long long)d->Nin, d->M, d->D, d->L, d->P);
    if (d->L > MSDA_MAX_LEVELS)
        return fail(MSDA_ERR_UNSUPPORTED, "L = %d exceeds MSDA_MAX_LEVELS = %d", d->L,
                    MSDA_MAX_LEVELS);
    if (d->P > MSDA_MAX_POINTS)
        return fail(MSDA_ERR_UNSUPPORTED, "P = %d exceeds MSDA_MAX_POINTS = %d", d->P,
                    MSDA_MAX_POINTS);
    if (d->Nin > (int64_t(1) << 30))
        return fail(MSDA_ERR_UNSUPPORTED, "Nin = %lld must be at most 2^30", (long long)d->Nin);
    if (!shapes || !level_start)
        return fail(MSDA_ERR_INVALID_ARG, "spatial_shapes / level_start_index is NULL");

    const int esize = d->value_dtype == MSDA_F32 ? 4 : 2;
    const int64_t dbytes = int64_t(d->D) * esize;
    if (dbytes % 16 != 0 || dbytes > 512 || ((dbytes / 16) & (dbytes / 16 - 1)) != 0)
        return fail(MSDA_ERR_UNSUPPORTED,
                    "D * sizeof(dtype) = %lld bytes; supported: 16, 32, 64, 128, 256, 512",
                    (long long)dbytes);
    *G = int(dbytes / 16);
    if (int64_t(d->M) * dbytes > INT32_MAX)
        return fail(MSDA_ERR_UNSUPPORTED, "M * D * sizeof(dtype) = %lld bytes must be below 2^31",
                    (long long)(int64_t(d->M) * dbytes));

    int64_t total = 0;
    for (int l = 0; l < d->L; ++l) {
        int64_t size = 1;
        for (int k = 0; k < ndim; ++k) {
            const int64_t e = shapes[l * ndim + k];
            if (e < 1)
                return fail(MSDA_ERR_INVALID_ARG, "spatial_shapes[%d][%d] = %lld must be >= 1",
                            l, k, (long long)e);
            // the kernels form loc * extent - 0.5 exactly in fp32 (product error by FMA, the
            // subtraction exact), which holds while the product stays below 2^23
            if (e >= (int64_t(1) << 23))
                return fail(MSDA_ERR_UNSUPPORTED,
                            "spatial_shapes[%d][%d] = %lld: extents of 2^23 pixels or more "
                            "are not supported", l, k, (long long)e);
            if (!mul_ok(size, e, &size) || size > (int64_t(1) << 30))
                return fail(MSDA_ERR_INVALID_ARG, "level %d has too many pixels", l);
        }
        if (level_start[l] != total)
            return fail(MSDA_ERR_INVALID_ARG,
                        "level_start_index[%d] = %lld, expected the prefix sum %lld", l,
                        (long long)level_start[l], (long long)total);
        total += size;
        if (total > d->Nin) break;
    }
    if (total != d->Nin)
        return fail(MSDA_ERR_INVALID_ARG, "level sizes add up to %lld, Nin is %lld",
                    (long long)total, (long long)d->Nin);

    int64_t t;
    if (!mul_ok(d->B, d->Nin, &t) || !mul_ok(t, d->M, &t) || !mul_ok(t, d->D, &t) ||
        !mul_ok(t, 4, &t))
        return fail(MSDA_ERR_INVALID_ARG, "B * Nin * M * D overflows");
    int64_t items;
    if (!mul_ok(d->B, d->Nq, &items) || !mul_ok(items, d->M, &items) ||
        !mul_ok(items, int64_t(d->L) * d->P * 3 * 4, &t) || !mul_ok(items, 32, &t))
        return fail(MSDA_ERR_INVALID_ARG, "B * Nq * M * L * P overflows");

    std::memset(p, 0, sizeof(*p));
    p->B = d->B;
    p->Nin = d->Nin;
    p->Nq = d->Nq;
    p->M = d->M;
    p->D = d->D;
    p->L = d->L;
    p->P = d->P;
    p->n_items = items;
    p->row_bytes = int64_t(d->M) * dbytes;
    p->rb32 = int(p->row_bytes);
    p->pinv = int((65536 + d->P - 1) / d->P);
    // the forward's tap records may carry the corner-validity bits under the row of corner
    // 0 (4 bits in 2D, 8 in 3D) while that row, in [-(H*W + W + 1), N_in), fits the rest
    p->pack_taps = d->Nin < (int64_t(1) << (ndim == 2 ? 27 : 22)) ? 1 : 0;
    for (int l = 0; l < d->L; ++l) {
        const int64_t *s = shapes + l * ndim;
        p->W[l] = int(s[ndim - 1]);
        p->H[l] = int(s[ndim - 2]);
        p->Z[l] = ndim == 3 ? int(s[0]) : 1;
        p->fW[l] = float(p->W[l]);
        p->fH[l] = float(p->H[l]);
        p->fZ[l] = float(p->Z[l]);
        p->start[l] = int(level_start[l]);
        p->sy[l] = int64_t(p->W[l]) * p->row_bytes;
        p->sz[l] = int64_t(p->H[l]) * p->W[l] * p->row_bytes;
    }
    return MSDA_OK;
}

msda_status check_ptr(const void *ptr, const char *name) {
    if (!ptr) return fail(MSDA_ERR_INVALID_ARG, "%s is NULL", name);
    if (misaligned(ptr)) return fail(MSDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return MSDA_OK;
}

#define MSDA_TRY(expr)                         \
    do {                                       \
        const msda_status st_ = (expr);        \
        if (st_ != MSDA_OK) return st_;        \
    } while (0)

msda_status cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return MSDA_OK;
    return fail(MSDA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

msda_status forward_impl(int ndim, const msda_dims *dims, const void *value,
                         const int64_t *shapes, const int64_t *level_start, const float *loc,
                         const float *attn, const int32_t *order, bool ordered, void *out,
                         msda_stream_t stream, float prune = 0.f,
                         const float *ref = nullptr, bool fused = false) {
    msda::Params p;
    int G = 0;
    MSDA_TRY(build_params(dims, ndim, shapes, level_start, &p, &G));
    if (p.n_items == 0) return MSDA_OK;  // empty batch or no queries: nothing to compute
    MSDA_TRY(check_ptr(value, "value"));
    MSDA_TRY(check_ptr(loc, fused ? "sampling_offsets" : "sampling_locations"));
    MSDA_TRY(check_ptr(attn, fused ? "attention_logits" : "attention_weights"));
    MSDA_TRY(check_ptr(out, "out"));
    if (ordered) {
        if (!order) return fail(MSDA_ERR_INVALID_ARG, "query_order is NULL");
        if ((reinterpret_cast<uintptr_t>(order) & 3u) != 0)
            return fail(MSDA_ERR_INVALID_ARG, "query_order is not 4-byte aligned");
        if (dims->Nq > INT32_MAX)
            return fail(MSDA_ERR_UNSUPPORTED, "Nq = %lld: a query order needs Nq < 2^31",
                        (long long)dims->Nq);
    }
    p.value = value;
    p.loc = loc;
    p.attn = attn;
    p.out = out;
    if (fused) MSDA_TRY(check_ptr(ref, "reference_points"));
    p.order = ordered ? order : nullptr;
    p.prune = prune;
    p.ref = fused ? ref : nullptr;
#ifdef MSDA_DEBUG_BOUNDS
    MSDA_TRY(cuda_status(msda::debug_record(&p.dbg), "bounds-check record"));
#endif
    return cuda_status(msda::launch_forward(ndim, dims->value_dtype, G, p,
                                            reinterpret_cast<cudaStream_t>(stream)),
                       "forward launch");
}

msda_status backward_impl(int ndim, const msda_dims *dims, const void *value,
                          const int64_t *shapes, const int64_t *level_start, const float *loc,
                          const float *attn, const void *grad_out, float *grad_value,
                          float *grad_loc, float *grad_attn, msda_stream_t stream,
                          const float *ref = nullptr, float *grad_ref = nullptr,
                          bool fused = false, const int32_t *order = nullptr,
                          bool ordered = false) {
    msda::Params p;
    int G = 0;
    MSDA_TRY(build_params(dims, ndim, shapes, level_start, &p, &G));
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dims->B == 0) return MSDA_OK;
    MSDA_TRY(check_ptr(grad_value, "grad_value"));
    if (p.n_items > 0) {
        MSDA_TRY(check_ptr(value, "value"));
        MSDA_TRY(check_ptr(loc, fused ? "sampling_offsets" : "sampling_locations"));
        MSDA_TRY(check_ptr(attn, fused ? "attention_logits" : "attention_weights"));
        MSDA_TRY(check_ptr(grad_out, "grad_out"));
        MSDA_TRY(check_ptr(grad_loc, fused ? "grad_sampling_offsets" : "grad_sampling_locations"));
        MSDA_TRY(check_ptr(grad_attn, fused ? "grad_attention_logits" : "grad_attention_weights"));
        if (fused) {
            MSDA_TRY(check_ptr(ref, "reference_points"));
            if (grad_ref) MSDA_TRY(check_ptr(grad_ref, "grad_reference_points"));
        }
        if (ordered) {
            if (!order) return fail(MSDA_ERR_INVALID_ARG, "query_order is NULL");
            if ((reinterpret_cast<uintptr_t>(order) & 3u) != 0)
                return fail(MSDA_ERR_INVALID_ARG, "query_order is not 4-byte aligned");
            if (dims->Nq > INT32_MAX)
                return fail(MSDA_ERR_UNSUPPORTED, "Nq = %lld: a query order needs Nq < 2^31",
                            (long long)dims->Nq);
        }
    }
    MSDA_TRY(cuda_status(msda::launch_zero_fill(grad_value, p.B * p.Nin * p.M * p.D, s),
                         "grad_value zero-fill launch"));
    p.value = value;
    p.loc = loc;
    p.attn = attn;
    p.grad_out = grad_out;
    p.grad_value = grad_value;
    p.grad_loc = grad_loc;
    p.grad_attn = grad_attn;
    p.ref = fused ? ref : nullptr;
    p.grad_ref = fused ? grad_ref : nullptr;
    p.order = ordered ? order : nullptr;
#ifdef MSDA_DEBUG_BOUNDS
    MSDA_TRY(cuda_status(msda::debug_record(&p.dbg), "bounds-check record"));
#endif
    return cuda_status(msda::launch_backward(ndim, dims->value_dtype, G, p, s),
                       fused ? "fused backward launch" : "backward launch");
}

// Workspace of msda_query_order: per-batch histogram, then per-query keys (256-byte aligned).
int64_t order_hist_bytes(int64_t B) { return B * msda::kOrderBuckets * int64_t(sizeof(int)); }
int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

msda_status order_dims(const msda_dims *d, int ndim, int64_t *bytes) {
    if (!d) return fail(MSDA_ERR_INVALID_ARG, "dims is NULL");
    if (ndim != 2 && ndim != 3) return fail(MSDA_ERR_INVALID_ARG, "ndim = %d must be 2 or 3", ndim);
    if (d->B < 0 || d->Nq < 0)
        return fail(MSDA_ERR_INVALID_ARG, "B (%lld) and Nq (%lld) must be >= 0",
                    (long long)d->B, (long long)d->Nq);
    if (d->M < 1 || d->L < 1 || d->P < 1)
        return fail(MSDA_ERR_INVALID_ARG, "M, L, P must be >= 1 (got %d %d %d)", d->M, d->L, d->P);
    if (d->Nq > INT32_MAX) return fail(MSDA_ERR_UNSUPPORTED, "Nq must be below 2^31");
    int64_t per = 0, t = 0;
    if (!mul_ok(int64_t(d->M) * d->L, d->P, &per) || !mul_ok(d->B, d->Nq, &t) ||
        !mul_ok(t, per * ndim * 4, &t) || !mul_ok(d->B, msda::kOrderBuckets * 4, &t) ||
        per > INT32_MAX)
        return fail(MSDA_ERR_INVALID_ARG, "sizes overflow");
    *bytes = align256(order_hist_bytes(d->B)) + align256(d->B * d->Nq * int64_t(sizeof(int)));
    return MSDA_OK;
}

}  // namespace

extern "C" {

msda_status msda_query_order_workspace_size(const msda_dims *dims, int32_t ndim, size_t *bytes) {
    if (!bytes) return fail(MSDA_ERR_INVALID_ARG, "bytes is NULL");
    int64_t b = 0;
    MSDA_TRY(order_dims(dims, ndim, &b));
    *bytes = static_cast<size_t>(b);
    return MSDA_OK;
}

msda_status msda_query_order(const msda_dims *dims, int32_t ndim, const float *sampling_locations,
                             int32_t *query_order, void *workspace, size_t workspace_bytes,
                             msda_stream_t stream) {
    int64_t need = 0;
    MSDA_TRY(order_dims(dims, ndim, &need));
    if (dims->B == 0 || dims->Nq == 0) return MSDA_OK;
    MSDA_TRY(check_ptr(sampling_locations, "sampling_locations"));
    if (!query_order) return fail(MSDA_ERR_INVALID_ARG, "query_order is NULL");
    if ((reinterpret_cast<uintptr_t>(query_order) & 3u) != 0)
        return fail(MSDA_ERR_INVALID_ARG, "query_order is not 4-byte aligned");
    MSDA_TRY(check_ptr(workspace, "workspace"));
    if (static_cast<int64_t>(workspace_bytes) < need)
        return fail(MSDA_ERR_INVALID_ARG, "workspace has %zu bytes, %lld needed", workspace_bytes,
                    (long long)need);
    msda::Params p;
    std::memset(&p, 0, sizeof(p));
    p.B = dims->B;
    p.Nq = dims->Nq;
    p.M = dims->M;
    p.L = dims->L;
    p.P = dims->P;
    p.loc = sampling_locations;
    char *ws = static_cast<char *>(workspace);
    int *hist = reinterpret_cast<int *>(ws);
    int *keys = reinterpret_cast<int *>(ws + align256(order_hist_bytes(dims->B)));
    return cuda_status(msda::launch_query_order(ndim, p, query_order, hist, keys,
                                                reinterpret_cast<cudaStream_t>(stream)),
                       "query order launch");
}

msda_status msda_query_order_static(const msda_dims *dims, int32_t ndim,
                                    const float *sampling_locations, int32_t *query_order,
                                    msda_stream_t stream) {
    int64_t need = 0;
    MSDA_TRY(order_dims(dims, ndim, &need));
    if (!msda::static_order_fits(dims->B, dims->Nq))
        return fail(MSDA_ERR_UNSUPPORTED,
                    "msda_query_order_static holds at most B = 64 and B * Nq = 1048576 queries "
                    "(got B = %lld, B * Nq = %lld); use msda_query_order with a workspace",
                    (long long)dims->B, (long long)(dims->B * dims->Nq));
    if (dims->B == 0 || dims->Nq == 0) return MSDA_OK;
    MSDA_TRY(check_ptr(sampling_locations, "sampling_locations"));
    if (!query_order) return fail(MSDA_ERR_INVALID_ARG, "query_order is NULL");
    if ((reinterpret_cast<uintptr_t>(query_order) & 3u) != 0)
        return fail(MSDA_ERR_INVALID_ARG, "query_order is not 4-byte aligned");
    msda::Params p;
    std::memset(&p, 0, sizeof(p));
    p.B = dims->B;
    p.Nq = dims->Nq;
    p.M = dims->M;
    p.L = dims->L;
    p.P = dims->P;
    p.loc = sampling_locations;
    return cuda_status(msda::launch_query_order_static(ndim, p, query_order,
                                                       reinterpret_cast<cudaStream_t>(stream)),
                       "query order (fixed scratch) launch");
}

msda_status msda2d_forward_fused(const msda_dims *dims, const void *value,
                                 const int64_t *spatial_shapes, const int64_t *level_start_index,
                                 const float *reference_points, const float *sampling_offsets,
                                 const float *attention_logits, void *out, msda_stream_t stream) {
    return forward_impl(2, dims, value, spatial_shapes, level_start_index, sampling_offsets,
                        attention_logits, nullptr, false, out, stream, 0.f, reference_points,
                        true);
}

msda_status msda3d_forward_fused(const msda_dims *dims, const void *value,
                                 const int64_t *spatial_shapes, const int64_t *level_start_index,
                                 const float *reference_points, const float *sampling_offsets,
                                 const float *attention_logits, void *out, msda_stream_t stream) {
    return forward_impl(3, dims, value, spatial_shapes, level_start_index, sampling_offsets,
                        attention_logits, nullptr, false, out, stream, 0.f, reference_points,
                        true);
}

msda_status msda2d_forward_pruned(const msda_dims *dims, const void *value,
                                  const int64_t *spatial_shapes, const int64_t *level_start_index,
                                  const float *sampling_locations, const float *attention_weights,
                                  float threshold, void *out, msda_stream_t stream) {
    if (!(threshold >= 0.f) || threshold == INFINITY)
        return fail(MSDA_ERR_INVALID_ARG, "threshold must be finite and >= 0");
    return forward_impl(2, dims, value, spatial_shapes, level_start_index, sampling_locations,
                        attention_weights, nullptr, false, out, stream, threshold);
}

msda_status msda3d_forward_pruned(const msda_dims *dims, const void *value,
                                  const int64_t *spatial_shapes, const int64_t *level_start_index,
                                  const float *sampling_locations, const float *attention_weights,
                                  float threshold, void *out, msda_stream_t stream) {
    if (!(threshold >= 0.f) || threshold == INFINITY)
        return fail(MSDA_ERR_INVALID_ARG, "threshold must be finite and >= 0");
    return forward_impl(3, dims, value, spatial_shapes, level_start_index, sampling_locations,
                        attention_weights, nullptr, false, out, stream, threshold);
}

msda_status msda2d_forward_ordered(const msda_dims *dims, const void *value,
                                   const int64_t *spatial_shapes, const int64_t *level_start_index,
                                   const float *sampling_locations, const float *attention_weights,
                                   const int32_t *query_order, void *out, msda_stream_t stream) {
    return forward_impl(2, dims, value, spatial_shapes, level_start_index, sampling_locations,
                        attention_weights, query_order, true, out, stream);
}

msda_status msda3d_forward_ordered(const msda_dims *dims, const void *value,
                                   const int64_t *spatial_shapes, const int64_t *level_start_index,
                                   const float *sampling_locations, const float *attention_weights,
                                   const int32_t *query_order, void *out, msda_stream_t stream) {
    return forward_impl(3, dims, value, spatial_shapes, level_start_index, sampling_locations,
                        attention_weights, query_order, true, out, stream);
}

msda_status msda2d_forward(const msda_dims *dims, const void *value,
                           const int64_t *spatial_shapes, const int64_t *level_start_index,
                           const float *sampling_locations, const float *attention_weights,
                           void *out, msda_stream_t stream) {
    return forward_impl(2, dims, value, spatial_shapes, level_start_index, sampling_locations,
                        attention_weights, nullptr, false, out, stream);
}

msda_status msda3d_forward(const msda_dims *dims, const void *value,
                           const int64_t *spatial_shapes, const int64_t *level_start_index,
                           const float *sampling_locations, const float *attention_weights,
                           void *out, msda_stream_t stream) {
    return forward_impl(3, dims, value, spatial_shapes, level_start_index, sampling_locations,
                        attention_weights, nullptr, false, out, stream);
}

msda_status msda2d_backward(const msda_dims *dims, const void *value,
                            const int64_t *spatial_shapes, const int64_t *level_start_index,
                            const float *sampling_locations, const float *attention_weights,
                            const void *grad_out, float *grad_value,
                            float *grad_sampling_locations, float *grad_attention_weights,
                            msda_stream_t stream) {
    return backward_impl(2, dims, value, spatial_shapes, level_start_index, sampling_locations,
                         attention_weights, grad_out, grad_value, grad_sampling_locations,
                         grad_attention_weights, stream);
}

msda_status msda3d_backward(const msda_dims *dims, const void *value,
                            const int64_t *spatial_shapes, const int64_t *level_start_index,
                            const float *sampling_locations, const float *attention_weights,
                            const void *grad_out, float *grad_value,
                            float *grad_sampling_locations, float *grad_attention_weights,
                            msda_stream_t stream) {
    return backward_impl(3, dims, value, spatial_shapes, level_start_index, sampling_locations,
                         attention_weights, grad_out, grad_value, grad_sampling_locations,
                         grad_attention_weights, stream);
}

msda_status msda2d_backward_ordered(const msda_dims *dims, const void *value,
                                    const int64_t *spatial_shapes,
                                    const int64_t *level_start_index,
                                    const float *sampling_locations,
                                    const float *attention_weights, const int32_t *query_order,
                                    const void *grad_out, float *grad_value,
                                    float *grad_sampling_locations,
                                    float *grad_attention_weights, msda_stream_t stream) {
    return backward_impl(2, dims, value, spatial_shapes, level_start_index, sampling_locations,
                         attention_weights, grad_out, grad_value, grad_sampling_locations,
                         grad_attention_weights, stream, nullptr, nullptr, false, query_order,
                         true);
}

msda_status msda3d_backward_ordered(const msda_dims *dims, const void *value,
                                    const int64_t *spatial_shapes,
                                    const int64_t *level_start_index,
                                    const float *sampling_locations,
                                    const float *attention_weights, const int32_t *query_order,
                                    const void *grad_out, float *grad_value,
                                    float *grad_sampling_locations,
                                    float *grad_attention_weights, msda_stream_t stream) {
    return backward_impl(3, dims, value, spatial_shapes, level_start_index, sampling_locations,
                         attention_weights, grad_out, grad_value, grad_sampling_locations,
                         grad_attention_weights, stream, nullptr, nullptr, false, query_order,
                         true);
}

msda_status msda2d_backward_fused(const msda_dims *dims, const void *value,
                                  const int64_t *spatial_shapes, const int64_t *level_start_index,
                                  const float *reference_points, const float *sampling_offsets,
                                  const float *attention_logits, const void *grad_out,
                                  float *grad_value, float *grad_sampling_offsets,
                                  float *grad_attention_logits, float *grad_reference_points,
                                  msda_stream_t stream) {
    return backward_impl(2, dims, value, spatial_shapes, level_start_index, sampling_offsets,
                         attention_logits, grad_out, grad_value, grad_sampling_offsets,
                         grad_attention_logits, stream, reference_points, grad_reference_points,
                         true);
}

msda_status msda3d_backward_fused(const msda_dims *dims, const void *value,
                                  const int64_t *spatial_shapes, const int64_t *level_start_index,
                                  const float *reference_points, const float *sampling_offsets,
                                  const float *attention_logits, const void *grad_out,
                                  float *grad_value, float *grad_sampling_offsets,
                                  float *grad_attention_logits, float *grad_reference_points,
                                  msda_stream_t stream) {
    return backward_impl(3, dims, value, spatial_shapes, level_start_index, sampling_offsets,
                         attention_logits, grad_out, grad_value, grad_sampling_offsets,
                         grad_attention_logits, stream, reference_points, grad_reference_points,
                         true);
}

int32_t msda_build_flags(void) {
#ifdef MSDA_DEBUG_BOUNDS
    return MSDA_BUILD_DEBUG_BOUNDS;
#else
    return 0;
#endif
}

msda_status msda_debug_bounds_status(void) {
#ifdef MSDA_DEBUG_BOUNDS
    msda::DebugRecord r;
    MSDA_TRY(cuda_status(msda::debug_record_take(&r), "reading the bounds-check record"));
    if (r.flag == 0) return MSDA_OK;
    const long long M = r.m_count > 0 ? r.m_count : 1, P = r.p_count > 0 ? r.p_count : 1;
    const long long Nq = r.nq > 0 ? r.nq : 1;
    const long long bq = r.item / M;
    return fail(MSDA_ERR_INTERNAL,
                "bounds check: corner row %lld outside [0, %lld) at batch %lld, query %lld, "
                "head %lld, level %lld, point %lld",
                r.row, r.nin, bq / Nq, bq % Nq, r.item % M, (long long)r.sample / P,
                (long long)r.sample % P);
#else
    return MSDA_OK;
#endif
}

msda_status msda_debug_bounds_selftest(msda_stream_t stream) {
#ifdef MSDA_DEBUG_BOUNDS
    // a made-up offender: N_in = 10, Nq = 7, M = 3, P = 2; row -5 at item (b=1, q=2, m=1),
    // sample (l=1, p=1); the check records it and nothing is accessed
    msda::Params p;
    std::memset(&p, 0, sizeof(p));
    p.Nin = 10;
    p.Nq = 7;
    p.M = 3;
    p.P = 2;
    MSDA_TRY(cuda_status(msda::debug_record(&p.dbg), "bounds-check record"));
    return cuda_status(msda::launch_debug_selftest(p, -5, (1 * 7 + 2) * 3 + 1, 1 * 2 + 1,
                                                   reinterpret_cast<cudaStream_t>(stream)),
                       "bounds-check self-test launch");
#else
    (void)stream;
    return fail(MSDA_ERR_UNSUPPORTED,
                "bounds checks are compiled only into the debug build (MSDA_DEBUG_BOUNDS)");
#endif
}

const char *msda_last_error(void) { return g_err; }

int32_t msda_abi_version(void) { return 10300; }

}  // extern "C"
