// Device-side building blocks shared by the libmsda kernels (sm_103a).
//
// Value rows are moved in 16-byte pieces: a "lane group" of G consecutive lanes owns one
// (batch, query, head) work item, and lane k of the group owns bytes [16k, 16k+16) of
// every D-channel value row the item touches (4 fp32 or 8 bf16 channels).  One warp-wide
// 16-byte load therefore fetches 32/G complete rows, each a contiguous, fully used span.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "msda_internal.h"

namespace msda {

// Channels held by one lane (16 bytes of the value dtype).
template <int DT> struct Vec;
template <> struct Vec<kF32> { static constexpr int N = 4; static constexpr int ESIZE = 4; };
template <> struct Vec<kBF16> { static constexpr int N = 8; static constexpr int ESIZE = 2; };

// Read-only 16-byte load through the non-coherent (texture/L1) path.
__device__ __forceinline__ uint4 ldg16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// 16 bytes of fp32 / bf16 channels -> fp32 registers.
__device__ __forceinline__ void unpack(const uint4 &u, float (&v)[4]) {
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack(const uint4 &u, float (&v)[8]) {
    // a bf16 is the high half of the fp32 with the same value
    v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
    v[4] = __uint_as_float(u.z << 16); v[5] = __uint_as_float(u.z & 0xffff0000u);
    v[6] = __uint_as_float(u.w << 16); v[7] = __uint_as_float(u.w & 0xffff0000u);
}

// fp32 registers -> 16 bytes of the value dtype (bf16: round to nearest even, once).
__device__ __forceinline__ uint4 pack(const float (&v)[4]) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[3]));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint4 pack(const float (&v)[8]) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                      pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

// Normalised location -> pixel coordinate on one axis: x = loc * extent - 0.5
// (align_corners = false).  Returns the cell index floor(x) and the fraction x - floor(x)
// of the EXACT coordinate, not of its fp32 rounding:
//
// * the product loc * extent is rounded once and its exact rounding error `err` is
//   recovered with an FMA; prod - 0.5 is exact for prod in [0.25, 2^23);
// * the fraction (x - floor(x)) + err is moved into [0, 1] by shifting the cell by one
//   when the error carries the coordinate across an integer.  The cell then agrees with
//   floor() of the exact coordinate, which matters for the location gradient: it jumps at
//   integer coordinates (the right-hand derivative of the cell chosen by floor() is used).
//   Rounding x itself to fp32 would also cost up to ~8e-6 px of accuracy at extent 150.
//
// Intrinsics with explicit rounding keep the compiler from contracting the product and
// the subtraction into one FMA, which would lose the error term.  The subtraction of 0.5
// is exact while |loc * extent| < 2^23 (the fp32 spacing there is at most 0.5); the ABI
// caps extents below 2^23, and a product beyond that belongs to a sample outside the level
// whichever way the subtraction rounds.
//
// A coordinate that is not finite or lies at or beyond -1 / the extent is reported as
// invalid (the function returns false; i0 = -2 and frac = 0 so no weight is NaN).  The
// caller ANDs the flags of all axes into every corner test: i0 = -2 alone does not fail
// the upper-bound test of the far corner.  When the flag is true, i0 is in [-1, extent-1],
// so a corner that passes its bound tests addresses a pixel inside the level.
__device__ __forceinline__ bool pixel_coord(float loc, float extent, int &i0, float &frac) {
    const float prod = __fmul_rn(loc, extent);
    const float err = __fmaf_rn(loc, extent, -prod);
    const float x = __fsub_rn(prod, 0.5f);
    float xf = floorf(x);
    float f = __fadd_rn(__fsub_rn(x, xf), err);
    if (f < 0.0f) {
        xf = __fsub_rn(xf, 1.0f);
        f = __fadd_rn(f, 1.0f);
    } else if (f >= 1.0f) {
        xf = __fadd_rn(xf, 1.0f);
        f = __fsub_rn(f, 1.0f);
    }
    // exact coordinate = xf + f with f in [0, 1]; it lies in (-1, extent) iff:
    const bool ok = (xf >= -1.0f) && (xf < extent) && (xf > -1.0f || f > 0.0f);
    frac = ok ? f : 0.0f;
    i0 = ok ? static_cast<int>(xf) : -2;
    return ok;
}

// Read-only 32-byte load (one 256-bit access; sm_100 and later).  `volatile` keeps the
// compiler from hoisting it above the caller's bounds test.
__device__ __forceinline__ void ldg32(const void *p, uint4 &a, uint4 &b) {
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                   "=r"(b.w)
                 : "l"(p));
}

// Vector reduction of 4 fp32 values into global memory (no return value).
__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    atomicAdd(reinterpret_cast<float4 *>(addr), make_float4(a, b, c, d));
}

// Sum over the G lanes of a lane group (G a power of two dividing 32); every lane of the
// warp must call it with the same G.
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Maximum over the G lanes of a lane group (same contract as group_sum).
template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Work item (b, q, m) at launch position `pos`.  Positions run over (b, i, m); the query
// is q = order[b * Nq + i] when a query order is given, else i.  Order entries are clamped
// into [0, Nq), so a malformed order gives wrong results but no out-of-range access.
__device__ __forceinline__ long long ordered_item(const Params &p, long long pos) {
    if (p.order == nullptr) return pos;
    const long long bi = pos / p.M;  // b * Nq + i
    const long long b = bi / p.Nq;
    int q = __ldg(p.order + bi);
    q = q < 0 ? 0 : (q >= p.Nq ? static_cast<int>(p.Nq - 1) : q);
    return (b * p.Nq + q) * p.M + (pos - bi * p.M);
}

// Fused prologue: normalised location of component k of a sample of level l of query
// (b, q): ref[b, q, l, k] + offset / extent, with IEEE round-to-nearest division and
// addition (an fp32 module computes the location the same way).
template <int NDIM>
__device__ __forceinline__ float fused_location(const Params &p, long long bq, int l, int k,
                                                float offset) {
    const float ext = k == 0 ? p.fW[l] : (k == 1 ? p.fH[l] : p.fZ[l]);
    const float r = __ldg(p.ref + (bq * p.L + l) * NDIM + k);
    return __fadd_rn(r, __fdiv_rn(offset, ext));
}

// Softmax statistics of an item's S logits (fused prologue, generic kernels and the
// backward epilogue): max and the sum of expf(z - max).
__device__ __forceinline__ void logit_stats(const float *z, int S, float &mx, float &sum) {
    mx = -INFINITY;
    for (int i = 0; i < S; ++i) mx = fmaxf(mx, __ldg(z + i));
    sum = 0.f;
    for (int i = 0; i < S; ++i) sum += expf(__ldg(z + i) - mx);
}

// ------------------------------------------------------------------ debug bounds checks

// row_ok(p, row, item, sample): true when the corner row index lies in [0, N_in).  In a
// build with MSDA_DEBUG_BOUNDS a row outside that range is recorded in *p.dbg (the first
// one only: the flag is claimed with atomicCAS, no trap, no wait) and the caller skips the
// access; in the normal build the function is the constant true and costs nothing.
__device__ __forceinline__ bool row_ok(const Params &p, long long row, long long item,
                                       int sample) {
#ifdef MSDA_DEBUG_BOUNDS
    if (row >= 0 && row < p.Nin) return true;
    DebugRecord *d = p.dbg;
    if (d != nullptr && atomicCAS(&d->flag, 0u, 1u) == 0u) {
        d->sample = sample;
        d->row = row;
        d->item = item;
        d->nin = p.Nin;
        d->nq = p.Nq;
        d->m_count = p.M;
        d->p_count = p.P;
        __threadfence();
        atomicExch(&d->flag, 2u);
    }
    return false;
#else
    (void)p; (void)row; (void)item; (void)sample;
    return true;
#endif
}

// ------------------------------------------------------------------ per-sample taps

constexpr unsigned kFull = 0xffffffffu;

// A sample whose attention weight is below p.prune in magnitude is treated like one that
// lies outside the level: no corner is valid, nothing is loaded, it contributes zero
// (probability-aware pruning; p.prune = 0 keeps every sample).
//
// Corner data ("taps") of one sample: value row of corner 0 (relative to the item's batch), one
// validity bit per corner (bit c: corner c lies inside the level) and the corner weights
// with the attention weight folded in (0 for corners outside).  Corner c has offsets
// dx = c & 1, dy = (c >> 1) & 1, dz = c >> 2.
template <int NC> struct Taps {
    int row;
    unsigned ok;
    float w[NC];
};

__device__ __forceinline__ void make_taps(const Params &p, int l, const float *xy, float a,
                                          Taps<4> &t, float *frac = nullptr) {
    int x0, y0;
    float fx, fy;
    const bool ok = pixel_coord(xy[0], p.fW[l], x0, fx) & pixel_coord(xy[1], p.fH[l], y0, fy) &
                    !(fabsf(a) < p.prune);
    const int W = p.W[l], H = p.H[l];
    const bool vx0 = ok && x0 >= 0, vx1 = ok && x0 < W - 1;
    const bool vy0 = y0 >= 0, vy1 = y0 < H - 1;
    t.ok = unsigned(vy0 && vx0) | unsigned(vy0 && vx1) << 1 | unsigned(vy1 && vx0) << 2 |
           unsigned(vy1 && vx1) << 3;
    const float ay0 = a * (1.f - fy), ay1 = a * fy;
    t.w[0] = (t.ok & 1u) ? ay0 * (1.f - fx) : 0.f;
    t.w[1] = (t.ok & 2u) ? ay0 * fx : 0.f;
    t.w[2] = (t.ok & 4u) ? ay1 * (1.f - fx) : 0.f;
    t.w[3] = (t.ok & 8u) ? ay1 * fx : 0.f;
    t.row = ok ? p.start[l] + y0 * W + x0 : 0;
    if (frac) {
        frac[0] = fx;
        frac[1] = fy;
    }
}

__device__ __forceinline__ void make_taps(const Params &p, int l, const float *xyz, float a,
                                          Taps<8> &t, float *frac = nullptr) {
    int x0, y0, z0;
    float fx, fy, fz;
    const bool ok = pixel_coord(xyz[0], p.fW[l], x0, fx) & pixel_coord(xyz[1], p.fH[l], y0, fy) &
                    pixel_coord(xyz[2], p.fZ[l], z0, fz) & !(fabsf(a) < p.prune);
    const int W = p.W[l], H = p.H[l], Z = p.Z[l];
    const bool vx[2] = {ok && x0 >= 0, ok && x0 < W - 1};
    const bool vy[2] = {y0 >= 0, y0 < H - 1};
    const bool vz[2] = {z0 >= 0, z0 < Z - 1};
    const float wx[2] = {1.f - fx, fx};
    const float wy[2] = {1.f - fy, fy};
    const float wz[2] = {a * (1.f - fz), a * fz};
    t.ok = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int dx = c & 1, dy = (c >> 1) & 1, dz = c >> 2;
        const bool in = vx[dx] && vy[dy] && vz[dz];
        t.ok |= unsigned(in) << c;
        t.w[c] = in ? (wz[dz] * wy[dy]) * wx[dx] : 0.f;
    }
    t.row = ok ? p.start[l] + (z0 * H + y0) * W + x0 : 0;
    if (frac) {
        frac[0] = fx;
        frac[1] = fy;
        frac[2] = fz;
    }
}

// Largest of 4, 2, 1 floats dividing x (alignment of a float offset, in floats).
__host__ __device__ constexpr int falign(int x) { return x % 4 == 0 ? 4 : (x % 2 == 0 ? 2 : 1); }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

// K consecutive floats starting at a pointer aligned to A floats, read once (streaming).
template <int K, int A>
__device__ __forceinline__ void load_stream(const float *src, float (&r)[K]) {
    if constexpr (A == 4 && K % 4 == 0) {
#pragma unroll
        for (int i = 0; i < K / 4; ++i) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(src) + i);
            r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
        }
    } else if constexpr (A >= 2 && K % 2 == 0) {
#pragma unroll
        for (int i = 0; i < K / 2; ++i) {
            const float2 v = __ldcs(reinterpret_cast<const float2 *>(src) + i);
            r[2 * i] = v.x; r[2 * i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i) r[i] = __ldcs(src + i);
    }
}

template <int NC>
__device__ __forceinline__ Taps<NC> shfl_taps(const Taps<NC> &t, int src, int width) {
    Taps<NC> r;
    r.row = __shfl_sync(kFull, t.row, src, width);
    r.ok = __shfl_sync(kFull, t.ok, src, width);
#pragma unroll
    for (int c = 0; c < NC; ++c) r.w[c] = __shfl_sync(kFull, t.w[c], src, width);
    return r;
}

// 2D taps with the four corner-validity bits carried under the row index: five shuffles
// instead of six.  The row of corner 0 lies in [-(W + 1), N_in), so it needs N_in < 2^27
// (and W < 2^23, which the ABI guarantees); the caller checks p.pack_taps.
__device__ __forceinline__ Taps<4> shfl_taps_packed(const Taps<4> &t, int src, int width) {
    Taps<4> r;
    const int v = __shfl_sync(kFull, static_cast<int>((static_cast<unsigned>(t.row) << 4) | t.ok),
                              src, width);
    r.row = v >> 4;
    r.ok = static_cast<unsigned>(v) & 15u;
#pragma unroll
    for (int c = 0; c < 4; ++c) r.w[c] = __shfl_sync(kFull, t.w[c], src, width);
    return r;
}

// ------------------------------------------------------------------ value-row slices

// VB bytes of one value row held by one lane (16: one 128-bit load; 32: one 256-bit load).
template <int VB> struct Slice;
template <> struct Slice<16> { uint4 a; };
template <> struct Slice<32> { uint4 a, b; };

__device__ __forceinline__ void load_slice(const char *p, Slice<16> &r) { r.a = ldg16(p); }
__device__ __forceinline__ void load_slice(const char *p, Slice<32> &r) { ldg32(p, r.a, r.b); }
__device__ __forceinline__ void zero_slice(Slice<16> &r) { r.a = make_uint4(0, 0, 0, 0); }
__device__ __forceinline__ void zero_slice(Slice<32> &r) {
    r.a = make_uint4(0, 0, 0, 0);
    r.b = r.a;
}

// Shared-memory slot of sample s of an item's tap records: one pad slot after every 8, so
// that the 8 lanes of a group writing their samples' records (two consecutive samples
// each) hit distinct banks.
__host__ __device__ constexpr int tap_slot(int s) { return s + (s >> 3); }

// Corner data ("tap record") of one sample, as the lane that computed it leaves it in
// shared memory for the other lanes of its group (forward and backward): x = value row of
// corner 0 (int bits; the forward may carry the validity bits under it), y = attention
// weight a, z / w = fractions fx / fy; 3D adds fz (and the validity bits when not packed)
// in second arrays.  A reader forms the corner weights from (a, fx, fy[, fz]) with
// tap_weights, the same expressions as make_taps, so its weights are bit-identical to the
// owner's.  Four words instead of the four weights: one shared-memory wavefront less per
// warp step in 2D.
template <int NC> struct TapView {
    int row;
    unsigned ok;
    float w[NC];
};

__device__ __forceinline__ void tap_weights(float a, float fx, float fy, float (&w)[4]) {
    const float ay0 = a * (1.f - fy), ay1 = a * fy;
    w[0] = ay0 * (1.f - fx);
    w[1] = ay0 * fx;
    w[2] = ay1 * (1.f - fx);
    w[3] = ay1 * fx;
}
__device__ __forceinline__ void tap_weights(float a, float fx, float fy, float fz, float (&w)[8]) {
    const float wx[2] = {1.f - fx, fx};
    const float wy[2] = {1.f - fy, fy};
    const float wz[2] = {a * (1.f - fz), a * fz};
#pragma unroll
    for (int c = 0; c < 8; ++c) w[c] = (wz[c >> 2] * wy[(c >> 1) & 1]) * wx[c & 1];
}

// Slice load under a predicate, without zeroing: when `pred` is false the destination
// holds an unspecified value and the caller must not read it (the matching FMAs are under
// the same predicate).  The empty asm gives the compiler a value to start from that costs
// no instruction; the load itself stays behind the branch.
__device__ __forceinline__ void load_slice_if(bool pred, const char *p, Slice<16> &r) {
    asm("" : "=r"(r.a.x), "=r"(r.a.y), "=r"(r.a.z), "=r"(r.a.w));
    if (pred) r.a = ldg16(p);
}
__device__ __forceinline__ void load_slice_if(bool pred, const char *p, Slice<32> &r) {
    asm("" : "=r"(r.a.x), "=r"(r.a.y), "=r"(r.a.z), "=r"(r.a.w), "=r"(r.b.x), "=r"(r.b.y),
             "=r"(r.b.z), "=r"(r.b.w));
    if (pred) ldg32(p, r.a, r.b);
}

}  // namespace msda
