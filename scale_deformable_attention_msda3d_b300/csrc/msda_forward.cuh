// Forward kernels: multi-scale deformable attention sampling + weighted sum.  This header
// holds the kernel templates; msda_forward_{f32,bf16}_{2d,3d}.cu instantiate them for one
// value dtype and dimensionality each (so the build compiles them in parallel), and
// msda_forward.cu dispatches.
//
// out[b,q,m,:] = sum_l sum_p A[b,q,m,l,p] * interp_l(value[b, level l, m, :], loc[b,q,m,l,p])
// ("Deformable Attention Module", DeformAttn equation; multi-scale blending and the 2D->3D
// changes from "3D Attention That Knows Where to Look").
//
// Mapping: a lane group of G lanes per (b, q, m) work item; lane k owns 16 bytes of
// channels, so a warp-wide 16-byte load brings 32/G whole value rows.  Corners outside
// the level are neither loaded nor weighted.  fp32 accumulation; one store of the item's
// D channels at the end.
//
// With a fused prologue (Params::ref set), `loc` holds per-sample offsets in pixels of the
// sampled level and `attn` the attention logits: the kernels form location = reference +
// offset / extent and the softmax of the item's L * P logits themselves.
//
// Two kernels:
// * fwd_tiled (the compiled (L, P) pairs): the locations and weights of an item are read
//   once with vector loads, spread over the lanes of its group; each lane works out the
//   cell, corner validity and fractions of its own samples and leaves them in shared
//   memory (one 16-byte record per sample), and the group then walks the samples in
//   order, reading each sample's record, loading the corner rows of the next AHEAD samples
//   (in-level corners only, without zeroing the others) before summing the current one
//   under the same per-corner predicates.  Optionally the item's samples are split over
//   SPLIT lane groups whose partial sums are added by shuffles at the end (fewer taps per
//   lane for narrow rows, more loads in flight when there are few items).  3D uses
//   32-byte (256-bit) loads per lane.
// * fwd{2,3}d_generic (any L, P): every lane of the group computes every sample itself.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace msda {

namespace {

template <int DT, int G, int LL, int PP, bool FUSED>
__global__ void __launch_bounds__(256)
fwd2d_generic(const __grid_constant__ Params p) {
    constexpr int N = Vec<DT>::N;
    const int L = LL > 0 ? LL : p.L;
    const int P = PP > 0 ? PP : p.P;
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t / G >= p.n_items) return;
    const long long item = ordered_item(p, t / G);
    const int sub = threadIdx.x & (G - 1);
    const int m = static_cast<int>(item % p.M);
    const long long b = item / p.M / p.Nq;
    const long long rb = p.row_bytes;
    const char *vb = static_cast<const char *>(p.value) + (b * p.Nin) * rb +
                     static_cast<long long>(m) * (rb / p.M) + sub * 16;
    const float2 *lp = reinterpret_cast<const float2 *>(p.loc) + item * L * P;
    const float *ap = p.attn + item * L * P;
    float zmax = 0.f, zsum = 1.f;
    if constexpr (FUSED) logit_stats(ap, L * P, zmax, zsum);

    float acc[N];
#pragma unroll
    for (int i = 0; i < N; ++i) acc[i] = 0.f;

#pragma unroll
    for (int l = 0; l < L; ++l) {
        const int W = p.W[l], H = p.H[l];
        const float fW = p.fW[l], fH = p.fH[l];
        const char *vl = vb + static_cast<long long>(p.start[l]) * rb;
#pragma unroll 4
        for (int k = 0; k < P; ++k) {
            float2 xy = __ldg(lp + l * P + k);
            float a = __ldg(ap + l * P + k);
            if constexpr (FUSED) {
                const long long bq = item / p.M;
                xy.x = fused_location<2>(p, bq, l, 0, xy.x);
                xy.y = fused_location<2>(p, bq, l, 1, xy.y);
                a = __fdiv_rn(expf(a - zmax), zsum);
            }
            int x0, y0;
            float fx, fy;
            const bool okx = pixel_coord(xy.x, fW, x0, fx);
            const bool oky = pixel_coord(xy.y, fH, y0, fy);
            const bool ok = okx && oky && !(fabsf(a) < p.prune);
            const bool vx0 = ok && x0 >= 0, vx1 = ok && x0 < W - 1;
            const bool vy0 = y0 >= 0, vy1 = y0 < H - 1;
            const long long r00 = p.start[l] + static_cast<long long>(y0) * W + x0;
            const int sidx = l * P + k;
            const bool k00 = vy0 && vx0 && row_ok(p, r00, item, sidx);
            const bool k01 = vy0 && vx1 && row_ok(p, r00 + 1, item, sidx);
            const bool k10 = vy1 && vx0 && row_ok(p, r00 + W, item, sidx);
            const bool k11 = vy1 && vx1 && row_ok(p, r00 + W + 1, item, sidx);
            const float ay0 = a * (1.f - fy), ay1 = a * fy;
            const float w00 = k00 ? ay0 * (1.f - fx) : 0.f;
            const float w01 = k01 ? ay0 * fx : 0.f;
            const float w10 = k10 ? ay1 * (1.f - fx) : 0.f;
            const float w11 = k11 ? ay1 * fx : 0.f;
            const char *c00 = vl + static_cast<long long>(y0 * W + x0) * rb;
            uint4 u00 = make_uint4(0, 0, 0, 0), u01 = u00, u10 = u00, u11 = u00;
            if (k00) u00 = ldg16(c00);
            if (k01) u01 = ldg16(c00 + rb);
            if (k10) u10 = ldg16(c00 + W * rb);
            if (k11) u11 = ldg16(c00 + (W + 1) * rb);
            float v[N];
            unpack(u00, v);
#pragma unroll
            for (int i = 0; i < N; ++i) acc[i] = fmaf(w00, v[i], acc[i]);
            unpack(u01, v);
#pragma unroll
            for (int i = 0; i < N; ++i) acc[i] = fmaf(w01, v[i], acc[i]);
            unpack(u10, v);
#pragma unroll
            for (int i = 0; i < N; ++i) acc[i] = fmaf(w10, v[i], acc[i]);
            unpack(u11, v);
#pragma unroll
            for (int i = 0; i < N; ++i) acc[i] = fmaf(w11, v[i], acc[i]);
        }
    }
    char *o = static_cast<char *>(p.out) + item * (rb / p.M) + sub * 16;
    *reinterpret_cast<uint4 *>(o) = pack(acc);
}

template <int DT, int G, int LL, int PP, bool FUSED>
__global__ void __launch_bounds__(256)
fwd3d_generic(const __grid_constant__ Params p) {
    constexpr int N = Vec<DT>::N;
    const int L = LL > 0 ? LL : p.L;
    const int P = PP > 0 ? PP : p.P;
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t / G >= p.n_items) return;
    const long long item = ordered_item(p, t / G);
    const int sub = threadIdx.x & (G - 1);
    const int m = static_cast<int>(item % p.M);
    const long long b = item / p.M / p.Nq;
    const long long rb = p.row_bytes;
    const char *vb = static_cast<const char *>(p.value) + (b * p.Nin) * rb +
                     static_cast<long long>(m) * (rb / p.M) + sub * 16;
    const float *lp = p.loc + item * L * P * 3;
    const float *ap = p.attn + item * L * P;
    float zmax = 0.f, zsum = 1.f;
    if constexpr (FUSED) logit_stats(ap, L * P, zmax, zsum);

    float acc[N];
#pragma unroll
    for (int i = 0; i < N; ++i) acc[i] = 0.f;

#pragma unroll
    for (int l = 0; l < L; ++l) {
        const int W = p.W[l], H = p.H[l], Z = p.Z[l];
        const float fW = p.fW[l], fH = p.fH[l], fZ = p.fZ[l];
        const char *vl = vb + static_cast<long long>(p.start[l]) * rb;
        const long long sy = W * rb, sz = static_cast<long long>(H) * W * rb;
#pragma unroll 2
        for (int k = 0; k < P; ++k) {
            const float *xyz = lp + (l * P + k) * 3;
            float lx = __ldg(xyz), ly = __ldg(xyz + 1), lz = __ldg(xyz + 2);
            float a = __ldg(ap + l * P + k);
            if constexpr (FUSED) {
                const long long bq = item / p.M;
                lx = fused_location<3>(p, bq, l, 0, lx);
                ly = fused_location<3>(p, bq, l, 1, ly);
                lz = fused_location<3>(p, bq, l, 2, lz);
                a = __fdiv_rn(expf(a - zmax), zsum);
            }
            int x0, y0, z0;
            float fx, fy, fz;
            const bool ok = pixel_coord(lx, fW, x0, fx) & pixel_coord(ly, fH, y0, fy) &
                            pixel_coord(lz, fZ, z0, fz) & !(fabsf(a) < p.prune);
            const bool vx[2] = {ok && x0 >= 0, ok && x0 < W - 1};
            const bool vy[2] = {y0 >= 0, y0 < H - 1};
            const bool vz[2] = {z0 >= 0, z0 < Z - 1};
            const float wx[2] = {1.f - fx, fx};
            const float wy[2] = {1.f - fy, fy};
            const float wz[2] = {a * (1.f - fz), a * fz};
            const char *c000 = vl + static_cast<long long>((z0 * H + y0) * W + x0) * rb;
            uint4 u[8];
            float w[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int dx = c & 1, dy = (c >> 1) & 1, dz = c >> 2;
                const bool inside =
                    vx[dx] && vy[dy] && vz[dz] &&
                    row_ok(p, p.start[l] + (static_cast<long long>(z0 + dz) * H + (y0 + dy)) * W +
                                  x0 + dx, item, l * P + k);
                w[c] = inside ? wz[dz] * wy[dy] * wx[dx] : 0.f;
                u[c] = make_uint4(0, 0, 0, 0);
                if (inside) u[c] = ldg16(c000 + dz * sz + dy * sy + dx * rb);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float v[N];
                unpack(u[c], v);
#pragma unroll
                for (int i = 0; i < N; ++i) acc[i] = fmaf(w[c], v[i], acc[i]);
            }
        }
    }
    char *o = static_cast<char *>(p.out) + item * (rb / p.M) + sub * 16;
    *reinterpret_cast<uint4 *>(o) = pack(acc);
}


// ------------------------------------------------------------------ compiled (L, P)

// acc += w * (the channels of one 16-byte piece), packed fp32x2 FMAs (same rounding as fmaf).
template <int DT>
__device__ __forceinline__ void fma16(float2 *acc, float w, const uint4 &u) {
    constexpr int NV = Vec<DT>::N;
    float v[NV];
    unpack(u, v);
    const float2 w2 = make_float2(w, w);
#pragma unroll
    for (int i = 0; i < NV / 2; ++i) acc[i] = __ffma2_rn(w2, make_float2(v[2 * i], v[2 * i + 1]), acc[i]);
}

template <int DT, int VB>
__device__ __forceinline__ void fma_slice(float2 *acc, float w, const Slice<VB> &r) {
    fma16<DT>(acc, w, r.a);
    if constexpr (VB == 32) fma16<DT>(acc + Vec<DT>::N / 2, w, r.b);
}

// 16 bytes of output channels from acc[half * NV/2 ...] (bf16: one RNE rounding).
template <int DT>
__device__ __forceinline__ uint4 pack16(const float2 *acc) {
    constexpr int NV = Vec<DT>::N;
    float r[NV];
#pragma unroll
    for (int i = 0; i < NV / 2; ++i) {
        r[2 * i] = acc[i].x;
        r[2 * i + 1] = acc[i].y;
    }
    return pack(r);
}

// Launch shape of the compiled path for one (ndim, dtype): bytes per lane and row (VB),
// samples whose corner rows are in flight ahead of the one being summed (AHEAD), and the
// minimum resident blocks of kFwdBlock threads per SM that caps registers (MINB).  Tuned
// on B300 with the encoder (fp32 2D), decoder (bf16 2D) and volume (bf16 3D) workloads.
// 16-byte lanes keep one L1 wavefront per 128-byte row (256-bit lanes over 128-byte rows
// cost about 1.5); 3D's 64-byte bf16 rows take 32-byte lanes (two lanes per row).
// Blocks are kFwdBlock = 128 threads: finished work is replaced at a finer grain than with
// 256 (items take uneven time, e.g. skipped out-of-level corners).
// PRED: out-of-level corners are skipped by predicating their loads and FMAs (no zeroed
// registers); without it (the wide 3D slices, where the predicated form needs more
// registers than the block budget) their slices are zeroed before the predicated load and
// their weights set to zero, and every FMA runs.
constexpr int kFwdBlock = 128;
template <int NDIM, int DT> struct Shape;
template <> struct Shape<2, kF32> { static constexpr int VB = 16, AHEAD = 1, MINB = 12; static constexpr bool PRED = true; };
template <> struct Shape<2, kBF16> { static constexpr int VB = 16, AHEAD = 1, MINB = 10; static constexpr bool PRED = false; };
template <> struct Shape<3, kF32> { static constexpr int VB = 32, AHEAD = 1, MINB = 6; static constexpr bool PRED = false; };
template <> struct Shape<3, kBF16> { static constexpr int VB = 32, AHEAD = 1, MINB = 6; static constexpr bool PRED = false; };

// One item = (b, q, m); LANES = G * SPLIT lanes per item; lane = (item, sp, sub).
// Subgroup sp handles samples [sp * SS, (sp + 1) * SS) of the item (sample index
// l * P + p); its lane `sub` computes the taps of SPL of them and leaves their records in
// shared memory.  The group then walks its samples: the corner rows of the next AHEAD
// samples are loaded (in-level corners only) before the current sample is summed.
//
// LL = 0 selects the runtime-(L, P) form: L and P come from the parameters, PP is the
// largest L * P it handles (SMAX), and the sample walk is a loop unrolled by DEPTH instead
// of a fully unrolled sequence; the level of sample j is (j * p.pinv) >> 16.
template <int DT, int G, int VB, int NDIM, int LL, int PP, int SPLIT, int AHEAD, int MINB,
          bool FUSED, bool PACK, bool PRED>
__global__ void __launch_bounds__(kFwdBlock, MINB)
fwd_tiled(const __grid_constant__ Params p) {
    constexpr bool RT = LL == 0;
    constexpr int N = VB / Vec<DT>::ESIZE;  // channels per lane
    constexpr int NC = 1 << NDIM;
    constexpr int SMAX = RT ? PP : LL * PP;           // samples per item (at most, if RT)
    static_assert(RT || SMAX % SPLIT == 0, "SPLIT must divide L * P");
    constexpr int SPLM = ((SMAX + SPLIT - 1) / SPLIT + G - 1) / G;  // taps per lane (at most)
    constexpr int LANES = G * SPLIT;
    static_assert(LANES <= 32 && (32 % LANES) == 0, "lanes per item must divide the warp");
    // compiled (L, P): when every lane owns exactly SPL samples, read them with vector loads
    constexpr int SSC = SMAX / SPLIT;
    constexpr bool EVEN = !RT && (SSC % G) == 0;
    constexpr int ALOC = cmin(cmin(falign(SMAX * NDIM), falign(SSC * NDIM)), falign(SPLM * NDIM));
    constexpr int AATT = cmin(cmin(falign(SMAX), falign(SSC)), falign(SPLM));
    constexpr int DEPTH = AHEAD + 1;
    constexpr int IPB = kFwdBlock / LANES;            // items per block
    constexpr int ISTR = tap_slot(SMAX - 1) + 2;      // slots per item (+1 pad between items)
    const int S = RT ? p.L * p.P : SMAX;              // samples per item
    const int SS = S / SPLIT;                         // samples per subgroup
    const int SPL = RT ? (SS + G - 1) / G : SPLM;     // taps per lane
    // level of sample j
    auto level = [&](int j) { return RT ? (j * p.pinv) >> 16 : j / PP; };
    constexpr int OKB = NDIM == 2 ? 4 : 8;            // validity bits under a packed row

    __shared__ float4 rec[IPB * ISTR];
    __shared__ float rec_z[NDIM == 3 ? IPB * ISTR : 1];               // fz (3D)
    __shared__ unsigned rec_ok[PACK ? 1 : IPB * ISTR];                // validity bits

    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    // whole warps leave together: the exchange below needs every lane of the warp
    if ((t & ~31LL) / LANES >= p.n_items) return;
    long long pos = t / LANES;
    const bool active = pos < p.n_items;
    if (!active) pos = p.n_items - 1;  // tail lanes redo a real item and store nothing
    long long item;
    int m;
    long long b;
    if (p.n_items <= 0x7fffffffLL) {
        // 32-bit index arithmetic while every item index fits
        const unsigned it = static_cast<unsigned>(pos);
        const unsigned bq = it / static_cast<unsigned>(p.M);       // b * Nq + i
        m = static_cast<int>(it - bq * static_cast<unsigned>(p.M));
        const unsigned bb = bq / static_cast<unsigned>(p.Nq);
        b = bb;
        if (p.order == nullptr) {
            item = it;
        } else {
            // query order: position i of batch b runs query order[b * Nq + i], clamped into
            // [0, Nq) (a malformed order gives wrong results, never an out-of-range access)
            int q = __ldg(p.order + bq);
            q = q < 0 ? 0 : (q >= p.Nq ? static_cast<int>(p.Nq - 1) : q);
            item = (static_cast<unsigned>(bb) * static_cast<unsigned>(p.Nq) + q) *
                       static_cast<unsigned>(p.M) + m;
        }
    } else {
        item = ordered_item(p, pos);
        m = static_cast<int>(item % p.M);
        b = item / p.M / p.Nq;
    }
    const int lane = threadIdx.x & 31;
    const int sub = lane & (G - 1);
    const int sp = SPLIT > 1 ? (lane / G) & (SPLIT - 1) : 0;
    const int ib = threadIdx.x / LANES;       // item within the block
    const int s0 = sp * SS;                  // first sample of this subgroup
    const int my0 = s0 + sub * SPL;          // first sample whose taps this lane computes

    // 1. locations and weights of this lane's samples, then their tap records
    float lv[SPLM * NDIM], av[SPLM];
    const float *lsrc = p.loc + (item * S + my0) * NDIM;
    const float *asrc = p.attn + item * S + my0;
    // sample my0 + i is this lane's and exists
    auto have = [&](int i) { return EVEN || ((!RT || i < SPL) && sub * SPL + i < SS); };
    if constexpr (EVEN) {
        load_stream<SPLM * NDIM, ALOC>(lsrc, lv);
        load_stream<SPLM, AATT>(asrc, av);
    } else {
#pragma unroll
        for (int i = 0; i < SPLM; ++i) {
            const bool h = have(i);
#pragma unroll
            for (int k = 0; k < NDIM; ++k) lv[i * NDIM + k] = h ? __ldcs(lsrc + i * NDIM + k) : 0.f;
            av[i] = h ? __ldcs(asrc + i) : 0.f;
        }
    }
    if constexpr (FUSED) {
        // prologue: softmax of the item's logits over all its lanes, then the locations
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < SPLM; ++i)
            if (have(i)) mx = fmaxf(mx, av[i]);
#pragma unroll
        for (int o = 1; o < LANES; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < SPLM; ++i) {
            av[i] = have(i) ? expf(av[i] - mx) : 0.f;
            sum += av[i];
        }
#pragma unroll
        for (int o = 1; o < LANES; o <<= 1) sum += __shfl_xor_sync(kFull, sum, o);
        const long long bq = item / p.M;
#pragma unroll
        for (int i = 0; i < SPLM; ++i) {
            av[i] = __fdiv_rn(av[i], sum);
            const int l = level(min(my0 + i, s0 + SS - 1));
#pragma unroll
            for (int k = 0; k < NDIM; ++k)
                lv[i * NDIM + k] = fused_location<NDIM>(p, bq, l, k, lv[i * NDIM + k]);
        }
    }
#pragma unroll
    for (int i = 0; i < SPLM; ++i) {
        if (!have(i)) continue;   // past the subgroup's samples
        const int j = my0 + i;
        Taps<NC> tp;
        float fr[NDIM];
        make_taps(p, level(j), lv + i * NDIM, av[i], tp, fr);
        const int slot = ib * ISTR + tap_slot(j);
        const int rbits = PACK ? static_cast<int>((static_cast<unsigned>(tp.row) << OKB) | tp.ok)
                               : tp.row;
        rec[slot] = make_float4(__int_as_float(rbits), av[i], fr[0], fr[1]);
        if constexpr (NDIM == 3) rec_z[slot] = fr[2];
        if constexpr (!PACK) rec_ok[slot] = tp.ok;
    }
    __syncwarp();

    // 2. walk the subgroup's samples; corner rows are VB-byte slices per lane
    const long long rb = p.row_bytes;
    const char *vb = static_cast<const char *>(p.value) + (b * p.Nin) * rb +
                     static_cast<long long>(m) * (rb / p.M) + sub * VB;
    float2 acc[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) acc[i] = make_float2(0.f, 0.f);

    TapView<NC> tq[DEPTH];
    Slice<VB> u[DEPTH][NC];
    // record of sample s0 + s, then its in-level corner rows
    auto fetch = [&](int s, int slot) {
        const int j = ib * ISTR + tap_slot(s0 + s);
        const float4 r = rec[j];
        if constexpr (PACK) {
            const int v = __float_as_int(r.x);
            tq[slot].row = v >> OKB;
            tq[slot].ok = static_cast<unsigned>(v) & ((1u << OKB) - 1u);
        } else {
            tq[slot].row = __float_as_int(r.x);
            tq[slot].ok = rec_ok[j];
        }
        if constexpr (NDIM == 2) tap_weights(r.y, r.z, r.w, tq[slot].w);
        else tap_weights(r.y, r.z, r.w, rec_z[j], tq[slot].w);
        if constexpr (!PRED) {
#pragma unroll
            for (int c = 0; c < NC; ++c) tq[slot].w[c] = ((tq[slot].ok >> c) & 1u) ? tq[slot].w[c] : 0.f;
        }
        const int l = level(s0 + s);  // a constant when SPLIT == 1 and (L, P) is compiled
        const char *c0 = vb + static_cast<long long>(tq[slot].row) * p.rb32;
        const char *cy[2] = {c0, c0 + p.sy[l]};
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const char *base = cy[(c >> 1) & 1];
            if (c >> 2) base += p.sz[l];
            bool in = (tq[slot].ok >> c) & 1u;
#ifdef MSDA_DEBUG_BOUNDS
            const long long crow = static_cast<long long>(tq[slot].row) + (c & 1) +
                                   (((c >> 1) & 1) ? p.W[l] : 0) +
                                   ((c >> 2) ? static_cast<long long>(p.W[l]) * p.H[l] : 0);
            if (in && !row_ok(p, crow, item, s0 + s)) {
                in = false;
                tq[slot].ok &= ~(1u << c);
            }
#endif
            if constexpr (PRED) {
                load_slice_if(in, base + ((c & 1) ? rb : 0), u[slot][c]);
            } else {
                zero_slice(u[slot][c]);
                if (in) load_slice(base + ((c & 1) ? rb : 0), u[slot][c]);
            }
        }
    };
#pragma unroll
    for (int k = 0; k < AHEAD; ++k)
        if (k < SS) fetch(k, k);
    // sample s sits in slot s % DEPTH; the loads of sample s + AHEAD are issued before s is
    // summed.  Compiled (L, P): fully unrolled; runtime (L, P): a loop unrolled by DEPTH, so
    // that every slot index stays a compile-time constant.
    auto step = [&](int s, int k) {
        if (s + AHEAD < SS) fetch(s + AHEAD, (k + AHEAD) % DEPTH);
#pragma unroll
        for (int c = 0; c < NC; ++c)
            if (!PRED || ((tq[k].ok >> c) & 1u)) fma_slice<DT, VB>(acc, tq[k].w[c], u[k][c]);
    };
    if constexpr (!RT) {
#pragma unroll
        for (int s = 0; s < SSC; ++s) step(s, s % DEPTH);
    } else {
#pragma unroll 1
        for (int sw = 0; sw < SS; sw += DEPTH) {
#pragma unroll
            for (int k = 0; k < DEPTH; ++k)
                if (sw + k < SS) step(sw + k, k);
        }
    }

    // 3. add the subgroups' partial sums, store the item's channels
    if constexpr (SPLIT > 1) {
#pragma unroll
        for (int o = G; o < LANES; o <<= 1)
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                acc[i].x += __shfl_xor_sync(kFull, acc[i].x, o);
                acc[i].y += __shfl_xor_sync(kFull, acc[i].y, o);
            }
    }
    if (active && sp == 0) {
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<char *>(p.out) + item * (rb / p.M) + sub * VB);
        __stcs(o, pack16<DT>(acc));
        if constexpr (VB == 32) __stcs(o + 1, pack16<DT>(acc + Vec<DT>::N / 2));
    }
}

// Lane groups per item for the compiled path.  Narrow rows (few lanes per row) split an
// item's samples until one lane computes the taps of at most MAX_SPL samples (their
// registers would spill otherwise); then the split grows while the launch has fewer than
// kWantThreads threads.
// kWantThreads: 1024 threads per SM of the B300, half its resident threads.  Measured on
// the decoder-shaped forward (19,200 items, 4 lanes per row): split 2 (153,600 threads)
// ran at 11.9 us, split 4 (two full waves, the earlier rule) at 12.7 us, split 1 at 14.4.
constexpr long long kWantThreads = 148LL * 1024;

template <int G, int S, int NDIM>
int pick_split(long long n_items) {
    constexpr int MAX_SPL = NDIM == 2 ? 4 : 2;
    auto can_double = [](int split) { return split < 4 && G * split * 2 <= 32 && S % (split * 2) == 0; };
    int split = 1;
    while (can_double(split) && S / split > MAX_SPL * G) split *= 2;
    while (can_double(split) && n_items * G * split < kWantThreads) split *= 2;
    return split;
}

// The runtime-(L, P) form keeps its whole prefetch pipeline live across the loop's back
// edge, so it takes a shallower window and more registers per thread than the fully
// unrolled compiled form.
template <int NDIM, int DT> struct RtShape;
template <> struct RtShape<2, kF32> { static constexpr int VB = 16, AHEAD = 1, MINB = 8; static constexpr bool PRED = true; };
template <> struct RtShape<2, kBF16> { static constexpr int VB = 16, AHEAD = 1, MINB = 8; static constexpr bool PRED = false; };
template <> struct RtShape<3, kF32> { static constexpr int VB = 32, AHEAD = 0, MINB = 5; static constexpr bool PRED = false; };
template <> struct RtShape<3, kBF16> { static constexpr int VB = 32, AHEAD = 0, MINB = 5; static constexpr bool PRED = false; };

// The launch shape of the compiled (LL > 0) or runtime-(L, P) (LL = 0) form.  The lanes per
// row (G) of a launch are derived from the same shape's VB, so that the G lanes of a group
// cover exactly one head's D channels.
template <int NDIM, int DT, int LL>
using TiledShape = typename std::conditional<LL == 0, RtShape<NDIM, DT>, Shape<NDIM, DT>>::type;

template <int DT, int G, int NDIM, int LL, int PP, int SPLIT>
cudaError_t launch_tiled(const Params &p, cudaStream_t s) {
    using SH = TiledShape<NDIM, DT, LL>;
    // a lane group must span one head's channels exactly: a wider group would read the
    // next head's (or past the row's) bytes
    if (static_cast<long long>(G) * SH::VB * p.M != p.row_bytes) return cudaErrorInvalidValue;
    const long long threads = p.n_items * G * SPLIT;
    const long long blocks = (threads + kFwdBlock - 1) / kFwdBlock;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (p.ref) {
        if (p.pack_taps)
            fwd_tiled<DT, G, SH::VB, NDIM, LL, PP, SPLIT, SH::AHEAD, SH::MINB, true, true, SH::PRED>
                <<<grid, kFwdBlock, 0, s>>>(p);
        else
            fwd_tiled<DT, G, SH::VB, NDIM, LL, PP, SPLIT, SH::AHEAD, SH::MINB, true, false, SH::PRED>
                <<<grid, kFwdBlock, 0, s>>>(p);
    } else {
        if (p.pack_taps)
            fwd_tiled<DT, G, SH::VB, NDIM, LL, PP, SPLIT, SH::AHEAD, SH::MINB, false, true, SH::PRED>
                <<<grid, kFwdBlock, 0, s>>>(p);
        else
            fwd_tiled<DT, G, SH::VB, NDIM, LL, PP, SPLIT, SH::AHEAD, SH::MINB, false, false, SH::PRED>
                <<<grid, kFwdBlock, 0, s>>>(p);
    }
    return cudaGetLastError();
}

// G16 = lanes per row at 16 bytes per lane; the kernel uses G = row bytes / VB lanes.
template <int DT, int G16, int NDIM, int LL, int PP>
cudaError_t launch_tiled_split(const Params &p, cudaStream_t s) {
    constexpr int VB = TiledShape<NDIM, DT, LL>::VB;
    constexpr int G = G16 * 16 / VB;
    static_assert(G >= 1, "rows narrower than one lane's slice take the generic path");
    const int split = pick_split<G, LL * PP, NDIM>(p.n_items);
    if constexpr (G <= 16) {
        if (split == 2) return launch_tiled<DT, G, NDIM, LL, PP, 2>(p, s);
    }
    if constexpr (G <= 8) {
        if (split == 4) return launch_tiled<DT, G, NDIM, LL, PP, 4>(p, s);
    }
    return launch_tiled<DT, G, NDIM, LL, PP, 1>(p, s);
}

// Runtime-(L, P) form of the compiled path: any L * P up to kRtMaxSamples, for rows of
// 2 to 16 sixteen-byte lanes.  The split follows pick_split with the runtime sample count.
constexpr int kRtMaxSamples = 32;

template <int G, int NDIM>
int pick_split_rt(int S, long long n_items) {
    constexpr int MAX_SPL = NDIM == 2 ? 4 : 2;
    auto can_double = [S](int split) { return split < 4 && G * split * 2 <= 32 && S % (split * 2) == 0; };
    int split = 1;
    while (can_double(split) && S / split > MAX_SPL * G) split *= 2;
    while (can_double(split) && n_items * G * split < kWantThreads) split *= 2;
    return split;
}

template <int DT, int G16, int NDIM>
cudaError_t launch_tiled_rt(const Params &p, cudaStream_t s) {
    constexpr int VB = TiledShape<NDIM, DT, 0>::VB;
    constexpr int G = G16 * 16 / VB;
    const int split = pick_split_rt<G, NDIM>(p.L * p.P, p.n_items);
    if constexpr (G <= 16) {
        if (split == 2) return launch_tiled<DT, G, NDIM, 0, kRtMaxSamples, 2>(p, s);
    }
    if constexpr (G <= 8) {
        if (split == 4) return launch_tiled<DT, G, NDIM, 0, kRtMaxSamples, 4>(p, s);
    }
    return launch_tiled<DT, G, NDIM, 0, kRtMaxSamples, 1>(p, s);
}

template <int DT, int G, int NDIM>
cudaError_t forward_nd(const Params &p, cudaStream_t s) {
    if constexpr (G * 16 >= Shape<NDIM, DT>::VB) {
        if (p.L == 4 && p.P == 4) return launch_tiled_split<DT, G, NDIM, 4, 4>(p, s);
        if (p.L == 1 && p.P == 4) return launch_tiled_split<DT, G, NDIM, 1, 4>(p, s);
    }
    if constexpr (G >= 2 && G <= 16 && G * 16 >= TiledShape<NDIM, DT, 0>::VB) {
        // the runtime-(L, P) instantiations live in msda_forward_rt_*.cu (compiled in
        // parallel with these)
        if (p.L * p.P <= kRtMaxSamples) {
            if constexpr (DT == kF32 && NDIM == 2) return launch_forward_rt_f32_2d(G, p, s);
            if constexpr (DT == kF32 && NDIM == 3) return launch_forward_rt_f32_3d(G, p, s);
            if constexpr (DT == kBF16 && NDIM == 2) return launch_forward_rt_bf16_2d(G, p, s);
            if constexpr (DT == kBF16 && NDIM == 3) return launch_forward_rt_bf16_3d(G, p, s);
        }
    }
    const long long threads = p.n_items * G;
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks)), block(256);
    if constexpr (NDIM == 2) {
        if (p.ref) fwd2d_generic<DT, G, 0, 0, true><<<grid, block, 0, s>>>(p);
        else fwd2d_generic<DT, G, 0, 0, false><<<grid, block, 0, s>>>(p);
    } else {
        if (p.ref) fwd3d_generic<DT, G, 0, 0, true><<<grid, block, 0, s>>>(p);
        else fwd3d_generic<DT, G, 0, 0, false><<<grid, block, 0, s>>>(p);
    }
    return cudaGetLastError();
}

// All lane-group widths G (lanes per value row at 16 bytes per lane) for one dtype and
// dimensionality.
template <int DT, int NDIM>
cudaError_t forward_dispatch(int G, const Params &p, cudaStream_t s) {
    switch (G) {
        case 1: return forward_nd<DT, 1, NDIM>(p, s);
        case 2: return forward_nd<DT, 2, NDIM>(p, s);
        case 4: return forward_nd<DT, 4, NDIM>(p, s);
        case 8: return forward_nd<DT, 8, NDIM>(p, s);
        case 16: return forward_nd<DT, 16, NDIM>(p, s);
        case 32: return forward_nd<DT, 32, NDIM>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

}  // namespace msda
