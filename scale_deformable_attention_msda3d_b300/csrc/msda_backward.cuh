// Backward kernels (templates; msda_backward_{2d,3d}.cu instantiate them, msda_backward.cu
// dispatches and holds the grad_value zero-fill): gradients of sum(grad_out * out) with
// respect to value, sampling
// locations and attention weights ("3D Attention That Knows Where to Look": gradients
// flow back into both the offsets and the weights; interpolation is differentiable).
//
// Per sample with weight a, corner weights w_c (without a) and corner rows v_c:
//   grad_A        = sum_c w_c <g, v_c>
//   grad_x (px)   = a * sum_c dw_c/dx <g, v_c>,   grad_loc_x = W_l * grad_x   (x = loc*W - 0.5)
//   grad_value[c] += a * w_c * g                  (corners inside the level only)
//
// Kernels:
// * bwd_tiled / bwd_tiled_wide (the compiled (L, P) pairs; the same body, rows of up to 8
//   lanes / wider rows, which differ only in the residency they ask of the compiler).  A CTA handles one (batch, head) and a run of
//   queries; a lane group of G lanes (16 bytes of channels each) handles one query.  Lane
//   j of the group owns samples j, G + j, 2G + j, ...: it reads their locations and
//   weights, computes their taps and leaves each sample's tap record (row, a, fractions,
//   validity bits) in shared memory for the group.  Every lane loads the in-level corner
//   rows of each sample (predicated, no zeroed registers) and forms its partial dot
//   products <g, v_c> over its channels (in 3D folded at once into partial grad_A, grad_x,
//   grad_y, grad_z, which are linear in them); after each batch of G samples a butterfly
//   reduce-scatter leaves each sample's sums on its owner, which writes grad_A and
//   grad_loc.  grad_value goes through 16-byte red.global.add.v4.f32, issued so that
//   the lanes of one instruction cover a contiguous run of the row (add_global_runs).
//   (Accumulating small levels in shared memory first was measured and dropped: on this
//   part shared-memory fp32 atomics ran about ten times slower than the L2 reductions.)
// * bwd{2,3}d_generic (any L, P): every lane of the group computes every sample, reduces
//   grad_A / grad_loc with xor shuffles and scatters with red.global.add.v4.f32 in runs.
// With FUSED (the backward of the fused-prologue forward) the kernels form the locations
// and softmax weights from reference points, offsets and logits as the fused forward does,
// and write offset gradients (d location / d offset = 1 / extent); bwd_tiled also forms
// the logit gradients, the generic kernels leave grad_A for an epilogue.
#pragma once

#include "common.cuh"

namespace msda {

namespace {

// grad_value += wgt * gr over this lane's N channels of one corner row, laid out in runs:
// reduction k (k < N / 4) of lane `sub` covers channels k * 4G + 4 sub .. + 3, so the G
// lanes of one instruction fill a contiguous 16 G-byte run of the fp32 row.  dst points at
// channel 4 sub of the row; gr holds those channels of grad_out (see run_channels).
template <int N, int G>
__device__ __forceinline__ void add_global_runs(float *dst, float wgt, const float (&gr)[N]) {
#pragma unroll
    for (int k = 0; k < N / 4; ++k)
        red_add_v4(dst + k * 4 * G, wgt * gr[4 * k], wgt * gr[4 * k + 1], wgt * gr[4 * k + 2],
                   wgt * gr[4 * k + 3]);
}

// The grad_out channels of lane `sub`'s reductions (channels k * 4G + 4 sub .. + 3), from
// the item's grad_out row: for fp32 (N = 4) they are the lane's own 16 bytes; for bf16
// (N = 8) two 8-byte pieces.  Why runs: a lane's 8 bf16 channels are 32 bytes of fp32
// gradient, and two reductions over the lanes' interleaved halves would write 16 bytes
// into each 32-byte sector of the line twice; the L2 reduction units work per sector, so
// runs of whole sectors halve their work.
template <int DT, int G>
__device__ __forceinline__ void run_channels(const char *go_row, int sub,
                                             const float (&g)[Vec<DT>::N],
                                             float (&gr)[Vec<DT>::N]) {
    constexpr int N = Vec<DT>::N;
    if constexpr (N == 4) {
#pragma unroll
        for (int i = 0; i < N; ++i) gr[i] = g[i];
    } else {
#pragma unroll
        for (int k = 0; k < N / 4; ++k) {
            const uint2 u = __ldg(reinterpret_cast<const uint2 *>(go_row) + k * G + sub);
            gr[4 * k] = __uint_as_float(u.x << 16);
            gr[4 * k + 1] = __uint_as_float(u.x & 0xffff0000u);
            gr[4 * k + 2] = __uint_as_float(u.y << 16);
            gr[4 * k + 3] = __uint_as_float(u.y & 0xffff0000u);
        }
    }
}

template <int N>
__device__ __forceinline__ float dot(const uint4 &u, const float (&g)[N]) {
    float v[N];
    unpack(u, v);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i) s = fmaf(g[i], v[i], s);
    return s;
}

template <int DT, int G, int LL, int PP, bool FUSED>
__global__ void __launch_bounds__(256)
bwd2d_generic(const __grid_constant__ Params p) {
    constexpr int N = Vec<DT>::N;
    const int L = LL > 0 ? LL : p.L;
    const int P = PP > 0 ? PP : p.P;
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    // whole warps leave together so that the group shuffles below see every lane
    if ((t - (threadIdx.x & 31)) / G >= p.n_items) return;
    long long pos = t / G;
    const bool active = pos < p.n_items;
    if (!active) pos = p.n_items - 1;  // tail lanes recompute a real item, write nothing
    const long long item = ordered_item(p, pos);  // the item itself without a query order
    const int sub = threadIdx.x & (G - 1);
    const int m = static_cast<int>(item % p.M);
    const long long b = item / p.M / p.Nq;
    const long long rb = p.row_bytes;
    const long long rowf = static_cast<long long>(p.M) * p.D;  // grad_value row stride (floats)
    const char *vb = static_cast<const char *>(p.value) + (b * p.Nin) * rb +
                     static_cast<long long>(m) * (rb / p.M) + sub * 16;
    // channel 4 sub of the head's grad_value row (reductions in runs, see add_global_runs)
    float *gvb = p.grad_value + (b * p.Nin) * rowf + static_cast<long long>(m) * p.D + sub * 4;
    const char *go_row = static_cast<const char *>(p.grad_out) + item * (rb / p.M);
    float g[N], gr[N];
    unpack(ldg16(go_row + sub * 16), g);
    run_channels<DT, G>(go_row, sub, g, gr);
    const long long s0 = item * L * P;
    const float2 *lp = reinterpret_cast<const float2 *>(p.loc) + s0;
    float zmax = 0.f, zsum = 1.f;
    if constexpr (FUSED) logit_stats(p.attn + s0, L * P, zmax, zsum);

#pragma unroll
    for (int l = 0; l < L; ++l) {
        const int W = p.W[l], H = p.H[l];
        const float fW = p.fW[l], fH = p.fH[l];
        // fused: the gradient goes to the offset, d location / d offset = 1 / extent
        const float eW = FUSED ? 1.f : fW, eH = FUSED ? 1.f : fH;
        const char *vl = vb + static_cast<long long>(p.start[l]) * rb;
        float *gl = gvb + static_cast<long long>(p.start[l]) * rowf;
#pragma unroll 2
        for (int k = 0; k < P; ++k) {
            const long long s = s0 + l * P + k;
            float2 xy = __ldg(lp + l * P + k);
            float a = __ldg(p.attn + s);
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
            const bool ok = okx && oky;
            const bool vx0 = ok && x0 >= 0, vx1 = ok && x0 < W - 1;
            const bool vy0 = y0 >= 0, vy1 = y0 < H - 1;
            const long long r00 = static_cast<long long>(y0 * W + x0);
            const long long a00 = p.start[l] + r00;  // row index within the batch
            const int sidx = l * P + k;
            const bool ok00 = vy0 && vx0 && row_ok(p, a00, item, sidx);
            const bool ok01 = vy0 && vx1 && row_ok(p, a00 + 1, item, sidx);
            const bool ok10 = vy1 && vx0 && row_ok(p, a00 + W, item, sidx);
            const bool ok11 = vy1 && vx1 && row_ok(p, a00 + W + 1, item, sidx);
            const char *c00 = vl + r00 * rb;
            uint4 u00 = make_uint4(0, 0, 0, 0), u01 = u00, u10 = u00, u11 = u00;
            if (ok00) u00 = ldg16(c00);
            if (ok01) u01 = ldg16(c00 + rb);
            if (ok10) u10 = ldg16(c00 + W * rb);
            if (ok11) u11 = ldg16(c00 + (W + 1) * rb);
            const float d00 = dot(u00, g), d01 = dot(u01, g), d10 = dot(u10, g),
                        d11 = dot(u11, g);
            const float wx0 = 1.f - fx, wy0 = 1.f - fy;
            float gA = wy0 * (wx0 * d00 + fx * d01) + fy * (wx0 * d10 + fx * d11);
            float gx = wy0 * (d01 - d00) + fy * (d11 - d10);
            float gy = wx0 * (d10 - d00) + fx * (d11 - d01);
            gA = group_sum<G>(gA);
            gx = group_sum<G>(gx);
            gy = group_sum<G>(gy);
            if (active) {
                if (sub == 0) {
                    const bool any = ok00 || ok01 || ok10 || ok11;
                    p.grad_attn[s] = gA;  // fused: grad_A, turned into d/d logits later
                    p.grad_loc[2 * s] = any ? a * gx * eW : 0.f;
                    p.grad_loc[2 * s + 1] = any ? a * gy * eH : 0.f;
                }
                float *d = gl + r00 * rowf;
                if (ok00) add_global_runs<N, G>(d, a * (wy0 * wx0), gr);
                if (ok01) add_global_runs<N, G>(d + rowf, a * (wy0 * fx), gr);
                if (ok10) add_global_runs<N, G>(d + W * rowf, a * (fy * wx0), gr);
                if (ok11) add_global_runs<N, G>(d + (W + 1) * rowf, a * (fy * fx), gr);
            }
        }
    }
}

template <int DT, int G, int LL, int PP, bool FUSED>
__global__ void __launch_bounds__(256)
bwd3d_generic(const __grid_constant__ Params p) {
    constexpr int N = Vec<DT>::N;
    const int L = LL > 0 ? LL : p.L;
    const int P = PP > 0 ? PP : p.P;
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if ((t - (threadIdx.x & 31)) / G >= p.n_items) return;
    long long pos = t / G;
    const bool active = pos < p.n_items;
    if (!active) pos = p.n_items - 1;
    const long long item = ordered_item(p, pos);
    const int sub = threadIdx.x & (G - 1);
    const int m = static_cast<int>(item % p.M);
    const long long b = item / p.M / p.Nq;
    const long long rb = p.row_bytes;
    const long long rowf = static_cast<long long>(p.M) * p.D;
    const char *vb = static_cast<const char *>(p.value) + (b * p.Nin) * rb +
                     static_cast<long long>(m) * (rb / p.M) + sub * 16;
    // channel 4 sub of the head's grad_value row (reductions in runs, see add_global_runs)
    float *gvb = p.grad_value + (b * p.Nin) * rowf + static_cast<long long>(m) * p.D + sub * 4;
    const char *go_row = static_cast<const char *>(p.grad_out) + item * (rb / p.M);
    float g[N], gr[N];
    unpack(ldg16(go_row + sub * 16), g);
    run_channels<DT, G>(go_row, sub, g, gr);
    const long long s0 = item * L * P;
    float zmax = 0.f, zsum = 1.f;
    if constexpr (FUSED) logit_stats(p.attn + s0, L * P, zmax, zsum);

#pragma unroll
    for (int l = 0; l < L; ++l) {
        const int W = p.W[l], H = p.H[l], Z = p.Z[l];
        const float fW = p.fW[l], fH = p.fH[l], fZ = p.fZ[l];
        const float eW = FUSED ? 1.f : fW, eH = FUSED ? 1.f : fH, eZ = FUSED ? 1.f : fZ;
        const char *vl = vb + static_cast<long long>(p.start[l]) * rb;
        float *gl = gvb + static_cast<long long>(p.start[l]) * rowf;
        const long long HW = static_cast<long long>(H) * W;
#pragma unroll 1
        for (int k = 0; k < P; ++k) {
            const long long s = s0 + l * P + k;
            float xyz[3] = {__ldg(p.loc + 3 * s), __ldg(p.loc + 3 * s + 1),
                            __ldg(p.loc + 3 * s + 2)};
            float a = __ldg(p.attn + s);
            if constexpr (FUSED) {
                const long long bq = item / p.M;
#pragma unroll
                for (int c = 0; c < 3; ++c) xyz[c] = fused_location<3>(p, bq, l, c, xyz[c]);
                a = __fdiv_rn(expf(a - zmax), zsum);
            }
            int x0, y0, z0;
            float fx, fy, fz;
            const bool valid = pixel_coord(xyz[0], fW, x0, fx) &
                               pixel_coord(xyz[1], fH, y0, fy) &
                               pixel_coord(xyz[2], fZ, z0, fz);
            const bool vx[2] = {valid && x0 >= 0, valid && x0 < W - 1};
            const bool vy[2] = {y0 >= 0, y0 < H - 1};
            const bool vz[2] = {z0 >= 0, z0 < Z - 1};
            const float wx[2] = {1.f - fx, fx};
            const float wy[2] = {1.f - fy, fy};
            const float wz[2] = {1.f - fz, fz};
            const long long r000 = static_cast<long long>((z0 * H + y0) * W + x0);
            const char *c000 = vl + r000 * rb;
            bool ok[8];
            long long off[8];
            float d[8];
            bool any = false;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int dx = c & 1, dy = (c >> 1) & 1, dz = c >> 2;
                off[c] = dz * HW + dy * W + dx;
                ok[c] = vx[dx] && vy[dy] && vz[dz] &&
                        row_ok(p, p.start[l] + r000 + off[c], item, static_cast<int>(l * P + k));
                any = any || ok[c];
                uint4 u = make_uint4(0, 0, 0, 0);
                if (ok[c]) u = ldg16(c000 + off[c] * rb);
                d[c] = dot(u, g);
            }
            float gA = 0.f, gx = 0.f, gy = 0.f, gz = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int dx = c & 1, dy = (c >> 1) & 1, dz = c >> 2;
                const float sx = dx ? 1.f : -1.f, sy = dy ? 1.f : -1.f, sz = dz ? 1.f : -1.f;
                gA = fmaf(wz[dz] * wy[dy] * wx[dx], d[c], gA);
                gx = fmaf(sx * wz[dz] * wy[dy], d[c], gx);
                gy = fmaf(sy * wz[dz] * wx[dx], d[c], gy);
                gz = fmaf(sz * wy[dy] * wx[dx], d[c], gz);
            }
            gA = group_sum<G>(gA);
            gx = group_sum<G>(gx);
            gy = group_sum<G>(gy);
            gz = group_sum<G>(gz);
            if (active) {
                if (sub == 0) {
                    p.grad_attn[s] = gA;  // fused: grad_A, turned into d/d logits later
                    p.grad_loc[3 * s] = any ? a * gx * eW : 0.f;
                    p.grad_loc[3 * s + 1] = any ? a * gy * eH : 0.f;
                    p.grad_loc[3 * s + 2] = any ? a * gz * eZ : 0.f;
                }
                float *dst = gl + r000 * rowf;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int dx = c & 1, dy = (c >> 1) & 1, dz = c >> 2;
                    if (ok[c])
                        add_global_runs<N, G>(dst + off[c] * rowf, a * (wz[dz] * wy[dy] * wx[dx]), gr);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ compiled (L, P)

// Sum over the G lanes of a group of v[j][k] (j = owner lane, k < K), scattered: lane
// `sub` ends with the group's sums for owner sub in v[0][0..K-1].  (G - 1) * K shuffles.
template <int G, int K>
__device__ __forceinline__ void reduce_scatter(float (&v)[G][K], int sub) {
#pragma unroll
    for (int o = G / 2; o >= 1; o >>= 1) {
        const bool hi = (sub & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i)
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const float send = hi ? v[i][k] : v[i + o][k];
                const float keep = hi ? v[i + o][k] : v[i][k];
                v[i][k] = keep + __shfl_xor_sync(kFull, send, o);
            }
    }
}

template <int DT, int G, int NDIM, int LL, int PP, int BT, bool FUSED>
__device__ __forceinline__ void bwd_tiled_body(const Params &p) {
    constexpr int N = Vec<DT>::N;  // channels per lane (16 bytes of value)
    constexpr int NC = 1 << NDIM;
    constexpr int S = LL * PP;
    constexpr int NB = (S + G - 1) / G;  // batches of G samples per item
    constexpr int GPB = BT / G;          // lane groups (queries in flight) per CTA

    const int cta = blockIdx.x;
    // CTA -> (batch, head, run of query positions).  Queries in the given order go
    // head-major: the CTAs in flight then cover one head, whose grad_value slice and value
    // lines stay in L2 whatever the queries' positions.  With a query order (locality
    // sorted) the head index runs fastest instead: the CTAs in flight cover a compact
    // region of the maps for all heads at once, and a value line shared by two heads'
    // 64-byte slices is fetched once for both.  Measured on the volume backward (random
    // voxel queries, inputs permuted on the host): head-major 738 us given, 712 us with
    // the queries sorted; head-fastest 877 us given, 695 us sorted.
    int m, chunk;
    long long b;
    if (p.order == nullptr) {
        const int bm = cta / p.nchunk;
        chunk = cta - bm * p.nchunk;
        m = bm % p.M;
        b = bm / p.M;
    } else {
        m = cta % p.M;
        const int rest = cta / p.M;
        chunk = rest % p.nchunk;
        b = rest / p.nchunk;
    }
    const long long q_lo = static_cast<long long>(chunk) * p.qchunk;
    const long long q_hi = q_lo + p.qchunk < p.Nq ? q_lo + p.qchunk : p.Nq;
    const int sub = threadIdx.x & (G - 1);
    const int grp = threadIdx.x / G;
    const int D = p.D;
    const long long rb = p.row_bytes;
    const long long rowf = static_cast<long long>(p.M) * D;  // grad_value row stride (floats)

    const char *vbase = static_cast<const char *>(p.value) + (b * p.Nin) * rb +
                        static_cast<long long>(m) * (rb / p.M) + sub * 16;
    constexpr int GS = 4 / Vec<DT>::ESIZE;  // grad_value (fp32) bytes per value byte
    // channel 4 sub of the head's grad_value row (reductions in runs, see add_global_runs)
    char *gbase = reinterpret_cast<char *>(p.grad_value + (b * p.Nin) * rowf +
                                           static_cast<long long>(m) * D + sub * 4);
    // tap records of the CTA's queries (see common.cuh): row, a, fx, fy (+ fz), validity
    constexpr int ISTR = tap_slot(S - 1) + 2;
    constexpr int OKB = NDIM == 2 ? 4 : 8;  // validity bits under a packed row
    __shared__ float4 rec[GPB * ISTR];
    __shared__ unsigned rec_ok[GPB * ISTR];
    __shared__ float rec_z[NDIM == 3 ? GPB * ISTR : 1];

    {
        // one lane group per query: the launch makes a CTA's query run exactly GPB long
        long long q = q_lo + grp;   // position among the batch's queries
        const bool active = q < q_hi;
        if (!active) q = q_hi - 1;  // recompute a real query, write nothing
        if (p.order != nullptr) {
            // query order: position q runs query order[b * Nq + q], clamped into [0, Nq)
            // (a malformed order gives wrong results, never an out-of-range access)
            const int o = __ldg(p.order + b * p.Nq + q);
            q = o < 0 ? 0 : (o >= p.Nq ? p.Nq - 1 : o);
        }
        const long long item = (b * p.Nq + q) * p.M + m;
        const char *go_row = static_cast<const char *>(p.grad_out) + item * (rb / p.M);
        float g[N], gr[N];
        unpack(ldg16(go_row + sub * 16), g);
        run_channels<DT, G>(go_row, sub, g, gr);
        // fused: softmax weights of the samples this lane owns (max and sum over the group)
        // and their grad_A, kept until the item's logit gradients can be formed
        float av[NB], gAs[NB];
#pragma unroll
        for (int bt = 0; bt < NB; ++bt) gAs[bt] = 0.f;
        if constexpr (FUSED) {
            float mx = -INFINITY;
#pragma unroll
            for (int bt = 0; bt < NB; ++bt) {
                const int own = bt * G + sub;
                av[bt] = own < S ? __ldcs(p.attn + item * S + own) : -INFINITY;
                mx = fmaxf(mx, av[bt]);
            }
            mx = group_max<G>(mx);
            float sum = 0.f;
#pragma unroll
            for (int bt = 0; bt < NB; ++bt) {
                av[bt] = bt * G + sub < S ? expf(av[bt] - mx) : 0.f;
                sum += av[bt];
            }
            sum = group_sum<G>(sum);
#pragma unroll
            for (int bt = 0; bt < NB; ++bt) av[bt] = __fdiv_rn(av[bt], sum);
        }

        // The group exchanges, per sample, either its 2^ndim partial dot products (the owner
        // then forms the gradients from its fractions) or, with FOLD, the partial gradients
        // each lane folds them into (see step 2).  Measured on B300: exchanging the dot
        // products is faster in 2D (the fused encoder backward 444 us against 462 us),
        // folding in 3D (the volume backward 722 us against 733 us, fused 796 against 819).
        constexpr bool FOLD = NDIM == 3;

        // 1. taps of the samples this lane owns (bt * G + sub), left in shared memory for
        //    the group; the owner keeps its weight, validity bits and (without FOLD) the
        //    fractions for its own outputs
        float aw[NB], frac[NB][NDIM];
        unsigned okw[NB];
#pragma unroll
        for (int bt = 0; bt < NB; ++bt) {
            const int own = bt * G + sub;
            const int so = own < S ? own : S - 1;
            float xyz[NDIM];
            const float *lsrc = p.loc + (item * S + so) * NDIM;
            if constexpr (NDIM == 2) {
                const float2 v = __ldcs(reinterpret_cast<const float2 *>(lsrc));
                xyz[0] = v.x;
                xyz[1] = v.y;
            } else {
#pragma unroll
                for (int k = 0; k < NDIM; ++k) xyz[k] = __ldcs(lsrc + k);
            }
            float a;
            if constexpr (FUSED) {
#pragma unroll
                for (int k = 0; k < NDIM; ++k)
                    xyz[k] = fused_location<NDIM>(p, item / p.M, so / PP, k, xyz[k]);
                a = av[bt];
            } else {
                a = __ldcs(p.attn + item * S + so);
            }
            Taps<NC> mine;
            float *fr = frac[bt];
            make_taps(p, so / PP, xyz, a, mine, fr);
            aw[bt] = a;
            okw[bt] = mine.ok;
            if (own < S) {
                // the validity bits ride under the row when it leaves room (p.pack_taps)
                const int j = grp * ISTR + tap_slot(own);
                const int rbits =
                    p.pack_taps ? static_cast<int>((static_cast<unsigned>(mine.row) << OKB) | mine.ok)
                                : mine.row;
                rec[j] = make_float4(__int_as_float(rbits), a, fr[0], fr[1]);
                if (!p.pack_taps) rec_ok[j] = mine.ok;
                if constexpr (NDIM == 3) rec_z[j] = fr[2];
            }
        }
        __syncwarp();

        // 2. per batch of G samples: corner rows (in-level corners only), the dot products
        //    d_c = <g, v_c> over this lane's channels, grad_value reductions.  A sample's
        //    gradients are linear in its dot products -- grad_A = sum_c w_c d_c and
        //    grad_x = sum_c (dw_c / dx) d_c, likewise y (and z), with w_c the bilinear
        //    (trilinear) weights without A.  One reduce-scatter over the group hands the
        //    owner of each sample the group's sums: of the dot products, or with FOLD of
        //    the partial gradients each lane folds its dot products into at once.
        constexpr int NG = FOLD ? 1 + NDIM : NC;  // values exchanged per sample
#pragma unroll
        for (int bt = 0; bt < NB; ++bt) {
            float pg[G][NG];  // this lane's partial values of every sample of the batch
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const int s = bt * G + j;
#pragma unroll
                for (int k = 0; k < NG; ++k) pg[j][k] = 0.f;
                if (s >= S) continue;
                const int jr = grp * ISTR + tap_slot(s);
                const float4 rr = rec[jr];
                const int rv = __float_as_int(rr.x);
                const int row = p.pack_taps ? rv >> OKB : rv;
                const unsigned ok = p.pack_taps ? static_cast<unsigned>(rv) & ((1u << OKB) - 1u)
                                                : rec_ok[jr];
                float w[NC];
                float fz = 0.f;
                if constexpr (NDIM == 2) {
                    tap_weights(rr.y, rr.z, rr.w, w);
                } else {
                    fz = rec_z[jr];
                    tap_weights(rr.y, rr.z, rr.w, fz, w);
                }
                // the per-axis factors of the corner weights, without A
                const float wx[2] = {1.f - rr.z, rr.z};
                const float wy[2] = {1.f - rr.w, rr.w};
                const float wz[2] = {NDIM == 3 ? 1.f - fz : 1.f, NDIM == 3 ? fz : 1.f};
                const int l = s / PP;
                // value and grad_value addresses of corner 0 and of the corner one image row
                // further; grad_value rows are fp32, GS times as wide as value rows
                const char *c0 = vbase + static_cast<long long>(row) * p.rb32;
                const char *cy[2] = {c0, c0 + p.sy[l]};
                char *g0 = gbase + static_cast<long long>(row) * (static_cast<long long>(p.rb32) * GS);
                char *gy[2] = {g0, g0 + p.sy[l] * GS};
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const int dx = c & 1, dy = (c >> 1) & 1, dz = c >> 2;
                    const bool in =
                        ((ok >> c) & 1u) &&
                        row_ok(p, static_cast<long long>(row) + dx + (dy ? p.W[l] : 0) +
                                      (dz ? static_cast<long long>(p.W[l]) * p.H[l] : 0),
                               item, s);
                    const char *src = cy[dy] + (dz ? p.sz[l] : 0) + (dx ? rb : 0);
                    Slice<16> u;
                    load_slice_if(in, src, u);
                    float v[N];
                    unpack(u.a, v);
                    float d = 0.f;
                    if (in) {
#pragma unroll
                        for (int i = 0; i < N; ++i) d = fmaf(g[i], v[i], d);
                    }
                    if constexpr (FOLD) {
                        const float sx = dx ? 1.f : -1.f, sy = dy ? 1.f : -1.f;
                        const float sz = dz ? 1.f : -1.f;
                        pg[j][0] = fmaf(wz[dz] * wy[dy] * wx[dx], d, pg[j][0]);
                        pg[j][1] = fmaf(sx * wz[dz] * wy[dy], d, pg[j][1]);
                        pg[j][2] = fmaf(sy * wz[dz] * wx[dx], d, pg[j][2]);
                        if constexpr (NDIM == 3) pg[j][3] = fmaf(sz * wy[dy] * wx[dx], d, pg[j][3]);
                    } else {
                        pg[j][c] = d;
                    }
                    if (active && in) {
                        char *dst = gy[dy] + (dz ? p.sz[l] * GS : 0) + (dx ? rb * GS : 0);
                        add_global_runs<N, G>(reinterpret_cast<float *>(dst), w[c], gr);
                    }
                }
            }
            reduce_scatter<G, NG>(pg, sub);
            const int own = bt * G + sub;
            if (active && own < S) {
                // the gradients of sample `own` before the factors A and extent
                float gA = 0.f, gx = 0.f, gy = 0.f, gz = 0.f;
                if constexpr (FOLD) {
                    gA = pg[0][0];
                    gx = pg[0][1];
                    gy = pg[0][2];
                    if constexpr (NDIM == 3) gz = pg[0][NDIM];
                } else {
                    // pg[0][c] = <g, v_c> of sample `own`; weight derivatives from frac
                    const float *fr = frac[bt];
                    const float wx[2] = {1.f - fr[0], fr[0]}, wy[2] = {1.f - fr[1], fr[1]};
                    const float wz[2] = {NDIM == 3 ? 1.f - fr[NDIM - 1] : 1.f,
                                         NDIM == 3 ? fr[NDIM - 1] : 1.f};
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const int dx = c & 1, dy = (c >> 1) & 1, dz = c >> 2;
                        const float d = pg[0][c];
                        const float sx = dx ? 1.f : -1.f, sy = dy ? 1.f : -1.f;
                        const float sz = dz ? 1.f : -1.f;
                        gA = fmaf(wz[dz] * wy[dy] * wx[dx], d, gA);
                        gx = fmaf(sx * wz[dz] * wy[dy], d, gx);
                        gy = fmaf(sy * wz[dz] * wx[dx], d, gy);
                        if constexpr (NDIM == 3) gz = fmaf(sz * wy[dy] * wx[dx], d, gz);
                    }
                }
                const long long s = item * S + own;
                const bool any = okw[bt] != 0u;
                const int l = own / PP;
                const float a = aw[bt];
                // fused: the offset gradient, d location / d offset = 1 / extent
                if constexpr (FUSED) gAs[bt] = gA;
                else p.grad_attn[s] = gA;
                p.grad_loc[NDIM * s] = any ? a * gx * (FUSED ? 1.f : p.fW[l]) : 0.f;
                p.grad_loc[NDIM * s + 1] = any ? a * gy * (FUSED ? 1.f : p.fH[l]) : 0.f;
                if constexpr (NDIM == 3)
                    p.grad_loc[NDIM * s + 2] = any ? a * gz * (FUSED ? 1.f : p.fZ[l]) : 0.f;
            }
        }
        if constexpr (FUSED) {
            // logit gradients (softmax Jacobian): A_s * (grad_A_s - sum_t A_t * grad_A_t)
            float dot = 0.f;
#pragma unroll
            for (int bt = 0; bt < NB; ++bt)
                if (bt * G + sub < S) dot = fmaf(av[bt], gAs[bt], dot);
            dot = group_sum<G>(dot);
            if (active) {
#pragma unroll
                for (int bt = 0; bt < NB; ++bt) {
                    const int own = bt * G + sub;
                    if (own < S) p.grad_attn[item * S + own] = av[bt] * (gAs[bt] - dot);
                }
            }
        }
    }

}

// Resident blocks per SM asked of the compiler for rows of up to 8 lanes: 3 x 256 threads
// in 2D (at most 85 registers) and 4 x 128 in 3D (at most 128).  The plain kernels reach
// that residency without the bound, but are scheduled better under it; the fused 2D kernel
// would otherwise take 86 registers and lose a block.  Measured on B300 against no bound:
// the encoder backward 407 us against 425 us, the volume one 984 against 1000, the fused
// encoder backward 456 against 508.  Wider rows (bwd_tiled_wide) keep the compiler's choice.
template <int NDIM> constexpr int bwd_min_blocks() { return NDIM == 2 ? 3 : 4; }

template <int DT, int G, int NDIM, int LL, int PP, int BT, bool FUSED>
__global__ void __launch_bounds__(BT, (bwd_min_blocks<NDIM>()))
bwd_tiled(const __grid_constant__ Params p) {
    bwd_tiled_body<DT, G, NDIM, LL, PP, BT, FUSED>(p);
}

template <int DT, int G, int NDIM, int LL, int PP, int BT, bool FUSED>
__global__ void __launch_bounds__(BT)
bwd_tiled_wide(const __grid_constant__ Params p) {
    bwd_tiled_body<DT, G, NDIM, LL, PP, BT, FUSED>(p);
}

// Block size of the tiled backward: 256 threads in 2D, 128 in 3D (measured on B300: the
// 3D kernel, 128 registers per thread, ran 17% faster with the finer blocks; 2D ran 2%
// slower).
template <int NDIM> constexpr int bwd_block() { return NDIM == 3 ? 128 : 256; }

template <int DT, int G, int NDIM, int LL, int PP, bool FUSED>
cudaError_t launch_bwd_tiled(Params p, cudaStream_t s) {
    constexpr int BT = bwd_block<NDIM>();
    // one lane group per query, one round per CTA: CTA = (b, m, run of BT / G queries)
    // (bwd_tiled_body relies on qchunk == BT / G)
    p.qchunk = BT / G;
    p.nchunk = static_cast<int>((p.Nq + p.qchunk - 1) / p.qchunk);
    const long long ctas = p.B * p.M * p.nchunk;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if constexpr (G <= 8)
        bwd_tiled<DT, G, NDIM, LL, PP, BT, FUSED><<<static_cast<unsigned>(ctas), BT, 0, s>>>(p);
    else
        bwd_tiled_wide<DT, G, NDIM, LL, PP, BT, FUSED>
            <<<static_cast<unsigned>(ctas), BT, 0, s>>>(p);
    return cudaGetLastError();
}

template <int DT, int G, int NDIM, bool FUSED>
cudaError_t backward_nd(const Params &p, cudaStream_t s) {
    if (backward_is_tiled(p)) {
        if (p.L == 4) return launch_bwd_tiled<DT, G, NDIM, 4, 4, FUSED>(p, s);
        return launch_bwd_tiled<DT, G, NDIM, 1, 4, FUSED>(p, s);
    }
    const long long threads = p.n_items * G;
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks)), block(256);
    if constexpr (NDIM == 2) bwd2d_generic<DT, G, 0, 0, FUSED><<<grid, block, 0, s>>>(p);
    else bwd3d_generic<DT, G, 0, 0, FUSED><<<grid, block, 0, s>>>(p);
    return cudaGetLastError();
}

// FUSED: `loc` holds pixel offsets and `attn` logits (as in the fused forward); the
// kernels write the offset gradients to grad_loc.  bwd_tiled writes the logit gradients
// itself; the generic kernels write grad_A to grad_attn, which the epilogue in
// msda_backward.cu turns into the logit gradients.
template <int NDIM, bool FUSED>
cudaError_t backward_dispatch(int dtype, int G, const Params &p, cudaStream_t s) {
#define MSDA_BWD_CASE(DT, GG) \
    if (dtype == DT && G == GG) return backward_nd<DT, GG, NDIM, FUSED>(p, s);
    MSDA_BWD_CASE(kF32, 1) MSDA_BWD_CASE(kF32, 2) MSDA_BWD_CASE(kF32, 4)
    MSDA_BWD_CASE(kF32, 8) MSDA_BWD_CASE(kF32, 16) MSDA_BWD_CASE(kF32, 32)
    MSDA_BWD_CASE(kBF16, 1) MSDA_BWD_CASE(kBF16, 2) MSDA_BWD_CASE(kBF16, 4)
    MSDA_BWD_CASE(kBF16, 8) MSDA_BWD_CASE(kBF16, 16) MSDA_BWD_CASE(kBF16, 32)
#undef MSDA_BWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

}  // namespace msda
