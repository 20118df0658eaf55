// Forward kernels: multi-scale deformable attention sampling + weighted sum.
//
// out[b,q,m,:] = sum_l sum_p A[b,q,m,l,p] * interp_l(value[b, level l, m, :], loc[b,q,m,l,p])
// ("Deformable Attention Module", DeformAttn equation; multi-scale blending and the 2D->3D
// changes from "3D Attention That Knows Where to Look").
//
// Mapping: a lane group of G lanes per (b, q, m) work item; lane k owns 16 bytes of
// channels.  Per sample the group computes the cell and corner weights redundantly
// (cheap ALU), then issues one predicated 16-byte load per existing corner: a warp-wide
// load brings 32/G whole value rows.  Corners outside the level are neither loaded nor
// weighted.  fp32 accumulation; one store of the item's D channels at the end.
#include "common.cuh"

namespace msda {

namespace {

template <int DT, int G, int LL, int PP>
__global__ void __launch_bounds__(256)
fwd2d_kernel(const __grid_constant__ Params p) {
    constexpr int N = Vec<DT>::N;
    const int L = LL > 0 ? LL : p.L;
    const int P = PP > 0 ? PP : p.P;
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long item = t / G;
    if (item >= p.n_items) return;
    const int sub = threadIdx.x & (G - 1);
    const int m = static_cast<int>(item % p.M);
    const long long b = item / p.M / p.Nq;
    const long long rb = p.row_bytes;
    const char *vb = static_cast<const char *>(p.value) + (b * p.Nin) * rb +
                     static_cast<long long>(m) * (rb / p.M) + sub * 16;
    const float2 *lp = reinterpret_cast<const float2 *>(p.loc) + item * L * P;
    const float *ap = p.attn + item * L * P;

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
            const float2 xy = __ldg(lp + l * P + k);
            const float a = __ldg(ap + l * P + k);
            int x0, y0;
            float fx, fy;
            const bool okx = pixel_coord(xy.x, fW, x0, fx);
            const bool oky = pixel_coord(xy.y, fH, y0, fy);
            const bool ok = okx && oky;
            const bool vx0 = ok && x0 >= 0, vx1 = ok && x0 < W - 1;
            const bool vy0 = y0 >= 0, vy1 = y0 < H - 1;
            const float ay0 = a * (1.f - fy), ay1 = a * fy;
            const float w00 = (vy0 && vx0) ? ay0 * (1.f - fx) : 0.f;
            const float w01 = (vy0 && vx1) ? ay0 * fx : 0.f;
            const float w10 = (vy1 && vx0) ? ay1 * (1.f - fx) : 0.f;
            const float w11 = (vy1 && vx1) ? ay1 * fx : 0.f;
            const char *c00 = vl + static_cast<long long>(y0 * W + x0) * rb;
            uint4 u00 = make_uint4(0, 0, 0, 0), u01 = u00, u10 = u00, u11 = u00;
            if (vy0 && vx0) u00 = ldg16(c00);
            if (vy0 && vx1) u01 = ldg16(c00 + rb);
            if (vy1 && vx0) u10 = ldg16(c00 + W * rb);
            if (vy1 && vx1) u11 = ldg16(c00 + (W + 1) * rb);
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

template <int DT, int G, int LL, int PP>
__global__ void __launch_bounds__(256)
fwd3d_kernel(const __grid_constant__ Params p) {
    constexpr int N = Vec<DT>::N;
    const int L = LL > 0 ? LL : p.L;
    const int P = PP > 0 ? PP : p.P;
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long item = t / G;
    if (item >= p.n_items) return;
    const int sub = threadIdx.x & (G - 1);
    const int m = static_cast<int>(item % p.M);
    const long long b = item / p.M / p.Nq;
    const long long rb = p.row_bytes;
    const char *vb = static_cast<const char *>(p.value) + (b * p.Nin) * rb +
                     static_cast<long long>(m) * (rb / p.M) + sub * 16;
    const float *lp = p.loc + item * L * P * 3;
    const float *ap = p.attn + item * L * P;

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
            const float lx = __ldg(xyz), ly = __ldg(xyz + 1), lz = __ldg(xyz + 2);
            const float a = __ldg(ap + l * P + k);
            int x0, y0, z0;
            float fx, fy, fz;
            const bool ok = pixel_coord(lx, fW, x0, fx) & pixel_coord(ly, fH, y0, fy) &
                            pixel_coord(lz, fZ, z0, fz);
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
                const bool inside = vx[dx] && vy[dy] && vz[dz];
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

template <int DT, int G>
cudaError_t forward_lp(int ndim, const Params &p, cudaStream_t s) {
    const long long threads = p.n_items * G;
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks)), block(256);
    if (ndim == 2) {
        if (p.L == 4 && p.P == 4) fwd2d_kernel<DT, G, 4, 4><<<grid, block, 0, s>>>(p);
        else if (p.L == 1 && p.P == 4) fwd2d_kernel<DT, G, 1, 4><<<grid, block, 0, s>>>(p);
        else fwd2d_kernel<DT, G, 0, 0><<<grid, block, 0, s>>>(p);
    } else {
        if (p.L == 4 && p.P == 4) fwd3d_kernel<DT, G, 4, 4><<<grid, block, 0, s>>>(p);
        else if (p.L == 1 && p.P == 4) fwd3d_kernel<DT, G, 1, 4><<<grid, block, 0, s>>>(p);
        else fwd3d_kernel<DT, G, 0, 0><<<grid, block, 0, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward(int ndim, int dtype, int G, const Params &p, cudaStream_t s) {
    if (p.n_items == 0) return cudaSuccess;
#define MSDA_FWD_CASE(DT, GG) \
    if (dtype == DT && G == GG) return forward_lp<DT, GG>(ndim, p, s);
    MSDA_FWD_CASE(kF32, 1) MSDA_FWD_CASE(kF32, 2) MSDA_FWD_CASE(kF32, 4)
    MSDA_FWD_CASE(kF32, 8) MSDA_FWD_CASE(kF32, 16) MSDA_FWD_CASE(kF32, 32)
    MSDA_FWD_CASE(kBF16, 1) MSDA_FWD_CASE(kBF16, 2) MSDA_FWD_CASE(kBF16, 4)
    MSDA_FWD_CASE(kBF16, 8) MSDA_FWD_CASE(kBF16, 16) MSDA_FWD_CASE(kBF16, 32)
#undef MSDA_FWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace msda
