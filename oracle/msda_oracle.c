/*
 * CPU oracle for the multi-scale deformable attention core (2D bilinear, 3D trilinear).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference leg may load or call this code.  The library that ships
 * (libmsda, the CUDA path) never calls it and shares no code with it.
 *
 * What it computes (the plain definition, evaluated in double precision):
 *
 *   out[b,q,m,:] = sum_l sum_p  A[b,q,m,l,p] * x_l( loc[b,q,m,l,p] )      (per head m)
 *
 * - "Deformable Attention Module" (Code with Papers), the DeformAttn equation: each head
 *   sums A_mqk times the (projected) feature map sampled at p_q + delta p_mqk, with
 *   bilinear interpolation at the fractional location.  Only this inner weighted sum
 *   is computed here; the projections W_m, W'_m are outside the core.
 * - "3D Attention That Knows Where to Look", the multi-scale paragraph: each query
 *   samples P points on every one of the L pyramid levels and blends all L x P samples
 *   in one weighted sum.
 * - same page, "What changes from 2D to 3D": locations (x, y) become (x, y, z), shapes
 *   (H, W) become (D, H, W), bilinear over 4 neighbours becomes trilinear over 8 corners.
 * - "What is Deformable Attention ...", "(3) Bilinear Interpolation": the value at a
 *   non-integer location is blended from the 4 nearest pixels.
 *
 * Readings where the pages are silent (each one is a stated convention):
 * - location -> pixel coordinate: x = loc_x * W_l - 0.5 (align_corners = False), per axis,
 *   with the extent of the sampled level.
 * - flattening: value row of pixel (h, w) of level l is level_start[l] + h*W_l + w, and
 *   of voxel (z, h, w) is level_start[l] + (z*H_l + h)*W_l + w.
 * - zero padding: a corner with an index outside the level contributes 0 and receives no
 *   gradient; a sample whose coordinate is not finite or lies at or beyond -1 / the extent
 *   on some axis contributes 0 (all its corners are outside).
 * - the attention weights are taken as given; nothing is renormalised.
 * - at an integer pixel coordinate the cell is the one chosen by floor(), so the location
 *   gradient there is that cell's (right-hand) derivative.
 *
 * Every floating-point input is passed as double (fp32 and bf16 values widen exactly).
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC (OpenMP only splits
 * the forward's queries across threads, for timing on all host cores; see the end).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* 2D                                                                        */
/* ------------------------------------------------------------------------- */

/* One bilinear tap of a sample: corner pixel (h, w) with weight wgt and the partial
 * derivatives of wgt with respect to the pixel coordinates x and y. */
typedef struct {
    int64_t h, w;
    double wgt, dwdx, dwdy;
    int inside;
} tap2d;

/* The four nearest pixels of pixel coordinate (x, y) in an H x W level.  Returns 0 when
 * the sample lies fully outside (or is not finite), in which case taps are not filled. */
static int bilinear_taps(double x, double y, int64_t H, int64_t W, tap2d t[4])
{
    if (!(x > -1.0 && x < (double)W && y > -1.0 && y < (double)H))
        return 0;
    double x0 = floor(x), y0 = floor(y);
    double fx = x - x0, fy = y - y0;
    int64_t ix = (int64_t)x0, iy = (int64_t)y0;
    /* corner (dy, dx): weight = (dx ? fx : 1-fx) * (dy ? fy : 1-fy) */
    for (int c = 0; c < 4; ++c) {
        int dx = c & 1, dy = c >> 1;
        double wx = dx ? fx : 1.0 - fx;
        double wy = dy ? fy : 1.0 - fy;
        double dwx = dx ? 1.0 : -1.0; /* d wx / d x */
        double dwy = dy ? 1.0 : -1.0; /* d wy / d y */
        t[c].h = iy + dy;
        t[c].w = ix + dx;
        t[c].wgt = wx * wy;
        t[c].dwdx = dwx * wy;
        t[c].dwdy = wx * dwy;
        t[c].inside = (t[c].h >= 0 && t[c].h < H && t[c].w >= 0 && t[c].w < W);
    }
    return 1;
}

static int check_common(int64_t B, int64_t Nin, int64_t Nq, int64_t M, int64_t D,
                        int64_t L, int64_t P)
{
    return (B >= 1 && Nin >= 1 && Nq >= 0 && M >= 1 && D >= 1 && L >= 1 && P >= 1) ? 0 : 1;
}

/* Forward, 2D.  shapes is [L][2] = (H, W); loc is [B,Nq,M,L,P,2] = (x, y). */
int oracle_msda2d_forward(int64_t B, int64_t Nin, int64_t Nq, int64_t M, int64_t D,
                          int64_t L, int64_t P, const int64_t *shapes,
                          const int64_t *level_start, const double *value,
                          const double *loc, const double *attn, double *out)
{
    if (check_common(B, Nin, Nq, M, D, L, P)) return 1;
    for (int64_t b = 0; b < B; ++b)
    for (int64_t q = 0; q < Nq; ++q)
    for (int64_t m = 0; m < M; ++m) {
        double *o = out + ((b * Nq + q) * M + m) * D;
        for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t l = 0; l < L; ++l) {
            int64_t H = shapes[2 * l + 0], W = shapes[2 * l + 1];
            for (int64_t p = 0; p < P; ++p) {
                int64_t s = (((b * Nq + q) * M + m) * L + l) * P + p;
                double x = loc[2 * s + 0] * (double)W - 0.5;
                double y = loc[2 * s + 1] * (double)H - 0.5;
                double a = attn[s];
                tap2d t[4];
                if (!bilinear_taps(x, y, H, W, t)) continue;
                for (int c = 0; c < 4; ++c) {
                    if (!t[c].inside) continue;
                    int64_t row = level_start[l] + t[c].h * W + t[c].w;
                    const double *v = value + ((b * Nin + row) * M + m) * D;
                    for (int64_t d = 0; d < D; ++d) o[d] += a * t[c].wgt * v[d];
                }
            }
        }
    }
    return 0;
}

/* Backward, 2D.  Gradients of sum(out * grad_out) with respect to value, loc and attn.
 * grad_value is overwritten (zeroed first) and accumulated serially. */
int oracle_msda2d_backward(int64_t B, int64_t Nin, int64_t Nq, int64_t M, int64_t D,
                           int64_t L, int64_t P, const int64_t *shapes,
                           const int64_t *level_start, const double *value,
                           const double *loc, const double *attn, const double *grad_out,
                           double *grad_value, double *grad_loc, double *grad_attn)
{
    if (check_common(B, Nin, Nq, M, D, L, P)) return 1;
    memset(grad_value, 0, sizeof(double) * (size_t)(B * Nin * M * D));
    for (int64_t b = 0; b < B; ++b)
    for (int64_t q = 0; q < Nq; ++q)
    for (int64_t m = 0; m < M; ++m) {
        const double *g = grad_out + ((b * Nq + q) * M + m) * D;
        for (int64_t l = 0; l < L; ++l) {
            int64_t H = shapes[2 * l + 0], W = shapes[2 * l + 1];
            for (int64_t p = 0; p < P; ++p) {
                int64_t s = (((b * Nq + q) * M + m) * L + l) * P + p;
                double x = loc[2 * s + 0] * (double)W - 0.5;
                double y = loc[2 * s + 1] * (double)H - 0.5;
                double a = attn[s];
                double gA = 0.0, gx = 0.0, gy = 0.0; /* d/dA, d/dx, d/dy of sum(g*out) */
                tap2d t[4];
                if (bilinear_taps(x, y, H, W, t)) {
                    for (int c = 0; c < 4; ++c) {
                        if (!t[c].inside) continue;
                        int64_t row = level_start[l] + t[c].h * W + t[c].w;
                        const double *v = value + ((b * Nin + row) * M + m) * D;
                        double *gv = grad_value + ((b * Nin + row) * M + m) * D;
                        double gdotv = 0.0;
                        for (int64_t d = 0; d < D; ++d) {
                            gdotv += g[d] * v[d];
                            gv[d] += a * t[c].wgt * g[d];
                        }
                        gA += t[c].wgt * gdotv;
                        gx += a * t[c].dwdx * gdotv;
                        gy += a * t[c].dwdy * gdotv;
                    }
                }
                grad_attn[s] = gA;
                /* chain rule through x = loc_x * W - 0.5, y = loc_y * H - 0.5 */
                grad_loc[2 * s + 0] = gx * (double)W;
                grad_loc[2 * s + 1] = gy * (double)H;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* 3D                                                                        */
/* ------------------------------------------------------------------------- */

typedef struct {
    int64_t z, h, w;
    double wgt, dwdx, dwdy, dwdz;
    int inside;
} tap3d;

/* The eight corners of the voxel cell around pixel coordinate (x, y, z) in a
 * Z x H x W level (trilinear interpolation). */
static int trilinear_taps(double x, double y, double z, int64_t Z, int64_t H, int64_t W,
                          tap3d t[8])
{
    if (!(x > -1.0 && x < (double)W && y > -1.0 && y < (double)H &&
          z > -1.0 && z < (double)Z))
        return 0;
    double x0 = floor(x), y0 = floor(y), z0 = floor(z);
    double fx = x - x0, fy = y - y0, fz = z - z0;
    int64_t ix = (int64_t)x0, iy = (int64_t)y0, iz = (int64_t)z0;
    for (int c = 0; c < 8; ++c) {
        int dx = c & 1, dy = (c >> 1) & 1, dz = c >> 2;
        double wx = dx ? fx : 1.0 - fx;
        double wy = dy ? fy : 1.0 - fy;
        double wz = dz ? fz : 1.0 - fz;
        double sx = dx ? 1.0 : -1.0, sy = dy ? 1.0 : -1.0, sz = dz ? 1.0 : -1.0;
        t[c].z = iz + dz;
        t[c].h = iy + dy;
        t[c].w = ix + dx;
        t[c].wgt = wx * wy * wz;
        t[c].dwdx = sx * wy * wz;
        t[c].dwdy = wx * sy * wz;
        t[c].dwdz = wx * wy * sz;
        t[c].inside = (t[c].z >= 0 && t[c].z < Z && t[c].h >= 0 && t[c].h < H &&
                       t[c].w >= 0 && t[c].w < W);
    }
    return 1;
}

/* Forward, 3D.  shapes is [L][3] = (Z, H, W); loc is [B,Nq,M,L,P,3] = (x, y, z). */
int oracle_msda3d_forward(int64_t B, int64_t Nin, int64_t Nq, int64_t M, int64_t D,
                          int64_t L, int64_t P, const int64_t *shapes,
                          const int64_t *level_start, const double *value,
                          const double *loc, const double *attn, double *out)
{
    if (check_common(B, Nin, Nq, M, D, L, P)) return 1;
    for (int64_t b = 0; b < B; ++b)
    for (int64_t q = 0; q < Nq; ++q)
    for (int64_t m = 0; m < M; ++m) {
        double *o = out + ((b * Nq + q) * M + m) * D;
        for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t l = 0; l < L; ++l) {
            int64_t Z = shapes[3 * l + 0], H = shapes[3 * l + 1], W = shapes[3 * l + 2];
            for (int64_t p = 0; p < P; ++p) {
                int64_t s = (((b * Nq + q) * M + m) * L + l) * P + p;
                double x = loc[3 * s + 0] * (double)W - 0.5;
                double y = loc[3 * s + 1] * (double)H - 0.5;
                double z = loc[3 * s + 2] * (double)Z - 0.5;
                double a = attn[s];
                tap3d t[8];
                if (!trilinear_taps(x, y, z, Z, H, W, t)) continue;
                for (int c = 0; c < 8; ++c) {
                    if (!t[c].inside) continue;
                    int64_t row = level_start[l] + (t[c].z * H + t[c].h) * W + t[c].w;
                    const double *v = value + ((b * Nin + row) * M + m) * D;
                    for (int64_t d = 0; d < D; ++d) o[d] += a * t[c].wgt * v[d];
                }
            }
        }
    }
    return 0;
}

/* Backward, 3D. */
int oracle_msda3d_backward(int64_t B, int64_t Nin, int64_t Nq, int64_t M, int64_t D,
                           int64_t L, int64_t P, const int64_t *shapes,
                           const int64_t *level_start, const double *value,
                           const double *loc, const double *attn, const double *grad_out,
                           double *grad_value, double *grad_loc, double *grad_attn)
{
    if (check_common(B, Nin, Nq, M, D, L, P)) return 1;
    memset(grad_value, 0, sizeof(double) * (size_t)(B * Nin * M * D));
    for (int64_t b = 0; b < B; ++b)
    for (int64_t q = 0; q < Nq; ++q)
    for (int64_t m = 0; m < M; ++m) {
        const double *g = grad_out + ((b * Nq + q) * M + m) * D;
        for (int64_t l = 0; l < L; ++l) {
            int64_t Z = shapes[3 * l + 0], H = shapes[3 * l + 1], W = shapes[3 * l + 2];
            for (int64_t p = 0; p < P; ++p) {
                int64_t s = (((b * Nq + q) * M + m) * L + l) * P + p;
                double x = loc[3 * s + 0] * (double)W - 0.5;
                double y = loc[3 * s + 1] * (double)H - 0.5;
                double z = loc[3 * s + 2] * (double)Z - 0.5;
                double a = attn[s];
                double gA = 0.0, gx = 0.0, gy = 0.0, gz = 0.0;
                tap3d t[8];
                if (trilinear_taps(x, y, z, Z, H, W, t)) {
                    for (int c = 0; c < 8; ++c) {
                        if (!t[c].inside) continue;
                        int64_t row = level_start[l] + (t[c].z * H + t[c].h) * W + t[c].w;
                        const double *v = value + ((b * Nin + row) * M + m) * D;
                        double *gv = grad_value + ((b * Nin + row) * M + m) * D;
                        double gdotv = 0.0;
                        for (int64_t d = 0; d < D; ++d) {
                            gdotv += g[d] * v[d];
                            gv[d] += a * t[c].wgt * g[d];
                        }
                        gA += t[c].wgt * gdotv;
                        gx += a * t[c].dwdx * gdotv;
                        gy += a * t[c].dwdy * gdotv;
                        gz += a * t[c].dwdz * gdotv;
                    }
                }
                grad_attn[s] = gA;
                grad_loc[3 * s + 0] = gx * (double)W;
                grad_loc[3 * s + 1] = gy * (double)H;
                grad_loc[3 * s + 2] = gz * (double)Z;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Forward over all host cores (for timing the oracle as a CPU baseline)     */
/* ------------------------------------------------------------------------- */

/* Every output row (b, q) of the forward depends only on its own locations and weights,
 * so the forward over all queries equals the forward over any split of the queries.
 * These entry points cut each batch's queries into blocks of OR_BLOCK and hand the
 * blocks to OpenMP threads; each block runs the serial forward above, unchanged, on its
 * slice (B = 1, Nq = block size), so every output is computed by the same arithmetic in
 * the same order as in the serial call.  nthreads <= 0 uses OpenMP's default. */
#define OR_BLOCK 64

typedef int (*oracle_fwd_fn)(int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t,
                             const int64_t *, const int64_t *, const double *, const double *,
                             const double *, double *);

static int forward_blocks(oracle_fwd_fn fn, int nd, int64_t B, int64_t Nin, int64_t Nq,
                          int64_t M, int64_t D, int64_t L, int64_t P, const int64_t *shapes,
                          const int64_t *level_start, const double *value, const double *loc,
                          const double *attn, double *out, int nthreads)
{
    if (check_common(B, Nin, Nq, M, D, L, P)) return 1;
    const int64_t per_b = (Nq + OR_BLOCK - 1) / OR_BLOCK;
    const int64_t total = B * per_b;
    const int64_t S = M * L * P; /* samples per query */
    int rc = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) reduction(| : rc) num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
#endif
    for (int64_t t = 0; t < total; ++t) {
        const int64_t b = t / per_b;
        const int64_t q0 = (t % per_b) * OR_BLOCK;
        const int64_t nq = (Nq - q0) < OR_BLOCK ? (Nq - q0) : OR_BLOCK;
        const int64_t first = b * Nq + q0; /* first (b, q) row of the block */
        rc |= fn(1, Nin, nq, M, D, L, P, shapes, level_start, value + b * Nin * M * D,
                 loc + first * S * nd, attn + first * S, out + first * M * D);
    }
    return rc;
}

int oracle_msda2d_forward_threads(int64_t B, int64_t Nin, int64_t Nq, int64_t M, int64_t D,
                                  int64_t L, int64_t P, const int64_t *shapes,
                                  const int64_t *level_start, const double *value,
                                  const double *loc, const double *attn, double *out,
                                  int nthreads)
{
    return forward_blocks(oracle_msda2d_forward, 2, B, Nin, Nq, M, D, L, P, shapes,
                          level_start, value, loc, attn, out, nthreads);
}

int oracle_msda3d_forward_threads(int64_t B, int64_t Nin, int64_t Nq, int64_t M, int64_t D,
                                  int64_t L, int64_t P, const int64_t *shapes,
                                  const int64_t *level_start, const double *value,
                                  const double *loc, const double *attn, double *out,
                                  int nthreads)
{
    return forward_blocks(oracle_msda3d_forward, 3, B, Nin, Nq, M, D, L, P, shapes,
                          level_start, value, loc, attn, out, nthreads);
}

/* Threads an OpenMP parallel region of this build gets by default (1 without OpenMP). */
int oracle_default_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
