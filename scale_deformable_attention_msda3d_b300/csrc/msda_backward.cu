// Backward entry of the kernel layer: the grad_value zero-fill, the dispatch to the 2D or
// 3D instantiation (msda_backward_{2d,3d}.cu, fused prologue msda_backward_fused_{2d,3d}.cu;
// kernels in msda_backward.cuh) and the two small kernels that finish the fused backward:
// the logit gradients after the generic kernels, and the reference-point gradients.
#include "common.cuh"

namespace msda {

namespace {

__global__ void zero_fill_kernel(float4 *__restrict__ p, long long n4) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += stride)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Fused backward through the generic kernels, logit gradients: those kernels leave grad_A
// in grad_attn; with the item's softmax weights A (recomputed from the logits),
//   d/d logit_s = A_s * (grad_A_s - sum_t A_t * grad_A_t)
// (softmax Jacobian), in place.  T lanes (a power of two, T <= 32) per (b, q, m) item; lane
// j takes samples j, j + T, ..., so a warp reads whole runs of consecutive items.
__global__ void logit_grad_kernel(const float *__restrict__ logits, float *grad, long long n_items,
                                  int S, int T) {
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if ((t & ~31LL) / T >= n_items) return;  // whole warps leave together (shuffles below)
    long long item = t / T;
    const bool active = item < n_items;
    if (!active) item = n_items - 1;
    const int j = static_cast<int>(t % T);
    const float *z = logits + item * S;
    float *g = grad + item * S;
    float mx = -INFINITY;
    for (int s = j; s < S; s += T) mx = fmaxf(mx, __ldg(z + s));
    for (int o = T / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o, T));
    float sum = 0.f;
    for (int s = j; s < S; s += T) sum += expf(__ldg(z + s) - mx);
    for (int o = T / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o, T);
    float dot = 0.f;
    for (int s = j; s < S; s += T) dot = fmaf(__fdiv_rn(expf(__ldg(z + s) - mx), sum), g[s], dot);
    for (int o = T / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o, T);
    if (!active) return;
    for (int s = j; s < S; s += T) g[s] = __fdiv_rn(expf(__ldg(z + s) - mx), sum) * (g[s] - dot);
}

// Fused backward, reference-point gradients: location = ref + offset / extent, so
//   d/d ref[b, q, l, k] = sum over m, p of d/d location = sum of extent_lk * d/d offset.
// One thread per (b, q, l, k), summing in the order m, p.
__global__ void ref_grad_kernel(const __grid_constant__ Params p, int ndim) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long n = p.B * p.Nq * p.L * ndim;
    if (i >= n) return;
    const int k = static_cast<int>(i % ndim);
    const int l = static_cast<int>((i / ndim) % p.L);
    const long long bq = i / ndim / p.L;
    const float ext = k == 0 ? p.fW[l] : (k == 1 ? p.fH[l] : p.fZ[l]);
    float acc = 0.f;
    for (int m = 0; m < p.M; ++m) {
        const float *g = p.grad_loc + (((bq * p.M + m) * p.L + l) * p.P) * ndim + k;
        for (int pp = 0; pp < p.P; ++pp) acc = fmaf(ext, g[pp * ndim], acc);
    }
    p.grad_ref[i] = acc;
}

cudaError_t launch_fused_epilogue(int ndim, const Params &p, cudaStream_t s) {
    const int S = p.L * p.P;
    const long long n = p.B * p.Nq * p.L * ndim;
    if ((n + 255) / 256 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaSuccess;
    if (!backward_is_tiled(p)) {  // bwd_tiled formed the logit gradients itself
        int T = 1;
        while (T < 32 && T < S) T <<= 1;
        const long long blocks = (p.n_items * T + 255) / 256;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        logit_grad_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(p.attn, p.grad_attn,
                                                                         p.n_items, S, T);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess || p.grad_ref == nullptr) return e;
    ref_grad_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(p, ndim);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_zero_fill(float *ptr, long long n_floats, cudaStream_t s) {
    if (n_floats <= 0) return cudaSuccess;
    const long long n4 = n_floats / 4;  // rows are whole multiples of 16 bytes
    long long blocks = (n4 + 255) / 256;
    if (blocks > 148LL * 16) blocks = 148LL * 16;
    zero_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        reinterpret_cast<float4 *>(ptr), n4);
    return cudaGetLastError();
}

cudaError_t launch_backward(int ndim, int dtype, int G, const Params &p, cudaStream_t s) {
    if (p.n_items == 0) return cudaSuccess;
    if (p.ref == nullptr)
        return ndim == 2 ? launch_backward_2d(dtype, G, p, s) : launch_backward_3d(dtype, G, p, s);
    const cudaError_t e = ndim == 2 ? launch_backward_fused_2d(dtype, G, p, s)
                                    : launch_backward_fused_3d(dtype, G, p, s);
    if (e != cudaSuccess) return e;
    return launch_fused_epilogue(ndim, p, s);
}

}  // namespace msda
