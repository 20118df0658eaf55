// Backward entry of the kernel layer: the grad_value zero-fill, the dispatch to the 2D or
// 3D instantiation (msda_backward_{2d,3d}.cu, fused prologue msda_backward_fused_{2d,3d}.cu;
// kernels in msda_backward.cuh) and the two small kernels that finish the fused backward's
// logit and reference-point gradients.
#include "common.cuh"

namespace msda {

namespace {

__global__ void zero_fill_kernel(float4 *__restrict__ p, long long n4) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += stride)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Fused backward, logit gradients: the kernels left grad_A in grad_attn; with the item's
// softmax weights A (recomputed from the logits as the kernels formed them),
//   d/d logit_s = A_s * (grad_A_s - sum_t A_t * grad_A_t)
// (softmax Jacobian).  One thread per (b, q, m) item, in place.
__global__ void logit_grad_kernel(const float *__restrict__ logits, float *grad, long long n_items,
                                  int S) {
    const long long item = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (item >= n_items) return;
    const float *z = logits + item * S;
    float *g = grad + item * S;
    float mx, sum;
    logit_stats(z, S, mx, sum);
    float dot = 0.f;
    for (int s = 0; s < S; ++s) dot = fmaf(__fdiv_rn(expf(__ldg(z + s) - mx), sum), g[s], dot);
    for (int s = 0; s < S; ++s) {
        const float a = __fdiv_rn(expf(__ldg(z + s) - mx), sum);
        g[s] = a * (g[s] - dot);
    }
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
    const long long blocks = (p.n_items + 255) / 256;
    const long long n = p.B * p.Nq * p.L * ndim;
    if (blocks > 0x7fffffffLL || (n + 255) / 256 > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    logit_grad_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(p.attn, p.grad_attn,
                                                                     p.n_items, S);
    cudaError_t e = cudaGetLastError();
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
