// Backward entry of the kernel layer: the grad_value zero-fill and the dispatch to the 2D
// or 3D instantiation (msda_backward_{2d,3d}.cu; kernels in msda_backward.cuh).
#include "common.cuh"

namespace msda {

namespace {

__global__ void zero_fill_kernel(float4 *__restrict__ p, long long n4) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += stride)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
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
    return ndim == 2 ? launch_backward_2d(dtype, G, p, s) : launch_backward_3d(dtype, G, p, s);
}

}  // namespace msda
