// Forward entry of the kernel layer: picks the instantiation for the value dtype and
// dimensionality (msda_forward_{f32,bf16}_{2d,3d}.cu; kernels in msda_forward.cuh).
#include "msda_internal.h"

namespace msda {

cudaError_t launch_forward(int ndim, int dtype, int G, const Params &p, cudaStream_t s) {
    if (p.n_items == 0) return cudaSuccess;
    if (dtype == kF32) return ndim == 2 ? launch_forward_f32_2d(G, p, s) : launch_forward_f32_3d(G, p, s);
    if (dtype == kBF16)
        return ndim == 2 ? launch_forward_bf16_2d(G, p, s) : launch_forward_bf16_3d(G, p, s);
    return cudaErrorInvalidValue;
}

}  // namespace msda
