// Forward kernels instantiated for bf16 values, 3D (see msda_forward.cuh).
#include "msda_forward.cuh"

namespace msda {

cudaError_t launch_forward_bf16_3d(int G, const Params &p, cudaStream_t s) {
    return forward_dispatch<kBF16, 3>(G, p, s);
}

}  // namespace msda
