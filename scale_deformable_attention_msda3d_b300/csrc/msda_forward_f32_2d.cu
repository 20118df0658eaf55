// Forward kernels instantiated for f32 values, 2D (see msda_forward.cuh).
#include "msda_forward.cuh"

namespace msda {

cudaError_t launch_forward_f32_2d(int G, const Params &p, cudaStream_t s) {
    return forward_dispatch<kF32, 2>(G, p, s);
}

}  // namespace msda
