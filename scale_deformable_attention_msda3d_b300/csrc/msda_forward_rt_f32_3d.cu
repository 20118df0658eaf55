// Runtime-(L, P) forward kernels instantiated for f32 values, 3D (see msda_forward.cuh).
#include "msda_forward.cuh"

namespace msda {

cudaError_t launch_forward_rt_f32_3d(int G, const Params &p, cudaStream_t s) {
    switch (G) {
        case 2: return launch_tiled_rt<kF32, 2, 3>(p, s);
        case 4: return launch_tiled_rt<kF32, 4, 3>(p, s);
        case 8: return launch_tiled_rt<kF32, 8, 3>(p, s);
        case 16: return launch_tiled_rt<kF32, 16, 3>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace msda
