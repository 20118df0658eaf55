// Runtime-(L, P) forward kernels instantiated for bf16 values, 2D (see msda_forward.cuh).
#include "msda_forward.cuh"

namespace msda {

cudaError_t launch_forward_rt_bf16_2d(int G, const Params &p, cudaStream_t s) {
    switch (G) {
        case 2: return launch_tiled_rt<kBF16, 2, 2>(p, s);
        case 4: return launch_tiled_rt<kBF16, 4, 2>(p, s);
        case 8: return launch_tiled_rt<kBF16, 8, 2>(p, s);
        case 16: return launch_tiled_rt<kBF16, 16, 2>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace msda
