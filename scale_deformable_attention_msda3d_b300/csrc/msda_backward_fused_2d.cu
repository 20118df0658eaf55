// Fused-prologue backward kernels instantiated for 2D, both value dtypes (see
// msda_backward.cuh; the logit and reference-point gradients are finished in msda_backward.cu).
#include "msda_backward.cuh"

namespace msda {

cudaError_t launch_backward_fused_2d(int dtype, int G, const Params &p, cudaStream_t s) {
    return backward_dispatch<2, true>(dtype, G, p, s);
}

}  // namespace msda
