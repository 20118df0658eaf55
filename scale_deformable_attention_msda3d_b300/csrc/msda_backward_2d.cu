// Backward kernels instantiated for 2D, both value dtypes (see msda_backward.cuh).
#include "msda_backward.cuh"

namespace msda {

cudaError_t launch_backward_2d(int dtype, int G, const Params &p, cudaStream_t s) {
    return backward_dispatch<2, false>(dtype, G, p, s);
}

}  // namespace msda
