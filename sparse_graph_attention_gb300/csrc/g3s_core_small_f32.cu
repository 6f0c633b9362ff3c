// Instantiations of the small-graph flavour of the fused CUDA-core kernel
// (one CTA per row) for float inputs.
#include "g3s_core.cuh"

namespace g3s {

cudaError_t core_small_launch_f32(bool out_f32, int mode, const CoreParams& p, cudaStream_t st) {
    using namespace core_detail;
    (void)out_f32;
    return launch_small_mode<float, float>(mode, p, st);
}

}  // namespace g3s
