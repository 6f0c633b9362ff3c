// Instantiations of the small-graph flavour of the fused CUDA-core kernel
// (one CTA per row) for __half inputs.
#include "g3s_core.cuh"

namespace g3s {

cudaError_t core_small_launch_f16(bool out_f32, int mode, const CoreParams& p, cudaStream_t st) {
    using namespace core_detail;
    return out_f32 ? launch_small_mode<__half, float>(mode, p, st) : launch_small_mode<__half, __half>(mode, p, st);
}

}  // namespace g3s
