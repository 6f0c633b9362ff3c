// Instantiations of the fused CUDA-core kernel for float inputs (one file per
// input type so the templates compile in parallel).
#include "g3s_core.cuh"

namespace g3s {

cudaError_t core_launch_f32(bool out_f32, int mode, const CoreParams& p, cudaStream_t st) {
    using namespace core_detail;
    (void)out_f32;
    return launch_core_mode<float, float>(mode, p, st);
}

cudaError_t merge_launch_f32(bool plain, const MergeParams& p, cudaStream_t st) {
    return core_detail::launch_merge<float>(plain, p, st);
}

}  // namespace g3s
