// Instantiations of the fused CUDA-core kernel for __nv_bfloat16 inputs (one file per
// input type so the templates compile in parallel).
#include "g3s_core.cuh"

namespace g3s {

cudaError_t core_launch_bf16(bool out_f32, int mode, const CoreParams& p, cudaStream_t st) {
    using namespace core_detail;
    if (out_f32) return launch_core_mode<__nv_bfloat16, float>(mode, p, st);
    return launch_core_mode<__nv_bfloat16, __nv_bfloat16>(mode, p, st);
}

cudaError_t merge_launch_bf16(bool plain, const MergeParams& p, cudaStream_t st) {
    return core_detail::launch_merge<__nv_bfloat16>(plain, p, st);
}

}  // namespace g3s
