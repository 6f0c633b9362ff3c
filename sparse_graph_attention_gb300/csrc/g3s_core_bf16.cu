// Instantiations of the fused CUDA-core kernel for __nv_bfloat16 inputs (one file per
// input type so the templates compile in parallel).
#include "g3s_core.cuh"

namespace g3s {

cudaError_t core_launch_bf16(bool out_f32, bool rtm, const CoreParams& p, cudaStream_t st) {
    using namespace core_detail;
    if (out_f32) return rtm ? launch_core<__nv_bfloat16, float, true>(p, st) : launch_core<__nv_bfloat16, float, false>(p, st);
    return rtm ? launch_core<__nv_bfloat16, __nv_bfloat16, true>(p, st) : launch_core<__nv_bfloat16, __nv_bfloat16, false>(p, st);
}

cudaError_t merge_launch_bf16(bool rtm, const MergeParams& p, cudaStream_t st) {
    return core_detail::launch_merge<__nv_bfloat16>(rtm, p, st);
}

}  // namespace g3s
