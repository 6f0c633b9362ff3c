// Instantiations of the fused CUDA-core kernel for __half inputs (one file per
// input type so the templates compile in parallel).
#include "g3s_core.cuh"

namespace g3s {

cudaError_t core_launch_f16(bool out_f32, bool rtm, const CoreParams& p, cudaStream_t st) {
    using namespace core_detail;
    if (out_f32) return rtm ? launch_core<__half, float, true>(p, st) : launch_core<__half, float, false>(p, st);
    return rtm ? launch_core<__half, __half, true>(p, st) : launch_core<__half, __half, false>(p, st);
}

cudaError_t merge_launch_f16(bool rtm, const MergeParams& p, cudaStream_t st) {
    return core_detail::launch_merge<__half>(rtm, p, st);
}

}  // namespace g3s
