// Instantiations of the fused CUDA-core kernel for float inputs (one file per
// input type so the templates compile in parallel).
#include "g3s_core.cuh"

namespace g3s {

cudaError_t core_launch_f32(bool out_f32, bool rtm, const CoreParams& p, cudaStream_t st) {
    using namespace core_detail;
    (void)out_f32;
    return rtm ? launch_core<float, float, true>(p, st) : launch_core<float, float, false>(p, st);
}

cudaError_t merge_launch_f32(bool rtm, const MergeParams& p, cudaStream_t st) {
    return core_detail::launch_merge<float>(rtm, p, st);
}

}  // namespace g3s
