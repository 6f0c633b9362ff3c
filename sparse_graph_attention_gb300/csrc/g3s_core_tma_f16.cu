// Instantiations of the TMA-fed fused kernel for __half inputs.
#include "g3s_core_tma.cuh"

namespace g3s {

cudaError_t core_tma_launch_f16(bool out_f32, const CoreParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t st) {
    using namespace core_detail;
    if (out_f32) return launch_core_tma<__half, float>(p, tk, tv, st);
    return launch_core_tma<__half, __half>(p, tk, tv, st);
}

}  // namespace g3s
