// Instantiations of the short-row pack flavour of the fused CUDA-core kernel
// for __half inputs (a file of its own so it compiles in parallel).
#include "g3s_core.cuh"

namespace g3s {

cudaError_t core_launch_pack_f16(bool out_f32, int mode, const CoreParams& p, cudaStream_t st) {
    using namespace core_detail;
    if (out_f32) return launch_core_packed_mode<__half, float>(mode, p, st);
    return launch_core_packed_mode<__half, __half>(mode, p, st);
}

}  // namespace g3s
