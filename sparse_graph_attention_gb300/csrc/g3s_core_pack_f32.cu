// Instantiations of the short-row pack flavour of the fused CUDA-core kernel
// for float inputs (a file of its own so it compiles in parallel).
#include "g3s_core.cuh"

namespace g3s {

cudaError_t core_launch_pack_f32(bool out_f32, int mode, const CoreParams& p, cudaStream_t st) {
    using namespace core_detail;
    (void)out_f32;
    return launch_core_packed_mode<float, float>(mode, p, st);
}

}  // namespace g3s
