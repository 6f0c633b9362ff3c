// Dispatch of the fused CUDA-core kernel and the heavy-row merge by input and
// output element type.  The kernels themselves are in g3s_core.cuh.
#include "g3s_internal.h"

namespace g3s {

bool core_supported(int dtype, int row_vecs) {
    if (dtype < 0 || dtype > 2) return false;
    if (row_vecs < 1 || row_vecs > 256 || (row_vecs & (row_vecs - 1))) return false;
    return true;
}

cudaError_t core_launch(int dtype, int out_dtype, int mode, const CoreParams& p, cudaStream_t st) {
    const bool out_f32 = out_dtype == 0;
    if (!out_f32 && out_dtype != dtype) return cudaErrorInvalidValue;
    switch (dtype) {
        case 0: return core_launch_f32(true, mode, p, st);
        case 1: return core_launch_f16(out_f32, mode, p, st);
        case 2: return core_launch_bf16(out_f32, mode, p, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t merge_launch(int out_dtype, bool plain, const MergeParams& p, cudaStream_t st) {
    switch (out_dtype) {
        case 0: return merge_launch_f32(plain, p, st);
        case 1: return merge_launch_f16(plain, p, st);
        case 2: return merge_launch_bf16(plain, p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace g3s
