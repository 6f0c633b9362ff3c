// Dispatch of the fused CUDA-core kernel and the heavy-row merge by input and
// output element type (the kernels themselves are in g3s_core.cuh), and the
// tensor-map encoder the projection GEMM's TMA copies use.
#include <mutex>

#include "g3s_internal.h"

namespace g3s {

namespace {

// cuTensorMapEncodeTiled, looked up once through the runtime (the library does
// not link the driver API).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

}  // namespace

bool tensor_maps_available() { return tensor_map_encoder() != nullptr; }

bool encode_tile(CUtensorMap* m, const void* base, long long rows, int row_elems, int elem_bytes, int box_rows,
                 int box_elems) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (enc == nullptr || rows < 1 || (elem_bytes != 2 && elem_bytes != 4)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_elems * elem_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_elems, (cuuint32_t)box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    return enc(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32, 2,
               const_cast<void*>(base), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool core_supported(int dtype, int row_vecs) {
    if (dtype < 0 || dtype > 2) return false;
    if (row_vecs < 1 || row_vecs > 256 || (row_vecs & (row_vecs - 1))) return false;
    return true;
}

cudaError_t core_launch(int dtype, int out_dtype, int mode, const CoreParams& p, cudaStream_t st) {
    const bool out_f32 = out_dtype == 0;
    if (!out_f32 && out_dtype != dtype) return cudaErrorInvalidValue;
    if (p.pack_rows && mode != 1 && p.row_vecs <= 16) {  // the short-row pack flavour
        switch (dtype) {
            case 0: return core_launch_pack_f32(true, mode, p, st);
            case 1: return core_launch_pack_f16(out_f32, mode, p, st);
            case 2: return core_launch_pack_bf16(out_f32, mode, p, st);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (dtype) {
        case 0: return core_launch_f32(true, mode, p, st);
        case 1: return core_launch_f16(out_f32, mode, p, st);
        case 2: return core_launch_bf16(out_f32, mode, p, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t core_small_launch(int dtype, int out_dtype, int mode, const CoreParams& p, cudaStream_t st) {
    const bool out_f32 = out_dtype == 0;
    if (!out_f32 && out_dtype != dtype) return cudaErrorInvalidValue;
    switch (dtype) {
        case 0: return core_small_launch_f32(true, mode, p, st);
        case 1: return core_small_launch_f16(out_f32, mode, p, st);
        case 2: return core_small_launch_bf16(out_f32, mode, p, st);
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
