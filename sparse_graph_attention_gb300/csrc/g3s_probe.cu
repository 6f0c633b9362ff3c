// Gather-rate probe: how fast random rows of a given size can be read from an
// array that fits in L2 (or one that does not).  A measurement aid for the
// roofline of the CUDA-core kernel on graphs whose K and V stay in L2, where
// the HBM copy rate is not the bound.  No counterpart on the pages.
//
// The j-th row read is row (j + 1) * 0x9E3779B97F4A7C15 >> (64 - log2 rows)
// (multiplicative hashing: spread uniformly over a power-of-two row count), so
// no index array stands between the loads.  Each warp of a persistent grid
// reads, per step, eight warp loads of 512 bytes of whole rows (four 128-byte
// rows, two 256-byte ones, one 512-byte row, or 512-byte slices of wider
// rows), all in flight before any is consumed; the pieces are XOR-ed together
// and one word per warp is written, so nothing is optimised away.
#include "g3s_internal.h"

namespace g3s {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kInFlight = 8;

__device__ __forceinline__ unsigned long long probe_row(unsigned long long j, int lg_rows) {
    return ((j + 1ull) * 0x9E3779B97F4A7C15ull) >> (64 - lg_rows);
}

template <bool kPlain>
__global__ void __launch_bounds__(kProbeThreads) gather_probe_kernel(const uint4* src, int lg_rows, int row_vecs,
                                                                     long long gathers, uint32_t* sink) {
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * kProbeThreads + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * kProbeThreads) >> 5;
    // a warp load covers 32 pieces: rows_per_load rows of row_vecs pieces, or
    // one row's 32-piece slice when a row is wider than 512 bytes
    const int rows_per_load = row_vecs >= 32 ? 1 : 32 / row_vecs;
    const int slices = row_vecs >= 32 ? row_vecs / 32 : 1;
    const int my_row = row_vecs >= 32 ? 0 : lane / row_vecs;
    const int my_vec = row_vecs >= 32 ? lane : lane % row_vecs;
    uint4 acc = make_uint4(0u, 0u, 0u, 0u);
    const long long rows_per_step = (long long)kInFlight * rows_per_load / slices;
    const long long steps = (gathers + rows_per_step * nwarps - 1) / (rows_per_step * nwarps);
    for (long long st = 0; st < steps; ++st) {
        const unsigned long long base = (unsigned long long)((st * nwarps + warp) * rows_per_step);
        uint4 v[kInFlight];
#pragma unroll
        for (int k = 0; k < kInFlight; ++k) {
            const int r_in_step = row_vecs >= 32 ? (k / slices) : k * rows_per_load + my_row;
            const int slice = row_vecs >= 32 ? k % slices : 0;
            const unsigned long long r = probe_row(base + (unsigned)r_in_step, lg_rows);
            const uint4* q = src + r * (unsigned)row_vecs + slice * 32 + my_vec;
            v[k] = kPlain ? *q : __ldg(q);
        }
#pragma unroll
        for (int k = 0; k < kInFlight; ++k) {
            acc.x ^= v[k].x;
            acc.y ^= v[k].y;
            acc.z ^= v[k].z;
            acc.w ^= v[k].w;
        }
    }
    uint32_t a = acc.x ^ acc.y ^ acc.z ^ acc.w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a ^= __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == 0) sink[warp] = a;
}

// rows one probe launch reads (whole warp steps)
long long probe_rows(long long gathers, int row_vecs, int ctas) {
    const long long nwarps = (long long)ctas * (kProbeThreads / 32);
    const int rows_per_load = row_vecs >= 32 ? 1 : 32 / row_vecs;
    const int slices = row_vecs >= 32 ? row_vecs / 32 : 1;
    const long long rows_per_step = (long long)kInFlight * rows_per_load / slices;
    const long long steps = (gathers + rows_per_step * nwarps - 1) / (rows_per_step * nwarps);
    return steps * nwarps * rows_per_step;
}

}  // namespace
}  // namespace g3s

using namespace g3s;
using namespace g3s::api;

extern "C" g3s_status g3s_gather_probe(const void* src, int64_t rows, int row_bytes, int64_t gathers, int ctas,
                                       int plain_loads, uint32_t* sink, int64_t* rows_read, g3s_stream_t stream) {
    if (!src || !sink) return fail(G3S_ERR_INVALID_ARG, "src and sink must be non-NULL");
    if (rows < 2 || (rows & (rows - 1)) || rows > (1ll << 40))
        return fail(G3S_ERR_INVALID_ARG, "rows must be a power of two in [2, 2^40]");
    if (gathers < 1 || ctas < 1 || ctas > 65535)
        return fail(G3S_ERR_INVALID_ARG, "gathers >= 1 and 1 <= ctas <= 65535 required");
    if (row_bytes < 16 || row_bytes > 4096 || (row_bytes & (row_bytes - 1)))
        return fail(G3S_ERR_INVALID_ARG, "row_bytes must be a power of two in [16, 4096]");
    if (!aligned16(src) || (reinterpret_cast<uintptr_t>(sink) & 3u))
        return fail(G3S_ERR_INVALID_ARG, "src must be 16-byte aligned, sink 4-byte aligned");
    int lg = 0;
    while ((1ll << lg) < rows) ++lg;
    if (rows_read) *rows_read = probe_rows(gathers, row_bytes / 16, ctas);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (plain_loads)
        gather_probe_kernel<true><<<ctas, kProbeThreads, 0, st>>>(static_cast<const uint4*>(src), lg, row_bytes / 16,
                                                                  gathers, sink);
    else
        gather_probe_kernel<false><<<ctas, kProbeThreads, 0, st>>>(static_cast<const uint4*>(src), lg, row_bytes / 16,
                                                                   gathers, sink);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? G3S_OK : cuda_fail(e, "gather probe launch");
}
