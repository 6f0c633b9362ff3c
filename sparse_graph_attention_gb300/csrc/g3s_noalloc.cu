// g3s_forward_noalloc: the fused forward pass for callers that cannot
// allocate device memory.
//
// Who needs it: code whose device memory is fixed before it runs -- an
// inference engine that hands out memory only when it is built, a process
// whose GPU memory is already reserved by another framework's caching
// allocator, a service with a hard memory budget -- cannot call cudaMalloc
// to get the planner workspace that g3s_plan_create expects, and cudaMalloc
// may also synchronise the device at a bad moment.  This entry point takes
// only inputs and outputs.  Its scratch (the planner arrays and the heavy-row
// partial results) lives in one file-scope device array of
// G3S_NOALLOC_SCRATCH_BYTES that every GPU loading this library keeps until
// the process exits.
//
// The work is the same as g3s_plan_create (without BSB tiles) followed by
// g3s_forward with the default options: the same planner kernels and the
// same fused and merge kernels, pointed at the static array instead of a
// caller workspace.  No cudaMalloc, cudaFree or other allocating call, on
// the device or the host, is made.
#include <mutex>

#include "g3s_internal.h"

using namespace g3s;
using namespace g3s::api;

static_assert(G3S_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// The scratch.  In host code this name is only a stand-in for the device
// symbol: its device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g3s_noalloc_scratch[G3S_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices];  // device address of the scratch on each device, once set up

// Device address of the scratch on the current device (set up on first use).
g3s_status scratch_on_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(G3S_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g3s_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g3s_noalloc_scratch)");
        if (p == nullptr || (reinterpret_cast<uintptr_t>(p) % kAlign) != 0)
            return fail(G3S_ERR_CUDA, "scratch symbol has no usable device address");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return G3S_OK;
}

#define NOALLOC_CUDA(x, where)                               \
    do {                                                     \
        cudaError_t e_ = (x);                                \
        if (e_ != cudaSuccess) return cuda_fail(e_, where);  \
    } while (0)

}  // namespace

extern "C" g3s_status g3s_forward_noalloc(const int32_t* row_ptr_d, const int32_t* col_idx_d, int64_t num_nodes,
                                          int64_t num_edges, int heads, int head_dim, g3s_dtype dtype,
                                          g3s_variant variant, const void* Q, const void* K, const void* V,
                                          const void* Eproj, void* O, void* Eout, g3s_stream_t stream_) {
    g3s_plan_options o;
    default_options(&o);
    o.bsb = 0;
    o.tile_path = 0;
    PlanShape s{};
    g3s_status st = check_shape(num_nodes, num_edges, heads, head_dim, dtype, variant, o, &s);
    if (st != G3S_OK) return st;
    PlanArrays a{};
    const size_t need = carve(s, &a, nullptr);
    if (need > (size_t)G3S_NOALLOC_SCRATCH_BYTES)
        return fail(G3S_ERR_WORKSPACE,
                    "graph needs %zu bytes of scratch but the static scratch holds %zu; use g3s_plan_create "
                    "with a caller workspace instead",
                    need, (size_t)G3S_NOALLOC_SCRATCH_BYTES);
    const bool rtm = variant == G3S_RTMSCORE;
    if (!row_ptr_d) return fail(G3S_ERR_INVALID_ARG, "row_ptr is NULL");
    if (num_edges > 0 && !col_idx_d) return fail(G3S_ERR_INVALID_ARG, "col_idx is NULL with E > 0");
    if ((reinterpret_cast<uintptr_t>(row_ptr_d) & 3u) || (reinterpret_cast<uintptr_t>(col_idx_d) & 3u))
        return fail(G3S_ERR_INVALID_ARG, "row_ptr / col_idx must be 4-byte aligned");
    if (num_nodes > 0 && (!Q || !K || !V || !O)) return fail(G3S_ERR_INVALID_ARG, "Q, K, V and O must be non-NULL");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(Eproj) || !aligned16(Eout))
        return fail(G3S_ERR_INVALID_ARG, "value pointers must be 16-byte aligned");
    if (rtm) {
        if (num_edges > 0 && !Eproj) return fail(G3S_ERR_INVALID_ARG, "RTMScore needs Eproj");
    } else if (Eproj || Eout) {
        return fail(G3S_ERR_INVALID_ARG, "Eproj / Eout are only valid for the RTMScore variant");
    }

    void* base = nullptr;
    st = scratch_on_current_device(&base);
    if (st != G3S_OK) return st;
    carve(s, &a, base);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

    // the planner (counters start at zero; every other array is fully written before it is read)
    PlanCounts hc;
    NOALLOC_CUDA(cudaMemsetAsync(a.counts, 0, sizeof(PlanCounts), stream), "cudaMemsetAsync(counts)");
    NOALLOC_CUDA(cudaMemsetAsync(a.fwd_status, 0, sizeof(int32_t), stream), "cudaMemsetAsync(status)");
    NOALLOC_CUDA(plan_validate(row_ptr_d, col_idx_d, s, a, stream), "CSR validation launch");
    NOALLOC_CUDA(cudaMemcpyAsync(&hc, a.counts, sizeof hc, cudaMemcpyDeviceToHost, stream), "cudaMemcpyAsync(counts)");
    NOALLOC_CUDA(cudaStreamSynchronize(stream), "cudaStreamSynchronize(validation)");
    if (hc.status) return fail(G3S_ERR_BAD_GRAPH, "CSR validation failed (error bits 0x%x)", (unsigned)hc.status);
    NOALLOC_CUDA(plan_build(row_ptr_d, col_idx_d, s, a, stream), "planner launch");
    NOALLOC_CUDA(cudaMemcpyAsync(&hc, a.counts, sizeof hc, cudaMemcpyDeviceToHost, stream), "cudaMemcpyAsync(counts)");
    NOALLOC_CUDA(cudaStreamSynchronize(stream), "cudaStreamSynchronize(planner)");
    if (s.N == 0) return G3S_OK;

    // the fused forward, heavy-row partials in the static scratch
    const int esz = dtype_size(dtype);
    CoreParams cp{};
    cp.W = nullptr;
    cp.normalize = 0;
    cp.edge_id = nullptr;  // E / Eout by CSR position
    cp.row_ptr = row_ptr_d;
    cp.col_idx = col_idx_d;
    cp.Q = Q;
    cp.K = K;
    cp.V = V;
    cp.E = Eproj;
    cp.O = O;
    cp.Eout = rtm ? Eout : nullptr;
    cp.chunks = a.chunks;
    cp.part_acc = a.part_acc;
    cp.part_ml = a.part_ml;
    cp.win_flags = nullptr;
    cp.work_counter = a.work_counter;
    cp.N = s.N;
    cp.n_chunks = hc.n_chunks;
    cp.H = s.H;
    cp.D = s.D;
    cp.heavy_threshold = s.heavy_threshold;
    cp.row_vecs = s.H * s.D * esz / 16;
    cp.lph = s.D * esz / 16;
    const float inv_sqrt_d = 1.0f / sqrtf((float)s.D);
    cp.qscale = rtm ? inv_sqrt_d : inv_sqrt_d * 1.4426950408889634f;
    cp.eps = o.rtm_epsilon;
    cp.elementwise_clamp = o.rtm_elementwise_clamp ? 1 : 0;
    cp.status = a.fwd_status;
    cp.pack_rows = use_packs(o.pack_rows, s, hc) ? 1 : 0;
    if (s.N <= s.small_rows) {  // as g3s_forward: one launch, a CTA per row
        NOALLOC_CUDA(core_small_launch(dtype, o.out_dtype, rtm, cp, stream), "small-graph kernel launch");
        return G3S_OK;
    }
    NOALLOC_CUDA(core_launch(dtype, o.out_dtype, rtm, cp, stream), "fused kernel launch");
    if (hc.n_chunks > 0) {
        MergeParams mp{};
        mp.heavy_rows = a.heavy_rows;
        mp.heavy_chunk_ptr = a.heavy_chunk_ptr;
        mp.part_acc = a.part_acc;
        mp.part_ml = a.part_ml;
        mp.O = O;
        mp.n_heavy = hc.n_heavy;
        mp.H = s.H;
        mp.D = s.D;
        mp.eps = o.rtm_epsilon;
        mp.normalize = 1;
        NOALLOC_CUDA(merge_launch(o.out_dtype, rtm, mp, stream), "merge kernel launch");
    }
    return G3S_OK;
}
