// C ABI of libg3s: argument checks, workspace layout, plan lifetime and the
// forward orchestration.  All compute runs in the kernels of g3s_core.cu,
// g3s_planner.cu (and the tile kernel); this file only validates and launches.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <new>
#include <string>

#include "g3s_internal.h"

using namespace g3s;

namespace {
thread_local std::string t_last_error;
}  // namespace

namespace g3s {
namespace api {

g3s_status fail(g3s_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

g3s_status cuda_fail(cudaError_t e, const char* where) {
    return fail(G3S_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define CUDA_OR_FAIL(x, where)                                     \
    do {                                                           \
        cudaError_t e_ = (x);                                      \
        if (e_ != cudaSuccess) return cuda_fail(e_, where);        \
    } while (0)

int dtype_size(int dt) { return dt == G3S_F32 ? 4 : 2; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Carver {
    char* base;
    size_t off = 0;
    template <class T>
    T* take(long long count) {
        off = (off + kAlign - 1) & ~(kAlign - 1);
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += (size_t)(count > 0 ? count : 0) * sizeof(T);
        return p;
    }
};

void default_options(g3s_plan_options* o) {
    memset(o, 0, sizeof *o);
    o->bucket_bounds[0] = 32;
    o->bucket_bounds[1] = 256;
    o->bucket_bounds[2] = 2048;
    o->heavy_threshold = 0;  // automatic: 10 x mean degree in [64, 512]
    o->chunk_edges = 0;  // automatic: 512 entries of rows up to 256 bytes, fewer for wider rows
    o->bsb = -1;
    o->tile_path = -1;
    o->tile_density_milli = 100;
    o->tile_pool_density_milli = 180;
    o->tile_max_tiles = 16;
    o->bsb_smem_edges = 2048;
    o->rtm_elementwise_clamp = 1;
    o->rtm_epsilon = 1e-6f;
    o->validate_graph = 1;
    o->out_dtype = G3S_F32;
    o->pack_rows = -1;
    o->degree_buckets = 0;
    o->small_graph_rows = kSmallGraphRows;
    o->tile_split_density_milli = 150;
    o->tile_split_parallel = 0;
}

bool tile_path_compiled(int dtype, int variant, int head_dim) { return tile_supported(dtype, variant, head_dim); }

g3s_status check_shape(int64_t N, int64_t E, int heads, int head_dim, int dtype, int variant,
                       const g3s_plan_options& o, PlanShape* s) {
    if (N < 0 || E < 0) return fail(G3S_ERR_INVALID_ARG, "negative size (N=%lld, E=%lld)", (long long)N, (long long)E);
    if (N > 0x7fffffffLL - 64) return fail(G3S_ERR_INVALID_ARG, "N=%lld does not fit int32 indices", (long long)N);
    if (E > 0x7fffffffLL) return fail(G3S_ERR_INVALID_ARG, "E=%lld does not fit int32 CSR offsets", (long long)E);
    if (dtype < G3S_F32 || dtype > G3S_BF16) return fail(G3S_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (variant != G3S_STANDARD && variant != G3S_RTMSCORE) return fail(G3S_ERR_INVALID_ARG, "unknown variant %d", variant);
    if (heads < 1) return fail(G3S_ERR_INVALID_ARG, "heads must be >= 1 (got %d)", heads);
    if (head_dim != 16 && head_dim != 32 && head_dim != 64 && head_dim != 128)
        return fail(G3S_ERR_UNSUPPORTED, "head_dim %d not in {16, 32, 64, 128}", head_dim);
    const long long row_bytes = (long long)heads * head_dim * dtype_size(dtype);
    const long long row_vecs = row_bytes / 16;
    if (!core_supported(dtype, (int)(row_vecs > 4096 ? 4096 : row_vecs)))
        return fail(G3S_ERR_UNSUPPORTED, "H*d*sizeof(dtype) = %lld bytes is not a power of two in [16, 4096]", row_bytes);
    for (int k = 0; k < G3S_NUM_BUCKETS - 2; ++k) {
        if (o.bucket_bounds[k] < 1 || (k > 0 && o.bucket_bounds[k] <= o.bucket_bounds[k - 1]))
            return fail(G3S_ERR_INVALID_ARG, "bucket_bounds must be positive and increasing");
    }
    if (o.heavy_threshold < 0) return fail(G3S_ERR_INVALID_ARG, "heavy_threshold must be >= 0 (0: automatic)");
    if (o.chunk_edges < 0) return fail(G3S_ERR_INVALID_ARG, "chunk_edges must be >= 0 (0: automatic)");
    if (o.bsb < -1 || o.bsb > 1 || o.tile_path < -1 || o.tile_path > 1)
        return fail(G3S_ERR_INVALID_ARG, "bsb and tile_path take -1, 0 or 1");
    if (o.tile_density_milli < 0 || o.tile_max_tiles < 1 || o.tile_pool_density_milli < 0)
        return fail(G3S_ERR_INVALID_ARG,
                    "tile_density_milli >= 0, tile_pool_density_milli >= 0 and tile_max_tiles >= 1 required");
    if (o.bsb_smem_edges < 1 || o.bsb_smem_edges > 16384)
        return fail(G3S_ERR_INVALID_ARG, "bsb_smem_edges must be in [1, 16384]");
    if (!(o.rtm_epsilon >= 0.f)) return fail(G3S_ERR_INVALID_ARG, "rtm_epsilon must be >= 0");
    if (o.out_dtype != G3S_F32 && o.out_dtype != dtype)
        return fail(G3S_ERR_INVALID_ARG, "out_dtype must be G3S_F32 or the input dtype");
    if (o.pack_rows < -1 || o.pack_rows > 1) return fail(G3S_ERR_INVALID_ARG, "pack_rows takes -1, 0 or 1");
    if (o.degree_buckets != 0 && o.degree_buckets != 1) return fail(G3S_ERR_INVALID_ARG, "degree_buckets takes 0 or 1");
    if (o.small_graph_rows < 0) return fail(G3S_ERR_INVALID_ARG, "small_graph_rows must be >= 0");
    if (o.tile_split_density_milli != 0 && (o.tile_split_density_milli < 100 || o.tile_split_density_milli > 1000))
        return fail(G3S_ERR_INVALID_ARG, "tile_split_density_milli takes 0 (off) or 100..1000");
    if (o.tile_split_parallel != 0 && o.tile_split_parallel != 1)
        return fail(G3S_ERR_INVALID_ARG, "tile_split_parallel takes 0 (node-parallel) or 1 (edge-parallel)");

    const bool tile_ok = tile_path_compiled(dtype, variant, head_dim);
    if (o.tile_path == 1 && !tile_ok)
        return fail(G3S_ERR_UNSUPPORTED, "tile path requested but not available for this dtype/variant/head_dim");
    s->N = N;
    s->E = E;
    s->H = heads;
    s->D = head_dim;
    // Heavy rows go to the front of the work queue as chunks.  Automatic
    // threshold: rows over ten times the mean degree (a long row taken late
    // in id order would otherwise finish last), between 64 and 512.
    if (o.heavy_threshold > 0) {
        s->heavy_threshold = o.heavy_threshold;
    } else {
        const long long t = N > 0 ? (10 * E + N / 2) / N : 512;
        s->heavy_threshold = (int)(t < 64 ? 64 : (t > 512 ? 512 : t));
    }
    s->pack_limit = pack_limit_for((int)row_vecs, s->heavy_threshold);
    // Automatic chunk length: one warp walks a chunk an edge step at a time,
    // and a step gathers fewer edges the wider the node row (one edge per
    // step from 512-byte rows on), so chunks hold 512 x 256 / row bytes
    // entries, between 64 and 512: 512 up to 256-byte rows, 128 for 1 KB.
    if (o.chunk_edges > 0) {
        s->chunk_edges = o.chunk_edges;
    } else {
        const long long c = 512LL * 256 / (row_bytes > 256 ? row_bytes : 256);
        s->chunk_edges = (int)(c < 64 ? 64 : c);
    }
    for (int k = 0; k < G3S_NUM_BUCKETS - 2; ++k) s->bounds[k] = o.bucket_bounds[k];
    s->bsb_smem_edges = o.bsb_smem_edges;
    s->bucket_lists = o.degree_buckets == 1;
    s->small_rows = o.small_graph_rows;
    s->tile_density_milli = o.tile_density_milli;
    s->tile_pool_milli = o.tile_pool_density_milli;
    s->tile_max_tiles = o.tile_max_tiles;
    s->tile_split_milli = o.tile_split_density_milli;
    s->split_edge_parallel = o.tile_split_parallel == 1;
    // automatic: on where compiled, unless the caller turned the BSB tiles off
    s->tile_enabled = tile_ok && (o.tile_path == 1 || (o.tile_path == -1 && o.bsb != 0));
    if (s->tile_enabled && o.tile_max_tiles > kTileMaxTilesPerWindow)
        return fail(G3S_ERR_INVALID_ARG, "tile_max_tiles must be <= %d with the tile path on", kTileMaxTilesPerWindow);
    s->build_bsb = o.bsb == 1 || (o.bsb == -1 && s->tile_enabled);
    if (s->tile_enabled && !s->build_bsb)
        return fail(G3S_ERR_INVALID_ARG, "the tile path needs the BSB tiles (bsb = 0 with tile_path on)");
    const long long T = s->heavy_threshold;
    s->max_heavy = N < E / (T + 1) ? N : E / (T + 1);
    s->max_chunks = E / s->chunk_edges + s->max_heavy;
    s->W = (N + kWinRows - 1) / kWinRows;
    s->max_tiles = s->build_bsb ? (E + 7 * s->W) / kTileCols : 0;
    // A split window of T > 16 tiles has S = ceil(T / 16) slices, 16 S < 2 T
    // partial rows, and T <= 1000 nnz / (128 split_milli) tiles.
    if (s->tile_enabled && s->tile_split_milli > 0) {
        const long long rows = 2000LL * E / (128LL * s->tile_split_milli) + 16;
        s->max_split_items = rows / 16 + 1;
        s->max_split_rows = s->split_edge_parallel ? rows : 0;  // partial states: edge-parallel only
    } else {
        s->tile_split_milli = 0;
        s->max_split_rows = s->max_split_items = 0;
    }
    s->bitmap_words = s->build_bsb ? (N + 31) / 32 : 0;
    const long long scan_n = N > s->W ? N : s->W;
    s->scan_blocks = (scan_n + 1023) / 1024 + 2;
    return G3S_OK;
}

size_t carve(const PlanShape& s, PlanArrays* a, void* base) {
    Carver c{static_cast<char*>(base)};
    a->counts = c.take<PlanCounts>(1);
    a->work_counter = c.take<unsigned long long>(1);
    a->tile_counter = c.take<unsigned int>(1);
    a->fwd_status = c.take<int32_t>(1);
    a->bucket_of = s.bucket_lists ? c.take<uint8_t>(s.N) : nullptr;
    a->bucket_ptr = c.take<int32_t>(G3S_NUM_BUCKETS + 1);
    a->bucket_rows = s.bucket_lists ? c.take<int32_t>(s.N) : nullptr;
    a->heavy_rows = c.take<int32_t>(s.max_heavy);
    a->heavy_chunk_ptr = c.take<int32_t>(s.max_heavy + 1);
    a->heavy_index = c.take<int32_t>(s.N);
    a->chunks = c.take<int32_t>(3 * s.max_chunks);
    a->part_acc = c.take<float>((s.max_chunks + s.max_split_rows) * s.H * s.D);
    a->part_ml = c.take<float>((s.max_chunks + s.max_split_rows) * s.H * 2);
    a->scan_blocks = c.take<int32_t>(s.scan_blocks);
    if (s.build_bsb) {
        a->win_tile_ptr = c.take<int32_t>(s.W + 1);
        a->win_ucount = c.take<int32_t>(s.W);
        a->win_nnz = c.take<int32_t>(s.W);
        a->win_flags = c.take<uint8_t>(s.W);
        a->tile_windows = c.take<int32_t>(s.W);
        a->tile_items = c.take<int4>(2 * (s.W + s.max_split_items));
        a->tile_sorted = c.take<int32_t>(s.W);
        a->tile_runs = c.take<int4>(32);
        a->core_windows = c.take<int32_t>(s.W);
        a->large_windows = c.take<int32_t>(s.W);
        a->tile_cols = c.take<int32_t>(s.max_tiles * kTileCols);
        a->tile_bits = c.take<uint32_t>(s.max_tiles * 4);
        a->bitmap_scratch = c.take<uint32_t>((long long)kLargeCtas * 3 * s.bitmap_words);
        const bool split = s.max_split_items > 0;
        a->win_split_base = split ? c.take<int32_t>(s.W) : nullptr;
        a->merge_rows = split ? c.take<int32_t>(s.N) : nullptr;
        a->merge_range = split ? c.take<int2>(s.N) : nullptr;
        a->chains = split && !s.split_edge_parallel ? c.take<int2>(s.W) : nullptr;
    } else {
        a->win_split_base = a->merge_rows = a->tile_sorted = nullptr;
        a->merge_range = a->chains = nullptr;
        a->tile_runs = nullptr;
        a->win_tile_ptr = a->win_ucount = a->win_nnz = a->tile_windows = a->large_windows = a->tile_cols = nullptr;
        a->core_windows = nullptr;
        a->tile_items = nullptr;
        a->win_flags = nullptr;
        a->tile_bits = a->bitmap_scratch = nullptr;
    }
    return (c.off + kAlign - 1) & ~(kAlign - 1);
}

}  // namespace api
}  // namespace g3s

using namespace g3s::api;

struct g3s_plan {
    PlanShape shape;
    PlanArrays arr;
    PlanCounts counts;  // host copy
    g3s_plan_options opts;
    int dtype, variant, device;
    const int32_t* row_ptr;
    const int32_t* col_idx;
    size_t ws_used;
    const int32_t* edge_id;  // optional CSR position -> physical edge slot
    long long edge_slots;    // rows of E / Eout / W (E without edge ids)
    // With tile windows, the CUDA-core kernel runs on this high-priority side
    // stream (forked from and joined back into the caller's stream with the
    // two events) while the tile kernel runs on the caller's; created with
    // the plan, destroyed with it.
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
};

extern "C" {

const char* g3s_version(void) { return "g3s 0.1 (sm_103a)"; }

const char* g3s_status_string(g3s_status s) {
    switch (s) {
        case G3S_OK: return "G3S_OK";
        case G3S_ERR_INVALID_ARG: return "G3S_ERR_INVALID_ARG";
        case G3S_ERR_UNSUPPORTED: return "G3S_ERR_UNSUPPORTED";
        case G3S_ERR_BAD_GRAPH: return "G3S_ERR_BAD_GRAPH";
        case G3S_ERR_WORKSPACE: return "G3S_ERR_WORKSPACE";
        case G3S_ERR_CUDA: return "G3S_ERR_CUDA";
        case G3S_ERR_TIMEOUT: return "G3S_ERR_TIMEOUT";
    }
    return "G3S_ERR_UNKNOWN";
}

const char* g3s_last_error(void) { return t_last_error.c_str(); }

void g3s_plan_options_init(g3s_plan_options* opts) {
    if (opts) default_options(opts);
}

g3s_status g3s_plan_workspace_size(int64_t num_nodes, int64_t num_edges, int heads, int head_dim, g3s_dtype dtype,
                                   g3s_variant variant, const g3s_plan_options* opts, size_t* bytes) {
    if (!bytes) return fail(G3S_ERR_INVALID_ARG, "bytes is NULL");
    g3s_plan_options o;
    if (opts)
        o = *opts;
    else
        default_options(&o);
    PlanShape s{};
    g3s_status st = check_shape(num_nodes, num_edges, heads, head_dim, dtype, variant, o, &s);
    if (st != G3S_OK) return st;
    PlanArrays a{};
    *bytes = carve(s, &a, nullptr);
    return G3S_OK;
}

g3s_status g3s_plan_create(const int32_t* row_ptr_d, const int32_t* col_idx_d, int64_t num_nodes, int64_t num_edges,
                           int heads, int head_dim, g3s_dtype dtype, g3s_variant variant,
                           const g3s_plan_options* opts, void* workspace_d, size_t workspace_bytes,
                           g3s_stream_t stream_, g3s_plan** out) {
    if (!out) return fail(G3S_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    g3s_plan_options o;
    if (opts)
        o = *opts;
    else
        default_options(&o);
    PlanShape s{};
    g3s_status st = check_shape(num_nodes, num_edges, heads, head_dim, dtype, variant, o, &s);
    if (st != G3S_OK) return st;
    if (!row_ptr_d) return fail(G3S_ERR_INVALID_ARG, "row_ptr is NULL");
    if (num_edges > 0 && !col_idx_d) return fail(G3S_ERR_INVALID_ARG, "col_idx is NULL with E > 0");
    if ((reinterpret_cast<uintptr_t>(row_ptr_d) & 3u) || (reinterpret_cast<uintptr_t>(col_idx_d) & 3u))
        return fail(G3S_ERR_INVALID_ARG, "row_ptr / col_idx must be 4-byte aligned");
    PlanArrays a{};
    const size_t need = carve(s, &a, nullptr);
    if (!workspace_d) return fail(G3S_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
    if (reinterpret_cast<uintptr_t>(workspace_d) % kAlign)
        return fail(G3S_ERR_WORKSPACE, "workspace must be %zu-byte aligned", kAlign);
    if (workspace_bytes < need)
        return fail(G3S_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
    carve(s, &a, workspace_d);

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    CUDA_OR_FAIL(cudaGetDevice(&dev), "cudaGetDevice");
    PlanCounts hc;
    CUDA_OR_FAIL(cudaMemsetAsync(a.counts, 0, sizeof(PlanCounts), stream), "cudaMemsetAsync(counts)");
    CUDA_OR_FAIL(cudaMemsetAsync(a.fwd_status, 0, sizeof(int32_t), stream), "cudaMemsetAsync(status)");
    if (s.build_bsb && s.bitmap_words > 0)
        CUDA_OR_FAIL(cudaMemsetAsync(a.bitmap_scratch, 0, (size_t)kLargeCtas * 3 * s.bitmap_words * sizeof(uint32_t), stream),
                     "cudaMemsetAsync(bitmaps)");
    if (o.validate_graph) {
        CUDA_OR_FAIL(plan_validate(row_ptr_d, col_idx_d, s, a, stream), "CSR validation launch");
        CUDA_OR_FAIL(cudaMemcpyAsync(&hc, a.counts, sizeof hc, cudaMemcpyDeviceToHost, stream), "cudaMemcpyAsync(counts)");
        CUDA_OR_FAIL(cudaStreamSynchronize(stream), "cudaStreamSynchronize(validation)");
        if (hc.status) {
            return fail(G3S_ERR_BAD_GRAPH, "CSR validation failed:%s%s%s%s",
                        (hc.status & kErrRowPtr0) ? " row_ptr[0] != 0;" : "",
                        (hc.status & kErrRowPtrOrder) ? " row_ptr decreases;" : "",
                        (hc.status & kErrRowPtrEnd) ? " row_ptr[N] != E;" : "",
                        (hc.status & kErrColRange) ? " a source index is outside [0, N);" : "");
        }
    }
    CUDA_OR_FAIL(plan_build(row_ptr_d, col_idx_d, s, a, stream), "planner launch");
    CUDA_OR_FAIL(cudaMemcpyAsync(&hc, a.counts, sizeof hc, cudaMemcpyDeviceToHost, stream), "cudaMemcpyAsync(counts)");
    CUDA_OR_FAIL(cudaStreamSynchronize(stream), "cudaStreamSynchronize(planner)");

    g3s_plan* p = new (std::nothrow) g3s_plan;
    if (!p) return fail(G3S_ERR_INVALID_ARG, "out of host memory for the plan struct");
    p->shape = s;
    p->arr = a;
    p->counts = hc;
    p->opts = o;
    p->dtype = dtype;
    p->variant = variant;
    p->device = dev;
    p->row_ptr = row_ptr_d;
    p->col_idx = col_idx_d;
    p->ws_used = need;
    p->edge_id = nullptr;
    p->edge_slots = num_edges;
    if (any_tile(hc)) {
        // the CUDA-core kernel runs here, at the highest priority, so its few
        // CTAs are placed before the tile kernel's waves take every SM
        int least = 0, greatest = 0;
        cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&p->side, cudaStreamNonBlocking, greatest);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            g3s_plan_destroy(p);
            return cuda_fail(e, "side stream / events of the tile path");
        }
    }
    *out = p;
    return G3S_OK;
}

g3s_status g3s_plan_get_stats(const g3s_plan* p, g3s_plan_stats* st) {
    if (!p || !st) return fail(G3S_ERR_INVALID_ARG, "NULL plan or stats");
    memset(st, 0, sizeof *st);
    st->num_nodes = p->shape.N;
    st->num_edges = p->shape.E;
    st->heads = p->shape.H;
    st->head_dim = p->shape.D;
    st->dtype = p->dtype;
    st->variant = p->variant;
    st->out_dtype = p->opts.out_dtype;
    for (int b = 0; b < G3S_NUM_BUCKETS; ++b) st->bucket_count[b] = p->counts.bucket_count[b];
    st->heavy_rows = p->counts.n_heavy;
    st->chunks = p->counts.n_chunks;
    st->has_bsb = p->shape.build_bsb ? 1 : 0;
    st->tile_path = p->shape.tile_enabled ? 1 : 0;
    st->windows = p->shape.build_bsb ? p->shape.W : 0;
    st->tiles = p->counts.n_tiles;
    st->tile_windows = p->counts.n_tile_windows + p->counts.n_split_windows;
    st->dup_windows = p->counts.n_dup_windows;
    st->large_windows = p->counts.n_large_windows;
    st->tile_window_nnz = p->counts.tile_window_nnz + p->counts.split_nnz;
    st->pack_rows = use_packs(p->opts.pack_rows, p->shape, p->counts) ? 1 : 0;
    st->pack_limit = p->shape.pack_limit;
    st->heavy_threshold = p->shape.heavy_threshold;
    st->chunk_edges = p->shape.chunk_edges;
    st->short_rows = p->counts.n_short;
    st->workspace_used = p->ws_used;
    st->tile_items = p->counts.n_tile_items + p->counts.n_split_items;
    st->small_graph = p->shape.N <= p->shape.small_rows && !any_tile(p->counts) ? 1 : 0;
    st->split_windows = p->counts.n_split_windows;
    st->split_items = p->counts.n_split_items;
    st->merge_rows = p->counts.n_split_windows > 0 ? p->counts.n_merge : p->counts.n_heavy;
    return G3S_OK;
}

g3s_status g3s_plan_export(const g3s_plan* p, g3s_plan_array which, void* host_dst, size_t bytes, size_t* bytes_needed) {
    if (!p) return fail(G3S_ERR_INVALID_ARG, "NULL plan");
    const void* src = nullptr;
    size_t n = 0;
    const PlanShape& s = p->shape;
    const PlanCounts& c = p->counts;
    const bool bsb_arr = which >= G3S_ARR_WIN_TILE_PTR;
    if (bsb_arr && !s.build_bsb) return fail(G3S_ERR_UNSUPPORTED, "plan was built without BSB tiles");
    switch (which) {
        case G3S_ARR_BUCKET_PTR: src = p->arr.bucket_ptr; n = 4 * (G3S_NUM_BUCKETS + 1); break;
        case G3S_ARR_BUCKET_ROWS:
            if (!s.bucket_lists) return fail(G3S_ERR_UNSUPPORTED, "plan was built without the bucket row lists");
            src = p->arr.bucket_rows;
            n = 4 * (size_t)s.N;
            break;
        case G3S_ARR_HEAVY_ROWS: src = p->arr.heavy_rows; n = 4 * (size_t)c.n_heavy; break;
        case G3S_ARR_HEAVY_CHUNK_PTR: src = p->arr.heavy_chunk_ptr; n = 4 * ((size_t)c.n_heavy + 1); break;
        case G3S_ARR_CHUNKS: src = p->arr.chunks; n = 12 * (size_t)c.n_chunks; break;
        case G3S_ARR_WIN_TILE_PTR: src = p->arr.win_tile_ptr; n = 4 * ((size_t)s.W + 1); break;
        case G3S_ARR_TILE_COLS: src = p->arr.tile_cols; n = 4 * kTileCols * (size_t)c.n_tiles; break;
        case G3S_ARR_TILE_BITS: src = p->arr.tile_bits; n = 16 * (size_t)c.n_tiles; break;
        case G3S_ARR_WIN_NNZ: src = p->arr.win_nnz; n = 4 * (size_t)s.W; break;
        case G3S_ARR_WIN_FLAGS: src = p->arr.win_flags; n = (size_t)s.W; break;
        case G3S_ARR_TILE_WINDOWS: src = p->arr.tile_windows; n = 4 * (size_t)c.n_tile_windows; break;
        case G3S_ARR_CORE_WINDOWS:
            src = p->arr.core_windows;
            n = 4 * (size_t)(s.W - c.n_tile_windows - c.n_split_windows);
            break;
        case G3S_ARR_TILE_ITEMS:
            if (!s.tile_enabled) return fail(G3S_ERR_UNSUPPORTED, "plan was built without the tile path");
            src = p->arr.tile_items;
            n = 32 * (size_t)(c.n_tile_items + c.n_split_items);
            break;
        case G3S_ARR_MERGE_ROWS:
        case G3S_ARR_MERGE_RANGES:
            if (s.max_split_items == 0)
                return fail(G3S_ERR_UNSUPPORTED, "plan was built without split windows (tile path or option off)");
            src = which == G3S_ARR_MERGE_ROWS ? (const void*)p->arr.merge_rows : (const void*)p->arr.merge_range;
            n = (which == G3S_ARR_MERGE_ROWS ? 4 : 8) * (size_t)(c.n_split_windows > 0 ? c.n_merge : 0);
            break;
        default: return fail(G3S_ERR_INVALID_ARG, "unknown plan array %d", (int)which);
    }
    if (bytes_needed) *bytes_needed = n;
    if (!host_dst) return G3S_OK;
    if (bytes < n) return fail(G3S_ERR_INVALID_ARG, "destination has %zu bytes, %zu needed", bytes, n);
    if (n == 0) return G3S_OK;
    CUDA_OR_FAIL(cudaDeviceSynchronize(), "cudaDeviceSynchronize(export)");
    CUDA_OR_FAIL(cudaMemcpy(host_dst, src, n, cudaMemcpyDeviceToHost), "cudaMemcpy(export)");
    return G3S_OK;
}

g3s_status g3s_forward(const g3s_plan* p, const void* Q, const void* K, const void* V, const void* Eproj, void* O,
                       void* Eout, g3s_stream_t stream_) {
    if (!p) return fail(G3S_ERR_INVALID_ARG, "NULL plan");
    const PlanShape& s = p->shape;
    const bool rtm = p->variant == G3S_RTMSCORE;
    if (s.N > 0 && (!Q || !K || !V || !O)) return fail(G3S_ERR_INVALID_ARG, "Q, K, V and O must be non-NULL");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(Eproj) || !aligned16(Eout))
        return fail(G3S_ERR_INVALID_ARG, "value pointers must be 16-byte aligned");
    if (rtm) {
        if (s.E > 0 && !Eproj) return fail(G3S_ERR_INVALID_ARG, "RTMScore plan needs Eproj");
    } else if (Eproj || Eout) {
        return fail(G3S_ERR_INVALID_ARG, "Eproj / Eout are only valid for an RTMScore plan");
    }
    int dev = -1;
    CUDA_OR_FAIL(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev != p->device) return fail(G3S_ERR_INVALID_ARG, "plan was built on device %d, current is %d", p->device, dev);
    if (s.N == 0) return G3S_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

    const int esz = dtype_size(p->dtype);
    CoreParams cp{};
    cp.W = nullptr;
    cp.normalize = 0;
    cp.edge_id = p->edge_id;
    cp.row_ptr = p->row_ptr;
    cp.col_idx = p->col_idx;
    cp.Q = Q;
    cp.K = K;
    cp.V = V;
    cp.E = Eproj;
    cp.O = O;
    cp.Eout = rtm ? Eout : nullptr;
    cp.chunks = p->arr.chunks;
    cp.part_acc = p->arr.part_acc;
    cp.part_ml = p->arr.part_ml;
    const bool tiles = any_tile(p->counts);
    const bool split = p->counts.n_split_windows > 0;
    cp.win_flags = tiles ? p->arr.win_flags : nullptr;
    if (tiles) {
        cp.core_windows = p->arr.core_windows;
        cp.n_core_windows = s.W - p->counts.n_tile_windows - p->counts.n_split_windows;
    }
    cp.work_counter = p->arr.work_counter;
    cp.N = s.N;
    cp.n_chunks = p->counts.n_chunks;
    cp.H = s.H;
    cp.D = s.D;
    cp.heavy_threshold = s.heavy_threshold;
    cp.row_vecs = s.H * s.D * esz / 16;
    cp.lph = s.D * esz / 16;
    const float inv_sqrt_d = 1.0f / sqrtf((float)s.D);
    cp.qscale = rtm ? inv_sqrt_d : inv_sqrt_d * 1.4426950408889634f;
    cp.eps = p->opts.rtm_epsilon;
    cp.elementwise_clamp = p->opts.rtm_elementwise_clamp ? 1 : 0;
    cp.status = p->arr.fwd_status;
    cp.pack_rows = use_packs(p->opts.pack_rows, p->shape, p->counts) ? 1 : 0;
    if (s.N <= s.small_rows && !tiles) {  // one launch: a CTA per row
        CUDA_OR_FAIL(core_small_launch(p->dtype, p->opts.out_dtype, rtm, cp, stream), "small-graph kernel launch");
        return G3S_OK;
    }
    if (tiles) {
        TileParams tp{};
        tp.Q = Q;
        tp.K = K;
        tp.V = V;
        tp.O = O;
        tp.N = s.N;
        tp.H = s.H;
        tp.tile_items = p->arr.tile_items;
        tp.n_single_items = p->counts.n_tile_items + (s.split_edge_parallel ? p->counts.n_split_items : 0);
        tp.chains = p->arr.chains;
        tp.n_chains = s.split_edge_parallel ? 0 : p->counts.n_split_windows;
        tp.part_acc = p->arr.part_acc;
        tp.part_ml = p->arr.part_ml;
        tp.tile_cols = p->arr.tile_cols;
        tp.tile_bits = p->arr.tile_bits;
        tp.scale_log2 = inv_sqrt_d * 1.4426950408889634f;
        tp.status = p->arr.fwd_status;
        tp.work_counter = p->arr.tile_counter;
        // the CUDA-core kernel first, on the plan's high-priority side stream,
        // then the tile kernel on the caller's stream; the two overlap
        CUDA_OR_FAIL(cudaEventRecord(p->ev_fork, stream), "cudaEventRecord(fork)");
        CUDA_OR_FAIL(cudaStreamWaitEvent(p->side, p->ev_fork, 0), "cudaStreamWaitEvent(fork)");
        CUDA_OR_FAIL(core_launch(p->dtype, p->opts.out_dtype, rtm, cp, p->side),
                     "fused kernel launch");
        CUDA_OR_FAIL(cudaEventRecord(p->ev_join, p->side), "cudaEventRecord(join)");
        CUDA_OR_FAIL(cudaMemsetAsync(p->arr.tile_counter, 0, sizeof(unsigned int), stream), "cudaMemsetAsync(tile queue)");
        CUDA_OR_FAIL(tile_launch(p->dtype, p->opts.out_dtype, tp, stream), "tile kernel launch");
        CUDA_OR_FAIL(cudaStreamWaitEvent(stream, p->ev_join, 0), "cudaStreamWaitEvent(join)");
    } else {
        CUDA_OR_FAIL(core_launch(p->dtype, p->opts.out_dtype, rtm, cp, stream),
                     "fused kernel launch");
    }
    if (split ? p->counts.n_merge > 0 : p->counts.n_chunks > 0) {
        // with split windows the merge list holds the heavy rows outside them
        // (their chunks) and every row of a split window (its slices)
        MergeParams mp{};
        mp.heavy_rows = split ? p->arr.merge_rows : p->arr.heavy_rows;
        mp.heavy_chunk_ptr = p->arr.heavy_chunk_ptr;
        mp.ranges = split ? p->arr.merge_range : nullptr;
        mp.part_acc = p->arr.part_acc;
        mp.part_ml = p->arr.part_ml;
        mp.O = O;
        mp.n_heavy = split ? p->counts.n_merge : p->counts.n_heavy;
        mp.H = s.H;
        mp.D = s.D;
        mp.eps = p->opts.rtm_epsilon;
        mp.normalize = 1;
        CUDA_OR_FAIL(merge_launch(p->opts.out_dtype, rtm, mp, stream), "merge kernel launch");
    }
    return G3S_OK;
}

g3s_status g3s_aggregate(const g3s_plan* p, const void* W, const void* X, void* O, int normalize, float eps,
                         g3s_stream_t stream_) {
    if (!p) return fail(G3S_ERR_INVALID_ARG, "NULL plan");
    const PlanShape& s = p->shape;
    const int esz = dtype_size(p->dtype);
    if (s.N > 0 && (!X || !O)) return fail(G3S_ERR_INVALID_ARG, "X and O must be non-NULL");
    if (p->edge_slots > 0 && s.E > 0 && !W) return fail(G3S_ERR_INVALID_ARG, "W must be non-NULL when the graph has edges");
    if (!aligned16(X) || !aligned16(O) || (reinterpret_cast<uintptr_t>(W) % esz))
        return fail(G3S_ERR_INVALID_ARG, "X and O must be 16-byte aligned, W aligned to its element size");
    if (!(eps >= 0.f)) return fail(G3S_ERR_INVALID_ARG, "eps must be >= 0");
    int dev = -1;
    CUDA_OR_FAIL(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev != p->device) return fail(G3S_ERR_INVALID_ARG, "plan was built on device %d, current is %d", p->device, dev);
    if (s.N == 0) return G3S_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    CoreParams cp{};
    cp.row_ptr = p->row_ptr;
    cp.col_idx = p->col_idx;
    cp.Q = nullptr;
    cp.K = nullptr;
    cp.V = X;
    cp.E = nullptr;
    cp.W = W;
    cp.edge_id = p->edge_id;
    cp.O = O;
    cp.Eout = nullptr;
    cp.chunks = p->arr.chunks;
    cp.part_acc = p->arr.part_acc;
    cp.part_ml = p->arr.part_ml;
    cp.win_flags = nullptr;  // every row, including tile-path windows
    cp.work_counter = p->arr.work_counter;
    cp.N = s.N;
    cp.n_chunks = p->counts.n_chunks;
    cp.H = s.H;
    cp.D = s.D;
    cp.heavy_threshold = s.heavy_threshold;
    cp.row_vecs = s.H * s.D * esz / 16;
    cp.lph = s.D * esz / 16;
    cp.qscale = 0.f;
    cp.eps = eps;
    cp.elementwise_clamp = 0;
    cp.normalize = normalize ? 1 : 0;
    cp.status = p->arr.fwd_status;
    cp.pack_rows = use_packs(p->opts.pack_rows, p->shape, p->counts) ? 1 : 0;
    if (s.N <= s.small_rows) {  // one launch: a CTA per row
        CUDA_OR_FAIL(core_small_launch(p->dtype, p->opts.out_dtype, 2, cp, stream), "small-graph kernel launch");
        return G3S_OK;
    }
    CUDA_OR_FAIL(core_launch(p->dtype, p->opts.out_dtype, 2, cp, stream), "aggregation kernel launch");
    if (p->counts.n_chunks > 0) {
        MergeParams mp{};
        mp.heavy_rows = p->arr.heavy_rows;
        mp.heavy_chunk_ptr = p->arr.heavy_chunk_ptr;
        mp.part_acc = p->arr.part_acc;
        mp.part_ml = p->arr.part_ml;
        mp.O = O;
        mp.n_heavy = p->counts.n_heavy;
        mp.H = s.H;
        mp.D = s.D;
        mp.eps = eps;
        mp.normalize = normalize ? 1 : 0;
        CUDA_OR_FAIL(merge_launch(p->opts.out_dtype, true, mp, stream), "merge kernel launch");
    }
    return G3S_OK;
}

g3s_status g3s_host_staging_size(const g3s_plan* p, size_t* bytes) {
    if (!p || !bytes) return fail(G3S_ERR_INVALID_ARG, "NULL plan or bytes");
    const size_t hd = (size_t)p->shape.H * p->shape.D;
    const size_t node = (size_t)p->shape.N * hd * dtype_size(p->dtype);
    const size_t node_out = (size_t)p->shape.N * hd * dtype_size(p->opts.out_dtype);
    const size_t edge = (size_t)p->edge_slots * hd * dtype_size(p->dtype);
    const size_t edge_out = (size_t)p->edge_slots * hd * dtype_size(p->opts.out_dtype);
    auto up = [](size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); };
    size_t n = 3 * up(node) + up(node_out);
    if (p->variant == G3S_RTMSCORE) n += up(edge) + up(edge_out);
    *bytes = n;
    return G3S_OK;
}

g3s_status g3s_forward_host(const g3s_plan* p, const void* Qh, const void* Kh, const void* Vh, const void* Eh, void* Oh,
                            void* Eouth, void* staging, size_t staging_bytes, g3s_stream_t stream_) {
    if (!p) return fail(G3S_ERR_INVALID_ARG, "NULL plan");
    size_t need = 0;
    g3s_host_staging_size(p, &need);
    if (!staging || staging_bytes < need || reinterpret_cast<uintptr_t>(staging) % kAlign)
        return fail(G3S_ERR_WORKSPACE, "staging needs %zu bytes, %zu-byte aligned", need, kAlign);
    const bool rtm = p->variant == G3S_RTMSCORE;
    const size_t hd = (size_t)p->shape.H * p->shape.D;
    const size_t node = (size_t)p->shape.N * hd * dtype_size(p->dtype);
    const size_t node_out = (size_t)p->shape.N * hd * dtype_size(p->opts.out_dtype);
    const size_t edge = (size_t)p->edge_slots * hd * dtype_size(p->dtype);
    const size_t edge_out = (size_t)p->edge_slots * hd * dtype_size(p->opts.out_dtype);
    if (p->shape.N > 0 && (!Qh || !Kh || !Vh || !Oh)) return fail(G3S_ERR_INVALID_ARG, "host Q, K, V, O must be non-NULL");
    if (rtm && p->shape.E > 0 && !Eh) return fail(G3S_ERR_INVALID_ARG, "RTMScore plan needs host Eproj");
    if (!rtm && (Eh || Eouth)) return fail(G3S_ERR_INVALID_ARG, "Eproj / Eout are only valid for an RTMScore plan");
    auto up = [](size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); };
    char* b = static_cast<char*>(staging);
    void* dQ = b;
    void* dK = b + up(node);
    void* dV = b + 2 * up(node);
    void* dO = b + 3 * up(node);
    void* dE = rtm ? b + 3 * up(node) + up(node_out) : nullptr;
    void* dEo = rtm ? b + 3 * up(node) + up(node_out) + up(edge) : nullptr;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (node) {
        CUDA_OR_FAIL(cudaMemcpyAsync(dQ, Qh, node, cudaMemcpyHostToDevice, stream), "H2D Q");
        CUDA_OR_FAIL(cudaMemcpyAsync(dK, Kh, node, cudaMemcpyHostToDevice, stream), "H2D K");
        CUDA_OR_FAIL(cudaMemcpyAsync(dV, Vh, node, cudaMemcpyHostToDevice, stream), "H2D V");
    }
    if (rtm && edge) CUDA_OR_FAIL(cudaMemcpyAsync(dE, Eh, edge, cudaMemcpyHostToDevice, stream), "H2D Eproj");
    g3s_status st = g3s_forward(p, dQ, dK, dV, rtm ? dE : nullptr, dO, (rtm && Eouth) ? dEo : nullptr, stream_);
    if (st != G3S_OK) return st;
    if (node_out) CUDA_OR_FAIL(cudaMemcpyAsync(Oh, dO, node_out, cudaMemcpyDeviceToHost, stream), "D2H O");
    if (rtm && Eouth && edge_out)
        CUDA_OR_FAIL(cudaMemcpyAsync(Eouth, dEo, edge_out, cudaMemcpyDeviceToHost, stream), "D2H Eout");
    return G3S_OK;
}

g3s_status g3s_plan_set_edge_ids(g3s_plan* p, const int32_t* edge_id_d, int64_t num_edge_slots,
                                 g3s_stream_t stream_) {
    if (!p) return fail(G3S_ERR_INVALID_ARG, "NULL plan");
    if (!edge_id_d) {
        p->edge_id = nullptr;
        p->edge_slots = p->shape.E;
        return G3S_OK;
    }
    if (reinterpret_cast<uintptr_t>(edge_id_d) & 3u) return fail(G3S_ERR_INVALID_ARG, "edge ids must be 4-byte aligned");
    if (num_edge_slots < 1 || num_edge_slots > 0x7fffffffLL)
        return fail(G3S_ERR_INVALID_ARG, "num_edge_slots must be in [1, 2^31)");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    PlanCounts hc;
    CUDA_OR_FAIL(cudaMemsetAsync(&p->arr.counts->status, 0, sizeof(int32_t), stream), "cudaMemsetAsync(status)");
    CUDA_OR_FAIL(validate_edge_ids(edge_id_d, p->shape.E, num_edge_slots, p->arr.counts, stream), "edge id validation");
    CUDA_OR_FAIL(cudaMemcpyAsync(&hc, p->arr.counts, sizeof hc, cudaMemcpyDeviceToHost, stream), "cudaMemcpyAsync(counts)");
    CUDA_OR_FAIL(cudaStreamSynchronize(stream), "cudaStreamSynchronize(edge ids)");
    if (hc.status & kErrEdgeId) return fail(G3S_ERR_BAD_GRAPH, "an edge id is outside [0, %lld)", (long long)num_edge_slots);
    p->edge_id = edge_id_d;
    p->edge_slots = num_edge_slots;
    return G3S_OK;
}

g3s_status g3s_forward_check(const g3s_plan* p, g3s_stream_t stream_) {
    if (!p) return fail(G3S_ERR_INVALID_ARG, "NULL plan");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int32_t st = 0;
    CUDA_OR_FAIL(cudaMemcpyAsync(&st, p->arr.fwd_status, sizeof st, cudaMemcpyDeviceToHost, stream), "cudaMemcpyAsync(status)");
    CUDA_OR_FAIL(cudaStreamSynchronize(stream), "cudaStreamSynchronize(check)");
    if (st & kErrTimeout) {
        CUDA_OR_FAIL(cudaMemsetAsync(p->arr.fwd_status, 0, sizeof(int32_t), stream), "cudaMemsetAsync(status)");
        CUDA_OR_FAIL(cudaStreamSynchronize(stream), "cudaStreamSynchronize(check)");
        return fail(G3S_ERR_TIMEOUT, "a forward kernel's bounded device wait gave up; its outputs are incomplete");
    }
    return G3S_OK;
}

g3s_status g3s_selftest_wait_timeout(const g3s_plan* p, uint64_t limit_ns, g3s_stream_t stream_) {
    if (!p) return fail(G3S_ERR_INVALID_ARG, "NULL plan");
    if (limit_ns == 0 || limit_ns > 2000000000ull) return fail(G3S_ERR_INVALID_ARG, "limit_ns must be in (0, 2e9]");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    CUDA_OR_FAIL(wait_selftest_launch(limit_ns, p->arr.fwd_status, stream), "self-test launch");
    return g3s_forward_check(p, stream_);
}

g3s_status g3s_linear(const void* X, const void* W, int64_t M, int Kin, int Nout, g3s_dtype dtype, void* const* Y,
                      int seg_cols, g3s_dtype out_dtype, int32_t* status_d, g3s_stream_t stream_) {
    if (M < 0 || Kin <= 0 || Nout <= 0 || seg_cols <= 0) return fail(G3S_ERR_INVALID_ARG, "negative or zero size");
    if (dtype != G3S_F16 && dtype != G3S_BF16) return fail(G3S_ERR_UNSUPPORTED, "g3s_linear takes fp16 or bf16 inputs");
    if (out_dtype != G3S_F32 && out_dtype != dtype)
        return fail(G3S_ERR_INVALID_ARG, "out_dtype must be G3S_F32 or the input dtype");
    if (Kin % 8 != 0 || seg_cols % 64 != 0 || Nout % seg_cols != 0 || Nout / seg_cols > 3)
        return fail(G3S_ERR_INVALID_ARG, "need Kin %% 8 == 0, seg_cols %% 64 == 0, Nout = 1..3 x seg_cols");
    if (M > 0x7fffffffLL) return fail(G3S_ERR_INVALID_ARG, "M must fit in int32");
    if (M == 0) return G3S_OK;
    if (!X || !W || !Y) return fail(G3S_ERR_INVALID_ARG, "X, W and Y must be non-NULL");
    const int nseg = Nout / seg_cols;
    LinearParams lp{};
    lp.A = X;
    lp.W = W;
    for (int i = 0; i < nseg; ++i) {
        if (!Y[i] || !aligned16(Y[i])) return fail(G3S_ERR_INVALID_ARG, "output %d is NULL or not 16-byte aligned", i);
        lp.out[i] = Y[i];
    }
    if (!aligned16(X) || !aligned16(W)) return fail(G3S_ERR_INVALID_ARG, "X and W must be 16-byte aligned");
    if (!linear_supported(dtype, out_dtype, Kin, seg_cols)) return fail(G3S_ERR_UNSUPPORTED, "shape without a kernel");
    if (!tensor_maps_available()) return fail(G3S_ERR_UNSUPPORTED, "the driver offers no tensor-map encoding");
    lp.seg_cols = seg_cols;
    lp.M = M;
    lp.Kin = Kin;
    lp.Nout = Nout;
    lp.status = status_d;
    CUDA_OR_FAIL(linear_launch(dtype, out_dtype, lp, reinterpret_cast<cudaStream_t>(stream_)), "projection launch");
    return G3S_OK;
}

g3s_status g3s_layer_forward(const g3s_plan* p, const void* X, const void* Wqkv, int Kin, const void* Xe,
                             const void* We, int Ke, void* Q, void* K, void* V, void* Eproj, void* O, void* Eout,
                             g3s_stream_t stream_) {
    if (!p) return fail(G3S_ERR_INVALID_ARG, "NULL plan");
    const bool rtm = p->variant == G3S_RTMSCORE;
    if (p->dtype != G3S_F16 && p->dtype != G3S_BF16) return fail(G3S_ERR_UNSUPPORTED, "layer needs a 16-bit plan");
    const int hd = p->shape.H * p->shape.D;
    if (rtm != (Xe != nullptr || We != nullptr))
        return fail(G3S_ERR_INVALID_ARG, "Xe / We are needed for an RTMScore plan and only then");
    const g3s_dtype dt = (g3s_dtype)p->dtype;
    void* qkv[3] = {Q, K, V};
    g3s_status st = g3s_linear(X, Wqkv, p->shape.N, Kin, 3 * hd, dt, qkv, hd, dt, p->arr.fwd_status, stream_);
    if (st != G3S_OK) return st;
    if (rtm) {
        void* e1[1] = {Eproj};
        st = g3s_linear(Xe, We, p->edge_slots, Ke, hd, dt, e1, hd, dt, p->arr.fwd_status, stream_);
        if (st != G3S_OK) return st;
    }
    return g3s_forward(p, Q, K, V, rtm ? Eproj : nullptr, O, rtm ? Eout : nullptr, stream_);
}

void g3s_plan_destroy(g3s_plan* p) {
    if (!p) return;
    if (p->ev_join) cudaEventDestroy(p->ev_join);
    if (p->ev_fork) cudaEventDestroy(p->ev_fork);
    if (p->side) cudaStreamDestroy(p->side);
    delete p;
}

}  // extern "C"
