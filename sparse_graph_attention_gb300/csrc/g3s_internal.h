// Internal declarations shared by the libg3s translation units.
#pragma once

#include <cuda.h>  // CUtensorMap (the type only; driver entry points are looked up at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/g3s.h"

namespace g3s {

constexpr int kWinRows = 16;   // rows per BSB row window
constexpr int kTileCols = 8;   // columns per BSB tile (16x8 tiles)
constexpr int kFlagDup = 1;    // window holds a repeated (row, source) pair
constexpr int kFlagTile = 2;   // window takes the tensor-core tile path
constexpr int kFlagElig = 4;   // planner scratch: window eligible for the tile path (cleared before the plan is done)
constexpr int kFlagSplit = 8;  // tile-path window cut into 128-column slices (set with kFlagTile)
constexpr int kWarpsPerCta = 8;

// Error bits written by the CSR validation kernel.
enum : int32_t {
    kErrRowPtr0 = 1,      // row_ptr[0] != 0
    kErrRowPtrOrder = 2,  // row_ptr decreasing somewhere
    kErrRowPtrEnd = 4,    // row_ptr[N] != E
    kErrColRange = 8,     // a source outside [0, N)
    kErrTimeout = 16,     // a bounded device-side wait gave up (forward status word)
    kErrEdgeId = 32,      // an edge id outside [0, edge slots)
};

constexpr int kTileMaxTilesPerWindow = 16;  // tile-path windows have at most this many 16x8 tiles (128 columns)
// A tile-kernel item holds one or two tile-path windows, each starting at a
// 16-column boundary of the item, together at most 128 columns: a window of T
// tiles takes ceil(T/2) units of 16 columns, and two windows pair when their
// units sum to <= 8 (matched over the whole list, g3s_planner.cu).
// Stored as two int4: (w0, first tile of w0, T0, nwin | units0 << 8) and
// (w1, first tile of w1, T1, 0).  A slice s of the S slices of a split window
// w (one item per 16 tiles) is (w, first tile + 16 s, its tiles, 1 | units <<
// 8 | flag) and, edge-parallel (kItemPartial), (partial index of its row 0,
// S, 0, 0): row r writes its partial softmax state to index base + r S; or,
// node-parallel (kItemChain: the CTA takes the window's slices in order),
// (s, S, 0, 0).
constexpr int kTileItemUnits = 8;
constexpr int kItemPartial = 1 << 16;
constexpr int kItemChain = 1 << 17;

// Small device-resident counters filled by the planner and read back once.
struct PlanCounts {
    int32_t status;
    int32_t bucket_count[G3S_NUM_BUCKETS];
    int32_t n_heavy;
    int32_t n_chunks;
    int32_t n_tiles;
    int32_t n_tile_windows;
    int32_t n_dup_windows;
    int32_t n_large_windows;
    int32_t n_short;  // rows with at most PlanShape::pack_limit entries
    long long tile_window_nnz;
    long long elig_nnz, elig_tiles;  // CSR entries and tiles of the tile-eligible windows
    int32_t n_tile_items;  // work items of the tile kernel (one or two tile-path windows each)
    int32_t n_split_windows;  // tile-path windows cut into 128-column slices
    int32_t n_split_items;    // their slices (tile items after the n_tile_items pairs)
    int32_t n_merge;          // rows a forward merges (with split windows; else the heavy rows)
    long long split_nnz;      // CSR entries of the split windows
    int32_t unit_count[kTileItemUnits + 1];  // tile-path windows by 16-column units (index 1..8)
    int32_t n_match_runs;     // runs of the item matching (planner scratch)
};

// Device views the planner writes into (all inside the caller's workspace).
struct PlanArrays {
    uint8_t* bucket_of;        // [N] (with the bucket lists only)
    int32_t* bucket_ptr;       // [NB+1]
    int32_t* bucket_rows;      // [N] (with the bucket lists only)
    int32_t* heavy_rows;       // [max_heavy]
    int32_t* heavy_chunk_ptr;  // [max_heavy+1]
    int32_t* heavy_index;      // [N] scratch: heavy ordinal of a heavy row
    int32_t* chunks;           // [max_chunks][3]
    float* part_acc;           // [max_chunks + max_split_rows][H*d]
    float* part_ml;            // [max_chunks + max_split_rows][H][2]
    // BSB
    int32_t* win_tile_ptr;     // [W+1]
    int32_t* win_ucount;       // [W] unique sources per window (scratch)
    int32_t* win_nnz;          // [W]
    uint8_t* win_flags;        // [W]
    int32_t* tile_windows;     // [W]
    int4* tile_items;          // [2 (W + max_split_items)] tile kernel items: two int4 per item (kTileItemUnits)
    int32_t* tile_sorted;      // [W] tile-path windows sorted by (units, id) (planner scratch)
    int4* tile_runs;           // [32] runs of the item matching (planner scratch)
    int32_t* win_split_base;   // [W] split windows: slices of the split windows before this one
    int32_t* merge_rows;       // [N] rows a forward merges when the plan has split windows
    int2* merge_range;         // [N] their partial index ranges
    int2* chains;              // [W] node-parallel split windows: (first slice item, slices)
    int32_t* core_windows;     // [W] the other windows, ascending (rows left to the CUDA-core kernel)
    int32_t* large_windows;    // [W]
    int32_t* tile_cols;        // [max_tiles][8]
    uint32_t* tile_bits;       // [max_tiles][4]
    uint32_t* bitmap_scratch;  // [kLargeCtas][3][words]
    // scan scratch
    int32_t* scan_blocks;      // [scan_block_capacity]
    PlanCounts* counts;
    unsigned long long* work_counter;  // the fused kernel's work queue head
    unsigned int* tile_counter;        // the tile kernel's work queue head
    int32_t* fwd_status;               // error bits set by forward kernels (kErrTimeout)
};

constexpr int kLargeCtas = 32;  // CTAs of the global-bitmap window compaction

struct PlanShape {
    int64_t N, E;
    int H, D;
    int heavy_threshold, chunk_edges;
    int bounds[G3S_NUM_BUCKETS - 2];
    int bsb_smem_edges;
    int tile_density_milli, tile_max_tiles, tile_pool_milli, tile_split_milli;
    bool split_edge_parallel;  // split windows: slices merged from partial states (else chains)
    bool build_bsb, tile_enabled, bucket_lists;
    int64_t max_heavy, max_chunks, W, max_tiles, bitmap_words;
    int64_t max_split_rows, max_split_items;  // partial rows (edge-parallel) and items of split windows
    int64_t scan_blocks;
    int pack_limit;  // most entries of a row a short-row pack takes (0: the row width does not pack)
    long long small_rows;  // graphs of at most this many rows take the small-graph flavour
};

// Most CSR entries of a row that a short-row pack takes, for node rows of
// row_vecs 16-byte vectors: packs exist where a row is at most 16 vectors
// (G = 32 / row_vecs >= 2 lane groups); a group walks its row 4 entries a
// step and holds its indices two per lane; never above the heavy threshold.
inline int pack_limit_for(int row_vecs, int heavy_threshold) {
    if (row_vecs < 1 || row_vecs > 16) return 0;
    const int G = 32 / row_vecs;
    int t = 4 * G < 2 * row_vecs ? 4 * G : 2 * row_vecs;
    return t < heavy_threshold ? t : heavy_threshold;
}

// Whether forwards run the short-row pack flavour: option 1 forces it where
// the row width packs, -1 (auto) takes it when at least a quarter of the rows
// are short, 0 never.
inline bool use_packs(int option, const PlanShape& s, const PlanCounts& c) {
    if (s.pack_limit <= 0 || option == 0) return false;
    return option == 1 || 4LL * c.n_short >= s.N;
}

// Whether a plan has windows on the tile path (pairs or split windows).
inline bool any_tile(const PlanCounts& c) { return c.n_tile_windows + c.n_split_windows > 0; }

// ---- planner (g3s_planner.cu) --------------------------------------------
cudaError_t plan_validate(const int32_t* row_ptr, const int32_t* col_idx, const PlanShape& s,
                          const PlanArrays& a, cudaStream_t st);
cudaError_t plan_build(const int32_t* row_ptr, const int32_t* col_idx, const PlanShape& s,
                       const PlanArrays& a, cudaStream_t st);
cudaError_t validate_edge_ids(const int32_t* edge_id, long long E, long long slots, PlanCounts* c, cudaStream_t st);

// ---- CUDA-core fused kernel (g3s_core.cu) ---------------------------------
struct CoreParams {
    const int32_t* row_ptr;
    const int32_t* col_idx;
    const void* Q;
    const void* K;
    const void* V;
    const void* E;
    const void* W;  // aggregation weights [slots][H] (input type), mode 2 only
    const int32_t* edge_id;  // CSR position -> physical edge slot of E/Eout/W, or nullptr
    void* O;
    void* Eout;
    const int32_t* chunks;
    float* part_acc;
    float* part_ml;
    const uint8_t* win_flags;  // nullptr when no window takes the tile path
    // With tile windows: the windows of 16 rows left to this kernel (ascending)
    // and their count; its row items then run over these windows only.
    const int32_t* core_windows;
    long long n_core_windows;
    unsigned long long* work_counter;  // device scratch word, zeroed before every launch
    long long N;
    long long n_chunks;
    int H, D;
    int heavy_threshold;
    int row_vecs;  // H*D*sizeof(T)/16
    int lph;       // 16-byte vectors per head = D*sizeof(T)/16
    float qscale;  // standard: log2(e)/sqrt(d); RTMScore: 1/sqrt(d)
    float eps;
    int elementwise_clamp;
    int normalize;  // aggregation: divide by (sum of weights + eps)
    int32_t* status;  // forward status word: kErrTimeout is OR-ed in when a bounded wait gives up
    int static_items;  // set by the launcher: one item per warp, by warp id (no work counter)
    int pack_rows;     // run the short-row pack flavour (the plan's choice)
    int pack;          // set by the launcher: rows per item (1, or the lane-group count)
    int pack_max_deg;  // set by the launcher: a pack runs packed when no row has more entries
};

struct MergeParams {
    const int32_t* heavy_rows;
    const int32_t* heavy_chunk_ptr;
    const int2* ranges;  // when set: entry k merges partials [ranges[k].x, ranges[k].y), not the chunk_ptr range
    const float* part_acc;
    const float* part_ml;
    void* O;
    int n_heavy;
    int H, D;
    float eps;
    int normalize;  // plain (RTMScore / aggregation) merges: divide by (sum + eps)
};

// dtype / out_dtype: 0 f32, 1 f16, 2 bf16; out_dtype is f32 or the input dtype.
// mode: 0 standard softmax, 1 RTMScore, 2 weighted aggregation.
// Launchers return cudaErrorInvalidValue for shapes without a kernel.
// Tensor maps for TMA, encoded through the driver entry point looked up at
// run time (g3s_core.cu).
bool tensor_maps_available();
// A 2-D map over `rows` rows of `row_elems` elements of elem_bytes (2 or 4)
// with a box of box_rows x box_elems and the 128-byte swizzle
// (box_elems * elem_bytes == 128).
bool encode_tile(CUtensorMap* m, const void* base, long long rows, int row_elems, int elem_bytes, int box_rows,
                 int box_elems);

bool core_supported(int dtype, int row_vecs);
cudaError_t core_launch(int dtype, int out_dtype, int mode, const CoreParams& p, cudaStream_t st);
// The default of the small_graph_rows option: graphs of at most this many
// rows run the small-graph flavour (one CTA per row) when no window takes the
// tile path, so the whole forward is one launch.
constexpr int kSmallGraphRows = 1024;
cudaError_t core_small_launch(int dtype, int out_dtype, int mode, const CoreParams& p, cudaStream_t st);
cudaError_t merge_launch(int out_dtype, bool plain, const MergeParams& p, cudaStream_t st);
cudaError_t core_launch_f32(bool out_f32, int mode, const CoreParams& p, cudaStream_t st);
cudaError_t core_launch_f16(bool out_f32, int mode, const CoreParams& p, cudaStream_t st);
cudaError_t core_launch_bf16(bool out_f32, int mode, const CoreParams& p, cudaStream_t st);
// the short-row pack flavour: p.row_vecs <= 16, mode 0 or 2
cudaError_t core_launch_pack_f32(bool out_f32, int mode, const CoreParams& p, cudaStream_t st);
cudaError_t core_launch_pack_f16(bool out_f32, int mode, const CoreParams& p, cudaStream_t st);
cudaError_t core_launch_pack_bf16(bool out_f32, int mode, const CoreParams& p, cudaStream_t st);
// the small-graph flavour (one CTA per row, no chunks or merge launch)
cudaError_t core_small_launch_f32(bool out_f32, int mode, const CoreParams& p, cudaStream_t st);
cudaError_t core_small_launch_f16(bool out_f32, int mode, const CoreParams& p, cudaStream_t st);
cudaError_t core_small_launch_bf16(bool out_f32, int mode, const CoreParams& p, cudaStream_t st);
cudaError_t merge_launch_f32(bool plain, const MergeParams& p, cudaStream_t st);
cudaError_t merge_launch_f16(bool plain, const MergeParams& p, cudaStream_t st);
cudaError_t merge_launch_bf16(bool plain, const MergeParams& p, cudaStream_t st);

// ---- tensor-core tile kernel (g3s_tile.cu) -------------------------------
struct TileParams {
    const void* Q;
    const void* K;
    const void* V;
    void* O;
    long long N;
    int H;
    const int4* tile_items;  // two int4 per item (kTileItemUnits above)
    long long n_single_items;  // items taken one work index each (pairs, edge-parallel slices)
    const int2* chains;        // node-parallel split windows: (first slice item, slices), one work index each
    int n_chains;
    const int32_t* tile_cols;
    const uint32_t* tile_bits;
    float scale_log2;  // log2(e)/sqrt(d)
    int32_t* status;   // kErrTimeout is OR-ed in when a wait gives up
    unsigned int* work_counter;  // zeroed before the launch; CTAs take work indices from it
    float* part_acc;             // partial states of split-window slices: [index][H*d] unnormalised output,
    float* part_ml;              // [index][H][2] (row max in the log2 domain, row sum)
};
bool tile_supported(int dtype, int variant, int head_dim);
cudaError_t wait_selftest_launch(unsigned long long limit_ns, int32_t* status, cudaStream_t st);
cudaError_t tile_launch(int dtype, int out_dtype, const TileParams& p, cudaStream_t st);


// ---- dense projection on the tensor cores (g3s_linear.cu) -------------------
struct LinearParams {
    const void* A;    // X (M, Kin) row-major
    const void* W;    // W (Nout, Kin) row-major
    void* out[3];     // output segments, each (M, seg_cols) row-major
    int seg_cols;
    long long M;
    int Kin, Nout;
    int32_t* status;  // kErrTimeout is OR-ed in when a bounded wait gives up (may be null)
};
bool linear_supported(int dtype, int out_dtype, int kin, int seg_cols);
cudaError_t linear_launch(int dtype, int out_dtype, const LinearParams& p, cudaStream_t st);

// ---- host helpers shared by the ABI translation units (g3s_api.cu) ---------
namespace api {
constexpr size_t kAlign = 256;
g3s_status fail(g3s_status st, const char* fmt, ...);
g3s_status cuda_fail(cudaError_t e, const char* where);
int dtype_size(int dt);
bool aligned16(const void* p);
void default_options(g3s_plan_options* o);
g3s_status check_shape(int64_t N, int64_t E, int heads, int head_dim, int dtype, int variant,
                       const g3s_plan_options& o, PlanShape* s);
size_t carve(const PlanShape& s, PlanArrays* a, void* base);
}  // namespace api

}  // namespace g3s
