/*
 * g3s.h -- C ABI of libg3s, fused sparse graph attention ("3S") on GB300.
 *
 * For every destination row i of a CSR graph (rows = destinations, columns =
 * sources) and every head h, one pass computes
 *   SDDMM    l_ij = <q_i, k_j> / sqrt(d)              over the in-edges of i
 *   softmax  a_ij = exp(l_ij - max_j l_ij) / sum_j exp(l_ij - max_j l_ij)
 *   SpMM     o_i  = sum_j a_ij v_j                    (o_i = 0 when i has no in-edge)
 * This is the three-step pattern named in the Fused3S abstract
 * (sciencestack.ai/paper/2505.08098, Abstract: "SDDMM, softmax normalization,
 * and SpMM") and the per-node gather of the Triton article
 * (stondelli.it/articles/gattn-triton, "Using the CSC index for fast edge
 * lookup").
 *
 * The RTMScore edge-modulated variant (same article, "Background" list and
 * "Fusing the full graph attention", the eager torch_attn listing) replaces
 * the logit and the softmax by
 *   t_ij = clamp(q_i * k_j / sqrt(d), -5, 5)   (elementwise; optional)
 *   u_ij = t_ij * e_ij                          (elementwise, stored as Eout)
 *   s_ij = exp(clamp(sum_f u_ij, -5, 5)),  a_ij = s_ij / (sum_j s_ij + eps)
 *
 * Memory model.  Every array belongs to the caller: this library allocates no
 * device or host memory after g3s_plan_create returns (the plan's small host
 * struct is the only allocation it ever makes).  Device pointers must stay
 * valid while a plan or a call uses them.  All work is enqueued on the given
 * stream; g3s_plan_create synchronises that stream (once, or twice with
 * validation on) to read back the plan's sizes, g3s_forward never does.
 *
 * Errors.  Every entry point returns a g3s_status; no exception or abort
 * crosses the ABI.  g3s_last_error() gives a human-readable detail of the
 * last failure on the calling thread.
 *
 * Layouts (row-major, contiguous, little-endian):
 *   row_ptr  int32 [N+1]      row_ptr[0] = 0, non-decreasing, row_ptr[N] = E
 *   col_idx  int32 [E]        sources of row i at col_idx[row_ptr[i] .. row_ptr[i+1])
 *   Q, K, V      [N][H][d]    element type = the plan's dtype
 *   O            [N][H][d]    element type = the plan's out_dtype (fp32 by default)
 *   Eproj        [E][H][d]    the plan's dtype, indexed by CSR position (RTMScore only)
 *   Eout         [E][H][d]    the plan's out_dtype, indexed by CSR position
 * Limits: E < 2^31; d in {16, 32, 64, 128}; H*d*sizeof(dtype) a power of two
 * between 16 B and 4 KiB; every value pointer 16-byte aligned.
 */
#ifndef G3S_H
#define G3S_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *g3s_stream_t;

typedef enum g3s_status {
    G3S_OK = 0,
    G3S_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size, plan mismatch */
    G3S_ERR_UNSUPPORTED = 2, /* shape or dtype without a compiled kernel */
    G3S_ERR_BAD_GRAPH = 3,   /* CSR failed validation (see g3s_last_error) */
    G3S_ERR_WORKSPACE = 4,   /* workspace missing, misaligned or too small */
    G3S_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
    G3S_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up */
} g3s_status;

typedef enum g3s_dtype { G3S_F32 = 0, G3S_F16 = 1, G3S_BF16 = 2 } g3s_dtype;

typedef enum g3s_variant {
    G3S_STANDARD = 0, /* softmax(<q,k>/sqrt d) */
    G3S_RTMSCORE = 1  /* exp(clip(sum clamp(q*k/sqrt d)*e)) / (sum + eps), with Eout */
} g3s_variant;

#define G3S_NUM_BUCKETS 5

/*
 * Planner options.  Fill with g3s_plan_options_init, then override.
 *  bucket_bounds   inclusive upper degree bounds of buckets 1..3 (bucket 0 is
 *                  degree 0, bucket 4 is above bucket_bounds[2]); default 32, 256, 2048
 *  heavy_threshold rows with more in-edges are cut into chunks processed by
 *                  several warps and merged; chunks are taken before the rows,
 *                  so long rows do not finish last.  0 (default): ten times
 *                  the mean degree E/N, clamped to [64, 512] (stats.heavy_threshold
 *                  reports the value used)
 *  chunk_edges     CSR positions per chunk of a heavy row (default 0:
 *                  automatic, 512 x 256 / (node row bytes) between 64 and 512:
 *                  512 for rows up to 256 bytes, 128 for 1 KB rows, since a
 *                  warp walks a chunk one edge step at a time and a step takes
 *                  fewer edges of wider rows)
 *  bsb             build the 16x8 BSB tiles: 1 on, 0 off, -1 when the tile path
 *                  is eligible (default -1)
 *  tile_path       route dense row windows to the tensor-core kernel: 1 on,
 *                  0 off, -1 automatic (default -1: on where compiled, which
 *                  is the standard form with fp16/bf16 inputs and d = 64,
 *                  unless bsb = 0)
 *  tile_density_milli  a window is eligible for the tile path when
 *                  1000 * nnz >= tile_density_milli * 128 * tiles (default 100)
 *                  and it has no repeated (row, source) pair, at most
 *                  tile_max_tiles tiles and no heavy row
 *  tile_pool_density_milli  the eligible windows take the tile path together
 *                  when 1000 * (their CSR entries) >= tile_pool_density_milli *
 *                  128 * (their tiles), and none does otherwise (default 180).
 *                  Measured on one GB300 with batched 20-60-node graphs (8 x 64
 *                  bf16, ms per forward, CUDA-core kernel against tensor-core
 *                  kernel): edge probability 0.18 (pooled density 0.16-0.18)
 *                  0.084 against 0.086, 0.22 (0.18-0.20) 0.094 against 0.088,
 *                  0.3 (0.24) 0.115 against 0.091, complete graphs 0.305
 *                  against 0.098; a plan that splits a batch between the two
 *                  kernels pays the slower one's tail (edge probability 0.3
 *                  with a per-window floor of 0.15: 0.095), so the choice is
 *                  made for the batch
 *  tile_max_tiles  most 16x8 tiles a tile-path window may have (default and
 *                  maximum with the tile path on: 16, i.e. 128 source columns,
 *                  the M side of the kernel's tcgen05 product)
 *  tile_split_density_milli  windows wider than 16 tiles (128 source
 *                  columns) whose density reaches tile_split_density_milli /
 *                  1000 take the tile path as split windows, cut into
 *                  128-column slices (the columns split as in the Fused3S
 *                  page's Figure 3 caption); heavy rows inside a split window
 *                  are computed there, not as chunks.  Decided per window,
 *                  outside the pooled rule.  0 turns split windows off;
 *                  otherwise 100..1000 (default 150: node-parallel slices beat
 *                  the CUDA-core path from a density between 0.125 and 0.17).
 *  tile_split_parallel  how split windows run (the node- and edge-parallel
 *                  blocks of the Fused3S page's Figure 2 caption): 0 (default)
 *                  node-parallel, one CTA takes all slices of a window and head,
 *                  O accumulating in tensor memory with the row maxima carried
 *                  over the slices; 1 edge-parallel, every slice a work item of
 *                  its own that writes a partial softmax state per row (row
 *                  max, row sum, unnormalised output), merged per row after the
 *                  kernels the way heavy-row chunks are.  Edge-parallel partial
 *                  states take workspace: up to 2000 * E / (128 *
 *                  tile_split_density_milli) rows of 4 * H * (d + 2) bytes.
 *                  Measured on one GB300 (1024 windows whose rows share
 *                  2048-node pools, 12.6 M entries, 8 x 64 bf16, ms per
 *                  forward): CUDA-core path 1.86, node-parallel 0.80,
 *                  edge-parallel 1.29; windows whose 16 rows each draw 1024 of
 *                  a shared pool, 4.2 M entries, CUDA-core chunks against
 *                  slices before the merge: density 1 0.87 against 0.11, 0.5
 *                  0.85 against 0.21, 0.25 0.85 against 0.40
 *  bsb_smem_edges  windows with more CSR entries than this are compacted by
 *                  the global-bitmap planner kernel instead of the shared-
 *                  memory sort (default 2048; a testing knob)
 *  rtm_elementwise_clamp  1: clamp q*k/sqrt(d) elementwise before *e, the
 *                  order of the article's code (default); 0: skip that clamp
 *  rtm_epsilon     the variant's denominator epsilon (default 1e-6)
 *  validate_graph  1: check the CSR on the device before planning (default)
 *  out_dtype       element type of O and Eout: G3S_F32 (default) or the input
 *                  dtype.  fp32 keeps the fp32 accumulation; a 16-bit store adds
 *                  up to one half-ulp of rounding (2^-8 relative for bf16)
 *  degree_buckets  1: also list the rows of each degree bucket (ascending
 *                  id), readable with g3s_plan_export; 0 (default): only
 *                  count them (stats.bucket_count).  No forward kernel reads
 *                  the lists: rows run in id order, so neighbouring rows'
 *                  sources meet in L2, heavy rows as chunks taken first, short
 *                  rows in packs; the lists cost five stable scans of N rows
 *  small_graph_rows  graphs of at most this many rows, with no window on
 *                  the tile path, run one CTA per row: its eight warps each
 *                  take an eighth of the row's entries and merge their partial
 *                  softmax states in shared memory, so the forward is one
 *                  launch whose latency is about one step of edges per row
 *                  (default 1024; 0: never; heavy-row chunks are then not used)
 *  pack_rows       short-row packs, where a node row is at most 256 bytes
 *                  (G = 32 * 16 / row bytes >= 2 lane groups per warp): a warp
 *                  takes G consecutive rows together, one per lane group,
 *                  when each has at most min(4 G, 2 * 32 / G, heavy_threshold)
 *                  entries (stats.pack_limit), else one row at a time.  The
 *                  kernel with packs needs more registers, so it is a second
 *                  flavour: -1 (default) uses it when at least a quarter of
 *                  the rows are that short (stats.short_rows), 1 whenever the
 *                  row width packs, 0 never.  Same arithmetic per row; a
 *                  packed row's terms are summed in CSR order by one lane
 *                  group (no lane-group merge).
 */
typedef struct g3s_plan_options {
    int32_t bucket_bounds[G3S_NUM_BUCKETS - 2];
    int32_t heavy_threshold;
    int32_t chunk_edges;
    int32_t bsb;
    int32_t tile_path;
    int32_t tile_density_milli;
    int32_t tile_max_tiles;
    int32_t bsb_smem_edges;
    int32_t rtm_elementwise_clamp;
    float rtm_epsilon;
    int32_t validate_graph;
    int32_t out_dtype;
    int32_t pack_rows;
    int32_t tile_pool_density_milli;
    int32_t degree_buckets;
    int32_t small_graph_rows;
    int32_t tile_split_density_milli;
    int32_t tile_split_parallel;
} g3s_plan_options;

typedef struct g3s_plan_stats {
    int64_t num_nodes, num_edges;
    int32_t heads, head_dim, dtype, variant, out_dtype;
    int64_t bucket_count[G3S_NUM_BUCKETS];
    int64_t heavy_rows, chunks;
    int32_t has_bsb, tile_path;
    int64_t windows, tiles, tile_windows, dup_windows, large_windows;
    int64_t tile_window_nnz; /* CSR entries handled by the tile path */
    int32_t pack_rows;       /* 1 when standard-form forwards and aggregations use short-row
                                packs (an RTMScore forward never does) */
    int32_t pack_limit;      /* most entries of a packed row (0: this row width does not pack) */
    int32_t heavy_threshold; /* the heavy-row threshold in use (option 0 resolved) */
    int32_t chunk_edges;     /* CSR positions per heavy-row chunk */
    int64_t short_rows;      /* rows with at most pack_limit entries */
    size_t workspace_used;
    int64_t tile_items;      /* work items of the tile kernel: one or two tile-path windows each,
                                or one 128-column slice of a split window */
    int32_t small_graph;     /* 1 when forwards and aggregations run the small-graph flavour */
    int64_t split_windows;   /* tile-path windows cut into 128-column slices (included in
                                tile_windows) */
    int64_t split_items;     /* items of the split windows (included in tile_items) */
    int64_t merge_rows;      /* rows a forward merges from partial states: heavy rows outside
                                split windows and every row of a split window */
} g3s_plan_stats;

/* Planner arrays readable with g3s_plan_export (all int32 unless noted). */
typedef enum g3s_plan_array {
    G3S_ARR_BUCKET_PTR = 0,      /* [G3S_NUM_BUCKETS+1] scan of bucket sizes */
    G3S_ARR_BUCKET_ROWS = 1,     /* [N] rows by bucket, ascending id inside (degree_buckets = 1) */
    G3S_ARR_HEAVY_ROWS = 2,      /* [heavy_rows] ascending */
    G3S_ARR_HEAVY_CHUNK_PTR = 3, /* [heavy_rows+1] */
    G3S_ARR_CHUNKS = 4,          /* [chunks][3] (row, e_begin, e_end) */
    G3S_ARR_WIN_TILE_PTR = 5,    /* [W+1], W = ceil(N/16) */
    G3S_ARR_TILE_COLS = 6,       /* [tiles][8], -1 padded */
    G3S_ARR_TILE_BITS = 7,       /* uint32 [tiles][4], bit r*8+c of a 128-bit word */
    G3S_ARR_WIN_NNZ = 8,         /* [W] CSR entries per window */
    G3S_ARR_WIN_FLAGS = 9,       /* uint8 [W]: bit0 repeated edge, bit1 tile path, bit3 split
                                    window (with bit1) */
    G3S_ARR_TILE_WINDOWS = 10,   /* [tile_windows - split_windows] ascending: the tile-path
                                    windows of at most 16 tiles */
    G3S_ARR_CORE_WINDOWS = 11,   /* [windows - tile_windows] ascending: the windows whose rows the
                                    CUDA-core kernel takes (every window without bit 1) */
    G3S_ARR_TILE_ITEMS = 12,     /* [tile_items][8]: the tile kernel's items.  First the windows
                                    of the tile-path list, one or two per item: a window of T
                                    tiles takes u = ceil(T/2) units of 16 columns; the list sorted
                                    by (u, id) is matched from both ends, the widest remaining
                                    window taking the narrowest remaining one when their units
                                    sum to <= 8, else alone; per item (w0, first tile of w0, T0,
                                    nwin | u0 << 8, w1, first tile of w1, T1, 0), window 0 the
                                    narrower of a pair, the second window zero when nwin = 1.
                                    Then the split windows in ascending order, one
                                    item per 128-column slice s of S = ceil(T/16):
                                    (w, first tile + 16 s, its tiles, 1 | units << 8 | 1 << 16,
                                     chunks + B_w + s, S, 0, 0), where B_w = 16 x (the slices of
                                    the split windows before w); row r of the window writes its
                                    partial state to partial index chunks + B_w + r S + s */
    G3S_ARR_MERGE_ROWS = 13,     /* [merge_rows] ascending: the rows a forward merges */
    G3S_ARR_MERGE_RANGES = 14    /* [merge_rows][2]: partial indices [begin, end) of each merged
                                    row (heavy-row chunks, or the slices of a split window) */
} g3s_plan_array;

typedef struct g3s_plan g3s_plan; /* opaque */

/* Library version string, e.g. "g3s 0.1 sm_103a". Never NULL.
 * (No counterpart on the pages: library plumbing, as are the next three.) */
const char *g3s_version(void);

/* Name of a status code. Never NULL. */
const char *g3s_status_string(g3s_status status);

/* Detail of the last failing call on this thread ("" when none). Never NULL. */
const char *g3s_last_error(void);

/* Fill *opts with the defaults listed above. */
void g3s_plan_options_init(g3s_plan_options *opts);

/*
 * Upper bound of the workspace bytes a plan for these sizes needs, for any
 * graph with N nodes and E edges.  opts may be NULL (defaults).
 * No counterpart on the pages: every device array belongs to the caller here
 * (the Triton article's "Conclusions": allocation on the host side costs more
 * than the kernels), so the caller asks for the size first.
 * INVALID_ARG for negative sizes or a NULL *bytes; UNSUPPORTED for shapes
 * without a kernel.
 */
g3s_status g3s_plan_workspace_size(int64_t num_nodes, int64_t num_edges, int heads, int head_dim,
                                   g3s_dtype dtype, g3s_variant variant,
                                   const g3s_plan_options *opts, size_t *bytes);

/*
 * Build a plan for one graph on the current CUDA device (the degree
 * buckets, heavy-row chunks and BSB tiles, all on the device).
 * Sources: the BSB tiles are the Fused3S row-window compaction
 * (sciencestack.ai/paper/2505.08098, Figure 1: a 16-row window compacted to
 * its unique columns, tiled into 16x8 blocks with bitmaps); the per-node
 * index ranges the CUDA-core kernel walks are the Triton article's CSC lookup
 * (stondelli.it/articles/gattn-triton, "Using the CSC index for fast edge
 * lookup"); the degree buckets and heavy-row chunks are this library's
 * scheduling (the pages have no counterpart; Fused3S Figure 2 shows blocks
 * sharing a row's work, which the chunks restate for heavy rows).
 *   row_ptr_d, col_idx_d  device CSR arrays; must outlive the plan
 *   workspace_d           device memory of workspace_bytes, 256-byte aligned,
 *                         owned by the caller, must outlive the plan
 *   stream                all planner kernels run here; synchronised before return
 *   out                   receives the plan; free with g3s_plan_destroy
 * Besides its host struct, a plan with tile-path windows holds one CUDA
 * stream (created at the device's highest stream priority) and two events:
 * g3s_forward runs the CUDA-core kernel on that stream, forked from and
 * joined back into the caller's stream, and the tile kernel on the caller's
 * stream after it (so both kernels overlap, the few CUDA-core CTAs are
 * placed first, and the call stays capturable in a CUDA graph).
 * Returns BAD_GRAPH when validation finds row_ptr[0] != 0, a decreasing
 * row_ptr, row_ptr[N] != E or a source outside [0, N).  With validation off
 * a malformed CSR is undefined behaviour.
 */
g3s_status g3s_plan_create(const int32_t *row_ptr_d, const int32_t *col_idx_d, int64_t num_nodes,
                           int64_t num_edges, int heads, int head_dim, g3s_dtype dtype,
                           g3s_variant variant, const g3s_plan_options *opts, void *workspace_d,
                           size_t workspace_bytes, g3s_stream_t stream, g3s_plan **out);

/*
 * Attach a physical edge numbering to the plan, as the Triton article's CSC
 * index does with its position-to-edge-id vector (stondelli.it/articles/
 * gattn-triton, "Using the CSC index for fast edge lookup"): edge features
 * live in their own storage order and several sparse indices can share them.
 *   edge_id_d       device int32 [E]: CSR position e -> slot in [0, num_edge_slots);
 *                   must outlive the plan.  NULL restores CSR-position indexing.
 *   num_edge_slots  rows of the edge arrays (Eproj, Eout and the aggregation W)
 * From then on g3s_forward reads Eproj[edge_id[e]] and writes
 * Eout[edge_id[e]] (RTMScore), g3s_aggregate reads W[edge_id[e]], and the
 * host staging holds num_edge_slots edge rows.  Validates every id on the
 * device (synchronises `stream`): BAD_GRAPH when one is out of range.
 */
g3s_status g3s_plan_set_edge_ids(g3s_plan *plan, const int32_t *edge_id_d, int64_t num_edge_slots,
                                 g3s_stream_t stream);

/* Sizes and counts of a plan.  (No counterpart on the pages.) */
g3s_status g3s_plan_get_stats(const g3s_plan *plan, g3s_plan_stats *stats);

/*
 * Copy one planner array to host memory (no counterpart on the pages: it lets
 * tests compare the device planner bit for bit).  bytes_needed (may be NULL)
 * receives its size; host_dst may be NULL to query only.  Otherwise bytes
 * must be at least that size.  Synchronous (blocks on the plan's stream).
 * UNSUPPORTED for BSB arrays of a plan built without BSB.
 */
g3s_status g3s_plan_export(const g3s_plan *plan, g3s_plan_array which, void *host_dst, size_t bytes,
                           size_t *bytes_needed);

/*
 * One fused forward pass over the whole graph, enqueued on `stream`: SDDMM,
 * row softmax and SpMM in one pass with nothing of S written to memory (the
 * Fused3S abstract and TL;DR, sciencestack.ai/paper/2505.08098), and for the
 * RTMScore variant the fused kernel of the Triton article
 * (stondelli.it/articles/gattn-triton, "Fusing the full graph attention"),
 * whose outputs are the node features and the updated edge features.
 *   Q, K, V  device [N][H][d] inputs
 *   Eproj    device [E][H][d] edge projections; RTMScore only, else NULL
 *            ([slots][H][d] in physical edge order after g3s_plan_set_edge_ids)
 *   O        device [N][H][d] output in out_dtype (fully overwritten)
 *   Eout     device [E][H][d] updated edge features in out_dtype (RTMScore;
 *            NULL skips the store)
 * Uses the plan's workspace for heavy-row partials, so calls that share a
 * plan must not overlap on the device.  Asynchronous: returns after the
 * launches are enqueued.  INVALID_ARG for NULL / misaligned pointers or an
 * Eproj that does not match the variant; CUDA when a launch fails.
 */
g3s_status g3s_forward(const g3s_plan *plan, const void *Q, const void *K, const void *V,
                       const void *Eproj, void *O, void *Eout, g3s_stream_t stream);

/*
 * Weighted aggregation over the plan's graph, enqueued on `stream`:
 *   O_i^h = sum_e W[e][h] * X[col_idx[e]][h][:]                 normalize = 0
 *   O_i^h = sum_e W[e][h] * X[...][h][:] / (sum_e W[e][h] + eps) normalize = 1
 * over the CSR entries e of row i: the normalised scatter-add of the Triton
 * article (stondelli.it/articles/gattn-triton, "Optimizing the scatter add in
 * Triton" and "Using the CSC index for fast edge lookup") and the CSR weighted
 * aggregation of the POPCORNBENCH task (normalize = 0).  Rows without edges
 * give 0.
 *   W  device [E][H] weights in the plan's dtype, indexed by CSR position
 *   X  device [N][H][d] features in the plan's dtype
 *   O  device [N][H][d] output in the plan's out_dtype (fully overwritten)
 * Works with a plan of either variant (it needs only the graph, H, d and
 * dtype) and uses its workspace, so it must not overlap another call on the
 * same plan.  INVALID_ARG for NULL or misaligned pointers or eps < 0.
 */
g3s_status g3s_aggregate(const g3s_plan *plan, const void *W, const void *X, void *O, int normalize, float eps,
                         g3s_stream_t stream);

/*
 * Dense projection on the tensor cores: Y = X W^T with fp32 accumulation.
 * The projection of node (or edge) features into the attention's inputs; the
 * Triton article (stondelli.it/articles/gattn-triton, closing section) notes
 * that once the attention is fused these GEMMs dominate the layer.  No
 * counterpart on the pages beyond that remark: the layout is this library's.
 *   X  device (M, Kin) row-major, 16-bit (dtype G3S_F16 or G3S_BF16)
 *   W  device (Nout, Kin) row-major (a linear layer's weight), same dtype
 *   Y  host array of Nout / seg_cols device pointers (1 to 3): output i holds
 *      columns [i * seg_cols, (i + 1) * seg_cols) of Y as an (M, seg_cols)
 *      row-major array in out_dtype (G3S_F32 or dtype), fully overwritten
 *   status_d  optional device int32: the bit 0x10 is OR-ed in if a bounded
 *      device wait gives up (the outputs are then incomplete); may be NULL
 * Kin must be a positive multiple of 8 and seg_cols a positive multiple of
 * 64 (Nout = 1, 2 or 3 times seg_cols); all pointers 16-byte aligned.
 * INVALID_ARG otherwise; UNSUPPORTED for other dtypes or when the driver
 * offers no tensor-map encoding; CUDA when the launch fails.
 */
g3s_status g3s_linear(const void *X, const void *W, int64_t M, int Kin, int Nout, g3s_dtype dtype,
                      void *const *Y, int seg_cols, g3s_dtype out_dtype, int32_t *status_d, g3s_stream_t stream);

/*
 * One attention layer on the plan's graph (the Triton article's closing
 * remark on the projections around the fused attention; the Fused3S abstract's
 * Graph Transformer layer; the layout is this library's): Q | K | V = X Wqkv^T with
 * g3s_linear (Wqkv is (3 H d, Kin), rows for Q, then K, then V), then
 * g3s_forward.  For an RTMScore plan also Eproj = Xe We^T (Xe (edge slots,
 * Ke), We (H d, Ke)) feeds the edge term; NULL Xe/We on a standard plan.
 * Q, K, V (each (N, H, d)) and Eproj ((edge slots, H, d)) are caller device
 * buffers of the plan's dtype that receive the projections; O and Eout as in
 * g3s_forward.  The plan's dtype must be 16-bit and H d a multiple of 64.
 * Uses the plan's workspace and status word.  Errors as g3s_linear and
 * g3s_forward.
 */
g3s_status g3s_layer_forward(const g3s_plan *plan, const void *X, const void *Wqkv, int Kin, const void *Xe,
                             const void *We, int Ke, void *Q, void *K, void *V, void *Eproj, void *O, void *Eout,
                             g3s_stream_t stream);

/*
 * (No counterpart on the pages, as g3s_forward_host.)
 * Bytes of device staging g3s_forward_host needs for this plan: room for
 * Q, K, V, O (and Eproj, Eout for RTMScore), each 256-byte aligned.
 */
g3s_status g3s_host_staging_size(const g3s_plan *plan, size_t *bytes);

/*
 * No counterpart on the pages: a convenience for callers whose features live
 * in host memory.
 * g3s_forward on HOST buffers: copies Q, K, V (and Eproj) host->device into
 * the caller's device staging area, runs the forward pass, and copies O (and
 * Eout when non-NULL) device->host, all enqueued on `stream` (one
 * cudaMemcpyAsync per array).  Host buffers should be pinned for the copies
 * to be asynchronous; the caller synchronises the stream before reading O.
 */
g3s_status g3s_forward_host(const g3s_plan *plan, const void *Q_h, const void *K_h, const void *V_h,
                            const void *Eproj_h, void *O_h, void *Eout_h, void *staging_d,
                            size_t staging_bytes, g3s_stream_t stream);

/*
 * (No counterpart on the pages: error reporting of the bounded device waits.)
 * Synchronise `stream` and report whether a kernel of an earlier g3s_forward
 * on this plan gave up a bounded device-side wait (the tensor-core tile
 * kernel waits on its MMAs for at most about one second).  Returns
 * G3S_ERR_TIMEOUT once per such event (the flag is then cleared): the
 * outputs of that forward are incomplete.  G3S_OK otherwise.
 */
g3s_status g3s_forward_check(const g3s_plan *plan, g3s_stream_t stream);

/*
 * (No counterpart on the pages.)
 * Self-test of the device-side timeout path: launches one CTA that waits, with
 * the same bounded wait the tile kernel uses, on an mbarrier that nothing ever
 * completes; after limit_ns (at most 2 s) it gives up and sets the plan's
 * status word.  Then behaves as g3s_forward_check: synchronises `stream` and
 * returns G3S_ERR_TIMEOUT, clearing the flag.  The context stays usable.
 */
g3s_status g3s_selftest_wait_timeout(const g3s_plan *plan, uint64_t limit_ns, g3s_stream_t stream);

/*
 * Gather-rate probe (no counterpart on the pages: a measurement aid for the
 * roofline of the CUDA-core kernel where K and V stay in L2).  Reads at least
 * `gathers` rows of row_bytes each (a power of two in [16, 4096]) from src
 * ([rows][row_bytes], 16-byte aligned, rows a power of two >= 2): the j-th row
 * read is (j + 1) * 0x9E3779B97F4A7C15 >> (64 - log2 rows) (64-bit wrap-around
 * product), spread uniformly over the rows.  `ctas` CTAs of 8 warps, eight
 * 512-byte warp loads in flight per warp, through the read-only path the
 * CUDA-core kernel uses (plain_loads = 0) or plain global loads
 * (plain_loads = 1); what is read is XOR-ed into one word
 * per warp of sink (ctas * 8 uint32).  *rows_read (may be NULL) receives the
 * rows read (whole warp steps).  Enqueued on `stream`; time it with events.
 */
g3s_status g3s_gather_probe(const void *src, int64_t rows, int row_bytes, int64_t gathers, int ctas, int plain_loads,
                            uint32_t *sink, int64_t *rows_read, g3s_stream_t stream);

/* Release the plan's host struct, stream and events (the caller still owns the workspace). NULL is a no-op.
 * (No counterpart on the pages.) */
void g3s_plan_destroy(g3s_plan *plan);

/*
 * Bytes of device scratch built into the library for g3s_forward_noalloc.
 */
#define G3S_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * g3s_forward_noalloc -- plan and forward in one call, with no allocation.
 *
 * The pages have no counterpart of this call; it exists for callers that
 * cannot allocate device memory: an inference engine that hands out device
 * memory only when it is built, a process whose GPU memory is already held
 * by another framework's caching allocator, or a service under a fixed
 * memory budget.  Such callers cannot provide the workspace g3s_plan_create
 * needs, and a cudaMalloc may also synchronise the device at a bad time.
 *
 * Same arguments and result as g3s_plan_create (default options, no BSB
 * tiles) followed by g3s_forward: O (and Eout) come out in fp32, the
 * caller passes the CSR, inputs and outputs only.  The planner arrays and
 * heavy-row partial results live in a static device array of
 * G3S_NOALLOC_SCRATCH_BYTES (32 MiB) that every GPU loading this library
 * holds until the process exits.  A graph whose plan needs more -- the size
 * g3s_plan_workspace_size reports with bsb = 0, about 9 bytes per node plus
 * 4*(H*d + 2*H + 3) bytes per possible chunk, E/512 + E/(T+1) of them for
 * the automatic heavy-row threshold T -- is rejected with
 * G3S_ERR_WORKSPACE before any device work.
 *
 * Calls no cudaMalloc, cudaFree or other allocating routine.  The first call
 * on a device looks up the scratch's device address (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture.
 * The address is kept for the life of the process: after cudaDeviceReset on
 * a device (which ends its context and the library's device memory with
 * it) do not call this entry point on that device again.
 * Every call on a device shares the one scratch array and leaves its
 * contents behind (the counters it needs are cleared at the start of each
 * call), so calls that overlap on the GPU, from any stream or thread, race:
 * serialise them.  Synchronises `stream` twice (validation and planner
 * sizes) before enqueueing the forward kernels, which run asynchronously.
 */
g3s_status g3s_forward_noalloc(const int32_t *row_ptr_d, const int32_t *col_idx_d, int64_t num_nodes,
                               int64_t num_edges, int heads, int head_dim, g3s_dtype dtype,
                               g3s_variant variant, const void *Q, const void *K, const void *V,
                               const void *Eproj, void *O, void *Eout, g3s_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* G3S_H */
