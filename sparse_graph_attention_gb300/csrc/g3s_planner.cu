// Device-side planner: CSR validation, degree buckets, heavy-row chunks and
// the Binary Sparse Block (BSB) compaction of 16-row windows into 16x8
// bitmap tiles (Fused3S, sciencestack.ai/paper/2505.08098, Figure 1: a row
// window is compacted, tiled and stored in BSB format).
//
// Everything is deterministic: positions come from exclusive scans (no
// atomics whose order can leak into an output), bitmaps are built with
// atomicOr (order-independent), counts with atomicAdd (order-independent).
#include <stdint.h>

#include "g3s_internal.h"

namespace g3s {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kScanThreads = 256;
constexpr int kScanItems = 4;
constexpr int kScanTile = kScanThreads * kScanItems;

// Block-wide exclusive prefix sum of one int per thread (blockDim.x a
// multiple of 32, at most 1024).  *total receives the block sum.
__device__ int block_exclusive_scan(int x, int* total) {
    __shared__ int warp_sums[32];
    __shared__ int block_total;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int inc = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(kFull, inc, off);
        if (lane >= off) inc += y;
    }
    if (lane == 31) warp_sums[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        const int ws = lane < nw ? warp_sums[lane] : 0;
        int wi = ws;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(kFull, wi, off);
            if (lane >= off) wi += y;
        }
        if (lane < nw) warp_sums[lane] = wi - ws;
        if (lane == 31) block_total = wi;
    }
    __syncthreads();
    const int res = warp_sums[wid] + inc - x;
    *total = block_total;
    __syncthreads();
    return res;
}

__device__ int block_sum(int x) {
    int t;
    block_exclusive_scan(x, &t);
    return t;
}

__device__ int block_max(int x) {
    __shared__ int wm[32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = max(x, __shfl_xor_sync(kFull, x, off));
    if (lane == 0) wm[wid] = x;
    __syncthreads();
    int r = wm[0];
    for (int k = 1; k < nw; ++k) r = max(r, wm[k]);
    __syncthreads();
    return r;
}

__device__ int block_min(int x) { return -block_max(-x); }

// ---------------------------------------------------------------------------
// Generic three-kernel exclusive scan over n items: val(i) gives the item's
// count, out(i, prefix, count) consumes the exclusive prefix.
// ---------------------------------------------------------------------------
template <class Val>
__global__ void __launch_bounds__(kScanThreads) k_scan_reduce(Val val, long long n, int32_t* block_sums) {
    const long long base = (long long)blockIdx.x * kScanTile + (long long)threadIdx.x * kScanItems;
    int s = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k)
        if (base + k < n) s += val(base + k);
    s = block_sum(s);
    if (threadIdx.x == 0) block_sums[blockIdx.x] = s;
}

__global__ void __launch_bounds__(1024) k_scan_blocks(int32_t* block_sums, long long nblocks, int32_t* total_out) {
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (long long base = 0; base < nblocks; base += blockDim.x) {
        const long long i = base + threadIdx.x;
        const int x = i < nblocks ? block_sums[i] : 0;
        int tot;
        const int ex = block_exclusive_scan(x, &tot);
        if (i < nblocks) block_sums[i] = carry + ex;
        __syncthreads();
        if (threadIdx.x == 0) carry += tot;
        __syncthreads();
    }
    if (threadIdx.x == 0 && total_out != nullptr) *total_out = carry;
}

template <class Val, class Out>
__global__ void __launch_bounds__(kScanThreads) k_scan_apply(Val val, Out out, long long n, const int32_t* block_sums) {
    const long long base = (long long)blockIdx.x * kScanTile + (long long)threadIdx.x * kScanItems;
    int v[kScanItems];
    int s = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        v[k] = base + k < n ? val(base + k) : 0;
        s += v[k];
    }
    int tot;
    int ex = block_exclusive_scan(s, &tot) + block_sums[blockIdx.x];
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        if (base + k < n) out(base + k, ex, v[k]);
        ex += v[k];
    }
}

template <class Val, class Out>
cudaError_t scan(Val val, Out out, long long n, int32_t* block_sums, int32_t* total, cudaStream_t st) {
    if (n <= 0) {
        if (total != nullptr) return cudaMemsetAsync(total, 0, sizeof(int32_t), st);
        return cudaSuccess;
    }
    const long long nb = (n + kScanTile - 1) / kScanTile;
    k_scan_reduce<<<(unsigned)nb, kScanThreads, 0, st>>>(val, n, block_sums);
    k_scan_blocks<<<1, 1024, 0, st>>>(block_sums, nb, total);
    k_scan_apply<<<(unsigned)nb, kScanThreads, 0, st>>>(val, out, n, block_sums);
    return cudaGetLastError();
}

inline unsigned grid_for(long long n, int threads) {
    long long b = (n + threads - 1) / threads;
    if (b < 1) b = 1;
    if (b > 1048576) b = 1048576;  // grid-stride loops cover the rest
    return (unsigned)b;
}

// ---------------------------------------------------------------------------
// Validation
// ---------------------------------------------------------------------------
__global__ void k_validate_rows(const int32_t* row_ptr, long long N, long long E, PlanCounts* c) {
    int err = 0;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i <= N; i += (long long)gridDim.x * blockDim.x) {
        const int a = row_ptr[i];
        if (i == 0 && a != 0) err |= kErrRowPtr0;
        if (i < N && row_ptr[i + 1] < a) err |= kErrRowPtrOrder;
        if (i == N && (long long)a != E) err |= kErrRowPtrEnd;
    }
    if (err) atomicOr(&c->status, err);
}

__global__ void k_validate_cols(const int32_t* col_idx, long long N, long long E, PlanCounts* c) {
    int err = 0;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += (long long)gridDim.x * blockDim.x) {
        const int s = col_idx[e];
        if (s < 0 || (long long)s >= N) err |= kErrColRange;
    }
    if (err) atomicOr(&c->status, err);
}

// ---------------------------------------------------------------------------
// Degree buckets
// ---------------------------------------------------------------------------
struct Bounds {
    int b[G3S_NUM_BUCKETS - 2];
};

__device__ __forceinline__ int bucket_of_degree(int d, const Bounds& bd) {
    if (d == 0) return 0;
    int k = 1;
#pragma unroll
    for (int x = 0; x < G3S_NUM_BUCKETS - 2; ++x)
        if (d > bd.b[x]) k = x + 2;
    return k;
}

// Also counts the rows with at most short_limit entries (the short-row packs'
// candidates; short_limit 0: none counted).
__global__ void k_bucket_classify(const int32_t* row_ptr, long long N, Bounds bd, int short_limit, uint8_t* bucket_of,
                                  PlanCounts* c) {
    __shared__ int cnt[G3S_NUM_BUCKETS + 1];
    if (threadIdx.x <= G3S_NUM_BUCKETS) cnt[threadIdx.x] = 0;
    __syncthreads();
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < N; i += (long long)gridDim.x * blockDim.x) {
        const int d = row_ptr[i + 1] - row_ptr[i];
        const int b = bucket_of_degree(d, bd);
        if (bucket_of != nullptr) bucket_of[i] = (uint8_t)b;
        atomicAdd(&cnt[b], 1);
        if (short_limit > 0 && d <= short_limit) atomicAdd(&cnt[G3S_NUM_BUCKETS], 1);
    }
    __syncthreads();
    if (threadIdx.x < G3S_NUM_BUCKETS && cnt[threadIdx.x]) atomicAdd(&c->bucket_count[threadIdx.x], cnt[threadIdx.x]);
    if (threadIdx.x == G3S_NUM_BUCKETS && cnt[threadIdx.x]) atomicAdd(&c->n_short, cnt[threadIdx.x]);
}

__global__ void k_bucket_ptr(const PlanCounts* c, int32_t* bucket_ptr) {
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        int s = 0;
        for (int b = 0; b < G3S_NUM_BUCKETS; ++b) {
            bucket_ptr[b] = s;
            s += c->bucket_count[b];
        }
        bucket_ptr[G3S_NUM_BUCKETS] = s;
    }
}

struct BucketFlag {
    const uint8_t* bucket_of;
    int b;
    __device__ int operator()(long long i) const { return bucket_of[i] == b ? 1 : 0; }
};
struct BucketOut {
    const int32_t* bucket_ptr;
    int32_t* bucket_rows;
    int b;
    __device__ void operator()(long long i, int p, int v) const {
        if (v) bucket_rows[bucket_ptr[b] + p] = (int32_t)i;
    }
};

// ---------------------------------------------------------------------------
// Heavy rows and their chunks
// ---------------------------------------------------------------------------
struct HeavyFlag {
    const int32_t* row_ptr;
    int threshold;
    __device__ int operator()(long long i) const { return (row_ptr[i + 1] - row_ptr[i]) > threshold ? 1 : 0; }
};
struct HeavyOut {
    int32_t* heavy_rows;
    int32_t* heavy_index;
    __device__ void operator()(long long i, int p, int v) const {
        if (v) {
            heavy_rows[p] = (int32_t)i;
            heavy_index[i] = p;
        }
    }
};
struct ChunkCount {
    const int32_t* row_ptr;
    int threshold, chunk;
    __device__ int operator()(long long i) const {
        const int d = row_ptr[i + 1] - row_ptr[i];
        return d > threshold ? (d + chunk - 1) / chunk : 0;
    }
};
struct ChunkOut {
    const int32_t* row_ptr;
    const int32_t* heavy_index;
    int32_t* heavy_chunk_ptr;
    int32_t* chunks;
    int chunk;
    __device__ void operator()(long long i, int p, int v) const {
        if (!v) return;
        heavy_chunk_ptr[heavy_index[i]] = p;
        const int a = row_ptr[i], b = row_ptr[i + 1];
        for (int c = 0; c < v; ++c) {
            const int s = a + c * chunk;
            int32_t* d = chunks + 3LL * (p + c);
            d[0] = (int32_t)i;
            d[1] = s;
            d[2] = min(s + chunk, b);
        }
    }
};

__global__ void k_heavy_tail(const PlanCounts* c, int32_t* heavy_chunk_ptr) {
    if (threadIdx.x == 0 && blockIdx.x == 0) heavy_chunk_ptr[c->n_heavy] = c->n_chunks;
}

// ---------------------------------------------------------------------------
// BSB compaction
// ---------------------------------------------------------------------------
__global__ void k_win_nnz(const int32_t* row_ptr, long long N, long long W, int32_t* win_nnz) {
    for (long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x; w < W; w += (long long)gridDim.x * blockDim.x) {
        const long long r0 = w * kWinRows, r1 = min(r0 + kWinRows, N);
        win_nnz[w] = row_ptr[r1] - row_ptr[r0];
    }
}

struct LargeFlag {
    const int32_t* win_nnz;
    int cap;
    __device__ int operator()(long long w) const { return win_nnz[w] > cap ? 1 : 0; }
};
struct ListOut {
    int32_t* list;
    __device__ void operator()(long long i, int p, int v) const {
        if (v) list[p] = (int32_t)i;
    }
};

// Sort the window's (source << 4 | row) keys in shared memory (bitonic).
__device__ int load_and_sort_window(const int32_t* row_ptr, const int32_t* col_idx, long long N, long long w,
                                    unsigned long long* keys, int* n_out) {
    const long long r0 = w * kWinRows;
    const long long r1 = min(r0 + kWinRows, N);
    const int e_lo = row_ptr[r0];
    const int n = row_ptr[r1] - e_lo;
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    // row of every CSR position: walk the <=16 row boundaries
    for (int x = threadIdx.x; x < n2; x += blockDim.x) {
        unsigned long long key = ~0ull;
        if (x < n) {
            const int e = e_lo + x;
            int r = 0;
            while (r0 + r + 1 < r1 && row_ptr[r0 + r + 1] <= e) ++r;
            key = ((unsigned long long)(unsigned)col_idx[e] << 4) | (unsigned)r;
        }
        keys[x] = key;
    }
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int x = threadIdx.x; x < n2; x += blockDim.x) {
                const int y = x ^ j;
                if (y > x) {
                    const unsigned long long a = keys[x], b = keys[y];
                    const bool up = (x & k) == 0;
                    if ((a > b) == up) {
                        keys[x] = b;
                        keys[y] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    *n_out = n;
    return e_lo;
}

constexpr int kSmallThreads = 256;

__global__ void __launch_bounds__(kSmallThreads) k_bsb_count_small(const int32_t* row_ptr, const int32_t* col_idx,
                                                                   long long N, int cap, const int32_t* win_nnz,
                                                                   int32_t* win_ucount, uint8_t* win_flags) {
    extern __shared__ unsigned long long keys[];
    const long long w = blockIdx.x;
    if (win_nnz[w] > cap) return;  // the global-bitmap kernel owns it
    int n;
    load_and_sort_window(row_ptr, col_idx, N, w, keys, &n);
    int uniq = 0, dup = 0;
    for (int x = threadIdx.x; x < n; x += blockDim.x) {
        const unsigned long long k = keys[x];
        if (x == 0 || (keys[x - 1] >> 4) != (k >> 4)) ++uniq;
        if (x > 0 && keys[x - 1] == k) dup = 1;
    }
    uniq = block_sum(uniq);
    dup = block_sum(dup);
    if (threadIdx.x == 0) {
        win_ucount[w] = uniq;
        win_flags[w] = dup ? (uint8_t)kFlagDup : (uint8_t)0;
    }
}

__global__ void __launch_bounds__(kSmallThreads) k_bsb_fill_small(const int32_t* row_ptr, const int32_t* col_idx,
                                                                  long long N, int cap, const int32_t* win_nnz,
                                                                  const int32_t* win_tile_ptr, int32_t* tile_cols,
                                                                  uint32_t* tile_bits) {
    extern __shared__ unsigned long long keys[];
    const long long w = blockIdx.x;
    if (win_nnz[w] > cap) return;
    int n2 = 1;
    while (n2 < cap) n2 <<= 1;
    int* uniq = reinterpret_cast<int*>(keys + n2);  // [cap]
    uint32_t* bits = reinterpret_cast<uint32_t*>(uniq + cap);  // [4 * ceil(cap/8)]
    const int t0 = win_tile_ptr[w];
    const int nt = win_tile_ptr[w + 1] - t0;
    for (int x = threadIdx.x; x < 4 * nt; x += blockDim.x) bits[x] = 0;
    int n;
    load_and_sort_window(row_ptr, col_idx, N, w, keys, &n);  // ends with __syncthreads
    int carry = 0;
    for (int base = 0; base < n; base += blockDim.x) {
        const int x = base + threadIdx.x;
        int first = 0;
        unsigned long long k = 0;
        if (x < n) {
            k = keys[x];
            first = (x == 0 || (keys[x - 1] >> 4) != (k >> 4)) ? 1 : 0;
        }
        int tot;
        const int ex = block_exclusive_scan(first, &tot);
        if (x < n) {
            const int pos = carry + ex + first - 1;  // rank of this key's source in U_w
            const int src = (int)(k >> 4), r = (int)(k & 15);
            if (first) uniq[pos] = src;
            const int bit = r * kTileCols + (pos % kTileCols);
            atomicOr(&bits[(pos / kTileCols) * 4 + bit / 32], 1u << (bit % 32));
        }
        carry += tot;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < nt * kTileCols; x += blockDim.x)
        tile_cols[(long long)t0 * kTileCols + x] = x < carry ? uniq[x] : -1;
    for (int x = threadIdx.x; x < 4 * nt; x += blockDim.x) tile_bits[(long long)t0 * 4 + x] = bits[x];
}

// Large windows: one CTA at a time per window, a global bitmap of all N
// sources per CTA.  Bitmaps are all-zero between windows.
constexpr int kLargeThreads = 1024;

struct WinRange {
    long long r0, r1;
    int e_lo, e_hi;
};

__device__ WinRange win_range(const int32_t* row_ptr, long long N, long long w) {
    WinRange q;
    q.r0 = w * kWinRows;
    q.r1 = min(q.r0 + kWinRows, N);
    q.e_lo = row_ptr[q.r0];
    q.e_hi = row_ptr[q.r1];
    return q;
}

// set the window bitmap, return [min, max] source through smin/smax
__device__ void large_set(const int32_t* col_idx, const WinRange& q, uint32_t* winmap, int* smin, int* smax) {
    int lo = 0x7fffffff, hi = -1;
    for (int e = q.e_lo + threadIdx.x; e < q.e_hi; e += blockDim.x) {
        const int s = col_idx[e];
        atomicOr(&winmap[s >> 5], 1u << (s & 31));
        lo = min(lo, s);
        hi = max(hi, s);
    }
    *smin = block_min(lo);
    *smax = block_max(hi);
    __syncthreads();
}

__global__ void __launch_bounds__(kLargeThreads) k_bsb_count_large(const int32_t* row_ptr, const int32_t* col_idx,
                                                                   long long N, const int32_t* large_windows,
                                                                   const PlanCounts* c, uint32_t* scratch,
                                                                   long long words, int32_t* win_ucount,
                                                                   uint8_t* win_flags) {
    uint32_t* winmap = scratch + (long long)blockIdx.x * 3 * words;
    uint32_t* rowmap = winmap + words;
    const int nl = c->n_large_windows;
    for (int k = blockIdx.x; k < nl; k += gridDim.x) {
        const long long w = large_windows[k];
        const WinRange q = win_range(row_ptr, N, w);
        int lo, hi;
        large_set(col_idx, q, winmap, &lo, &hi);
        int dup = 0;
        for (long long r = q.r0; r < q.r1; ++r) {
            const int a = row_ptr[r], b = row_ptr[r + 1];
            for (int e = a + threadIdx.x; e < b; e += blockDim.x) {
                const int s = col_idx[e];
                const uint32_t bit = 1u << (s & 31);
                if (atomicOr(&rowmap[s >> 5], bit) & bit) dup = 1;
            }
            __syncthreads();
            for (int e = a + threadIdx.x; e < b; e += blockDim.x) rowmap[col_idx[e] >> 5] = 0;
            __syncthreads();
        }
        int u = 0;
        if (hi >= 0)
            for (int x = (lo >> 5) + threadIdx.x; x <= (hi >> 5); x += blockDim.x) u += __popc(winmap[x]);
        u = block_sum(u);
        dup = block_sum(dup);
        if (hi >= 0)
            for (int x = (lo >> 5) + threadIdx.x; x <= (hi >> 5); x += blockDim.x) winmap[x] = 0;
        if (threadIdx.x == 0) {
            win_ucount[w] = u;
            win_flags[w] = dup ? (uint8_t)kFlagDup : (uint8_t)0;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kLargeThreads) k_bsb_fill_large(const int32_t* row_ptr, const int32_t* col_idx,
                                                                  long long N, const int32_t* large_windows,
                                                                  const PlanCounts* c, uint32_t* scratch,
                                                                  long long words, const int32_t* win_tile_ptr,
                                                                  int32_t* tile_cols, uint32_t* tile_bits) {
    uint32_t* winmap = scratch + (long long)blockIdx.x * 3 * words;
    uint32_t* pre = winmap + 2 * words;
    const int nl = c->n_large_windows;
    for (int k = blockIdx.x; k < nl; k += gridDim.x) {
        const long long w = large_windows[k];
        const WinRange q = win_range(row_ptr, N, w);
        int lo, hi;
        large_set(col_idx, q, winmap, &lo, &hi);
        const long long t0 = win_tile_ptr[w];
        const int nt = win_tile_ptr[w + 1] - (int)t0;
        int carry = 0;
        if (hi >= 0) {
            for (int base = lo >> 5; base <= (hi >> 5); base += blockDim.x) {
                const int x = base + threadIdx.x;
                const uint32_t word = x <= (hi >> 5) ? winmap[x] : 0u;
                const int pc = __popc(word);
                int tot;
                const int ex = block_exclusive_scan(pc, &tot);
                if (x <= (hi >> 5)) {
                    pre[x] = carry + ex;
                    uint32_t m = word;
                    int j = 0;
                    while (m) {
                        const int b = __ffs(m) - 1;
                        tile_cols[t0 * kTileCols + carry + ex + j] = x * 32 + b;
                        m &= m - 1;
                        ++j;
                    }
                }
                carry += tot;
            }
        }
        __syncthreads();
        for (long long r = q.r0; r < q.r1; ++r) {
            const int a = row_ptr[r], b = row_ptr[r + 1];
            const int rr = (int)(r - q.r0);
            for (int e = a + threadIdx.x; e < b; e += blockDim.x) {
                const int s = col_idx[e];
                const int pos = pre[s >> 5] + __popc(winmap[s >> 5] & ((1u << (s & 31)) - 1u));
                const int bit = rr * kTileCols + (pos % kTileCols);
                atomicOr(&tile_bits[(t0 + pos / kTileCols) * 4 + bit / 32], 1u << (bit % 32));
            }
        }
        for (int x = carry + threadIdx.x; x < nt * kTileCols; x += blockDim.x) tile_cols[t0 * kTileCols + x] = -1;
        __syncthreads();
        if (hi >= 0)
            for (int x = (lo >> 5) + threadIdx.x; x <= (hi >> 5); x += blockDim.x) winmap[x] = 0;
        __syncthreads();
    }
}

struct TileCount {
    const int32_t* win_ucount;
    __device__ int operator()(long long w) const { return (win_ucount[w] + kTileCols - 1) / kTileCols; }
};
struct TilePtrOut {
    int32_t* win_tile_ptr;
    __device__ void operator()(long long w, int p, int) const { win_tile_ptr[w] = p; }
};
__global__ void k_tile_ptr_tail(const PlanCounts* c, int32_t* win_tile_ptr, long long W) {
    if (threadIdx.x == 0 && blockIdx.x == 0) win_tile_ptr[W] = c->n_tiles;
}

// Tile-path selection, two passes.  A window is eligible when it has no
// repeated (row, source) pair, 1..max_tiles tiles, no heavy row and a density
// (CSR entries / (128 tiles)) of at least density_milli / 1000.  The eligible
// windows then take the tile path together when their pooled density
// (their entries / (128 x their tiles)) reaches pool_milli / 1000, and none does
// otherwise: the two kernels run concurrently but a plan that splits a batch of
// similar windows between them pays the slower kernel's tail, so the choice is
// made for the batch.  A window of more than 16 tiles (wider than the kernel's
// 128 columns) with no repeated pair and a density of at least split_milli /
// 1000 takes the tile path on its own as a split window, heavy rows included
// (split_milli = 0: never).
__global__ void k_tile_eligible(const int32_t* row_ptr, long long N, long long W, const int32_t* win_tile_ptr,
                                const int32_t* win_nnz, uint8_t* win_flags, bool enabled, int heavy_threshold,
                                int max_tiles, int density_milli, int split_milli, PlanCounts* c) {
    int ndup = 0, nsplit = 0;
    unsigned long long nnz_sum = 0, tile_sum = 0, split_nnz = 0;
    for (long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x; w < W; w += (long long)gridDim.x * blockDim.x) {
        uint8_t f = win_flags[w];
        if (f & kFlagDup) ++ndup;
        if (enabled && !(f & kFlagDup)) {
            const long long nt = win_tile_ptr[w + 1] - win_tile_ptr[w];
            const long long r0 = w * kWinRows, r1 = min(r0 + kWinRows, N);
            int md = 0;
            for (long long r = r0; r < r1; ++r) md = max(md, row_ptr[r + 1] - row_ptr[r]);
            const long long nnz = win_nnz[w];
            if (split_milli > 0 && nt > kTileMaxTilesPerWindow && 1000LL * nnz >= (long long)split_milli * 128LL * nt) {
                f |= kFlagTile | kFlagSplit;
                ++nsplit;
                split_nnz += (unsigned long long)nnz;
            } else if (nt >= 1 && nt <= max_tiles && md <= heavy_threshold &&
                       1000LL * nnz >= (long long)density_milli * 128LL * nt) {
                f |= kFlagElig;
                nnz_sum += (unsigned long long)nnz;
                tile_sum += (unsigned long long)nt;
            }
        }
        win_flags[w] = f;
    }
    if (ndup) atomicAdd(&c->n_dup_windows, ndup);
    if (nsplit) atomicAdd(&c->n_split_windows, nsplit);
    if (split_nnz) atomicAdd(reinterpret_cast<unsigned long long*>(&c->split_nnz), split_nnz);
    if (nnz_sum) atomicAdd(reinterpret_cast<unsigned long long*>(&c->elig_nnz), nnz_sum);
    if (tile_sum) atomicAdd(reinterpret_cast<unsigned long long*>(&c->elig_tiles), tile_sum);
}

__global__ void k_tile_pool(long long W, uint8_t* win_flags, int pool_milli, PlanCounts* c) {
    const unsigned long long nnz = (unsigned long long)c->elig_nnz, tiles = (unsigned long long)c->elig_tiles;
    const bool take = tiles > 0 && 1000ull * nnz >= (unsigned long long)pool_milli * 128ull * tiles;
    for (long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x; w < W; w += (long long)gridDim.x * blockDim.x) {
        const uint8_t f = win_flags[w];
        win_flags[w] = (uint8_t)((f & ~kFlagElig) | ((take && (f & kFlagElig)) ? kFlagTile : 0));
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) c->tile_window_nnz = take ? (long long)nnz : 0;
}

// Tile-kernel items.  A tile-path window of T tiles takes u = ceil(T/2)
// units of 16 columns (1..8); two windows share an item when their units sum
// to at most kTileItemUnits.  The list is sorted by (u, window id) -- eight
// stable scans put each unit bucket in place -- and matched from both ends:
// the widest remaining window takes the narrowest remaining one when the two
// fit, else it is an item on its own (the fewest items any pairing reaches).
// The walk runs over the eight bucket counts in one thread as at most 17
// runs of identical steps; a parallel kernel then writes the items.
constexpr int kMaxMatchRuns = 32;
__device__ __forceinline__ int window_units(const int32_t* win_tile_ptr, int w) {
    return (win_tile_ptr[w + 1] - win_tile_ptr[w] + 1) / 2;
}
struct UnitFlag {
    const int32_t* tile_windows;
    const int32_t* win_tile_ptr;
    const PlanCounts* c;
    int u;
    __device__ int operator()(long long i) const {
        return i < c->n_tile_windows && window_units(win_tile_ptr, tile_windows[i]) == u ? 1 : 0;
    }
};
struct UnitOut {
    const int32_t* tile_windows;
    const PlanCounts* c;
    int32_t* sorted;
    int u;
    __device__ void operator()(long long i, int p, int v) const {
        if (!v) return;
        int base = 0;
        for (int b = 1; b < u; ++b) base += c->unit_count[b];
        sorted[base + p] = tile_windows[i];
    }
};
// runs[r] = (count << 1 | pair, low position, high position, first item)
__global__ void k_match_runs(PlanCounts* c, int4* runs) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int base[kTileItemUnits + 2];
    base[1] = 0;
    for (int b = 1; b <= kTileItemUnits; ++b) base[b + 1] = base[b] + c->unit_count[b];
    auto bucket = [&](int pos) {
        int b = 1;
        while (b < kTileItemUnits && pos >= base[b + 1]) ++b;
        return b;
    };
    int lo = 0, hi = base[kTileItemUnits + 1] - 1, nr = 0, items = 0;
    while (lo <= hi && nr < kMaxMatchRuns) {
        const int bl = bucket(lo), bh = bucket(hi);
        const bool pair = lo < hi && bl + bh <= kTileItemUnits;
        int k;
        if (pair)
            k = bl == bh ? (hi - lo + 1) / 2 : min(base[bl + 1] - lo, hi - base[bh] + 1);
        else
            k = hi - max(base[bh], lo) + 1;  // the rest of the high bucket, each on its own
        runs[nr++] = make_int4(k << 1 | (pair ? 1 : 0), lo, hi, items);
        items += k;
        if (pair) lo += k;
        hi -= k;
    }
    c->n_tile_items = items;
    c->n_match_runs = nr;
}
__global__ void k_match_items(const PlanCounts* c, const int4* runs, const int32_t* sorted,
                              const int32_t* win_tile_ptr, int4* items, long long W) {
    const int n = c->n_tile_items, nr = c->n_match_runs;
    for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += (long long)gridDim.x * blockDim.x) {
        int r = 0;
        while (r + 1 < nr && runs[r + 1].w <= k) ++r;
        const int4 R = runs[r];
        const int j = (int)k - R.w;
        const int wh = sorted[R.z - j];
        const int th = win_tile_ptr[wh];
        const int4 high = make_int4(wh, th, win_tile_ptr[wh + 1] - th, 0);
        if (R.x & 1) {
            const int wl = sorted[R.y + j];
            const int tl = win_tile_ptr[wl];
            items[2 * k] = make_int4(wl, tl, win_tile_ptr[wl + 1] - tl, 2 | (window_units(win_tile_ptr, wl) << 8));
            items[2 * k + 1] = high;
        } else {
            items[2 * k] = make_int4(wh, th, high.z, 1 | (window_units(win_tile_ptr, wh) << 8));
            items[2 * k + 1] = make_int4(0, 0, 0, 0);
        }
    }
    (void)W;
}

struct TileFlag {  // tile-path windows of at most 16 tiles (the pairs' list)
    const uint8_t* win_flags;
    __device__ int operator()(long long w) const { return (win_flags[w] & (kFlagTile | kFlagSplit)) == kFlagTile ? 1 : 0; }
};

// Split windows: S = ceil(T / 16) slices each, numbered in window order after
// the pairs' items.  Edge-parallel, the slices before window w
// (win_split_base) place its partial states at chunks + 16 x base: row r,
// slice s at + r S + s; node-parallel, a slice carries (s, S) and the
// window's chain entry (first slice item, S) is one work unit.
struct SplitCount {
    const uint8_t* win_flags;
    const int32_t* win_tile_ptr;
    __device__ int operator()(long long w) const {
        if (!(win_flags[w] & kFlagSplit)) return 0;
        return (win_tile_ptr[w + 1] - win_tile_ptr[w] + kTileMaxTilesPerWindow - 1) / kTileMaxTilesPerWindow;
    }
};
struct SplitOut {
    const int32_t* win_tile_ptr;
    const PlanCounts* c;
    int32_t* win_split_base;
    int4* items;
    bool edge_parallel;
    __device__ void operator()(long long w, int p, int v) const {
        if (!v) return;
        win_split_base[w] = p;
        const int t0 = win_tile_ptr[w], T = win_tile_ptr[w + 1] - t0;
        const int base = c->n_chunks + kWinRows * p;
        int4* it = items + 2LL * (c->n_tile_items + p);
        for (int sl = 0; sl < v; ++sl) {
            const int ts = min(kTileMaxTilesPerWindow, T - kTileMaxTilesPerWindow * sl);
            it[2 * sl] = make_int4((int)w, t0 + kTileMaxTilesPerWindow * sl, ts,
                                   1 | (((ts + 1) / 2) << 8) | (edge_parallel ? kItemPartial : kItemChain));
            it[2 * sl + 1] = make_int4(edge_parallel ? base + sl : sl, v, 0, 0);
        }
    }
};
struct SplitFlag {
    const uint8_t* win_flags;
    __device__ int operator()(long long w) const { return (win_flags[w] & kFlagSplit) ? 1 : 0; }
};
struct ChainOut {
    const int32_t* win_tile_ptr;
    const int32_t* win_split_base;
    const PlanCounts* c;
    int2* chains;
    __device__ void operator()(long long w, int p, int v) const {
        if (!v) return;
        const int S = (win_tile_ptr[w + 1] - win_tile_ptr[w] + kTileMaxTilesPerWindow - 1) / kTileMaxTilesPerWindow;
        chains[p] = make_int2(c->n_tile_items + win_split_base[w], S);
    }
};

// The rows a forward merges when the plan has split windows: the heavy rows
// outside split windows (their chunks) and, edge-parallel, every row of a
// split window (its slices' partial states), with the partial index range of
// each.  (Node-parallel, a split window's rows are final in the tile kernel.)
struct MergeFlag {
    const int32_t* row_ptr;
    const uint8_t* win_flags;
    int threshold;
    bool edge_parallel;
    __device__ int operator()(long long r) const {
        if (win_flags[r / kWinRows] & kFlagSplit) return edge_parallel ? 1 : 0;
        return (row_ptr[r + 1] - row_ptr[r]) > threshold ? 1 : 0;
    }
};
struct MergeOut {
    const uint8_t* win_flags;
    const int32_t* win_tile_ptr;
    const int32_t* win_split_base;
    const int32_t* heavy_index;
    const int32_t* heavy_chunk_ptr;
    const PlanCounts* c;
    int32_t* merge_rows;
    int2* merge_range;
    __device__ void operator()(long long r, int p, int v) const {
        if (!v) return;
        merge_rows[p] = (int32_t)r;
        const long long w = r / kWinRows;
        if (win_flags[w] & kFlagSplit) {
            const int S = (win_tile_ptr[w + 1] - win_tile_ptr[w] + kTileMaxTilesPerWindow - 1) / kTileMaxTilesPerWindow;
            const int b = c->n_chunks + kWinRows * win_split_base[w] + (int)(r % kWinRows) * S;
            merge_range[p] = make_int2(b, b + S);
        } else {
            const int h = heavy_index[r];
            merge_range[p] = make_int2(heavy_chunk_ptr[h], heavy_chunk_ptr[h + 1]);
        }
    }
};
struct CoreWindowFlag {
    const uint8_t* win_flags;
    __device__ int operator()(long long w) const { return (win_flags[w] & kFlagTile) ? 0 : 1; }
};

#define G3S_TRY(x)                          \
    do {                                    \
        cudaError_t err_ = (x);             \
        if (err_ != cudaSuccess) return err_; \
    } while (0)

}  // namespace

__global__ void k_validate_edge_ids(const int32_t* ids, long long E, long long slots, PlanCounts* c) {
    int err = 0;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += (long long)gridDim.x * blockDim.x) {
        const int v = ids[e];
        if (v < 0 || (long long)v >= slots) err = kErrEdgeId;
    }
    if (err) atomicOr(&c->status, err);
}

cudaError_t validate_edge_ids(const int32_t* edge_id, long long E, long long slots, PlanCounts* c, cudaStream_t st) {
    if (E <= 0) return cudaSuccess;
    k_validate_edge_ids<<<grid_for(E, 256), 256, 0, st>>>(edge_id, E, slots, c);
    return cudaGetLastError();
}

cudaError_t plan_validate(const int32_t* row_ptr, const int32_t* col_idx, const PlanShape& s, const PlanArrays& a,
                          cudaStream_t st) {
    k_validate_rows<<<grid_for(s.N + 1, 256), 256, 0, st>>>(row_ptr, s.N, s.E, a.counts);
    G3S_TRY(cudaGetLastError());
    if (s.E > 0) {
        k_validate_cols<<<grid_for(s.E, 256), 256, 0, st>>>(col_idx, s.N, s.E, a.counts);
        G3S_TRY(cudaGetLastError());
    }
    return cudaSuccess;
}

cudaError_t plan_build(const int32_t* row_ptr, const int32_t* col_idx, const PlanShape& s, const PlanArrays& a,
                       cudaStream_t st) {
    PlanCounts* c = a.counts;
    // 1. degree buckets
    Bounds bd;
    for (int k = 0; k < G3S_NUM_BUCKETS - 2; ++k) bd.b[k] = s.bounds[k];
    if (s.N > 0) {
        k_bucket_classify<<<grid_for(s.N, 256), 256, 0, st>>>(row_ptr, s.N, bd, s.pack_limit, a.bucket_of, c);
        G3S_TRY(cudaGetLastError());
    }
    k_bucket_ptr<<<1, 32, 0, st>>>(c, a.bucket_ptr);
    G3S_TRY(cudaGetLastError());
    // the per-bucket row lists (five stable scans) only on request: no forward
    // kernel reads them (rows run in id order, heavy rows as chunks)
    for (int b = 0; s.bucket_lists && b < G3S_NUM_BUCKETS; ++b)
        G3S_TRY(scan(BucketFlag{a.bucket_of, b}, BucketOut{a.bucket_ptr, a.bucket_rows, b}, s.N, a.scan_blocks,
                     nullptr, st));

    // 2. heavy rows and chunks
    G3S_TRY(scan(HeavyFlag{row_ptr, s.heavy_threshold}, HeavyOut{a.heavy_rows, a.heavy_index}, s.N, a.scan_blocks,
                 &c->n_heavy, st));
    G3S_TRY(scan(ChunkCount{row_ptr, s.heavy_threshold, s.chunk_edges},
                 ChunkOut{row_ptr, a.heavy_index, a.heavy_chunk_ptr, a.chunks, s.chunk_edges}, s.N, a.scan_blocks,
                 &c->n_chunks, st));
    k_heavy_tail<<<1, 32, 0, st>>>(c, a.heavy_chunk_ptr);
    G3S_TRY(cudaGetLastError());

    if (!s.build_bsb) return cudaSuccess;

    // 3. BSB tiles
    const long long W = s.W;
    if (W > 0) {
        k_win_nnz<<<grid_for(W, 256), 256, 0, st>>>(row_ptr, s.N, W, a.win_nnz);
        G3S_TRY(cudaGetLastError());
    }
    G3S_TRY(scan(LargeFlag{a.win_nnz, s.bsb_smem_edges}, ListOut{a.large_windows}, W, a.scan_blocks,
                 &c->n_large_windows, st));
    int n2 = 1;
    while (n2 < s.bsb_smem_edges) n2 <<= 1;
    const size_t smem_count = (size_t)n2 * sizeof(unsigned long long);
    const size_t smem_fill = smem_count + (size_t)s.bsb_smem_edges * sizeof(int) +
                             (size_t)4 * ((s.bsb_smem_edges + kTileCols - 1) / kTileCols) * sizeof(uint32_t);
    G3S_TRY(cudaFuncSetAttribute(k_bsb_count_small, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_count));
    G3S_TRY(cudaFuncSetAttribute(k_bsb_fill_small, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_fill));
    if (W > 0) {
        k_bsb_count_small<<<(unsigned)W, kSmallThreads, smem_count, st>>>(row_ptr, col_idx, s.N, s.bsb_smem_edges,
                                                                          a.win_nnz, a.win_ucount, a.win_flags);
        G3S_TRY(cudaGetLastError());
    }
    k_bsb_count_large<<<kLargeCtas, kLargeThreads, 0, st>>>(row_ptr, col_idx, s.N, a.large_windows, c,
                                                            a.bitmap_scratch, s.bitmap_words, a.win_ucount,
                                                            a.win_flags);
    G3S_TRY(cudaGetLastError());
    G3S_TRY(scan(TileCount{a.win_ucount}, TilePtrOut{a.win_tile_ptr}, W, a.scan_blocks, &c->n_tiles, st));
    k_tile_ptr_tail<<<1, 32, 0, st>>>(c, a.win_tile_ptr, W);
    G3S_TRY(cudaGetLastError());
    if (s.max_tiles > 0) G3S_TRY(cudaMemsetAsync(a.tile_bits, 0, (size_t)s.max_tiles * 4 * sizeof(uint32_t), st));
    if (W > 0) {
        k_bsb_fill_small<<<(unsigned)W, kSmallThreads, smem_fill, st>>>(row_ptr, col_idx, s.N, s.bsb_smem_edges,
                                                                        a.win_nnz, a.win_tile_ptr, a.tile_cols,
                                                                        a.tile_bits);
        G3S_TRY(cudaGetLastError());
    }
    k_bsb_fill_large<<<kLargeCtas, kLargeThreads, 0, st>>>(row_ptr, col_idx, s.N, a.large_windows, c,
                                                           a.bitmap_scratch, s.bitmap_words, a.win_tile_ptr,
                                                           a.tile_cols, a.tile_bits);
    G3S_TRY(cudaGetLastError());

    // 4. tile-path selection
    if (W > 0) {
        k_tile_eligible<<<grid_for(W, 256), 256, 0, st>>>(row_ptr, s.N, W, a.win_tile_ptr, a.win_nnz, a.win_flags,
                                                          s.tile_enabled, s.heavy_threshold, s.tile_max_tiles,
                                                          s.tile_density_milli, s.tile_split_milli, c);
        G3S_TRY(cudaGetLastError());
        k_tile_pool<<<grid_for(W, 256), 256, 0, st>>>(W, a.win_flags, s.tile_pool_milli, c);
        G3S_TRY(cudaGetLastError());
    }
    G3S_TRY(scan(TileFlag{a.win_flags}, ListOut{a.tile_windows}, W, a.scan_blocks, &c->n_tile_windows, st));
    if (s.tile_enabled && W > 0) {
        for (int u = 1; u <= kTileItemUnits; ++u)
            G3S_TRY(scan(UnitFlag{a.tile_windows, a.win_tile_ptr, c, u}, UnitOut{a.tile_windows, c, a.tile_sorted, u}, W,
                         a.scan_blocks, &c->unit_count[u], st));
        k_match_runs<<<1, 32, 0, st>>>(c, a.tile_runs);
        G3S_TRY(cudaGetLastError());
        k_match_items<<<grid_for(W, 256), 256, 0, st>>>(c, a.tile_runs, a.tile_sorted, a.win_tile_ptr, a.tile_items, W);
        G3S_TRY(cudaGetLastError());
    }
    if (s.max_split_items > 0) {
        G3S_TRY(scan(SplitCount{a.win_flags, a.win_tile_ptr},
                     SplitOut{a.win_tile_ptr, c, a.win_split_base, a.tile_items, s.split_edge_parallel}, W,
                     a.scan_blocks, &c->n_split_items, st));
        if (!s.split_edge_parallel)
            G3S_TRY(scan(SplitFlag{a.win_flags}, ChainOut{a.win_tile_ptr, a.win_split_base, c, a.chains}, W,
                         a.scan_blocks, nullptr, st));
        G3S_TRY(scan(MergeFlag{row_ptr, a.win_flags, s.heavy_threshold, s.split_edge_parallel},
                     MergeOut{a.win_flags, a.win_tile_ptr, a.win_split_base, a.heavy_index, a.heavy_chunk_ptr, c,
                              a.merge_rows, a.merge_range},
                     s.N, a.scan_blocks, &c->n_merge, st));
    }
    G3S_TRY(scan(CoreWindowFlag{a.win_flags}, ListOut{a.core_windows}, W, a.scan_blocks, nullptr, st));
    return cudaSuccess;
}

}  // namespace g3s
