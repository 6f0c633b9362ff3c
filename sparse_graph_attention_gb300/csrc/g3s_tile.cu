// Tensor-core tile path: fused SDDMM -> masked softmax -> SpMM over the BSB
// tiles of dense row windows, with tcgen05.mma accumulating in TMEM.
//
// Source: the Fused3S design (sciencestack.ai/paper/2505.08098): a 16-row
// window is compacted to its unique source columns and tiled into 16x8 tiles
// with bitmaps (Figure 1); one thread block owns a window's Q and O rows
// (node-parallel, Figure 2); SDDMM, softmax and SpMM stay on chip (TL;DR).
// Its warp-level MMA layout is not reused: on sm_103a one thread issues
// tcgen05.mma for the whole CTA, an MMA has 64 or 128 rows (M), and the
// accumulators live in tensor memory.
//
// Mapping (the transposed products).  A window has 16 rows but up to 128
// source columns, so the columns go on the MMA's M side and the rows on N.
// A work item is one head of one or two consecutive tile-path windows whose
// columns, each window starting at a 16-column boundary, fill at most the
// 128 rows of M (the planner's items):
//   S^T = K_cols Q_w^T   M = 128 item columns, N = 16 rows per window, K = d
//   O^T = V_cols^T P^T   per window: M = d (64, issued as 128: see below),
//                        N = its 16 rows, K = its columns, 16 at a time
// so every column of the item serves its own window's rows in one MMA round
// trip, and the second product runs only over each window's own columns.
//
// Per item: cp.async gathers the head's 128-byte K and V rows of the item's
// columns and its windows' Q rows into 128-byte-swizzled shared memory; one
// thread issues S^T into TMEM; thread c reads column c of S^T (the 16 logits
// of its window's rows) and masks it by the tile bitmap.  The row maxima and
// the row sums of P = 2^(s - m), rounded to the input type, are reduced in
// registers: a half-warp (16 columns, always inside one window, since
// windows start at 16-column boundaries) reduce-scatters its 16 x 16 values
// with shuffles so that lane l holds row l, and 32 threads combine the eight
// half-warps' partials per row.  A window has at most 128 columns, so the max
// is final before any P is formed and the softmax needs no online rescale.
// Each column's thread writes its 16 values of P as one 32-byte row of P^T,
// the MN-major B operand of the second product.  O^T uses the V rows as its
// MN-major A operand; its 64 feature rows are issued as M = 128 with the
// second half reading the same rows again (atom stride 0), so TMEM lanes
// 64-127 repeat lanes 0-63 and all four warps store rows.
//
// Pipeline: one item in flight per CTA and five CTAs per SM (shared memory
// for one stage of K, V, Q and P^T: about 44 KB), so the SM, not the CTA,
// hides the gathers' latency.  At the start of item i (S^T of item i and
// O^T of item i-1 complete) the CTA requests item i+1's K, Q and bitmaps and
// item i's V rows, stores item i-1's rows, and turns item i's logits into
// row maxima; S^T of item i+1 is issued as soon as its K and Q have landed,
// and runs while item i forms P; O^T of item i follows once its V rows are
// in.  Work indices come from one counter; one thread keeps the descriptors
// of the next three items in a shared-memory ring.  The serial roles are
// spread over the four warps (mbarrier polling and the row-max combine in
// warp 0, S^T issued from warp 1, O^T from warp 2, the row-sum combine and
// the descriptor fetch in warp 3), so no warp holds the others at a barrier.
//
// Windows wider than 128 columns (split windows) are cut into 128-column
// slices, taken either edge-parallel (each slice an item of its own that
// writes a partial softmax state per row, merged per row afterwards) or
// node-parallel (a chain: one CTA takes all slices of a window and head in a
// row, O^T accumulating in TMEM across them, with a lazily moved reference
// max per row: O^T and the row sums are rescaled only when a slice's max
// exceeds the reference by more than 2^8; the rows are stored after the last
// slice).  Every mbarrier wait is
// bounded (about one second of %globaltimer); on expiry the CTA sets the
// plan's status word, frees its TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstddef>
#include <type_traits>

#include "g3s_internal.h"
#include "g3s_ptx.cuh"

namespace g3s {
namespace {

constexpr int kThreads = 128;
constexpr int kMinCtasPerSm = 5;
constexpr int kD = 64;                         // head_dim of this kernel
constexpr int kRows = kWinRows;                // 16 rows per window: the N of a window
constexpr int kCols = kTileItemUnits * 16;     // 128 item columns: the MMA's M
constexpr int kTiles = kCols / kTileCols;      // 16 tile slots per item
constexpr int kMaxWin = 2;                     // windows per item
constexpr int kItemRows = kMaxWin * kRows;     // 32
constexpr int kHalfWarps = kCols / 16;         // 8 half-warps of 16 columns
constexpr uint32_t kTmemCols = 64;             // S^T [0, 32), O^T [32, 64) (window j at +16 j)
constexpr int kRing = 8;                       // item descriptor ring
constexpr float kLazyRescale = 8.f;            // a chain moves its reference max only past +8 (P <= 2^8)
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

struct TileSmem {
    uint8_t k[kCols * 128];            // K rows: K-major A operand of S^T
    uint8_t v[kCols * 128];            // V rows: MN-major A operand of O^T (M rows 0-63)
    uint8_t q[kItemRows * 128];        // Q rows (row 16 j + r of window j): K-major B operand of S^T
    uint8_t pt[kCols * 32];            // P^T: [column][16 rows of its window], MN-major B operand, 32-byte swizzle
    float part[kHalfWarps][kRows];     // per half-warp: partial row maxima, later partial row sums
    float rowmax[kItemRows];           // row maxima of the item's windows (row 16 j + r)
    float inv_l[kItemRows];            // 1 / row sum of P (0 for a row without entries)
    float rowsum[kItemRows];           // row sums of P (a split window's slice stores them)
    float mref[kRows];                 // a chain's reference row maxima (log2 domain), carried over its slices
    float fac[kRows];                  // this slice's rescale of the chain's O and row sums (1: none)
    float lacc[kRows];                 // a chain's row sums so far
    uint32_t bits[2][kTiles][4];       // tile bitmaps, item i in stage i % 2
    int cols[2][kCols];                // source ids of the item columns, item i in slot i % 2 (-1: none)
    int4 desc[kRing][2];               // item descriptors, item i in slot i % kRing (the head in [1].w)
    unsigned long long bar_s, bar_o;
    uint32_t tmem_base;
};
static_assert(offsetof(TileSmem, v) % 1024 == 0 && offsetof(TileSmem, q) % 1024 == 0 &&
                  offsetof(TileSmem, pt) % 1024 == 0,
              "operand alignment");
static_assert(kMinCtasPerSm * (sizeof(TileSmem) + 2048) <= 228 * 1024, "CTAs per SM by shared memory");
static_assert(kMinCtasPerSm * kTmemCols <= 512, "CTAs per SM by tensor memory");

using namespace ptx;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// two floats rounded to the input type, packed (first in the low half); and
// such a pair back as floats
template <typename T>
struct Half2;
template <>
struct Half2<__nv_bfloat16> {
    __device__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static void unpack(uint32_t w, float& lo, float& hi) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    }
};
template <>
struct Half2<__half> {
    __device__ static uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static void unpack(uint32_t w, float& lo, float& hi) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
        lo = f.x;
        hi = f.y;
    }
};

template <typename OutT>
__device__ __forceinline__ void store_out(void* O, long long idx, float v);
template <>
__device__ __forceinline__ void store_out<float>(void* O, long long idx, float v) {
    __stcs(static_cast<float*>(O) + idx, v);
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(void* O, long long idx, float v) {
    static_cast<__nv_bfloat16*>(O)[idx] = __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ void store_out<__half>(void* O, long long idx, float v) {
    static_cast<__half*>(O)[idx] = __float2half_rn(v);
}

// An item descriptor: (w0, t0, T0, nwin | units0 << 8), (w1, t1, T1, head).
// Window j of the item covers rows 16 w_j .. 16 w_j + 15 and tiles t_j ..
// t_j + T_j - 1; window 1 starts at item column 16 units0.  A slice of a
// split window (kItemPartial set, one window) has (partial index of row 0,
// row stride, 0, head) in place of the second window.
__device__ __forceinline__ int item_nwin(const int4& a) { return a.w & 0xff; }
__device__ __forceinline__ int item_split(const int4& a) { return 16 * ((a.w >> 8) & 0xff); }

// Source id of item column c (-1: padding or no column).
__device__ __forceinline__ int item_column(const TileParams& p, const int4& a, const int4& b, int c) {
    const int nw = item_nwin(a);
    if (nw == 0) return -1;
    const int split = item_split(a);
    const bool second = nw == 2 && c >= split;
    const int local = second ? c - split : c;
    const int wt = second ? b.z : a.z, wy = second ? b.y : a.y;
    if (local >= kTileCols * min(wt, kTiles)) return -1;
    return p.tile_cols[(long long)wy * kTileCols + local];
}

// Reduce 16 values over the 16 lanes of a half-warp so that lane l ends with
// the reduction of every lane's x[l] (a reduce-scatter: 8 + 4 + 2 + 1
// shuffles, each lane keeping the half of its values its partner sends it).
template <bool kMax>
__device__ __forceinline__ float halfwarp_reduce_scatter(const float (&x)[16]) {
    const int l = threadIdx.x & 15;
    auto op = [](float u, float w) { return kMax ? fmaxf(u, w) : u + w; };
    float a[8], b[4], c[2];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const bool up = l & 8;
        const float got = __shfl_xor_sync(0xffffffffu, up ? x[r] : x[r + 8], 8);
        a[r] = op(up ? x[r + 8] : x[r], got);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const bool up = l & 4;
        const float got = __shfl_xor_sync(0xffffffffu, up ? a[r] : a[r + 4], 4);
        b[r] = op(up ? a[r + 4] : a[r], got);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const bool up = l & 2;
        const float got = __shfl_xor_sync(0xffffffffu, up ? b[r] : b[r + 2], 2);
        c[r] = op(up ? b[r + 2] : b[r], got);
    }
    const bool up = l & 1;
    const float got = __shfl_xor_sync(0xffffffffu, up ? c[0] : c[1], 1);
    return op(up ? c[1] : c[0], got);
}

// ---------------------------------------------------------------------------
// kChains: the flavour for plans with node-parallel split windows (its chain
// bookkeeping costs the other plans registers, so they run the one without).
template <typename T, typename OutT, bool kChains>
__global__ void __launch_bounds__(kThreads, kMinCtasPerSm) tile_kernel(const TileParams p) {
    extern __shared__ uint8_t smem_raw[];
    TileSmem& sm = *reinterpret_cast<TileSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const T* Q = static_cast<const T*>(p.Q);
    const T* K = static_cast<const T*>(p.K);
    const T* V = static_cast<const T*>(p.V);
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdescO = idesc_f16(kBf16, true, 128, kRows, true);  // A and B MN-major
    // Work indices: k H + h for item k < n_single and head h (every item on its
    // own); then, with node-parallel split windows, n_single H + j H + h for the
    // chain of split window j (its slices, consecutive items, all taken by the
    // CTA that drew the index).
    const int n_single_work = (int)(p.n_single_items * p.H);
    const int n_work = n_single_work + (kChains ? p.n_chains * p.H : 0);
    const long long node_stride = (long long)p.H * kD;
    // Roles, spread over the four warps so no warp is the others' barrier wait:
    // thread 0 polls the mbarriers and warp 0 combines the row maxima, thread 32
    // issues S^T, thread 64 issues O^T, warp 3 combines the row sums and thread
    // 96 takes work indices and loads item descriptors.
    constexpr int kIssueS = 32, kIssueO = 64, kFetcher = 96;

    // The fetcher's state: the next work index (taken from the counter one
    // item ahead) and the rest of the chain it is expanding.
    int wk_next = 0, chain_k = 0, chain_left = 0, chain_h = 0;
    // the next item's descriptor (an empty one past the end); true when it
    // took wk_next, which the caller then replaces
    auto next_desc = [&](int4& a, int4& b) {
        if (kChains && chain_left > 0) {
            a = p.tile_items[2 * chain_k];
            b = p.tile_items[2 * chain_k + 1];
            b.w = chain_h;
            ++chain_k;
            --chain_left;
            return false;
        }
        a = b = make_int4(0, 0, 0, 0);
        const int wk = wk_next;
        if (wk < n_single_work) {
            const int k = wk / p.H;
            a = p.tile_items[2 * k];
            b = p.tile_items[2 * k + 1];
            b.w = wk - k * p.H;
        } else if (kChains && wk < n_work) {
            const int j = (wk - n_single_work) / p.H;
            const int2 u = p.chains[j];  // (first slice item, slices)
            chain_h = wk - n_single_work - j * p.H;
            a = p.tile_items[2 * u.x];
            b = p.tile_items[2 * u.x + 1];
            b.w = chain_h;
            chain_k = u.x + 1;
            chain_left = u.y - 1;
        }
        return true;
    };

    if (warp == 0) tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    if (tid == 0) {
        mbar_init(smem_u32(&sm.bar_s), 1);
        mbar_init(smem_u32(&sm.bar_o), 1);
        fence_mbar_init();
    }
    if (tid == kFetcher) {
        // items 0-2 now, and the next work index (a CTA that starts late takes fewer)
        wk_next = (int)atomicAdd(p.work_counter, 1u);
#pragma unroll 1
        for (int j = 0; j < 3; ++j)
            if (next_desc(sm.desc[j][0], sm.desc[j][1])) wk_next = (int)atomicAdd(p.work_counter, 1u);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lanes
    const uint32_t kbase = smem_u32(sm.k), vbase = smem_u32(sm.v), qbase = smem_u32(sm.q),
                   ptbase = smem_u32(sm.pt);

    // K rows of an item, its Q rows and its tile bitmaps (stage bs), column ids
    // from slot cs.  Eight threads share a row (one 16-byte piece each), so a
    // warp's copy covers four whole 128-byte rows.
    auto load_kq = [&](const int4& a, const int4& b, int cs, int bs) {
        const int nw = item_nwin(a);
        if (nw == 0) return;
        const int x = tid & 7, h = b.w;
        const T* kh = K + (long long)h * kD + x * 8;  // this thread's piece of head h of node 0
        const uint32_t kdst = kbase + (tid >> 3) * 128 + ((x ^ ((tid >> 3) & 7)) << 4);
#pragma unroll
        for (int rep = 0; rep < kCols / 16; ++rep) {
            const int col = sm.cols[cs][(tid >> 3) + 16 * rep];
            if (col >= 0) cp_async16(kdst + rep * 16 * 128, kh + col * node_stride);
        }
#pragma unroll
        for (int half = 0; half < kMaxWin; ++half) {
            const int R = (tid >> 3) + kRows * half;
            const long long node = (long long)(half ? b.x : a.x) * kRows + (R & 15);
            const bool ok = half < nw && node < p.N;
            const T* qsrc = ok ? Q + (node * p.H + h) * kD + x * 8 : Q;
            cp_async16(qbase + R * 128 + ((x ^ (R & 7)) << 4), qsrc, ok ? 16u : 0u);
        }
        if (tid < kTiles) {
            const int split = item_split(a) >> 3;
            const bool second = nw == 2 && tid >= split;
            const int t = second ? tid - split : tid;
            const int wt = second ? b.z : a.z, wy = second ? b.y : a.y;
            if (t < min(wt, kTiles)) cp_async16(smem_u32(&sm.bits[bs][tid][0]), p.tile_bits + ((long long)wy + t) * 4);
        }
    };
    // V rows of an item: every column of each window's 16-column MMA steps,
    // padding ones zero-filled (their P is 0, and 0 * stale data could be NaN)
    auto load_v = [&](const int4& a, const int4& b, int cs) {
        const int nw = item_nwin(a);
        if (nw == 0) return;
        const int x = tid & 7;
        const int used = item_split(a) + (nw == 2 ? 16 * ((min(b.z, kTiles) + 1) / 2) : 0);
        const T* vh = V + (long long)b.w * kD + x * 8;
        const uint32_t vdst = vbase + (tid >> 3) * 128 + ((x ^ ((tid >> 3) & 7)) << 4);
#pragma unroll
        for (int rep = 0; rep < kCols / 16; ++rep) {
            const int c = (tid >> 3) + 16 * rep;
            if (c < used) {
                const int col = sm.cols[cs][c];
                cp_async16(vdst + rep * 16 * 128, col >= 0 ? vh + col * node_stride : V, col >= 0 ? 16u : 0u);
            }
        }
    };
    // S^T = K Q^T of an item into TMEM columns [0, 16 nw)
    auto issue_s = [&](const int4& a) {
        const uint32_t idesc = idesc_f16(kBf16, false, 128, kRows * item_nwin(a));
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
            mma_f16(tmem, sdesc_sw128(kbase + kk * 32, 16, 1024), sdesc_sw128(qbase + kk * 32, 16, 1024), idesc,
                    kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&sm.bar_s));
    };
    // read back O^T of an item, normalise and store its windows' rows: TMEM
    // lanes 0-63 and again 64-127 hold the 64 features; warps 0 and 1 take
    // rows 0-7 of each window, warps 2 and 3 rows 8-15, 32 features per warp.
    auto epilogue = [&](const int4& a, const int4& b) {
        if (kChains && (a.w & kItemChain) && b.x != b.y - 1) return;  // a chain's rows are stored after its last slice
        const int nw = item_nwin(a);
        const int f = (warp & 1) * 32 + (tid & 31);
        const int r0 = (warp >> 1) * 8;
        if (a.w & kItemPartial) {
            // a split window's slice: the unnormalised rows, and (row max in the
            // log2 domain, row sum) per row, -inf for a row without entries here
            float o[kRows];
            tmem_ld16(tmem + 32 + lane_base, o);
            const long long rows_left = p.N - ((long long)a.x * kRows + r0);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float v = r0 == 0 ? o[r] : o[8 + r];  // static register indices
                if (r < rows_left) {
                    const long long idx = (long long)b.x + (long long)(r0 + r) * b.y;
                    __stcs(p.part_acc + idx * node_stride + (long long)b.w * kD + f, v);
                    if (f == 0) {
                        const float l = sm.rowsum[r0 + r];
                        const float2 ml = make_float2(l > 0.f ? sm.rowmax[r0 + r] : -INFINITY, l);
                        *reinterpret_cast<float2*>(p.part_ml + idx * 2 * p.H + 2 * b.w) = ml;
                    }
                }
            }
            return;
        }
        for (int j = 0; j < nw; ++j) {
            float o[kRows];
            tmem_ld16(tmem + 32 + 16 * j + lane_base, o);
            const long long node0 = (long long)(j ? b.x : a.x) * kRows + r0;
            const long long rows_left = p.N - node0;
            OutT* dst = static_cast<OutT*>(p.O) + (node0 * p.H + b.w) * kD + f;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float v = r0 == 0 ? o[r] : o[8 + r];  // static register indices
                if (r < rows_left) store_out<OutT>(dst, r * node_stride, v * sm.inv_l[kRows * j + r0 + r]);
            }
        }
    };

    // column ids of items 0 and 1, then item 0's K, Q and bitmaps and its S^T
    sm.cols[0][tid] = item_column(p, sm.desc[0][0], sm.desc[0][1], tid);
    sm.cols[1][tid] = item_column(p, sm.desc[1][0], sm.desc[1][1], tid);
    __syncthreads();
    load_kq(sm.desc[0][0], sm.desc[0][1], 0, 0);
    cp_async_commit();
    cp_async_wait_group<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == kIssueS && item_nwin(sm.desc[0][0]) > 0) issue_s(sm.desc[0][0]);
    const float scale = p.scale_log2;
    const int hw = tid >> 4;  // this thread's half-warp: columns 16 hw .. 16 hw + 15
    bool failed = false;
    int done = 0;  // items whose O^T was issued

    // Work indices are taken from one counter in increasing order, so the first
    // empty item ends the CTA's sequence.
    for (int i = 0;; ++i) {
        const int4 a0 = sm.desc[i % kRing][0], b0 = sm.desc[i % kRing][1];
        const int nw = item_nwin(a0);
        if (nw == 0) break;
        // (a) S^T of item i and O^T of item i-1 complete: K, Q, V and P^T are free
        {
            bool ok = true;
            if (tid == 0) {
                if (i > 0) ok = mbar_wait_bounded_sleep(smem_u32(&sm.bar_o), (uint32_t)((i - 1) & 1), kWaitLimitNs);
                if (ok) ok = mbar_wait_bounded_sleep(smem_u32(&sm.bar_s), (uint32_t)(i & 1), kWaitLimitNs);
            }
            if (__syncthreads_or(!ok)) {
                failed = true;
                break;
            }
            tc_fence_after();
        }
        // the fetcher: the descriptor of item i+3 (and a new work index when it
        // took the last one)
        int4 fa = make_int4(0, 0, 0, 0), fb = fa;
        bool took = false;
        int grab = 0;
        if (tid == kFetcher) {
            took = next_desc(fa, fb);
            if (took) grab = (int)atomicAdd(p.work_counter, 1u);
        }
        // (b) item i+1's K, Q and bitmaps, then item i's V rows
        const int4 a1 = sm.desc[(i + 1) % kRing][0], b1 = sm.desc[(i + 1) % kRing][1];
        load_kq(a1, b1, (i + 1) & 1, (i + 1) & 1);
        cp_async_commit();
        load_v(a0, b0, i & 1);
        cp_async_commit();
        // (c) item i-1's rows
        if (i > 0) epilogue(sm.desc[(i - 1) % kRing][0], sm.desc[(i - 1) % kRing][1]);
        // this thread's column id of item i+2 (stored at the end of the iteration)
        const int col2 = item_column(p, sm.desc[(i + 2) % kRing][0], sm.desc[(i + 2) % kRing][1], tid);

        // (d) this thread's column of item i's logits, masked and scaled
        const int c = tid;
        const int split = item_split(a0);
        const bool second = nw == 2 && c >= split;
        float x[kRows];
        {
            float t16[kRows];
            tmem_ld16(tmem + lane_base, t16);  // warp-collective: window 0's rows, every column
#pragma unroll
            for (int r = 0; r < kRows; ++r) x[r] = t16[r];
        }
        if (nw == 2) {
            float t16[kRows];
            tmem_ld16(tmem + 16 + lane_base, t16);  // window 1's rows
            if (second) {
#pragma unroll
                for (int r = 0; r < kRows; ++r) x[r] = t16[r];
            }
        }
        {
            const uint4 bw = *reinterpret_cast<const uint4*>(&sm.bits[i & 1][c >> 3][0]);
            const bool live = sm.cols[i & 1][c] >= 0;
            const uint32_t w4[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const bool on = live && ((w4[r >> 2] >> ((r & 3) * 8 + (c & 7))) & 1u);
                x[r] = on ? x[r] : -INFINITY;  // unscaled: the scale goes into the maxima and the exponent
            }
        }
        // (e) row maxima: per half-warp, then over the half-warps of each window.  A
        // slice of a chain (a split window taken node-parallel, one window) keeps a
        // reference max per row over its slices, moved only when a slice's max
        // exceeds it by more than 2^8; O and the row sums are rescaled then.
        const bool chain = kChains && (a0.w & kItemChain);
        const bool chain_first = chain && b0.x == 0;
        sm.part[hw][tid & 15] = halfwarp_reduce_scatter<true>(x);
        tc_fence_before();
        __syncthreads();
        int rescale = 0;
        if (tid < kItemRows) {
            const int j = tid >> 4, r = tid & 15;
            float m = -INFINITY;
#pragma unroll
            for (int g = 0; g < kHalfWarps; ++g)
                if ((nw == 2 && 16 * g >= split) == (j == 1)) m = fmaxf(m, sm.part[g][r]);
            m *= scale;  // log2 domain (scale > 0 keeps the max)
            if (chain && tid < kRows) {
                const float mref = chain_first ? -INFINITY : sm.mref[tid];
                const float mnew = m > mref + kLazyRescale ? m : mref;
                const float f = mnew == mref ? 1.f : ex2(mref - mnew);
                sm.mref[tid] = mnew;
                sm.fac[tid] = f;
                rescale = !chain_first && f != 1.f;
                m = mnew;
            }
            sm.rowmax[tid] = m == -INFINITY ? 0.f : m;  // a row without entries: every P is 0
        }
        cp_async_wait_group<1>();  // item i+1's K, Q and bitmaps (item i's V may still be in flight)
        fence_proxy_async_smem();
        if constexpr (kChains)
            rescale = __syncthreads_or(rescale);
        else
            __syncthreads();
        tc_fence_after();
        if (tid == kIssueS && item_nwin(a1) > 0) issue_s(a1);  // runs while item i forms P
        if (kChains && rescale) {  // CTA-uniform: the chain's O rows (TMEM columns) times their factors
            float o[kRows];
            tmem_ld16(tmem + 32 + lane_base, o);
#pragma unroll
            for (int r = 0; r < kRows; ++r) o[r] *= sm.fac[r];
            tmem_st16(tmem + 32 + lane_base, o);
        }
        // (f) this column's 16 values of P, one 32-byte row of P^T (rows 0-7 and 8-15 in
        // the two 16-byte halves, swapped on every other group of four columns), and
        // the row sums of the rounded values
        {
            const float4* mr = reinterpret_cast<const float4*>(&sm.rowmax[second ? kRows : 0]);
            uint32_t w[8];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float4 m = mr[q4];
                w[2 * q4] = Half2<T>::pack(ex2(fmaf(x[4 * q4], scale, -m.x)), ex2(fmaf(x[4 * q4 + 1], scale, -m.y)));
                w[2 * q4 + 1] =
                    Half2<T>::pack(ex2(fmaf(x[4 * q4 + 2], scale, -m.z)), ex2(fmaf(x[4 * q4 + 3], scale, -m.w)));
            }
            const uint32_t row = ptbase + c * 32, sw = (uint32_t)((c >> 2) & 1) << 4;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + sw), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (sw ^ 16u)), "r"(w[4]), "r"(w[5]),
                         "r"(w[6]), "r"(w[7])
                         : "memory");
#pragma unroll
            for (int q = 0; q < 8; ++q) Half2<T>::unpack(w[q], x[2 * q], x[2 * q + 1]);
            sm.part[hw][tid & 15] = halfwarp_reduce_scatter<false>(x);
        }
        // (g) item i's V rows; O^T = V^T P^T per window, over its columns 16 at a time
        cp_async_wait_group<0>();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == kIssueO) {
            for (int j = 0; j < nw; ++j) {
                const int c0 = j ? split : 0;
                const int ksteps = j ? (min(b0.z, kTiles) + 1) / 2 : split / 16;
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint32_t va = vbase + (uint32_t)(c0 + 16 * kk) * 128;
                    mma_f16(tmem + 32 + 16 * j, sdesc_sw128(va, 0, 1024),
                            sdesc_sw32(ptbase + (uint32_t)(c0 + 16 * kk) * 32, 0, 256), kIdescO,
                            kk > 0 || (chain && !chain_first) ? 1u : 0u);
                }
            }
            mma_commit(smem_u32(&sm.bar_o));
        }
        if (warp == 3) {
            const int t = tid - 96, j = t >> 4, r = t & 15;
            float l = 0.f;
#pragma unroll
            for (int g = 0; g < kHalfWarps; ++g)
                if ((nw == 2 && 16 * g >= split) == (j == 1)) l += sm.part[g][r];
            if (chain && t < kRows) {
                if (!chain_first) l += sm.lacc[t] * sm.fac[t];
                sm.lacc[t] = l;
            }
            sm.inv_l[t] = l > 0.f ? 1.0f / l : 0.f;
            sm.rowsum[t] = l;
        }
        // read after the next iteration's first barrier
        sm.cols[i & 1][tid] = col2;
        if (tid == kFetcher) {
            sm.desc[(i + 3) % kRing][0] = fa;
            sm.desc[(i + 3) % kRing][1] = fb;
            if (took) wk_next = grab;
        }
        ++done;
    }
    if (!failed && done > 0) {
        bool ok = true;
        if (tid == 0) ok = mbar_wait_bounded_sleep(smem_u32(&sm.bar_o), (uint32_t)((done - 1) & 1), kWaitLimitNs);
        if (__syncthreads_or(!ok)) {
            failed = true;
        } else {
            tc_fence_after();
            epilogue(sm.desc[(done - 1) % kRing][0], sm.desc[(done - 1) % kRing][1]);
        }
    }
    cp_async_wait_all();
    if (failed && tid == 0) atomicOr(p.status, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Self-test of the bounded wait: one CTA waits on an mbarrier that nothing
// arrives at, gives up after limit_ns, and reports it through *status the way
// the tile kernel does.
__global__ void wait_selftest_kernel(unsigned long long limit_ns, int32_t* status) {
    __shared__ unsigned long long mbar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&mbar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(smem_u32(&mbar), 0, limit_ns);
    if (__syncthreads_or(!ok) && threadIdx.x == 0) atomicOr(status, kErrTimeout);
}

template <typename T, typename OutT, bool kChains>
cudaError_t launch_flavour(const TileParams& p, cudaStream_t st) {
    const long long work = (p.n_single_items + p.n_chains) * p.H;
    if (work <= 0) return cudaSuccess;
    // work indices are 32-bit (one counter, every CTA taking a few past the end)
    if (work > (1ll << 30)) return cudaErrorInvalidValue;
    const size_t smem = sizeof(TileSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(tile_kernel<T, OutT, kChains>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // all of the SM's unified L1/shared storage as shared memory, so five CTAs fit
    e = cudaFuncSetAttribute(tile_kernel<T, OutT, kChains>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    // resident CTAs per SM from shared memory, registers and TMEM (the
    // occupancy query does not see the carveout set above)
    int dev = 0, sms = 0, smem_sm = 0, reserved = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, tile_kernel<T, OutT, kChains>)) != cudaSuccess) return e;
    int per_sm = smem_sm / (int)(smem + reserved);
    const int regs = (fa.numRegs + 7) / 8 * 8 * kThreads;
    if (regs > 0 && 65536 / regs < per_sm) per_sm = 65536 / regs;
    if ((int)(512 / kTmemCols) < per_sm) per_sm = (int)(512 / kTmemCols);
    if (per_sm < 1) per_sm = 1;
    long long grid = (long long)sms * (per_sm > 0 ? per_sm : 1);
    if (grid > work) grid = work;
    tile_kernel<T, OutT, kChains><<<(unsigned)grid, kThreads, smem, st>>>(p);
    return cudaGetLastError();
}

template <typename T, typename OutT>
cudaError_t launch(const TileParams& p, cudaStream_t st) {
    return p.n_chains > 0 ? launch_flavour<T, OutT, true>(p, st) : launch_flavour<T, OutT, false>(p, st);
}

}  // namespace

cudaError_t wait_selftest_launch(unsigned long long limit_ns, int32_t* status, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns, status);
    return cudaGetLastError();
}

bool tile_supported(int dtype, int variant, int head_dim) {
    return (dtype == G3S_F16 || dtype == G3S_BF16) && variant == G3S_STANDARD && head_dim == kD;
}

cudaError_t tile_launch(int dtype, int out_dtype, const TileParams& p, cudaStream_t st) {
    if (dtype == G3S_BF16) {
        if (out_dtype == G3S_F32) return launch<__nv_bfloat16, float>(p, st);
        if (out_dtype == G3S_BF16) return launch<__nv_bfloat16, __nv_bfloat16>(p, st);
    } else if (dtype == G3S_F16) {
        if (out_dtype == G3S_F32) return launch<__half, float>(p, st);
        if (out_dtype == G3S_F16) return launch<__half, __half>(p, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace g3s
