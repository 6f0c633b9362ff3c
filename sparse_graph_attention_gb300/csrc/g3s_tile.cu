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
// thread issues S^T into TMEM; each thread reads its column of S^T (the 16
// logits of its window's rows) and masks it by the tile bitmap.  The row
// maxima need all of a window's columns: the scaled logits go through a
// transposed buffer where eight threads per row take the max and the row
// sum of P = 2^(s - m) rounded to the input type.  A window has at most 128
// columns, so the max is final before any P is formed and the softmax needs
// no online rescale.  Each column's thread then forms its own 16 values of P
// (the same rounded values the row sums were taken over) and writes them as
// one 32-byte row of P^T, the MN-major B operand of the second product.  O^T
// uses the V rows as its MN-major A operand; its 64 feature rows are issued
// as M = 128 with the second half reading the same rows again (atom stride
// 0), so TMEM lanes 64-127 repeat lanes 0-63 and all four warps store rows.
//
// Pipeline (persistent CTAs, three per SM, static item order): K, Q and the
// bitmaps are double-buffered and V single-buffered; S^T is double-buffered
// in TMEM.  Item i+1's S^T is issued as soon as item i's logits are out of
// TMEM, and item i+2's K, Q and bitmaps are requested once item i's row maxima
// are done (the transposed logits live in item i's K buffer), so both have a
// whole item's time to complete; item i's V rows are requested once O^T of
// item i-1 is done, and arrive while item i-1's rows are stored and item i
// goes through its softmax.  Item descriptors and column ids are loaded three
// and two items ahead.  Every mbarrier wait is bounded (about one second of
// %globaltimer); on expiry the CTA sets the plan's status word, frees its TMEM
// and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstddef>
#include <type_traits>

#include "g3s_internal.h"
#include "g3s_ptx.cuh"

namespace g3s {
namespace {

constexpr int kThreads = 128;
constexpr int kD = 64;                         // head_dim of this kernel
constexpr int kRows = kWinRows;                // 16 rows per window: the N of a window
constexpr int kCols = kTileItemUnits * 16;     // 128 item columns: the MMA's M
constexpr int kTiles = kCols / kTileCols;      // 16 tile slots per item
constexpr int kMaxWin = 2;                     // windows per item
constexpr int kItemRows = kMaxWin * kRows;     // 32
constexpr int kXtPitch = 20;                   // words per column of the transposed logits (16 used)
constexpr uint32_t kTmemCols = 128;            // S^T by item parity [0, 32) and [32, 64), O^T [64, 96)
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

struct TileSmem {
    uint8_t k[2][kCols * 128];         // K rows by stage: K-major A operand of S^T; then the transposed logits
    uint8_t v[kCols * 128];            // V rows: MN-major A operand of O^T (M rows 0-63)
    uint8_t q[2][kItemRows * 128];     // Q rows by stage (row 16 j + r of window j): K-major B operand of S^T
    uint8_t pt[kCols * 32];            // P^T: [column][16 rows of its window], MN-major B operand, 32-byte swizzle
    float rowmax[kItemRows];           // row maxima of the item's windows (row 16 j + r)
    float inv_l[kItemRows];            // 1 / row sum of P (0 for a row without entries)
    uint32_t bits[2][kTiles][4];       // tile bitmaps by stage and item tile slot
    int cols[3][kCols];                // source ids of the item columns, item i in slot i % 3 (-1: none)
    int ring[8];                       // work indices of this CTA's items, item j in slot j % 8
    unsigned long long bar_s, bar_o;
    uint32_t tmem_base;
};
static_assert(sizeof(TileSmem) + 1024 <= 75 * 1024, "three CTAs per SM");
static_assert(kCols * kXtPitch * 4 <= kCols * 128, "transposed logits fit a K stage");
static_assert(offsetof(TileSmem, pt) % 1024 == 0, "operand alignment");

using namespace ptx;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// two floats rounded to the input type, packed (first in the low half); and
// one float rounded to it, back as a float
template <typename T>
struct Half2;
template <>
struct Half2<__nv_bfloat16> {
    __device__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static float round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
};
template <>
struct Half2<__half> {
    __device__ static uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static float round(float x) { return __half2float(__float2half_rn(x)); }
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

// An item: its windows (w, first tile, tiles), the 16-column units of window
// 0 (window 1 starts there) and the head.
struct Item {
    int4 a, b;  // (w0, t0, T0, nwin | units0 << 8), (w1, t1, T1, 0)
    int h;
    __device__ int nwin() const { return a.w & 0xff; }
    __device__ int units0() const { return a.w >> 8; }
};

// ---------------------------------------------------------------------------
template <typename T, typename OutT>
__global__ void __launch_bounds__(kThreads) tile_kernel(const TileParams p) {
    extern __shared__ uint8_t smem_raw[];
    TileSmem& sm = *reinterpret_cast<TileSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const T* Q = static_cast<const T*>(p.Q);
    const T* K = static_cast<const T*>(p.K);
    const T* V = static_cast<const T*>(p.V);
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdescO = idesc_f16(kBf16, true, 128, kRows, true);  // A and B MN-major
    const int n_work = (int)(p.n_tile_items * p.H);  // work index k H + h: item k, head h

    if (warp == 0) tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    if (tid == 0) {
        mbar_init(smem_u32(&sm.bar_s), 1);
        mbar_init(smem_u32(&sm.bar_o), 1);
        fence_mbar_init();
        // the first five work indices of this CTA (a CTA that starts late takes fewer)
#pragma unroll
        for (int j = 0; j < 5; ++j) sm.ring[j] = (int)atomicAdd(p.work_counter, 1u);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lanes

    // Wait for an MMA commit: thread 0 polls the mbarrier (bounded), the
    // other threads block in the CTA barrier, which issues nothing, instead of
    // spinning beside the other CTAs of the SM.  False when the wait gave up.
    auto cta_wait = [&](uint32_t bar, uint32_t parity) {
        bool ok = true;
        if (tid == 0) ok = mbar_wait_bounded_sleep(bar, parity, kWaitLimitNs);
        return __syncthreads_or(!ok) == 0;
    };
    // item j of this CTA from its work index in the ring (a zero item past the end)
    auto fetch_item = [&](int j) {
        Item it;
        it.a = it.b = make_int4(0, 0, 0, 0);
        it.h = 0;
        const int wk = sm.ring[j & 7];
        if (wk < n_work) {
            const int k = wk / p.H;
            it.h = wk - k * p.H;
            it.a = p.tile_items[2 * k];
            it.b = p.tile_items[2 * k + 1];
        }
        return it;
    };
    // source id of item column c (-1: padding or no column)
    auto column_of = [&](const Item& it, int c) {
        const int nw = it.nwin();
        if (nw == 0) return -1;
        const int split = 16 * it.units0();
        const bool second = nw == 2 && c >= split;
        const int local = second ? c - split : c;
        const int wt = second ? it.b.z : it.a.z, wy = second ? it.b.y : it.a.y;
        if (local >= kTileCols * min(wt, kTiles)) return -1;
        return p.tile_cols[(long long)wy * kTileCols + local];
    };
    // K rows of the item, its Q rows and its tile bitmaps into stage s.  Eight
    // threads share a row (one 16-byte piece each), so a warp's copy covers
    // four whole 128-byte rows; the column ids come from slot cs.
    auto load_kq = [&](const Item& it, int cs, int s) {
        const int nw = it.nwin();
        if (nw == 0) return;
        const int x = tid & 7;
        const T* kh = K + (long long)it.h * kD + x * 8;  // this thread's piece of head h of node 0
        const long long node_stride = (long long)p.H * kD;
        const uint32_t kdst = smem_u32(sm.k[s]) + (tid >> 3) * 128 + ((x ^ ((tid >> 3) & 7)) << 4);
#pragma unroll
        for (int rep = 0; rep < kCols / 16; ++rep) {
            const int col = sm.cols[cs][(tid >> 3) + 16 * rep];
            if (col >= 0) cp_async16(kdst + rep * 16 * 128, kh + col * node_stride);
        }
#pragma unroll
        for (int half = 0; half < kMaxWin; ++half) {
            const int R = (tid >> 3) + kRows * half;
            const long long node = (long long)(half ? it.b.x : it.a.x) * kRows + (R & 15);
            const bool ok = half < nw && node < p.N;
            const T* qsrc = ok ? Q + (node * p.H + it.h) * kD + x * 8 : Q;
            cp_async16(smem_u32(sm.q[s]) + R * 128 + ((x ^ (R & 7)) << 4), qsrc, ok ? 16u : 0u);
        }
        if (tid < kTiles) {
            const int split = 2 * it.units0();
            const bool second = nw == 2 && tid >= split;
            const int t = second ? tid - split : tid;
            const int wt = second ? it.b.z : it.a.z, wy = second ? it.b.y : it.a.y;
            if (t < min(wt, kTiles)) cp_async16(smem_u32(&sm.bits[s][tid][0]), p.tile_bits + ((long long)wy + t) * 4);
        }
    };
    // V rows of the item: every column of each window's 16-column MMA steps,
    // padding ones zero-filled (their P is 0, and 0 * stale data could be NaN)
    auto load_v = [&](const Item& it, int cs) {
        const int nw = it.nwin();
        if (nw == 0) return;
        const int x = tid & 7;
        const int used = 16 * (it.units0() + (nw == 2 ? (min(it.b.z, kTiles) + 1) / 2 : 0));
        const T* vh = V + (long long)it.h * kD + x * 8;
        const long long node_stride = (long long)p.H * kD;
        const uint32_t vdst = smem_u32(sm.v) + (tid >> 3) * 128 + ((x ^ ((tid >> 3) & 7)) << 4);
#pragma unroll
        for (int rep = 0; rep < kCols / 16; ++rep) {
            const int c = (tid >> 3) + 16 * rep;
            if (c < used) {
                const int col = sm.cols[cs][c];
                cp_async16(vdst + rep * 16 * 128, col >= 0 ? vh + col * node_stride : V, col >= 0 ? 16u : 0u);
            }
        }
    };
    // read back O^T of an item, normalise and store its windows' rows: TMEM
    // lanes 0-63 and again 64-127 hold the 64 features; warps 0 and 1 take
    // rows 0-7 of each window, warps 2 and 3 rows 8-15, 32 features per warp.
    auto epilogue = [&](const Item& it) {
        const int nw = it.nwin();
        const int f = (warp & 1) * 32 + (tid & 31);
        const int r0 = (warp >> 1) * 8;
        const long long stride = (long long)p.H * kD;
        for (int j = 0; j < nw; ++j) {
            float o[kRows];
            tmem_ld16(tmem + 64 + 16 * j + lane_base, o);
            const long long node0 = (long long)(j ? it.b.x : it.a.x) * kRows + r0;
            const long long rows_left = p.N - node0;
            OutT* dst = static_cast<OutT*>(p.O) + (node0 * p.H + it.h) * kD + f;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float v = r0 == 0 ? o[r] : o[8 + r];  // static register indices
                if (r < rows_left) store_out<OutT>(dst, r * stride, v * sm.inv_l[kRows * j + r0 + r]);
            }
        }
    };

    // descriptors of items i .. i+3 and this thread's column ids of items i .. i+2
    Item it0 = fetch_item(0), it1 = fetch_item(1), it2 = fetch_item(2), it3 = fetch_item(3);
    int col0 = column_of(it0, tid), col1 = column_of(it1, tid), col2 = column_of(it2, tid);
    Item itp = it0;  // the previous item (for its epilogue)
    sm.cols[0][tid] = col0;
    sm.cols[1][tid] = col1;
    __syncthreads();
    // cp.async groups, oldest first: KQ(0), KQ(1), then per item i: V(i), KQ(i+2).
    load_kq(it0, 0, 0);
    cp_async_commit();
    load_kq(it1, 1, 1);
    cp_async_commit();
    const float scale = p.scale_log2;
    const uint32_t vbase = smem_u32(sm.v), ptbase = smem_u32(sm.pt);
    // S^T = K Q^T of an item from K/Q stage ks into TMEM S buffer ks (columns [32 ks, 32 ks + 16 nw))
    auto issue_s = [&](const Item& it, int ks) {
        const uint32_t idesc = idesc_f16(kBf16, false, 128, kRows * it.nwin());
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
            mma_f16(tmem + 32 * ks, sdesc_sw128(smem_u32(sm.k[ks]) + kk * 32, 16, 1024),
                    sdesc_sw128(smem_u32(sm.q[ks]) + kk * 32, 16, 1024), idesc, kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&sm.bar_s));
    };
    cp_async_wait_group<1>();  // item 0's K, Q and bitmaps
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && it0.nwin() > 0) issue_s(it0, 0);
    bool failed = false;
    int done = 0;  // items this CTA has finished

    // Work indices are taken from one counter in increasing order, so the first
    // empty item ends the CTA's sequence.
    for (int i = 0; it0.nwin() > 0; ++i) {
        // the work index of item i+5, stored at the end of this iteration
        int grab = 0;
        if (tid == 96) grab = (int)atomicAdd(p.work_counter, 1u);
        const int s = i & 1;
        const int cs = i % 3;
        sm.cols[(i + 2) % 3][tid] = col2;  // slot last read by item i-1's V copies, before the next barrier
        const int nw = it0.nwin();
        const int split = 16 * it0.units0();  // first column of window 1
        // (c) O^T of item i-1 complete: V and P^T are free.  Item i's V rows are
        // requested and item i-1's rows stored.
        {
            // thread 0 also takes item i's S^T (issued during item i-1, normally done by
            // now), so one barrier serves both waits
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
        load_v(it0, cs);
        cp_async_commit();
        if (i > 0) epilogue(itp);
        // column ids of item i+3 and the descriptor of item i+4, for the next iterations
        const int col3 = column_of(it3, tid);
        const Item it4 = fetch_item(i + 4);

        // (d) this thread's column of item i's logits, masked and scaled
        const int c = tid;
        const bool second = nw == 2 && c >= split;
        float x[kRows];
        {
            float t16[kRows];
            tmem_ld16(tmem + 32 * s + lane_base, t16);  // warp-collective: window 0's rows, every column
#pragma unroll
            for (int r = 0; r < kRows; ++r) x[r] = t16[r];
        }
        if (nw == 2) {
            float t16[kRows];
            tmem_ld16(tmem + 32 * s + 16 + lane_base, t16);  // window 1's rows
            if (second) {
#pragma unroll
                for (int r = 0; r < kRows; ++r) x[r] = t16[r];
            }
        }
        {
            uint4 b = make_uint4(0u, 0u, 0u, 0u);
            if (col0 >= 0) b = *reinterpret_cast<const uint4*>(&sm.bits[s][c >> 3][0]);
            const uint32_t w4[4] = {b.x, b.y, b.z, b.w};
            float* xt = reinterpret_cast<float*>(sm.k[s]);  // [column][kXtPitch]
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const bool on = (w4[r >> 2] >> ((r & 3) * 8 + (c & 7))) & 1u;
                x[r] = on ? x[r] * scale : -INFINITY;
            }
            float4* dst = reinterpret_cast<float4*>(xt + c * kXtPitch);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_float4(x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
        }
        cp_async_wait_group<1>();  // item i+1's K, Q and bitmaps (only item i's V may still be in flight)
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();  // transposed logits complete; S^T, item i's Q and bitmaps are no longer read
        tc_fence_after();
        if (tid == 0 && it1.nwin() > 0) issue_s(it1, s ^ 1);  // runs while item i goes through its softmax
        // (d2) row maxima and row sums of the rounded P: eight threads per row over
        // the item's columns 8 at a time (column 8 k + part)
        {
            const int r = tid >> 3, part = tid & 7;
            const int ksplit = split >> 3;
            const int nsteps = ksplit + (nw == 2 ? 2 * ((min(it0.b.z, kTiles) + 1) / 2) : 0);
            const float* xt = reinterpret_cast<const float*>(sm.k[s]);
            float xs[2 * kTileItemUnits];
            float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
            for (int k = 0; k < 2 * kTileItemUnits; ++k) {
                xs[k] = k < nsteps ? xt[(8 * k + part) * kXtPitch + r] : -INFINITY;
                if (k < ksplit)
                    m0 = fmaxf(m0, xs[k]);
                else
                    m1 = fmaxf(m1, xs[k]);
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
                m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
            }
            if (m0 == -INFINITY) m0 = 0.f;  // a row without entries: every P is 0
            if (m1 == -INFINITY) m1 = 0.f;
            float l0 = 0.f, l1 = 0.f;
#pragma unroll
            for (int k = 0; k < 2 * kTileItemUnits; ++k) {
                if (k < ksplit)
                    l0 += Half2<T>::round(ex2(xs[k] - m0));
                else
                    l1 += Half2<T>::round(ex2(xs[k] - m1));
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, o);
                l1 += __shfl_xor_sync(0xffffffffu, l1, o);
            }
            if (part == 0) {
                sm.rowmax[r] = m0;
                sm.rowmax[kRows + r] = m1;
                sm.inv_l[r] = l0 > 0.f ? 1.0f / l0 : 0.f;
                sm.inv_l[kRows + r] = l1 > 0.f ? 1.0f / l1 : 0.f;
            }
        }
        __syncthreads();  // row maxima published; item i's K stage is free
        // (e) item i+2's K, Q and bitmaps into stage s
        load_kq(it2, (i + 2) % 3, s);
        cp_async_commit();
        // (f) this column's 16 values of P, one 32-byte row of P^T (rows 0-7 and 8-15 in
        // the two 16-byte halves, swapped on every other group of four columns)
        {
            const float4* mr = reinterpret_cast<const float4*>(&sm.rowmax[second ? kRows : 0]);
            uint32_t w[8];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float4 m = mr[q4];
                w[2 * q4] = Half2<T>::pack(ex2(x[4 * q4] - m.x), ex2(x[4 * q4 + 1] - m.y));
                w[2 * q4 + 1] = Half2<T>::pack(ex2(x[4 * q4 + 2] - m.z), ex2(x[4 * q4 + 3] - m.w));
            }
            const uint32_t row = ptbase + c * 32, sw = (uint32_t)((c >> 2) & 1) << 4;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + sw), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (sw ^ 16u)), "r"(w[4]), "r"(w[5]),
                         "r"(w[6]), "r"(w[7])
                         : "memory");
        }
        // (g) item i's V rows; O^T = V^T P^T per window, over its columns 16 at a time
        cp_async_wait_group<1>();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            for (int j = 0; j < nw; ++j) {
                const int c0 = j ? split : 0;
                const int ksteps = j ? (min(it0.b.z, kTiles) + 1) / 2 : it0.units0();
                for (int kk = 0; kk < ksteps; ++kk) {
                    const uint32_t va = vbase + (uint32_t)(c0 + 16 * kk) * 128;
                    mma_f16(tmem + 64 + 16 * j, sdesc_sw128(va, 0, 1024),
                            sdesc_sw32(ptbase + (uint32_t)(c0 + 16 * kk) * 32, 0, 256), kIdescO, kk > 0 ? 1u : 0u);
                }
            }
            mma_commit(smem_u32(&sm.bar_o));
        }
        if (tid == 96) sm.ring[(i + 5) & 7] = grab;  // read by fetch_item(i + 5) after the next barriers
        ++done;
        itp = it0;
        it0 = it1;
        it1 = it2;
        it2 = it3;
        it3 = it4;
        col0 = col1;
        col1 = col2;
        col2 = col3;
    }
    if (!failed && done > 0) {
        if (!cta_wait(smem_u32(&sm.bar_o), (uint32_t)((done - 1) & 1))) {
            failed = true;
        } else {
            tc_fence_after();
            epilogue(itp);
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

template <typename T, typename OutT>
cudaError_t launch(const TileParams& p, cudaStream_t st) {
    if (p.n_tile_items <= 0) return cudaSuccess;
    const size_t smem = sizeof(TileSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(tile_kernel<T, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // all of the SM's unified L1/shared storage as shared memory, so three CTAs fit
    e = cudaFuncSetAttribute(tile_kernel<T, OutT>, cudaFuncAttributePreferredSharedMemoryCarveout,
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
    if ((e = cudaFuncGetAttributes(&fa, tile_kernel<T, OutT>)) != cudaSuccess) return e;
    int per_sm = smem_sm / (int)(smem + reserved);
    const int regs = (fa.numRegs + 7) / 8 * 8 * kThreads;
    if (regs > 0 && 65536 / regs < per_sm) per_sm = 65536 / regs;
    if ((int)(512 / kTmemCols) < per_sm) per_sm = (int)(512 / kTmemCols);
    if (per_sm < 1) per_sm = 1;
    const long long work = p.n_tile_items * p.H;
    long long grid = (long long)sms * (per_sm > 0 ? per_sm : 1);
    if (grid > work) grid = work;
    tile_kernel<T, OutT><<<(unsigned)grid, kThreads, smem, st>>>(p);
    return cudaGetLastError();
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
