// Tensor-core tile path: fused SDDMM -> masked softmax -> SpMM over the BSB
// tiles of dense row windows, with tcgen05.mma accumulating in TMEM.
//
// Source: the Fused3S design (sciencestack.ai/paper/2505.08098): a 16-row
// window is compacted to its unique source columns and tiled into 16x8 tiles
// with bitmaps (Figure 1); one thread block owns a window's Q and O rows
// (node-parallel, Figure 2); SDDMM, softmax and SpMM stay on chip with an
// online softmax (TL;DR).  Its warp-level MMA layout is not reused: on sm_103a
// one thread issues tcgen05.mma for the whole CTA and the accumulators live
// in tensor memory.
//
// Mapping.  A CTA (4 warps, 128 threads) takes one group of up to 8 tile
// windows and one head.  The 8 x 16 window rows stack into the 128 rows of
// the MMA; the group's tiles are concatenated (window by window) and walked
// 64 columns (8 tiles) at a time:
//   1. cp.async gathers the K and V rows of the 64 columns (head h, d = 64)
//      into 128-byte-swizzled shared memory (Q rows once per CTA); the
//      gathers of the next chunk (two buffers) and the column ids and bitmaps
//      of the chunk after it (three buffers) are in flight while this chunk
//      is computed;
//   2. S = Q K^T (M=128, N=64, K=64) into TMEM columns [0, 64);
//   3. thread i reads row i of S, masks entries outside its own window's
//      tiles or absent from the bitmap, updates its running max / sum and
//      writes P = 2^(s - m) in the input type to shared memory;
//   4. O += P V (M=128, N=64, K=64; V read as an MN-major operand) accumulates
//      in TMEM columns [64, 128); it is issued together with the next chunk's
//      S = Q K^T under one commit, so each chunk costs one MMA round trip.
//      When a row's reference max moves (rarely: only by more than 2^8), the
//      thread rescales its row of O in TMEM before the next accumulation.
// Rows are read back from TMEM, normalised and stored at the end.  Every wait on an mbarrier is
// bounded (about one second of %globaltimer); on expiry the CTA sets the
// plan's status word, frees its TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "g3s_internal.h"
#include "g3s_ptx.cuh"

namespace g3s {
namespace {

constexpr int kThreads = 128;
constexpr int kD = 64;               // head_dim of this kernel
constexpr int kNC = 64;              // columns per chunk (8 tiles)
constexpr int kGroupWindows = 8;     // windows per CTA: 8 x 16 rows = 128 MMA rows
constexpr int kMaxGroupTiles = kGroupWindows * kTileMaxTilesPerWindow;
constexpr uint32_t kTmemCols = 128;  // S chunk [0, 64) + O chunk [64, 128)
constexpr float kNegBig = -1e30f;
constexpr float kRescaleSlack = 8.0f;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

struct TileSmem {
    uint8_t q[128 * 128];     // Q rows, 128B-swizzled, K-major A operand
    uint8_t k[2][kNC * 128];  // K rows of a chunk (K-major B operand of S), two stages
    uint8_t v[2][kNC * 128];  // V rows of a chunk (MN-major B operand of O), two stages
    uint8_t p[128 * 128];     // P rows (K-major A operand of O)
    int cols[3][kNC];         // column ids of a chunk, three stages
    uint32_t bits[3][8][4];   // bitmaps of a chunk's 8 tiles, three stages
    int tile_g[kMaxGroupTiles];     // global tile index of each group tile
    int8_t tile_j[kMaxGroupTiles];  // window slot of each group tile
    int win[kGroupWindows];
    int win_t0[kGroupWindows], win_t1[kGroupWindows];  // group-tile range of each window
    unsigned long long mbar;
    uint32_t tmem_base;
    int nw, tt;
};

using namespace ptx;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T>
struct Pack2;
template <>
struct Pack2<__nv_bfloat16> {
    // round two floats to bf16, return the packed pair and the rounded values
    __device__ static uint32_t pack(float a, float b, float& ra, float& rb) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        float2 f = __bfloat1622float2(h);
        ra = f.x;
        rb = f.y;
        return *reinterpret_cast<uint32_t*>(&h);
    }
};
template <>
struct Pack2<__half> {
    __device__ static uint32_t pack(float a, float b, float& ra, float& rb) {
        __half2 h = __floats2half2_rn(a, b);
        float2 f = __half22float2(h);
        ra = f.x;
        rb = f.y;
        return *reinterpret_cast<uint32_t*>(&h);
    }
};

template <typename OutT>
__device__ __forceinline__ void store_row(void* O, long long off, const float (&o)[kD], float inv);
template <>
__device__ __forceinline__ void store_row<float>(void* O, long long off, const float (&o)[kD], float inv) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(O) + off);
#pragma unroll
    for (int i = 0; i < kD / 4; ++i) d[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
}
template <>
__device__ __forceinline__ void store_row<__nv_bfloat16>(void* O, long long off, const float (&o)[kD], float inv) {
    uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(O) + off);
#pragma unroll
    for (int i = 0; i < kD / 8; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(o[8 * i + 2 * k] * inv, o[8 * i + 2 * k + 1] * inv);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        d[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}
template <>
__device__ __forceinline__ void store_row<__half>(void* O, long long off, const float (&o)[kD], float inv) {
    uint4* d = reinterpret_cast<uint4*>(static_cast<__half*>(O) + off);
#pragma unroll
    for (int i = 0; i < kD / 8; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __half2 h = __floats2half2_rn(o[8 * i + 2 * k] * inv, o[8 * i + 2 * k + 1] * inv);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        d[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ---------------------------------------------------------------------------
template <typename T, typename OutT>
__global__ void __launch_bounds__(kThreads) tile_kernel(const TileParams p) {
    extern __shared__ uint8_t smem_raw[];
    TileSmem& sm = *reinterpret_cast<TileSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int group = blockIdx.x, h = blockIdx.y;
    const T* Q = static_cast<const T*>(p.Q);
    const T* K = static_cast<const T*>(p.K);
    const T* V = static_cast<const T*>(p.V);
    constexpr bool kBf16 = sizeof(T) == 2 && !std::is_same<T, __half>::value;
    constexpr uint32_t kIdescS = idesc_f16(kBf16, false, 128, kNC);
    constexpr uint32_t kIdescO = idesc_f16(kBf16, true, 128, kD);

    // ---- set-up: TMEM, mbarrier, the group's windows and tiles ---------------
    if (warp == 0) tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    if (tid == 0) {
        mbar_init(smem_u32(&sm.mbar), 1);
        fence_mbar_init();
    }
    // windows of the group and their tile ranges, read in parallel by the first warp
    if (warp == 0) {
        const int lane = tid;
        int w = -1, t0 = 0, cnt = 0;
        if (lane < kGroupWindows) {
            const long long idx = (long long)group * kGroupWindows + lane;
            if (idx < p.n_tile_windows) {
                w = p.tile_windows[idx];
                t0 = p.win_tile_ptr[w];
                cnt = min(p.win_tile_ptr[w + 1] - t0, kTileMaxTilesPerWindow);
            }
            sm.win[lane] = w;
        }
        int start = cnt;  // exclusive prefix of the tile counts over the 8 windows
#pragma unroll
        for (int o = 1; o < kGroupWindows; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, start, o);
            if (lane >= o) start += y;
        }
        start -= cnt;
        if (lane < kGroupWindows) {
            for (int k = 0; k < cnt; ++k) {
                sm.tile_g[start + k] = t0 + k;
                sm.tile_j[start + k] = (int8_t)lane;
            }
            sm.win_t0[lane] = start;
            sm.win_t1[lane] = start + cnt;
        }
        const int nw = __popc(__ballot_sync(0xffffffffu, w >= 0));
        const int tt = __shfl_sync(0xffffffffu, start + cnt, kGroupWindows - 1);
        if (lane == 0) {
            sm.nw = nw;
            sm.tt = tt;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t tmem_row = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's TMEM lanes
    const int tt = sm.tt;
    const int nchunks = (tt + 7) / 8;

    // chunk `ch`'s column ids and bitmaps into meta stage `ms` (24 copies of 16 B)
    auto issue_meta = [&](int ch, int ms) {
        if (tid < 24) {
            const int slot = tid / 3, part = tid - 3 * slot;
            const int t = ch * 8 + slot;
            const bool valid = t < tt;
            const long long g = valid ? sm.tile_g[t] : 0;
            if (part < 2)
                cp_async16(smem_u32(&sm.cols[ms][slot * 8 + part * 4]), p.tile_cols + g * kTileCols + part * 4,
                           valid ? 16u : 0u);
            else
                cp_async16(smem_u32(&sm.bits[ms][slot][0]), p.tile_bits + g * 4, valid ? 16u : 0u);
        }
    };
    // chunk `ch`'s K or V rows (64 rows x 8 pieces of 16 B) into stage `st`
    auto issue_gather = [&](const T* src, uint8_t* dst_base, int ch, int ms) {
#pragma unroll
        for (int it = 0; it < (kNC * 8) / kThreads; ++it) {
            const int piece = tid + kThreads * it;
            const int c = piece >> 3, x = piece & 7;
            const int col = (ch * 8 + (c >> 3)) < tt ? sm.cols[ms][c] : -1;
            const long long off = col >= 0 ? ((long long)col * p.H + h) * kD + x * 8 : 0;
            const uint32_t d = (uint32_t)(c * 128 + ((x ^ (c & 7)) << 4));
            cp_async16(smem_u32(dst_base) + d, src + off, col >= 0 ? 16u : 0u);
        }
    };

    // ---- this thread's row ------------------------------------------------------
    const int j = tid >> 4, r = tid & 15;
    long long node = -1;
    if (j < sm.nw) {
        const long long n = (long long)sm.win[j] * kWinRows + r;
        if (n < p.N) node = n;
    }
    const int my_t0 = j < sm.nw ? sm.win_t0[j] : 0;  // this row's window: group tiles [my_t0, my_t1)
    const int my_t1 = j < sm.nw ? sm.win_t1[j] : 0;
    const uint32_t tmem_S = tmem;             // S chunk, columns [0, 64)
    const uint32_t tmem_O = tmem + kNC;       // O accumulator, columns [64, 128)
    const uint32_t row_S = tmem_row;          // this warp's lanes of S
    const uint32_t row_O = tmem_row + kNC;    // and of O

    // ---- prologue: Q, chunk 0's metadata, then chunk 0's rows + chunk 1's metadata
    {
        const T* qrow = node >= 0 ? Q + (node * p.H + h) * kD : Q;
        const uint32_t qdst = smem_u32(sm.q) + tid * 128;
#pragma unroll
        for (int x = 0; x < 8; ++x) cp_async16(qdst + ((x ^ (tid & 7)) << 4), qrow + x * 8, node >= 0 ? 16u : 0u);
    }
    issue_meta(0, 0);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    if (nchunks > 0) {
        issue_gather(K, sm.k[0], 0, 0);
        issue_gather(V, sm.v[0], 0, 0);
    }
    if (nchunks > 1) issue_meta(1, 1);
    cp_async_commit();

    float m = kNegBig, l = 0.f;
    uint32_t phase = 0;
    bool failed = false;
    const float scale = p.scale_log2;

    for (int ch = 0; ch < nchunks; ++ch) {
        const int ks = ch & 1, ms = ch % 3;
        cp_async_wait_all();  // this chunk's K and V rows, the next chunk's metadata
        fence_proxy_async_smem();   // ... and the previous chunk's P: visible to the tensor core
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // O += P_{ch-1} V_{ch-1} (accumulated in TMEM), then S = Q K_ch^T; one commit covers both
        if (tid == 0) {
            if (ch > 0) {
#pragma unroll
                for (int kk = 0; kk < kNC / 16; ++kk)
                    mma_f16(tmem_O, sdesc_sw128(smem_u32(sm.p) + kk * 32, 16, 1024),
                            sdesc_sw128(smem_u32(sm.v[ks ^ 1]) + kk * 16 * 128, kNC * 128, 1024), kIdescO,
                            (ch > 1 || kk > 0) ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
                mma_f16(tmem_S, sdesc_sw128(smem_u32(sm.q) + kk * 32, 16, 1024),
                        sdesc_sw128(smem_u32(sm.k[ks]) + kk * 32, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
            mma_commit(smem_u32(&sm.mbar));
        }
        // the next chunk's K rows (that stage was last read by S_{ch-1}, complete) and
        // the metadata two chunks ahead
        if (ch + 1 < nchunks) issue_gather(K, sm.k[ks ^ 1], ch + 1, (ch + 1) % 3);
        if (ch + 2 < nchunks) issue_meta(ch + 2, (ch + 2) % 3);

        const bool ok = mbar_wait_bounded(smem_u32(&sm.mbar), phase, kWaitLimitNs);
        phase ^= 1u;
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        tc_fence_after();
        // the next chunk's V rows (that stage was last read by P_{ch-1} V_{ch-1}, now complete)
        if (ch + 1 < nchunks) issue_gather(V, sm.v[ks ^ 1], ch + 1, (ch + 1) % 3);
        cp_async_commit();

        // masked online softmax of this row of S_ch
        float s[kNC];
#pragma unroll
        for (int q4 = 0; q4 < kNC / 16; ++q4) {
            float v16[16];
            tmem_ld16(row_S + q4 * 16, v16);
#pragma unroll
            for (int i = 0; i < 16; ++i) s[q4 * 16 + i] = v16[i];
        }
        float cmax = -INFINITY;
#pragma unroll
        for (int slot = 0; slot < 8; ++slot) {
            const int t = ch * 8 + slot;
            uint32_t mask8 = 0;
            if (node >= 0 && t >= my_t0 && t < my_t1) mask8 = (sm.bits[ms][slot][r >> 2] >> ((r & 3) * 8)) & 0xffu;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float x = ((mask8 >> c) & 1u) ? s[slot * 8 + c] * scale : -INFINITY;
                s[slot * 8 + c] = x;
                cmax = fmaxf(cmax, x);
            }
        }
        // Move the reference max when a logit exceeds it by more than the slack.
        // The row of O in TMEM then needs the same factor -- unless nothing has
        // been accumulated for this row yet (l == 0: its O row is still zero).
        float corr = 1.f;
        bool rescale = false;
        if (cmax > m + kRescaleSlack) {
            corr = ex2(m - cmax);
            rescale = l > 0.f;
            l *= corr;
            m = cmax;
        }
        // tcgen05.ld / st are warp-collective: every thread takes part, the
        // ones that need no rescale multiply by 1.
        if (__syncthreads_or(rescale)) {  // rare; O_{ch-1} is complete, nothing is in flight on O
            const float f = rescale ? corr : 1.f;
#pragma unroll
            for (int q4 = 0; q4 < kD / 16; ++q4) {
                float v16[16];
                tmem_ld16(row_O + q4 * 16, v16);
#pragma unroll
                for (int i = 0; i < 16; ++i) v16[i] *= f;
                tmem_st16(row_O + q4 * 16, v16);
            }
        }
        {
            const uint32_t pdst = smem_u32(sm.p) + tid * 128;
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float ra, rb;
                    w[k] = Pack2<T>::pack(ex2(s[x * 8 + 2 * k] - m), ex2(s[x * 8 + 2 * k + 1] - m), ra, rb);
                    l += ra + rb;
                }
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(pdst + ((x ^ (tid & 7)) << 4)), "r"(w[0]),
                             "r"(w[1]), "r"(w[2]), "r"(w[3])
                             : "memory");
            }
        }
    }

    // the last chunk's P V
    if (!failed && nchunks > 0) {
        cp_async_wait_all();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < kNC / 16; ++kk)
                mma_f16(tmem_O, sdesc_sw128(smem_u32(sm.p) + kk * 32, 16, 1024),
                        sdesc_sw128(smem_u32(sm.v[(nchunks - 1) & 1]) + kk * 16 * 128, kNC * 128, 1024), kIdescO,
                        (nchunks > 1 || kk > 0) ? 1u : 0u);
            mma_commit(smem_u32(&sm.mbar));
        }
        const bool ok = mbar_wait_bounded(smem_u32(&sm.mbar), phase, kWaitLimitNs);
        phase ^= 1u;
        if (__syncthreads_or(!ok)) failed = true;
        tc_fence_after();
    }
    cp_async_wait_all();

    if (!failed) {  // uniform over the CTA
        float o[kD];
        if (nchunks > 0) {
            // warp-collective read of every row, padding rows included
#pragma unroll
            for (int q4 = 0; q4 < kD / 16; ++q4) {
                float v16[16];
                tmem_ld16(row_O + q4 * 16, v16);
#pragma unroll
                for (int i = 0; i < 16; ++i) o[q4 * 16 + i] = v16[i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < kD; ++i) o[i] = 0.f;
        }
        if (node >= 0) store_row<OutT>(p.O, (node * p.H + h) * kD, o, l > 0.f ? 1.0f / l : 0.f);
    }
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
    if (p.n_tile_windows <= 0) return cudaSuccess;
    const size_t smem = sizeof(TileSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(tile_kernel<T, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long groups = (p.n_tile_windows + kGroupWindows - 1) / kGroupWindows;
    dim3 grid((unsigned)groups, (unsigned)p.H);
    tile_kernel<T, OutT><<<grid, kThreads, smem, st>>>(p);
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
