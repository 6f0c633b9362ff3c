// CUDA-core fused 3S kernel: SDDMM -> softmax -> SpMM in one pass per
// destination row, plus the merge of heavy-row partial results.
//
// Mapping.  One warp owns one work item: a whole destination row, or one
// chunk of a heavy row.  A node's features for all heads, H*d values, are
// read as 16-byte vectors ("row_vecs" of them).  When a row is narrower than
// 32 vectors the warp splits into G = 32/row_vecs lane groups and every group
// gathers a different in-edge, so one warp load instruction covers G edges;
// wider rows give each lane NV = row_vecs/32 vectors of a single edge.  The
// lanes of one head (lph = d*sizeof(T)/16 of them) reduce the dot product
// with xor shuffles.  Every group keeps its own online-softmax state (running
// max m, denominator l, fp32 accumulator) in registers; the groups are merged
// with a fixed butterfly at the end, so the result does not depend on timing.
//
// This is the per-node gather of the Triton article (stondelli.it/articles/
// gattn-triton, "Using the CSC index for fast edge lookup" and "Fusing the
// full graph attention": one program per node walking its CSC range), with
// the online softmax of the Fused3S abstract (sciencestack.ai/paper/2505.08098)
// for the standard form, and the article's clipped, epsilon-normalised
// exponent for the RTMScore form (no running max needed there: the logit is
// clipped to [-5, 5] before exp).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "g3s_internal.h"

namespace g3s {
namespace core_detail {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -1e30f;  // finite start of the running max
constexpr unsigned kFull = 0xffffffffu;

template <typename T>
struct Vec;

template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void to_float(const uint4& r, float (&f)[4]) {
        f[0] = __uint_as_float(r.x);
        f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z);
        f[3] = __uint_as_float(r.w);
    }
    __device__ static uint4 from_float(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ static void store1(void* base, long long i, float x) { static_cast<float*>(base)[i] = x; }
};

__device__ __forceinline__ void bf2_to_float(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
}
__device__ __forceinline__ uint32_t float_to_bf2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
}

template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void to_float(const uint4& r, float (&f)[8]) {
        bf2_to_float(r.x, f[0], f[1]);
        bf2_to_float(r.y, f[2], f[3]);
        bf2_to_float(r.z, f[4], f[5]);
        bf2_to_float(r.w, f[6], f[7]);
    }
    __device__ static uint4 from_float(const float (&f)[8]) {
        return make_uint4(float_to_bf2(f[0], f[1]), float_to_bf2(f[2], f[3]), float_to_bf2(f[4], f[5]),
                          float_to_bf2(f[6], f[7]));
    }
    __device__ static void store1(void* base, long long i, float x) {
        static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(x);
    }
};

__device__ __forceinline__ void h2_to_float(uint32_t w, float& lo, float& hi) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
}
__device__ __forceinline__ uint32_t float_to_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <>
struct Vec<__half> {
    static constexpr int N = 8;
    __device__ static void to_float(const uint4& r, float (&f)[8]) {
        h2_to_float(r.x, f[0], f[1]);
        h2_to_float(r.y, f[2], f[3]);
        h2_to_float(r.z, f[4], f[5]);
        h2_to_float(r.w, f[6], f[7]);
    }
    __device__ static uint4 from_float(const float (&f)[8]) {
        return make_uint4(float_to_h2(f[0], f[1]), float_to_h2(f[2], f[3]), float_to_h2(f[4], f[5]),
                          float_to_h2(f[6], f[7]));
    }
    __device__ static void store1(void* base, long long i, float x) {
        static_cast<__half*>(base)[i] = __float2half_rn(x);
    }
};

__device__ __forceinline__ uint4 ldg16(const uint4* p) { return __ldg(p); }

__device__ __forceinline__ float clamp5(float x) { return fminf(fmaxf(x, -5.0f), 5.0f); }

// Store VE fp32 values as OutT at element offset `elem` (16-byte aligned).
template <typename OutT, int VE>
struct Store;
template <int VE>
struct Store<float, VE> {
    __device__ static void run(void* base, long long elem, const float (&f)[VE]) {
        float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + elem);
#pragma unroll
        for (int k = 0; k < VE / 4; ++k) d[k] = make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
    }
};
template <>
struct Store<__nv_bfloat16, 8> {
    __device__ static void run(void* base, long long elem, const float (&f)[8]) {
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + elem) = Vec<__nv_bfloat16>::from_float(f);
    }
};
template <>
struct Store<__half, 8> {
    __device__ static void run(void* base, long long elem, const float (&f)[8]) {
        *reinterpret_cast<uint4*>(static_cast<__half*>(base) + elem) = Vec<__half>::from_float(f);
    }
};

// ---------------------------------------------------------------------------
// The fused kernel.  T: input element type; OutT: type of O and Eout (fp32
// or T); NV: 16-byte vectors per lane per edge; RTM: edge-modulated variant.
// ---------------------------------------------------------------------------
template <typename T, typename OutT, int NV, bool RTM>
__global__ void __launch_bounds__(kWarpsPerCta * 32) core_kernel(const CoreParams p) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;                   // elements per 16-byte vector
    constexpr int U = NV >= 4 ? 1 : 4 / NV;     // edges per lane group per step
    const int lane = threadIdx.x & 31;
    const long long w = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);

    int row;
    long long e0, e1;
    bool is_chunk;
    if (w < p.n_chunks) {
        const int32_t* c = p.chunks + 3 * w;
        row = c[0];
        e0 = c[1];
        e1 = c[2];
        is_chunk = true;
    } else {
        const long long r = w - p.n_chunks;
        if (r >= p.N) return;
        row = (int)r;
        e0 = p.row_ptr[row];
        e1 = p.row_ptr[row + 1];
        if (e1 - e0 > p.heavy_threshold) return;  // done by chunks + merge
        if (p.win_flags != nullptr && (p.win_flags[row >> 4] & kFlagTile)) return;  // tile path
        is_chunk = false;
    }

    const int rv = p.row_vecs;
    const int gsize = rv < 32 ? rv : 32;
    const int G = 32 / gsize;
    const int g = lane / gsize;
    const int sub = lane - g * gsize;
    const int lph = p.lph;

    const uint4* Q4 = static_cast<const uint4*>(p.Q);
    const uint4* K4 = static_cast<const uint4*>(p.K);
    const uint4* V4 = static_cast<const uint4*>(p.V);
    const uint4* E4 = static_cast<const uint4*>(p.E);

    float q[NV][VE];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        VT::to_float(ldg16(Q4 + (long long)row * rv + sub + 32 * j), q[j]);
#pragma unroll
        for (int k = 0; k < VE; ++k) q[j][k] *= p.qscale;
    }

    float m[NV], l[NV], acc[NV][VE];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        m[j] = kNegBig;
        l[j] = 0.f;
#pragma unroll
        for (int k = 0; k < VE; ++k) acc[j][k] = 0.f;
    }

    const long long step = (long long)G * U;
    for (long long base = e0; base < e1; base += step) {
        const long long eb = base + (long long)g * U;
        int src[U];
#pragma unroll
        for (int u = 0; u < U; ++u) src[u] = (eb + u < e1) ? __ldg(p.col_idx + eb + u) : -1;

        uint4 kr[U][NV], vr[U][NV];
        uint4 er[RTM ? U : 1][RTM ? NV : 1];
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (src[u] >= 0) {
                    const long long o = (long long)src[u] * rv + sub + 32 * j;
                    kr[u][j] = ldg16(K4 + o);
                    vr[u][j] = ldg16(V4 + o);
                    if constexpr (RTM) er[u][j] = ldg16(E4 + (eb + u) * rv + sub + 32 * j);
                } else {
                    kr[u][j] = make_uint4(0, 0, 0, 0);
                    vr[u][j] = make_uint4(0, 0, 0, 0);
                    if constexpr (RTM) er[u][j] = make_uint4(0, 0, 0, 0);
                }
            }
        }

        float lg[U][NV];
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                float kf[VE];
                VT::to_float(kr[u][j], kf);
                float s = 0.f;
                if constexpr (RTM) {
                    float ef[VE], uo[VE];
                    VT::to_float(er[u][j], ef);
#pragma unroll
                    for (int k = 0; k < VE; ++k) {
                        float t = q[j][k] * kf[k];
                        if (p.elementwise_clamp) t = clamp5(t);
                        uo[k] = t * ef[k];
                        s += uo[k];
                    }
                    if (p.Eout != nullptr && src[u] >= 0)
                        Store<OutT, VE>::run(p.Eout, ((eb + u) * rv + sub + 32 * j) * VE, uo);
                } else {
#pragma unroll
                    for (int k = 0; k < VE; ++k) s = fmaf(q[j][k], kf[k], s);
                }
                for (int off = 1; off < lph; off <<= 1) s += __shfl_xor_sync(kFull, s, off);
                lg[u][j] = s;
            }
        }

#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if constexpr (RTM) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float sc = src[u] >= 0 ? exp2f(clamp5(lg[u][j]) * kLog2e) : 0.f;
                    float vf[VE];
                    VT::to_float(vr[u][j], vf);
                    l[j] += sc;
#pragma unroll
                    for (int k = 0; k < VE; ++k) acc[j][k] = fmaf(sc, vf[k], acc[j][k]);
                }
            } else {
                float mx = m[j];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (src[u] >= 0) mx = fmaxf(mx, lg[u][j]);
                const float corr = exp2f(m[j] - mx);
                l[j] *= corr;
#pragma unroll
                for (int k = 0; k < VE; ++k) acc[j][k] *= corr;
                m[j] = mx;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float pw = src[u] >= 0 ? exp2f(lg[u][j] - mx) : 0.f;
                    float vf[VE];
                    VT::to_float(vr[u][j], vf);
                    l[j] += pw;
#pragma unroll
                    for (int k = 0; k < VE; ++k) acc[j][k] = fmaf(pw, vf[k], acc[j][k]);
                }
            }
        }
    }

    // merge the lane groups (fixed butterfly order)
    for (int off = gsize; off < 32; off <<= 1) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if constexpr (RTM) {
                l[j] += __shfl_xor_sync(kFull, l[j], off);
#pragma unroll
                for (int k = 0; k < VE; ++k) acc[j][k] += __shfl_xor_sync(kFull, acc[j][k], off);
            } else {
                const float mo = __shfl_xor_sync(kFull, m[j], off);
                const float lo = __shfl_xor_sync(kFull, l[j], off);
                const float mx = fmaxf(m[j], mo);
                const float ca = exp2f(m[j] - mx), cb = exp2f(mo - mx);
                l[j] = l[j] * ca + lo * cb;
#pragma unroll
                for (int k = 0; k < VE; ++k) {
                    const float ao = __shfl_xor_sync(kFull, acc[j][k], off);
                    acc[j][k] = acc[j][k] * ca + ao * cb;
                }
                m[j] = mx;
            }
        }
    }
    if (g != 0) return;

    if (is_chunk) {
        const long long HD = (long long)rv * VE;
        float* pa = p.part_acc + w * HD;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int v = sub + 32 * j;
            float4* dst = reinterpret_cast<float4*>(pa + (long long)v * VE);
#pragma unroll
            for (int k = 0; k < VE; k += 4) dst[k / 4] = make_float4(acc[j][k], acc[j][k + 1], acc[j][k + 2], acc[j][k + 3]);
            if (v % lph == 0) {
                float* ml = p.part_ml + (w * p.H + v / lph) * 2;
                ml[0] = m[j];
                ml[1] = l[j];
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float inv;
            if constexpr (RTM)
                inv = 1.0f / (l[j] + p.eps);
            else
                inv = l[j] > 0.f ? 1.0f / l[j] : 0.f;
            float o[VE];
#pragma unroll
            for (int k = 0; k < VE; ++k) o[k] = acc[j][k] * inv;
            Store<OutT, VE>::run(p.O, ((long long)row * rv + sub + 32 * j) * VE, o);
        }
    }
}

// ---------------------------------------------------------------------------
// Merge of heavy-row partials: one warp per heavy row, chunks combined in
// ascending order (m = max m_c, l = sum l_c 2^(m_c - m), O = sum acc_c 2^(m_c - m) / l;
// RTMScore: plain sums, epsilon added once).
// ---------------------------------------------------------------------------
template <typename OutT, bool RTM>
__global__ void __launch_bounds__(kWarpsPerCta * 32) merge_kernel(const MergeParams p) {
    const int lane = threadIdx.x & 31;
    const long long k = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (k >= p.n_heavy) return;
    const int row = p.heavy_rows[k];
    const int c0 = p.heavy_chunk_ptr[k], c1 = p.heavy_chunk_ptr[k + 1];
    const int HD = p.H * p.D;
    for (int x = lane; x < HD; x += 32) {
        const int h = x / p.D;
        float o;
        if constexpr (RTM) {
            float a = 0.f, s = 0.f;
            for (int c = c0; c < c1; ++c) {
                a += p.part_acc[(long long)c * HD + x];
                s += p.part_ml[((long long)c * p.H + h) * 2 + 1];
            }
            o = a / (s + p.eps);
        } else {
            float mx = kNegBig;
            for (int c = c0; c < c1; ++c) mx = fmaxf(mx, p.part_ml[((long long)c * p.H + h) * 2]);
            float a = 0.f, s = 0.f;
            for (int c = c0; c < c1; ++c) {
                const float* ml = p.part_ml + ((long long)c * p.H + h) * 2;
                const float f = exp2f(ml[0] - mx);
                s += ml[1] * f;
                a += p.part_acc[(long long)c * HD + x] * f;
            }
            o = s > 0.f ? a / s : 0.f;
        }
        Vec<OutT>::store1(p.O, (long long)row * HD + x, o);
    }
}


template <typename T, typename OutT, bool RTM>
cudaError_t launch_core(const CoreParams& p, cudaStream_t st) {
    const long long items = p.n_chunks + p.N;
    if (items <= 0) return cudaSuccess;
    const long long blocks = (items + kWarpsPerCta - 1) / kWarpsPerCta;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int nv = p.row_vecs <= 32 ? 1 : p.row_vecs / 32;
    dim3 grid((unsigned)blocks), block(kWarpsPerCta * 32);
    switch (nv) {
        case 1: core_kernel<T, OutT, 1, RTM><<<grid, block, 0, st>>>(p); break;
        case 2: core_kernel<T, OutT, 2, RTM><<<grid, block, 0, st>>>(p); break;
        case 4: core_kernel<T, OutT, 4, RTM><<<grid, block, 0, st>>>(p); break;
        case 8: core_kernel<T, OutT, 8, RTM><<<grid, block, 0, st>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename OutT>
cudaError_t launch_merge(bool rtm, const MergeParams& p, cudaStream_t st) {
    if (p.n_heavy <= 0) return cudaSuccess;
    dim3 grid((unsigned)((p.n_heavy + kWarpsPerCta - 1) / kWarpsPerCta)), block(kWarpsPerCta * 32);
    if (rtm)
        merge_kernel<OutT, true><<<grid, block, 0, st>>>(p);
    else
        merge_kernel<OutT, false><<<grid, block, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace core_detail
}  // namespace g3s
