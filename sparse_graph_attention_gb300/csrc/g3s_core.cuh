// CUDA-core fused 3S kernel: SDDMM -> softmax -> SpMM in one pass per
// destination row, plus the merge of heavy-row partial results.
//
// Mapping.  A warp processes one work item at a time: a whole destination
// row, or one chunk of a heavy row.  A node's features for all heads, H*d values, are
// read as 16-byte vectors ("row_vecs" of them).  When a row is narrower than
// 32 vectors the warp splits into G = 32/row_vecs lane groups and every group
// gathers a different in-edge, so one warp load instruction covers G edges;
// wider rows give each lane NV = row_vecs/32 vectors of a single edge.  The
// lanes of one head (lph = d*sizeof(T)/16 of them) reduce the dot product
// with xor shuffles (for 16-bit inputs the per-lane dot products take the
// stored 16-bit values directly into fp32 FMAs, and the 1/sqrt(d) scale is
// applied after the reduction).  Every group keeps its own online-softmax state (running
// max m, denominator l, fp32 accumulator) in registers; the groups are merged
// with a fixed butterfly at the end, so the result does not depend on timing.
// In the pack flavour a work item is instead G consecutive short rows, one
// per lane group, each walked by its group alone (no merge).
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

#include <type_traits>

#include "g3s_internal.h"

namespace g3s {
namespace core_detail {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kModeStd = 0;  // softmax(<q,k>/sqrt d)
constexpr int kModeRtm = 1;  // RTMScore edge-modulated form
constexpr int kModeAgg = 2;  // weighted aggregation with given weights
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
    __device__ static float load1(const void* base, long long i) { return __ldg(static_cast<const float*>(base) + i); }
    __device__ static void to_float2(const uint4& r, float2 (&f)[2]) {
        f[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
        f[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
    }
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
    __device__ static float load1(const void* base, long long i) {
        const unsigned short b = __ldg(static_cast<const unsigned short*>(base) + i);
        return __uint_as_float((uint32_t)b << 16);
    }
    // element 2k is the low half of word k
    __device__ static void to_float2(const uint4& r, float2 (&f)[4]) {
        f[0] = make_float2(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u));
        f[1] = make_float2(__uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
        f[2] = make_float2(__uint_as_float(r.z << 16), __uint_as_float(r.z & 0xffff0000u));
        f[3] = make_float2(__uint_as_float(r.w << 16), __uint_as_float(r.w & 0xffff0000u));
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
    __device__ static float load1(const void* base, long long i) {
        return __half2float(__ldg(static_cast<const __half*>(base) + i));
    }
    __device__ static void to_float2(const uint4& r, float2 (&f)[4]) {
        f[0] = __half22float2(*reinterpret_cast<const __half2*>(&r.x));
        f[1] = __half22float2(*reinterpret_cast<const __half2*>(&r.y));
        f[2] = __half22float2(*reinterpret_cast<const __half2*>(&r.z));
        f[3] = __half22float2(*reinterpret_cast<const __half2*>(&r.w));
    }
};

__device__ __forceinline__ uint4 ldg16(const uint4* p) { return __ldg(p); }

// Dot product of two 16-byte vectors of 16-bit values with fp32 FMAs that
// take the 16-bit operands directly (fma.rn.f32.bf16 / .f16: the product of
// two 16-bit values is exact in fp32, so this equals unpacking to fp32 and
// using fp32 FMAs in the same order).  Even and odd elements form two chains.
template <typename T>
struct MixedDot;
template <>
struct MixedDot<__nv_bfloat16> {
    __device__ static float run(const uint4& q, const uint4& k) {
        float a = 0.f, b = 0.f;
        asm("{\n .reg .b16 q0,q1,q2,q3,q4,q5,q6,q7,k0,k1,k2,k3,k4,k5,k6,k7;\n"
            " mov.b32 {q0,q1}, %2;\n mov.b32 {q2,q3}, %3;\n mov.b32 {q4,q5}, %4;\n mov.b32 {q6,q7}, %5;\n"
            " mov.b32 {k0,k1}, %6;\n mov.b32 {k2,k3}, %7;\n mov.b32 {k4,k5}, %8;\n mov.b32 {k6,k7}, %9;\n"
            " fma.rn.f32.bf16 %0, q0, k0, %0;\n fma.rn.f32.bf16 %1, q1, k1, %1;\n"
            " fma.rn.f32.bf16 %0, q2, k2, %0;\n fma.rn.f32.bf16 %1, q3, k3, %1;\n"
            " fma.rn.f32.bf16 %0, q4, k4, %0;\n fma.rn.f32.bf16 %1, q5, k5, %1;\n"
            " fma.rn.f32.bf16 %0, q6, k6, %0;\n fma.rn.f32.bf16 %1, q7, k7, %1;\n}"
            : "+f"(a), "+f"(b)
            : "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w), "r"(k.x), "r"(k.y), "r"(k.z), "r"(k.w));
        return a + b;
    }
};
template <>
struct MixedDot<__half> {
    __device__ static float run(const uint4& q, const uint4& k) {
        float a = 0.f, b = 0.f;
        asm("{\n .reg .b16 q0,q1,q2,q3,q4,q5,q6,q7,k0,k1,k2,k3,k4,k5,k6,k7;\n"
            " mov.b32 {q0,q1}, %2;\n mov.b32 {q2,q3}, %3;\n mov.b32 {q4,q5}, %4;\n mov.b32 {q6,q7}, %5;\n"
            " mov.b32 {k0,k1}, %6;\n mov.b32 {k2,k3}, %7;\n mov.b32 {k4,k5}, %8;\n mov.b32 {k6,k7}, %9;\n"
            " fma.rn.f32.f16 %0, q0, k0, %0;\n fma.rn.f32.f16 %1, q1, k1, %1;\n"
            " fma.rn.f32.f16 %0, q2, k2, %0;\n fma.rn.f32.f16 %1, q3, k3, %1;\n"
            " fma.rn.f32.f16 %0, q4, k4, %0;\n fma.rn.f32.f16 %1, q5, k5, %1;\n"
            " fma.rn.f32.f16 %0, q6, k6, %0;\n fma.rn.f32.f16 %1, q7, k7, %1;\n}"
            : "+f"(a), "+f"(b)
            : "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w), "r"(k.x), "r"(k.y), "r"(k.z), "r"(k.w));
        return a + b;
    }
};

__device__ __forceinline__ float clamp5(float x) { return fminf(fmaxf(x, -5.0f), 5.0f); }

// Store VE fp32 values as OutT at element offset `elem` (16-byte aligned),
// with the streaming hint (written once, never read back by this kernel).
template <typename OutT, int VE>
struct Store;
template <int VE>
struct Store<float, VE> {
    __device__ static void run(void* base, long long elem, const float (&f)[VE]) {
        float4* d = reinterpret_cast<float4*>(static_cast<float*>(base) + elem);
#pragma unroll
        for (int k = 0; k < VE / 4; ++k) __stcs(d + k, make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]));
    }
};
template <>
struct Store<__nv_bfloat16, 8> {
    __device__ static void run(void* base, long long elem, const float (&f)[8]) {
        __stcs(reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + elem), Vec<__nv_bfloat16>::from_float(f));
    }
};
template <>
struct Store<__half, 8> {
    __device__ static void run(void* base, long long elem, const float (&f)[8]) {
        __stcs(reinterpret_cast<uint4*>(static_cast<__half*>(base) + elem), Vec<__half>::from_float(f));
    }
};

// 2^x with the hardware approximation (relative error about 2^-22; -inf -> 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Lazy rescale: the running max used as the exponent's reference only moves
// up when a logit exceeds it by more than this (log2 units), so most batches
// skip the rescale; weights stay below 2^kRescaleSlack.
constexpr float kRescaleSlack = 8.0f;
constexpr int kItemsPerGrab = 2;  // work items a warp takes per atomic grab

// Per-lane constants of the lane mapping.
struct Lanes {
    int lane, rv, gsize, G, g, sub, lph;
    __device__ Lanes(int lane_, int rv_, int lph_) : lane(lane_), rv(rv_), lph(lph_) {
        gsize = rv < 32 ? rv : 32;
        G = 32 / gsize;
        g = lane / gsize;
        sub = lane - g * gsize;
    }
};

// ---------------------------------------------------------------------------
// Per-lane state of one work item.
// ---------------------------------------------------------------------------
template <int NV, int VP>
struct ItemState {
    float2 q[NV][VP];    // query, pre-scaled (pairs of features)
    uint4 qr[NV];        // query as stored (16-bit inputs, standard form)
    float2 acc[NV][VP];  // sum of weight * value
    float m[NV], l[NV];  // reference max (log2 units) and sum of weights
    int cbase, idx_lo, idx_hi;  // window of 64 source indices held one per lane
};

// The arithmetic of one step on fetched rows: logits, softmax weights and the
// weighted sum of values (kr/vr/er: the lane's 16-byte vectors of K, V and E
// for its U edges; ok: the slot holds a real edge; eid: its physical slot).
template <int U, typename T, typename OutT, int NV, int MODE, int VP, int LPH>
__device__ __forceinline__ void edge_math(const CoreParams& p, const Lanes& L, ItemState<NV, VP>& st,
                                          const uint4 (&kr)[MODE == kModeAgg ? 1 : U][MODE == kModeAgg ? 1 : NV],
                                          const uint4 (&vr)[U][NV],
                                          const uint4 (&er)[MODE == kModeRtm ? U : 1][MODE == kModeRtm ? NV : 1],
                                          const float (&wg)[MODE == kModeAgg ? U : 1][MODE == kModeAgg ? NV : 1],
                                          const bool (&ok)[U],
                                          const int (&eid)[(MODE == kModeRtm || MODE == kModeAgg) ? U : 1]) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    constexpr bool RTM = MODE == kModeRtm;
    constexpr bool AGG = MODE == kModeAgg;
    constexpr bool MIXED = MODE == kModeStd && VE == 8;  // 16-bit inputs
    const int rv = L.rv, lph = LPH > 0 ? LPH : L.lph;
    float lg[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if constexpr (AGG) {
                lg[u][j] = 0.f;
                continue;
            }
            float s;
            if constexpr (MIXED) {
                s = MixedDot<T>::run(st.qr[j], kr[u][j]);
            } else if constexpr (RTM) {
                float2 kf[VP];
                VT::to_float2(kr[u][j], kf);
                float2 ef[VP];
                VT::to_float2(er[u][j], ef);
                float uo[VE];
                s = 0.f;
#pragma unroll
                for (int k = 0; k < VP; ++k) {
                    float t0 = st.q[j][k].x * kf[k].x, t1 = st.q[j][k].y * kf[k].y;
                    if (p.elementwise_clamp) {
                        t0 = clamp5(t0);
                        t1 = clamp5(t1);
                    }
                    uo[2 * k] = t0 * ef[k].x;
                    uo[2 * k + 1] = t1 * ef[k].y;
                    s += uo[2 * k];
                    s += uo[2 * k + 1];
                }
                if (p.Eout != nullptr && ok[u])
                    Store<OutT, VE>::run(p.Eout, ((long long)eid[u] * rv + L.sub + 32 * j) * VE, uo);
            } else {
                float2 kf[VP];
                VT::to_float2(kr[u][j], kf);
                float2 s2 = make_float2(0.f, 0.f);  // packed fp32 FMA
#pragma unroll
                for (int k = 0; k < VP; ++k) s2 = __ffma2_rn(st.q[j][k], kf[k], s2);
                s = s2.x + s2.y;
            }
            if constexpr (LPH > 0) {  // lanes per head known at compile time
#pragma unroll
                for (int o2 = 1; o2 < LPH; o2 <<= 1) s += __shfl_xor_sync(kFull, s, o2);
            } else {
                for (int o2 = 1; o2 < lph; o2 <<= 1) s += __shfl_xor_sync(kFull, s, o2);
            }
            lg[u][j] = MIXED ? s * p.qscale : s;  // logit in log2 units
        }
    }

#pragma unroll
    for (int j = 0; j < NV; ++j) {
        float w[U];
        if constexpr (AGG) {
#pragma unroll
            for (int u = 0; u < U; ++u) w[u] = ok[u] ? wg[u][j] : 0.f;
        } else if constexpr (RTM) {
#pragma unroll
            for (int u = 0; u < U; ++u) w[u] = ok[u] ? ex2(clamp5(lg[u][j]) * kLog2e) : 0.f;
        } else {
            float mx = st.m[j];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (ok[u]) mx = fmaxf(mx, lg[u][j]);
            if (mx > st.m[j] + kRescaleSlack) {  // move the reference max
                const float corr = ex2(st.m[j] - mx);
                const float2 c2 = make_float2(corr, corr);
                st.l[j] *= corr;
#pragma unroll
                for (int k = 0; k < VP; ++k) st.acc[j][k] = __fmul2_rn(st.acc[j][k], c2);
                st.m[j] = mx;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) w[u] = ok[u] ? ex2(lg[u][j] - st.m[j]) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float2 vf[VP];
            VT::to_float2(vr[u][j], vf);
            st.l[j] += w[u];
            const float2 w2 = make_float2(w[u], w[u]);
#pragma unroll
            for (int k = 0; k < VP; ++k) st.acc[j][k] = __ffma2_rn(w2, vf[k], st.acc[j][k]);
        }
    }
}

// Gather the rows of U source nodes (K, V; E or the given weights through
// the slots' CSR positions) for this lane and run the step's arithmetic.
template <int U, typename T, typename OutT, int NV, int MODE, int VP, int LPH>
__device__ __forceinline__ void fetch_math(const CoreParams& p, const Lanes& L, ItemState<NV, VP>& st,
                                           const int (&src)[U], const bool (&ok)[U], const int (&epos)[U]) {
    constexpr bool RTM = MODE == kModeRtm;
    constexpr bool AGG = MODE == kModeAgg;
    const int rv = L.rv, lph = LPH > 0 ? LPH : L.lph;
    const uint4* K4 = static_cast<const uint4*>(p.K) + L.sub;
    const uint4* V4 = static_cast<const uint4*>(p.V) + L.sub;
    // physical slot of each edge's features (RTMScore) or weights (aggregation)
    int eid[(RTM || AGG) ? U : 1];
    if constexpr (RTM || AGG) {
#pragma unroll
        for (int u = 0; u < U; ++u) eid[u] = p.edge_id != nullptr ? __ldg(p.edge_id + epos[u]) : epos[u];
    }
    uint4 kr[AGG ? 1 : U][AGG ? 1 : NV], vr[U][NV];
    uint4 er[RTM ? U : 1][RTM ? NV : 1];
    float wg[AGG ? U : 1][AGG ? NV : 1];  // given weights (aggregation)
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const long long o = (long long)src[u] * rv;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if constexpr (!AGG) kr[u][j] = ldg16(K4 + o + 32 * j);
            vr[u][j] = ldg16(V4 + o + 32 * j);
            if constexpr (AGG) wg[u][j] = Vec<T>::load1(p.W, (long long)eid[u] * p.H + (L.sub + 32 * j) / lph);
            if constexpr (RTM) {
                er[u][j] = ldg16(static_cast<const uint4*>(p.E) + L.sub + (long long)eid[u] * rv + 32 * j);
            }
        }
    }

    edge_math<U, T, OutT, NV, MODE, VP, LPH>(p, L, st, kr, vr, er, wg, ok, eid);
}

// Edges a lane group takes per step (U): four 16-byte K and V vectors in
// flight per lane; the aggregation gathers no K, so it takes twice as many.
template <int NV, int MODE>
struct StepEdges {
    static constexpr int value = (NV >= 4 ? 1 : 4 / NV) * (MODE == kModeAgg ? 2 : 1);
};

// One step of S = G * U edges starting at CSR position `base`.  TAIL: the
// step runs past the row's end; slots beyond it re-read the row's last edge
// (a valid, cached address) and get weight 0, so no load is branched.
template <bool TAIL, typename T, typename OutT, int NV, int MODE, int VP, int LPH>
__device__ __forceinline__ void edge_step(const CoreParams& p, const Lanes& L, ItemState<NV, VP>& st, const int base,
                                          const int e1) {
    constexpr int U = StepEdges<NV, MODE>::value;
    const int g = L.g;
    const int S = L.G * U;
    if constexpr (U > 4) {  // aggregation: a step can span more than the 64-index window
        if (S > 64) {       // (16 lane groups): each slot loads its index itself
            int src[U], epos[U];
            bool ok[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int pos = base + g * U + u;
                ok[u] = !TAIL || pos < e1;
                epos[u] = ok[u] ? pos : e1 - 1;
                src[u] = __ldg(p.col_idx + epos[u]);
            }
            fetch_math<U, T, OutT, NV, MODE, VP, LPH>(p, L, st, src, ok, epos);
            return;
        }
    }
    if (base - st.cbase >= 64) {  // warp-uniform: the next 64 indices
        st.cbase += 64;
        st.idx_lo = (st.cbase + L.lane < e1) ? __ldg(p.col_idx + st.cbase + L.lane) : 0;
        st.idx_hi = (st.cbase + 32 + L.lane < e1) ? __ldg(p.col_idx + st.cbase + 32 + L.lane) : 0;
    }
    const int off = base - st.cbase;  // 0, S, 2S, ... < 64
    const int last = e1 - 1 - st.cbase;
    int src[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        int pos = off + g * U + u;
        ok[u] = !TAIL || pos <= last;
        if (TAIL) pos = ok[u] ? pos : last;
        if (S <= 32) {
            const int v = (off & 32) ? st.idx_hi : st.idx_lo;  // warp-uniform choice
            src[u] = __shfl_sync(kFull, v, pos & 31);
        } else {
            const int a = __shfl_sync(kFull, st.idx_lo, pos & 31);
            const int b = __shfl_sync(kFull, st.idx_hi, pos & 31);
            src[u] = pos < 32 ? a : b;
        }
    }

    int epos[U];  // CSR position of each slot's edge (a valid one for masked slots)
#pragma unroll
    for (int u = 0; u < U; ++u) epos[u] = ok[u] ? base + g * U + u : e1 - 1;
    fetch_math<U, T, OutT, NV, MODE, VP, LPH>(p, L, st, src, ok, epos);
}

// Start of a work item: the query, an empty softmax state, and the first 64
// source indices.
template <typename T, int NV, int MODE, int VP>
__device__ __forceinline__ void init_item(const CoreParams& p, const Lanes& L, ItemState<NV, VP>& st, const int row,
                                          const int e0, const int e1) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    const int rv = L.rv, sub = L.sub;
    st.cbase = e0;
    st.idx_lo = (e0 + L.lane < e1) ? __ldg(p.col_idx + e0 + L.lane) : 0;
    st.idx_hi = (e0 + 32 + L.lane < e1) ? __ldg(p.col_idx + e0 + 32 + L.lane) : 0;
    const uint4* Q4 = static_cast<const uint4*>(p.Q);
    const float2 qs = make_float2(p.qscale, p.qscale);
    constexpr bool MIXED = MODE == kModeStd && VE == 8;  // dot products on the stored 16-bit query
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        if constexpr (MIXED) st.qr[j] = ldg16(Q4 + (long long)row * rv + sub + 32 * j);
        else if constexpr (MODE != kModeAgg) VT::to_float2(ldg16(Q4 + (long long)row * rv + sub + 32 * j), st.q[j]);
#pragma unroll
        for (int k = 0; k < VP; ++k) {
            if constexpr (MODE != kModeAgg && !MIXED) st.q[j][k] = __fmul2_rn(st.q[j][k], qs);
            st.acc[j][k] = make_float2(0.f, 0.f);
        }
        st.m[j] = kNegBig;
        st.l[j] = 0.f;
    }

}

// End of a work item: merge the lane groups, then write the partial result of
// a heavy-row chunk (chunk >= 0) or the normalised output row.
template <typename T, typename OutT, int NV, int MODE, int VP, int LPH, bool MERGE = true>
__device__ __forceinline__ void finish_item(const CoreParams& p, const Lanes& L, ItemState<NV, VP>& st, const int row,
                                            const long long chunk) {
    using VT = Vec<T>;
    constexpr int VE = VT::N;
    constexpr bool PLAIN = MODE != kModeStd;  // weights need no running max
    const int rv = L.rv, g = L.g, sub = L.sub, lph = LPH > 0 ? LPH : L.lph;
    // merge the lane groups (fixed butterfly order); a packed item's groups
    // each hold their own row and skip this
    for (int off = L.gsize; MERGE && off < 32; off <<= 1) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if constexpr (PLAIN) {
                st.l[j] += __shfl_xor_sync(kFull, st.l[j], off);
#pragma unroll
                for (int k = 0; k < VP; ++k) {
                    st.acc[j][k].x += __shfl_xor_sync(kFull, st.acc[j][k].x, off);
                    st.acc[j][k].y += __shfl_xor_sync(kFull, st.acc[j][k].y, off);
                }
            } else {
                const float mo = __shfl_xor_sync(kFull, st.m[j], off);
                const float lo = __shfl_xor_sync(kFull, st.l[j], off);
                const float mx = fmaxf(st.m[j], mo);
                const float ca = ex2(st.m[j] - mx), cb = ex2(mo - mx);
                st.l[j] = st.l[j] * ca + lo * cb;
#pragma unroll
                for (int k = 0; k < VP; ++k) {
                    const float ax = __shfl_xor_sync(kFull, st.acc[j][k].x, off);
                    const float ay = __shfl_xor_sync(kFull, st.acc[j][k].y, off);
                    st.acc[j][k].x = st.acc[j][k].x * ca + ax * cb;
                    st.acc[j][k].y = st.acc[j][k].y * ca + ay * cb;
                }
                st.m[j] = mx;
            }
        }
    }
    if (MERGE && g != 0) return;

    if (chunk >= 0) {
        const long long HD = (long long)rv * VE;
        float* pa = p.part_acc + chunk * HD;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int v = sub + 32 * j;
            float4* dst = reinterpret_cast<float4*>(pa + (long long)v * VE);
#pragma unroll
            for (int k = 0; k < VP; k += 2)
                dst[k / 2] = make_float4(st.acc[j][k].x, st.acc[j][k].y, st.acc[j][k + 1].x, st.acc[j][k + 1].y);
            if (v % lph == 0) {
                float* ml = p.part_ml + (chunk * p.H + v / lph) * 2;
                ml[0] = st.m[j];
                ml[1] = st.l[j];
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float inv;
            if constexpr (MODE == kModeRtm)
                inv = 1.0f / (st.l[j] + p.eps);
            else if constexpr (MODE == kModeAgg)
                inv = p.normalize ? 1.0f / (st.l[j] + p.eps) : 1.0f;
            else
                inv = st.l[j] > 0.f ? 1.0f / st.l[j] : 0.f;
            float o[VE];
#pragma unroll
            for (int k = 0; k < VP; ++k) {
                o[2 * k] = st.acc[j][k].x * inv;
                o[2 * k + 1] = st.acc[j][k].y * inv;
            }
            Store<OutT, VE>::run(p.O, ((long long)row * rv + sub + 32 * j) * VE, o);
        }
    }
}

// ---------------------------------------------------------------------------
// One work item: destination `row`, CSR positions [e0, e1).  chunk >= 0 means
// this is chunk `chunk` of a heavy row: write the partial (m, l, acc) there;
// otherwise normalise and write O.
// ---------------------------------------------------------------------------
template <typename T, typename OutT, int NV, int MODE, int LPH>
__device__ __forceinline__ void process_item(const CoreParams& p, const Lanes& L, const int row, const int e0,
                                             const int e1, const long long chunk) {
    constexpr int VP = Vec<T>::N / 2;
    constexpr int U = StepEdges<NV, MODE>::value;
    const int S = L.G * U;
    ItemState<NV, VP> st;
    init_item<T, NV, MODE, VP>(p, L, st, row, e0, e1);
    const int full_end = e0 + ((e1 - e0) & ~(S - 1));  // S is a power of two
    for (int base = e0; base < full_end; base += S) edge_step<false, T, OutT, NV, MODE, VP, LPH>(p, L, st, base, e1);
    if (full_end < e1) edge_step<true, T, OutT, NV, MODE, VP, LPH>(p, L, st, full_end, e1);

    finish_item<T, OutT, NV, MODE, VP, LPH>(p, L, st, row, chunk);
}

// ---------------------------------------------------------------------------
// A pack of G consecutive rows, one per lane group (G = 32 / row_vecs >= 2):
// every group walks its own short row U edges per step, so a warp covers G
// rows at once and no lane-group merge is needed.  A short row has at most
// pack_max_deg <= 2 * group-size entries, held two per lane of the group.
// live: this group writes its row (a short row inside the graph; a long row
// of the pack is left to the whole warp afterwards and passes deg 0 here);
// deg: this group's row length; maxdeg: the largest among the pack's groups.
// ---------------------------------------------------------------------------
template <typename T, typename OutT, int NV, int MODE, int LPH>
__device__ __forceinline__ void process_pack(const CoreParams& p, const Lanes& L, const int row, const int e0,
                                             const int deg, const int maxdeg, const bool live) {
    constexpr int VP = Vec<T>::N / 2;
    constexpr int U = NV >= 4 ? 1 : 4 / NV;
    const int gs = L.gsize;
    ItemState<NV, VP> st;
    // the query of this group's row (row 0 stands in past the end) and an empty state
    init_item<T, NV, MODE, VP>(p, L, st, live ? row : 0, 0, 0);
    const int w0 = L.sub < deg ? __ldg(p.col_idx + e0 + L.sub) : 0;
    const int w1 = gs + L.sub < deg ? __ldg(p.col_idx + e0 + gs + L.sub) : 0;
    const int last = deg > 0 ? deg - 1 : 0;
    for (int base = 0; base < maxdeg; base += U) {
        int src[U], epos[U];
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            ok[u] = base + u < deg;
            const int slot = ok[u] ? base + u : last;  // the same on every lane of the group
            // the group's lane holding `slot` offers the word that has it
            const int w = slot >= gs ? w1 : w0;
            src[u] = __shfl_sync(kFull, w, L.g * gs + (slot & (gs - 1)));
            epos[u] = deg > 0 ? e0 + slot : 0;  // an empty row's slots: any valid position
        }
        fetch_math<U, T, OutT, NV, MODE, VP, LPH>(p, L, st, src, ok, epos);
    }
    if (live) finish_item<T, OutT, NV, MODE, VP, LPH, false>(p, L, st, row, -1);
}

// ---------------------------------------------------------------------------
// The fused kernel.  T: input element type; OutT: type of O and Eout (fp32
// or T); NV: 16-byte vectors per lane per edge; MODE: standard, RTMScore or
// weighted aggregation; LPH: lanes per head when known at compile time (0:
// from the parameters); PACK: the short-row pack flavour (items are packs of
// G rows); WINS: the window-list flavour (plans with tile windows: row items
// only over the windows the tile kernel leaves).  The flavours are separate
// instantiations because their extra code costs the plain one registers.
//
// Persistent: the grid fills the GPU once and every warp takes work items
// (heavy-row chunks first, then rows in ascending id) kItemsPerGrab at a
// time from an atomic counter, so a warp that drew a short row is never idle
// behind a long one, and the rows in flight stay a narrow band of ids (the
// L2 keeps serving the sources near them).  Each item's result depends only
// on its own data, so the dynamic order does not change any output.  When all
// items fit one resident wave of warps the launcher instead gives every warp
// exactly one item by its id (no counter, no memset launch): small graphs are
// bound by one row's latency chain, not by balance.
// ---------------------------------------------------------------------------
template <typename T, typename OutT, int NV, int MODE, int LPH, bool PACK, bool WINS>
__global__ void __launch_bounds__(kWarpsPerCta * 32, NV == 1 ? (MODE == kModeRtm ? 3 : 4) : (NV == 2 && MODE != kModeRtm ? 3 : 1))
    core_kernel(const CoreParams p) {
    static_assert(!PACK || (NV == 1 && MODE != kModeRtm), "packs: one vector per lane, no edge outputs");
    const Lanes L(threadIdx.x & 31, p.row_vecs, p.lph);
    const unsigned long long n_chunks = (unsigned long long)p.n_chunks;
    const int pack = PACK ? p.pack : 1;  // rows per item: 1, or G (the pack flavour; 16 % G == 0)
    // Row items: every row (pack) in id order; in the WINS flavour (plans with
    // tile windows) only the rows of the windows left to this kernel, 16 / pack
    // items a window.  (Kept apart: the extra mapping slows the plain flavour.)
    const int pack_shift = __ffs(pack) - 1, win_shift = 4 - pack_shift;
    const unsigned long long total =
        n_chunks + (WINS ? (unsigned long long)p.n_core_windows << win_shift
                         : (unsigned long long)((p.N + pack - 1) / pack));
    auto run = [&](unsigned long long it) {
        if (it < n_chunks) {
            const int32_t* c = p.chunks + 3 * it;
            // a heavy row inside a split window is the tile kernel's (its slices)
            if constexpr (WINS)
                if (p.win_flags[c[0] >> 4] & kFlagSplit) return;
            process_item<T, OutT, NV, MODE, LPH>(p, L, c[0], c[1], c[2], (long long)it);
            return;
        }
        int r0;
        if constexpr (WINS) {
            const int q = (int)(it - n_chunks);  // row item (< N)
            r0 = p.core_windows[q >> win_shift] * 16 + ((q & ((1 << win_shift) - 1)) << pack_shift);
            if (r0 >= p.N) return;  // past the last (partial) window
        } else {
            r0 = (int)(it - n_chunks) * pack;
            if (p.win_flags != nullptr && (p.win_flags[r0 >> 4] & kFlagTile)) return;  // tile path (whole window)
        }
        if constexpr (!PACK) {
            const int e0 = p.row_ptr[r0], e1 = p.row_ptr[r0 + 1];
            if (e1 - e0 > p.heavy_threshold) return;  // chunks + merge
            process_item<T, OutT, NV, MODE, LPH>(p, L, r0, e0, e1, -1);
        } else {
            // this group's row: the short ones are packed, one per group ...
            const int row = r0 + L.g;
            int e0 = 0, e1 = 0;
            if (row < p.N) {
                e0 = p.row_ptr[row];
                e1 = p.row_ptr[row + 1];
            }
            const bool is_short = e1 - e0 <= p.pack_max_deg;
            const int sdeg = is_short ? e1 - e0 : 0;
            process_pack<T, OutT, NV, MODE, LPH>(p, L, row, e0, sdeg, __reduce_max_sync(kFull, sdeg),
                                                 is_short && row < p.N);
            // ... then each longer one on the whole warp (heavy rows: chunks + merge)
            unsigned longs = __ballot_sync(kFull, !is_short && e1 - e0 <= p.heavy_threshold);
            const unsigned group_bits = (1u << L.gsize) - 1u;  // gsize <= 16 in a pack
            while (longs) {
                const int lane0 = __ffs(longs) - 1;  // first lane of the row's group
                longs &= ~(group_bits << lane0);      // the whole group
                const int a = __shfl_sync(kFull, e0, lane0), b = __shfl_sync(kFull, e1, lane0);
                process_item<T, OutT, NV, MODE, LPH>(p, L, r0 + lane0 / L.gsize, a, b, -1);
            }
        }
    };
    if (p.static_items) {  // at most one item per warp: item = global warp id, no counter
        const unsigned long long it = (unsigned long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
        if (it < total) run(it);
        return;
    }
    for (;;) {
        unsigned long long first = 0;
        if (L.lane == 0) first = atomicAdd(p.work_counter, (unsigned long long)kItemsPerGrab);
        first = __shfl_sync(kFull, first, 0);
        if (first >= total) break;
        const unsigned long long last = first + kItemsPerGrab < total ? first + kItemsPerGrab : total;
        for (unsigned long long it = first; it < last; ++it) run(it);
    }
}

// ---------------------------------------------------------------------------
// Merge of heavy-row partials: one warp per heavy row and 32-column block,
// chunks combined in ascending order (m = max m_c, l = sum l_c 2^(m_c - m), O = sum acc_c 2^(m_c - m) / l;
// RTMScore: plain sums, epsilon added once).  The same merge serves the rows
// of split windows (their slices' partial states, from the tile kernel; an
// empty slice has m = -inf and l = 0).
// ---------------------------------------------------------------------------
template <typename OutT, bool PLAIN>
__global__ void __launch_bounds__(kWarpsPerCta * 32) merge_kernel(const MergeParams p) {
    // one warp per (heavy row, block of 32 output columns); the chunk loops
    // are unrolled so several chunks' loads are in flight at once
    const int lane = threadIdx.x & 31;
    const int HD = p.H * p.D;
    const int col_blocks = (HD + 31) / 32;
    const long long w = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (w >= (long long)p.n_heavy * col_blocks) return;
    const long long k = w / col_blocks;
    const int x = (int)(w - k * col_blocks) * 32 + lane;
    if (x >= HD) return;
    const int row = p.heavy_rows[k];
    int c0, c1;
    if (p.ranges != nullptr) {  // explicit partial ranges (plans with split windows)
        const int2 r = p.ranges[k];
        c0 = r.x;
        c1 = r.y;
    } else {
        c0 = p.heavy_chunk_ptr[k];
        c1 = p.heavy_chunk_ptr[k + 1];
    }
    const int h = x / p.D;
    const float* ml = p.part_ml + (long long)h * 2;     // chunk c: ml[c * 2H], ml[c * 2H + 1]
    const float* acc = p.part_acc + x;                  // chunk c: acc[c * HD]
    float o;
    if constexpr (PLAIN) {
        float a = 0.f, s = 0.f;
#pragma unroll 8
        for (int c = c0; c < c1; ++c) {
            a += acc[(long long)c * HD];
            s += ml[(long long)c * 2 * p.H + 1];
        }
        o = p.normalize ? a / (s + p.eps) : a;
    } else {
        float mx = kNegBig;
#pragma unroll 8
        for (int c = c0; c < c1; ++c) mx = fmaxf(mx, ml[(long long)c * 2 * p.H]);
        float a = 0.f, s = 0.f;
#pragma unroll 8
        for (int c = c0; c < c1; ++c) {
            const float f = ex2(ml[(long long)c * 2 * p.H] - mx);
            s += ml[(long long)c * 2 * p.H + 1] * f;
            a += acc[(long long)c * HD] * f;
        }
        o = s > 0.f ? a / s : 0.f;
    }
    Vec<OutT>::store1(p.O, (long long)row * HD + x, o);
}


// ---------------------------------------------------------------------------
// Small graphs (a few hundred rows: far fewer rows than resident warps): one
// CTA per row, its eight warps each walking one eighth of the row's CSR
// positions as a chunk whose partial (m, l, acc) goes to shared memory; the
// CTA then merges the eight partials in warp order, as the heavy-row merge
// does, and writes the row.  A row's latency chain is then about one step of
// edges instead of deg / (edges per step) steps.  Every row, heavy or not, is
// done this way (no chunks, no merge launch); same arithmetic per edge.
// ---------------------------------------------------------------------------
template <typename T, typename OutT, int NV, int MODE, int LPH>
__global__ void __launch_bounds__(kWarpsPerCta * 32) small_kernel(const CoreParams p) {
    extern __shared__ float part[];  // [warp][H*d] accumulators, then [warp][H][2] (m, l)
    const int row = blockIdx.x;
    const int w = threadIdx.x >> 5;
    const Lanes L(threadIdx.x & 31, p.row_vecs, p.lph);
    const int HD = p.row_vecs * Vec<T>::N;
    const int e0 = p.row_ptr[row], e1 = p.row_ptr[row + 1];
    const int per = (e1 - e0 + kWarpsPerCta - 1) / kWarpsPerCta;
    const int a = min(e0 + w * per, e1), b = min(a + per, e1);
    CoreParams q = p;
    q.part_acc = part;
    q.part_ml = part + kWarpsPerCta * HD;
    process_item<T, OutT, NV, MODE, LPH>(q, L, row, a, b, (long long)w);
    __syncthreads();
    for (int x = threadIdx.x; x < HD; x += kWarpsPerCta * 32) {
        const int h = x / p.D;
        const float* ml = q.part_ml + h * 2;  // warp c: ml[c * 2H], ml[c * 2H + 1]
        float o;
        if constexpr (MODE != kModeStd) {
            float acc = 0.f, sum = 0.f;
#pragma unroll
            for (int c = 0; c < kWarpsPerCta; ++c) {
                acc += part[c * HD + x];
                sum += ml[c * 2 * p.H + 1];
            }
            o = (MODE == kModeRtm || p.normalize) ? acc / (sum + p.eps) : acc;
        } else {
            float mx = kNegBig;
#pragma unroll
            for (int c = 0; c < kWarpsPerCta; ++c) mx = fmaxf(mx, ml[c * 2 * p.H]);
            float acc = 0.f, sum = 0.f;
#pragma unroll
            for (int c = 0; c < kWarpsPerCta; ++c) {
                const float f = ex2(ml[c * 2 * p.H] - mx);
                sum += ml[c * 2 * p.H + 1] * f;
                acc += part[c * HD + x] * f;
            }
            o = sum > 0.f ? acc / sum : 0.f;
        }
        Vec<OutT>::store1(p.O, (long long)row * HD + x, o);
    }
}

template <typename T, typename OutT, int NV, int MODE, int LPH>
cudaError_t launch_small_nv(const CoreParams& p, cudaStream_t st) {
    if (p.N <= 0) return cudaSuccess;
    const int HD = p.row_vecs * Vec<T>::N;
    const size_t smem = (size_t)kWarpsPerCta * ((size_t)HD + 2 * (size_t)p.H) * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(small_kernel<T, OutT, NV, MODE, LPH>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    small_kernel<T, OutT, NV, MODE, LPH><<<(unsigned)p.N, kWarpsPerCta * 32, smem, st>>>(p);
    return cudaGetLastError();
}

template <typename T, typename OutT, int MODE>
cudaError_t launch_small(const CoreParams& p, cudaStream_t st) {
    const int nv = p.row_vecs <= 32 ? 1 : p.row_vecs / 32;
    switch (nv) {
        case 1: return launch_small_nv<T, OutT, 1, MODE, 0>(p, st);
        case 2: return launch_small_nv<T, OutT, 2, MODE, 0>(p, st);
        case 4: return launch_small_nv<T, OutT, 4, MODE, 0>(p, st);
        case 8: return launch_small_nv<T, OutT, 8, MODE, 0>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, typename OutT>
cudaError_t launch_small_mode(int mode, const CoreParams& p, cudaStream_t st) {
    switch (mode) {
        case kModeStd: return launch_small<T, OutT, kModeStd>(p, st);
        case kModeRtm: return launch_small<T, OutT, kModeRtm>(p, st);
        case kModeAgg: return launch_small<T, OutT, kModeAgg>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, typename OutT, int NV, int MODE, int LPH, bool PACK, bool WINS = false>
cudaError_t launch_core_nv(const CoreParams& p_in, cudaStream_t st) {
    CoreParams p = p_in;
    // Short-row packs: one row per lane group, where a row is narrower than
    // 16 vectors (G >= 2 groups) and its entries fit two per group lane.
    const int gsize = p.row_vecs < 32 ? p.row_vecs : 32, G = 32 / gsize;
    constexpr int U = NV >= 4 ? 1 : 4 / NV;
    p.pack = 1;
    p.pack_max_deg = 0;
    if (PACK && G >= 2 && G <= 16) {
        int t = G * U < 2 * gsize ? G * U : 2 * gsize;
        if (t > p.heavy_threshold) t = p.heavy_threshold;
        p.pack = G;
        p.pack_max_deg = t;
    }
    if (WINS != (p.core_windows != nullptr)) return cudaErrorInvalidValue;
    const long long items = p.n_chunks + (WINS ? p.n_core_windows * (16 / p.pack) : (p.N + p.pack - 1) / p.pack);
    if (items <= 0) return cudaSuccess;
    // one resident wave of CTAs (cached per instantiation and device)
    thread_local int cached_dev = -1, cached_ctas = 0;  // per host thread: no shared mutable state
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != cached_dev) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, core_kernel<T, OutT, NV, MODE, LPH, PACK, WINS>, kWarpsPerCta * 32,
                                                          0);
        if (e != cudaSuccess) return e;
        cached_ctas = sms * (per_sm > 0 ? per_sm : 1);
        cached_dev = dev;
    }
    if (items <= (long long)cached_ctas * kWarpsPerCta) {
        // Every item fits one resident wave of warps: one item per warp, no
        // work counter (no memset launch, no atomic round trip).
        CoreParams q = p;
        q.static_items = 1;
        const int ctas = (int)((items + kWarpsPerCta - 1) / kWarpsPerCta);
        core_kernel<T, OutT, NV, MODE, LPH, PACK, WINS><<<ctas, kWarpsPerCta * 32, 0, st>>>(q);
        return cudaGetLastError();
    }
    const long long need = (items + (long long)kWarpsPerCta * kItemsPerGrab - 1) / ((long long)kWarpsPerCta * kItemsPerGrab);
    const int ctas = (int)(need < cached_ctas ? need : cached_ctas);
    e = cudaMemsetAsync(p.work_counter, 0, sizeof(unsigned long long), st);
    if (e != cudaSuccess) return e;
    core_kernel<T, OutT, NV, MODE, LPH, PACK, WINS><<<ctas, kWarpsPerCta * 32, 0, st>>>(p);
    return cudaGetLastError();
}

// The WINS flavour: plans with tile windows, which exist for the standard
// form with 16-bit inputs and head_dim 64 (8 vectors a head).
template <typename T, typename OutT, bool PACK>
cudaError_t launch_core_wins(const CoreParams& p, cudaStream_t st) {
    if constexpr (std::is_same<T, float>::value) {
        return cudaErrorInvalidValue;
    } else {
        if (p.lph != 8) return cudaErrorInvalidValue;
        if constexpr (PACK) {
            return launch_core_nv<T, OutT, 1, kModeStd, 8, true, true>(p, st);
        } else {
            switch (p.row_vecs <= 32 ? 1 : p.row_vecs / 32) {
                case 1: return launch_core_nv<T, OutT, 1, kModeStd, 8, false, true>(p, st);
                case 2: return launch_core_nv<T, OutT, 2, kModeStd, 0, false, true>(p, st);
                case 4: return launch_core_nv<T, OutT, 4, kModeStd, 0, false, true>(p, st);
                case 8: return launch_core_nv<T, OutT, 8, kModeStd, 0, false, true>(p, st);
                default: return cudaErrorInvalidValue;
            }
        }
    }
}

template <typename T, typename OutT, int MODE>
cudaError_t launch_core(const CoreParams& p, cudaStream_t st) {
    if (p.core_windows != nullptr) {
        if constexpr (MODE == kModeStd) return launch_core_wins<T, OutT, false>(p, st);
        return cudaErrorInvalidValue;
    }
    const int nv = p.row_vecs <= 32 ? 1 : p.row_vecs / 32;
    if (nv == 1) {  // one vector per lane: the head-lane reduction is unrolled
        switch (p.lph) {
            case 2: return launch_core_nv<T, OutT, 1, MODE, 2, false>(p, st);
            case 4: return launch_core_nv<T, OutT, 1, MODE, 4, false>(p, st);
            case 8: return launch_core_nv<T, OutT, 1, MODE, 8, false>(p, st);
            case 16: return launch_core_nv<T, OutT, 1, MODE, 16, false>(p, st);
            case 32: return launch_core_nv<T, OutT, 1, MODE, 32, false>(p, st);
            default: return launch_core_nv<T, OutT, 1, MODE, 0, false>(p, st);
        }
    }
    switch (nv) {
        case 2: return launch_core_nv<T, OutT, 2, MODE, 0, false>(p, st);
        case 4: return launch_core_nv<T, OutT, 4, MODE, 0, false>(p, st);
        case 8: return launch_core_nv<T, OutT, 8, MODE, 0, false>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, typename OutT>
cudaError_t launch_core_mode(int mode, const CoreParams& p, cudaStream_t st) {
    switch (mode) {
        case kModeStd: return launch_core<T, OutT, kModeStd>(p, st);
        case kModeRtm: return launch_core<T, OutT, kModeRtm>(p, st);
        case kModeAgg: return launch_core<T, OutT, kModeAgg>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

// The pack flavour: node rows of at most 16 vectors (two or more lane groups),
// standard and aggregation modes.
template <typename T, typename OutT, int MODE>
cudaError_t launch_core_packed(const CoreParams& p, cudaStream_t st) {
    if (p.row_vecs > 16) return cudaErrorInvalidValue;
    if (p.core_windows != nullptr) {
        if constexpr (MODE == kModeStd) return launch_core_wins<T, OutT, true>(p, st);
        return cudaErrorInvalidValue;
    }
    switch (p.lph) {
        case 2: return launch_core_nv<T, OutT, 1, MODE, 2, true>(p, st);
        case 4: return launch_core_nv<T, OutT, 1, MODE, 4, true>(p, st);
        case 8: return launch_core_nv<T, OutT, 1, MODE, 8, true>(p, st);
        case 16: return launch_core_nv<T, OutT, 1, MODE, 16, true>(p, st);
        default: return launch_core_nv<T, OutT, 1, MODE, 0, true>(p, st);
    }
}

template <typename T, typename OutT>
cudaError_t launch_core_packed_mode(int mode, const CoreParams& p, cudaStream_t st) {
    switch (mode) {
        case kModeStd: return launch_core_packed<T, OutT, kModeStd>(p, st);
        case kModeAgg: return launch_core_packed<T, OutT, kModeAgg>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename OutT>
cudaError_t launch_merge(bool plain, const MergeParams& p, cudaStream_t st) {
    if (p.n_heavy <= 0) return cudaSuccess;
    const long long warps = (long long)p.n_heavy * ((p.H * p.D + 31) / 32);
    dim3 grid((unsigned)((warps + kWarpsPerCta - 1) / kWarpsPerCta)), block(kWarpsPerCta * 32);
    if (plain)
        merge_kernel<OutT, true><<<grid, block, 0, st>>>(p);
    else
        merge_kernel<OutT, false><<<grid, block, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace core_detail
}  // namespace g3s
