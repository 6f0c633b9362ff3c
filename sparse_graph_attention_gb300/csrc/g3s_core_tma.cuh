// TMA-fed form of the fused kernel (standard softmax, 16-bit inputs, node
// rows of 128, 256 or 512 bytes, i.e. one 16-byte vector per lane).
//
// The arithmetic is the CUDA-core kernel's (edge_math, init_item and
// finish_item in g3s_core.cuh); only the way K and V reach the lanes differs.
// Each warp owns a ring of D stages in shared memory.  A stage holds the K
// and V rows of the S = 128/row_vecs edges of one step, gathered by the
// tensor memory accelerator (cp.async.bulk.tensor tile::gather4: four rows per
// instruction, row indices taken from the warp's index window) and counted on
// the stage's mbarrier.  The warp issues the gathers for step j + D as soon as
// it has finished reading step j, so D steps of rows are always in flight per
// warp without holding registers, and the lanes read their vectors from shared
// memory instead of computing addresses and issuing global loads.
//
// Every wait is bounded (1 s of the global timer); a warp that gives up sets
// kErrTimeout in the forward status word, waits (bounded) for its copies still
// in flight, and stops.
#pragma once
#include "g3s_core.cuh"
#include "g3s_ptx.cuh"

namespace g3s {
namespace core_detail {

constexpr int kTmaStageBytes = 4096;  // S edges x (K row + V row) = 128/rv x 2 x 16 rv bytes
constexpr int kTmaStages = 2;         // stages in flight per warp
constexpr uint64_t kTmaWaitLimitNs = 1000000000ull;

// The gathers of one step: K and V rows of the edges at window positions
// [pos0, pos0 + S), positions past `last` (the item's last edge) repeat it.
// All lanes take part in the index shuffles; lane 0 issues the copies.
template <int RV, int VP>
__device__ __forceinline__ void tma_issue_step(const ItemState<1, VP>& st, const Lanes& L, const CUtensorMap* tmK,
                                               const CUtensorMap* tmV, const uint32_t stage, const uint32_t bar,
                                               const int pos0, const int last) {
    constexpr int S = 128 / RV;
    constexpr int RB = RV * 16;
    int r[S];
#pragma unroll
    for (int i = 0; i < S; ++i) {
        const int pos = min(pos0 + i, last);           // warp-uniform, < 64
        const int v = pos < 32 ? st.idx_lo : st.idx_hi;  // warp-uniform choice
        r[i] = __shfl_sync(kFull, v, pos & 31);
    }
    if (L.lane == 0) {
        ptx::mbar_arrive_expect_tx(bar, kTmaStageBytes);
#pragma unroll
        for (int q = 0; q < S / 4; ++q) {
            ptx::tma_gather4(stage + 4 * q * RB, tmK, r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3], bar);
            ptx::tma_gather4(stage + (S + 4 * q) * RB, tmV, r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3], bar);
        }
    }
}

// One work item through the ring.  Returns false when a wait gave up.
template <typename T, typename OutT, int RV, int LPH, int D>
__device__ __forceinline__ bool process_item_tma(const CoreParams& p, const Lanes& L, const CUtensorMap* tmK,
                                                 const CUtensorMap* tmV, const unsigned char* ring,
                                                 const uint32_t bar0, uint32_t& t_issue, uint32_t& t_cons,
                                                 const int row, const int e0, const int e1, const long long chunk) {
    constexpr int NV = 1, U = 4, VP = Vec<T>::N / 2;
    constexpr int S = 128 / RV, RB = RV * 16;
    static_assert(S * 2 * RB == kTmaStageBytes, "one step per stage");
    static_assert(D * S <= 32, "the issue distance must stay inside the index window");
    ItemState<NV, VP> st;
    init_item<T, NV, kModeStd, VP>(p, L, st, row, e0, e1);
    const int nst = (e1 - e0 + S - 1) / S;
    const uint32_t ring_s = ptx::smem_u32(ring);

    // the first D steps (window positions below D*S <= 32)
    for (int j = 0; j < D && j < nst; ++j) {
        const uint32_t slot = t_issue % D;
        tma_issue_step<RV>(st, L, tmK, tmV, ring_s + slot * kTmaStageBytes, bar0 + 8 * slot, j * S,
                           e1 - 1 - st.cbase);
        ++t_issue;
    }
    for (int j = 0; j < nst; ++j) {
        const int base = e0 + j * S;
        if (base - st.cbase >= 32) {  // slide the index window by 32 (warp-uniform)
            st.cbase += 32;
            st.idx_lo = st.idx_hi;
            st.idx_hi = (st.cbase + 32 + L.lane < e1) ? __ldg(p.col_idx + st.cbase + 32 + L.lane) : 0;
        }
        const uint32_t slot = t_cons % D;
        if (!ptx::mbar_wait_bounded(bar0 + 8 * slot, (t_cons / D) & 1u, kTmaWaitLimitNs)) {
            if (L.lane == 0) atomicOr(p.status, (int32_t)kErrTimeout);
            for (uint32_t t = t_cons; t < t_issue; ++t)
                ptx::mbar_wait_bounded(bar0 + 8 * (t % D), (t / D) & 1u, kTmaWaitLimitNs);
            return false;
        }
        const unsigned char* stg = ring + slot * kTmaStageBytes;
        uint4 kr[U][NV], vr[U][NV], er[1][1];
        float wg[1][1];
        const int eid[1] = {0};
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = L.g * U + u;
            kr[u][0] = *reinterpret_cast<const uint4*>(stg + i * RB + L.sub * 16);
            vr[u][0] = *reinterpret_cast<const uint4*>(stg + (S + i) * RB + L.sub * 16);
        }
        if (base + S <= e1) {
#pragma unroll
            for (int u = 0; u < U; ++u) ok[u] = true;
            edge_math<U, T, OutT, NV, kModeStd, VP, LPH>(p, L, st, kr, vr, er, wg, ok, eid);
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) ok[u] = base + L.g * U + u < e1;
            edge_math<U, T, OutT, NV, kModeStd, VP, LPH>(p, L, st, kr, vr, er, wg, ok, eid);
        }
        ++t_cons;
        __syncwarp();  // every lane has read the stage
        if (j + D < nst) {
            if (L.lane == 0) ptx::fence_proxy_async_smem();
            const uint32_t s2 = t_issue % D;
            tma_issue_step<RV>(st, L, tmK, tmV, ring_s + s2 * kTmaStageBytes, bar0 + 8 * s2, base + D * S - st.cbase,
                               e1 - 1 - st.cbase);
            ++t_issue;
        }
    }
    finish_item<T, OutT, NV, kModeStd, VP, LPH>(p, L, st, row, chunk);
    return true;
}

// Persistent like core_kernel: warps take work items from the same atomic
// counter in the same order (heavy-row chunks, then rows by id).
template <typename T, typename OutT, int RV, int LPH, int D>
__global__ void __launch_bounds__(kWarpsPerCta * 32, D <= 2 ? 3 : 2)
    core_tma_kernel(const CoreParams p, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV) {
    extern __shared__ unsigned char tma_smem_raw[];
    __shared__ __align__(8) uint64_t bars[kWarpsPerCta * D];
    const int warp = threadIdx.x >> 5;
    const Lanes L(threadIdx.x & 31, p.row_vecs, p.lph);
    // stages start on a 1024-byte boundary (1 KB of slack is allocated for this)
    const uint32_t raw = ptx::smem_u32(tma_smem_raw);
    const unsigned char* ring = tma_smem_raw + (((raw + 1023u) & ~1023u) - raw) + warp * D * kTmaStageBytes;
    const uint32_t bar0 = ptx::smem_u32(&bars[warp * D]);
    if (L.lane == 0) {
        for (int s = 0; s < D; ++s) ptx::mbar_init(bar0 + 8 * s, 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();
    uint32_t t_issue = 0, t_cons = 0;
    const unsigned long long n_chunks = (unsigned long long)p.n_chunks;
    const unsigned long long total = n_chunks + (unsigned long long)p.N;
    for (;;) {
        unsigned long long first = 0;
        if (L.lane == 0) first = atomicAdd(p.work_counter, (unsigned long long)kItemsPerGrab);
        first = __shfl_sync(kFull, first, 0);
        if (first >= total) break;
        const unsigned long long last = first + kItemsPerGrab < total ? first + kItemsPerGrab : total;
        for (unsigned long long it = first; it < last; ++it) {
            bool ok = true;
            if (it < n_chunks) {
                const int32_t* c = p.chunks + 3 * it;
                ok = process_item_tma<T, OutT, RV, LPH, D>(p, L, &tmK, &tmV, ring, bar0, t_issue, t_cons, c[0], c[1],
                                                           c[2], (long long)it);
            } else {
                const int row = (int)(it - n_chunks);
                const int e0 = p.row_ptr[row], e1 = p.row_ptr[row + 1];
                if (e1 - e0 > p.heavy_threshold) continue;                                    // chunks + merge
                if (p.win_flags != nullptr && (p.win_flags[row >> 4] & kFlagTile)) continue;  // tile path
                ok = process_item_tma<T, OutT, RV, LPH, D>(p, L, &tmK, &tmV, ring, bar0, t_issue, t_cons, row, e0, e1,
                                                           -1);
            }
            if (!ok) return;
        }
    }
}

template <typename T, typename OutT, int RV, int LPH>
cudaError_t launch_core_tma_lph(const CoreParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
    constexpr int S = 128 / RV;  // edges per step
    constexpr int D = kTmaStages < 32 / S ? kTmaStages : 32 / S;
    const long long items = p.n_chunks + p.N;
    if (items <= 0) return cudaSuccess;
    auto kern = core_tma_kernel<T, OutT, RV, LPH, D>;
    const int smem = kWarpsPerCta * D * kTmaStageBytes + 1024;
    thread_local int cached_dev = -1, cached_ctas = 0;  // per host thread: no shared mutable state
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != cached_dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarpsPerCta * 32, smem);
        if (e != cudaSuccess) return e;
        cached_ctas = sms * (per_sm > 0 ? per_sm : 1);
        cached_dev = dev;
    }
    const long long need =
        (items + (long long)kWarpsPerCta * kItemsPerGrab - 1) / ((long long)kWarpsPerCta * kItemsPerGrab);
    const int ctas = (int)(need < cached_ctas ? need : cached_ctas);
    e = cudaMemsetAsync(p.work_counter, 0, sizeof(unsigned long long), st);
    if (e != cudaSuccess) return e;
    kern<<<ctas, kWarpsPerCta * 32, smem, st>>>(p, tk, tv);
    return cudaGetLastError();
}

template <typename T, typename OutT, int RV>
cudaError_t launch_core_tma_rv(const CoreParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
    switch (p.lph) {
        case 2: return launch_core_tma_lph<T, OutT, RV, 2>(p, tk, tv, st);
        case 4: return launch_core_tma_lph<T, OutT, RV, 4>(p, tk, tv, st);
        case 8: return launch_core_tma_lph<T, OutT, RV, 8>(p, tk, tv, st);
        case 16:
            if constexpr (RV >= 16) return launch_core_tma_lph<T, OutT, RV, 16>(p, tk, tv, st);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, typename OutT>
cudaError_t launch_core_tma(const CoreParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
    switch (p.row_vecs) {
        case 8: return launch_core_tma_rv<T, OutT, 8>(p, tk, tv, st);
        case 16: return launch_core_tma_rv<T, OutT, 16>(p, tk, tv, st);
        case 32: return launch_core_tma_rv<T, OutT, 32>(p, tk, tv, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace core_detail
}  // namespace g3s
