// Dense projection Y = X W^T on the tensor cores (tcgen05.mma, TMEM
// accumulators, TMA tiles).
//
// This is the projection of node (or edge) features into the queries, keys
// and values that the attention consumes (the Triton article,
// stondelli.it/articles/gattn-triton, notes that once the attention is fused
// these GEMMs take most of the time).  X is (M, Kin) row-major, W is
// (Nout, Kin) row-major -- the layout of a linear layer's weight -- so both
// operands are K-major.  The Nout output columns are written to up to three
// row-major outputs of seg_cols columns each (Q | K | V of a layer).
//
// Kernel: persistent CTAs over 128 x BN output tiles (BN = 256, 128 or 64 by
// what seg_cols allows), tiles in row-block-major order so the
// CTAs in flight share X row blocks through L2.  Six warps:
//   warp 0, one thread: TMA loads of the X and W tiles of each 64-wide K
//     step (128-byte swizzle) into a ring of 4 stages;
//   warp 1, one thread: tcgen05.mma (M = 128, N = BN, K = 16 per
//     instruction) into one of two TMEM accumulators, alternating by tile so
//     the epilogue of a tile overlaps the MMAs of the next;
//   warps 2-5: the epilogue, one output row per thread: tcgen05.ld of the
//     accumulator row, conversion into a 128-byte-swizzled staging block in
//     shared memory, and a TMA tile store of each 128 x 128-byte block.
// Every mbarrier wait is bounded (1 s of %globaltimer, or until another role
// has given up); on expiry the kernel records kErrTimeout in the status word,
// lets the copies and MMAs in flight finish, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "g3s_internal.h"
#include "g3s_ptx.cuh"

namespace g3s {
namespace {

constexpr int kBM = 128;        // output rows per tile (MMA M)
constexpr int kBK = 64;         // K per stage: 64 16-bit elements = one 128-byte swizzle row
constexpr int kStagesL = 4;
constexpr int kWarpsL = 6;
constexpr uint64_t kLimitL = 1000000000ull;

template <int BN>
struct __align__(1024) LinSmem {
    uint8_t a[kStagesL][kBM * 128];  // X tile: 128 rows x 64 K (K-major, 128-byte swizzle)
    uint8_t b[kStagesL][BN * 128];   // W tile: BN rows x 64 K
    uint8_t o[2][kBM * 128];         // output staging: 128 rows x 128 bytes (128-byte swizzle), two buffers
    uint64_t full[kStagesL], empty[kStagesL];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

using namespace ptx;

// the 128 epilogue threads
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// the same barrier, returning whether `ok` holds on all 128 threads (so that
// they all leave the loop together: a named barrier has no timeout)
__device__ __forceinline__ bool epi_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}

// K-major operand with the 128-byte swizzle: 8-row groups 1024 B apart
__device__ __forceinline__ uint64_t sdesc_l(uint32_t saddr) { return sdesc_sw128(saddr, 16, 1024); }

template <int BN>
__device__ __forceinline__ bool wait_l(LinSmem<BN>& sm, uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int*>(&sm.abort)) return false;
        if (globaltimer() - t0 > kLimitL) {
            *reinterpret_cast<volatile int*>(&sm.abort) = 1;
            return false;
        }
    }
}

// One row of a 128-byte output block into the staging buffer (128-byte
// swizzle: 16-byte chunk x of row r at r * 128 + ((x ^ (r & 7)) << 4)) from
// 128 / sizeof(OutT) fp32 accumulator values.
template <typename OutT>
__device__ __forceinline__ void stage_row(uint32_t buf, int row, const uint32_t* r) {
    const uint32_t base = buf + row * 128;
#pragma unroll
    for (int x = 0; x < 8; ++x) {
        uint32_t w[4];
        if constexpr (std::is_same<OutT, float>::value) {
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = r[4 * x + k];
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float a = __uint_as_float(r[8 * x + 2 * k]), b = __uint_as_float(r[8 * x + 2 * k + 1]);
                if constexpr (std::is_same<OutT, __half>::value) {
                    __half2 h = __floats2half2_rn(a, b);
                    w[k] = *reinterpret_cast<uint32_t*>(&h);
                } else {
                    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
                    w[k] = *reinterpret_cast<uint32_t*>(&h);
                }
            }
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + ((x ^ (row & 7)) << 4)), "r"(w[0]),
                     "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
    }
}

template <typename T, typename OutT, int BN>
__global__ void __launch_bounds__(kWarpsL * 32, 1)
    linear_kernel(const LinearParams p, const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                  const __grid_constant__ CUtensorMap to0, const __grid_constant__ CUtensorMap to1,
                  const __grid_constant__ CUtensorMap to2) {
    extern __shared__ uint8_t lin_smem_raw[];
    LinSmem<BN>& sm =
        *reinterpret_cast<LinSmem<BN>*>((reinterpret_cast<uintptr_t>(lin_smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool kBf16 = !std::is_same<T, __half>::value;
    constexpr uint32_t kId = idesc_f16(kBf16, false, kBM, BN);
    constexpr uint32_t kStageBytes = (kBM + BN) * 128;
    const long long m_tiles = (p.M + kBM - 1) / kBM;
    const int n_tiles = (p.Nout + BN - 1) / BN;
    const long long tiles = m_tiles * n_tiles;
    const int k_steps = (p.Kin + kBK - 1) / kBK;

    if (warp == 1) tmem_alloc(smem_u32(&sm.tmem_base), 2 * BN);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesL; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sm.acc_full[b]), 1);
            mbar_init(smem_u32(&sm.acc_empty[b]), 128);
        }
        mbar_init(smem_u32(&sm.mma_done), 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        if (lane == 0) {  // loads
            uint32_t it = 0;  // stage uses
            bool ok = true;
            for (long long t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int m0 = (int)(t / n_tiles) * kBM, n0 = (int)(t % n_tiles) * BN;
                for (int ks = 0; ks < k_steps; ++ks, ++it) {
                    const int s = (int)(it % kStagesL);
                    const uint32_t u = it / kStagesL;
                    if (u >= 1 && !wait_l(sm, smem_u32(&sm.empty[s]), (u - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_u32(&sm.full[s]);
                    mbar_arrive_expect_tx(bar, kStageBytes);
                    tma_load_2d(smem_u32(sm.a[s]), &ta, ks * kBK, m0, bar);
                    tma_load_2d(smem_u32(sm.b[s]), &tb, ks * kBK, n0, bar);
                }
            }
            // every armed copy lands before the CTA may exit
            for (int s = 0; s < kStagesL; ++s) {
                const uint32_t uses = it / kStagesL + ((uint32_t)s < it % kStagesL ? 1u : 0u);
                if (uses > 0) mbar_wait_bounded(smem_u32(&sm.full[s]), (uses - 1) & 1, kLimitL);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {  // MMAs
            uint32_t it = 0, tl = 0;  // stage uses, local tiles
            bool ok = true;
            for (long long t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++tl) {
                const uint32_t buf = tl & 1, use = tl >> 1;
                if (use >= 1 && !wait_l(sm, smem_u32(&sm.acc_empty[buf]), (use - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * BN;
                for (int ks = 0; ks < k_steps; ++ks, ++it) {
                    const int s = (int)(it % kStagesL);
                    if (!wait_l(sm, smem_u32(&sm.full[s]), (it / kStagesL) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = smem_u32(sm.a[s]), b = smem_u32(sm.b[s]);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_f16(d, sdesc_l(a + kk * 32), sdesc_l(b + kk * 32), kId, (ks > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&sm.empty[s]));  // the stage is free once these MMAs are done
                }
                if (ok) mma_commit(smem_u32(&sm.acc_full[buf]));
            }
            mma_commit(smem_u32(&sm.mma_done));
            mbar_wait_bounded(smem_u32(&sm.mma_done), 0, kLimitL);
        }
        __syncwarp();
    } else {  // epilogue: warps 2-5, TMEM lane quarter warp % 4
        // A tile leaves in blocks of 128 bytes per row (64 16-bit or 32 fp32
        // columns): every thread converts its row of the block into a staging
        // buffer, then one thread stores the block with TMA.  Two buffers: a
        // buffer is rewritten only after the store two blocks back has read it.
        constexpr int kBC = 128 / (int)sizeof(OutT);  // output columns per block
        const int row = 32 * (warp & 3) + lane;
        const bool leader = threadIdx.x == 64;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const CUtensorMap* maps[3] = {&to0, &to1, &to2};
        uint32_t tl = 0, blocks = 0;
        for (long long t = blockIdx.x; t < tiles; t += gridDim.x, ++tl) {
            const uint32_t buf = tl & 1, use = tl >> 1;
            if (!epi_all(wait_l(sm, smem_u32(&sm.acc_full[buf]), use & 1))) break;
            tc_fence_after();
            const int m0 = (int)(t / n_tiles) * kBM;
            const int n0 = (int)(t % n_tiles) * BN;
            const int seg = n0 / p.seg_cols, c0 = n0 - seg * p.seg_cols;
#pragma unroll 1
            for (int j = 0; j < BN / kBC; ++j, ++blocks) {
                const uint32_t sb = smem_u32(sm.o[blocks & 1]);
                if (leader && blocks >= 2) bulk_wait_read<1>();
                epi_sync();  // the staging buffer is free
                uint32_t r[32 * (kBC / 32)];
#pragma unroll
                for (int q = 0; q < kBC / 32; ++q)
                    tmem_ld32(tmem + lane_off + buf * BN + j * kBC + q * 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * q));
                if (j == BN / kBC - 1) {  // the accumulator is read: the MMAs may reuse it
                    tc_fence_before();
                    mbar_arrive(smem_u32(&sm.acc_empty[buf]));
                }
                stage_row<OutT>(sb, row, r);
                fence_proxy_async_smem();
                epi_sync();  // the block is staged
                if (leader) {
                    tma_store_2d(maps[seg], c0 + j * kBC, m0, sb);
                    bulk_commit();
                }
            }
        }
        if (leader) bulk_wait_all();  // the stores have completed before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && sm.abort && p.status != nullptr) atomicOr(p.status, (int32_t)kErrTimeout);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * BN);
    }
}

struct LinMaps {
    const void* A = nullptr;
    const void* B = nullptr;
    const void* O[3] = {nullptr, nullptr, nullptr};
    long long M = -1;
    int Kin = 0, Nout = 0, BN = 0, seg = 0, esz = 0;
    CUtensorMap a, b, o[3];
};
thread_local LinMaps lin_maps;

// A 2-D K-major map: rows x kin 16-bit elements, box of box_rows x 64, 128-byte swizzle.
bool encode_kmajor(CUtensorMap* m, const void* base, long long rows, int kin, int box_rows);

template <typename T, typename OutT, int BN>
cudaError_t launch_lin(const LinearParams& p, cudaStream_t st) {
    LinMaps& mp = lin_maps;
    constexpr int esz = (int)sizeof(OutT);
    const int nseg = p.Nout / p.seg_cols;
    bool same = mp.A == p.A && mp.B == p.W && mp.M == p.M && mp.Kin == p.Kin && mp.Nout == p.Nout && mp.BN == BN &&
                mp.seg == p.seg_cols && mp.esz == esz;
    for (int i = 0; i < 3; ++i) same = same && mp.O[i] == (i < nseg ? p.out[i] : nullptr);
    if (!same) {
        mp.A = nullptr;
        if (!encode_kmajor(&mp.a, p.A, p.M, p.Kin, kBM) || !encode_kmajor(&mp.b, p.W, p.Nout, p.Kin, BN))
            return cudaErrorInvalidValue;
        for (int i = 0; i < 3; ++i) {  // unused segments get a copy of the first map (never stored through)
            if (!encode_tile(&mp.o[i], p.out[i < nseg ? i : 0], p.M, p.seg_cols, esz, kBM, 128 / esz))
                return cudaErrorInvalidValue;
            mp.O[i] = i < nseg ? p.out[i] : nullptr;
        }
        mp.A = p.A;
        mp.B = p.W;
        mp.M = p.M;
        mp.Kin = p.Kin;
        mp.Nout = p.Nout;
        mp.BN = BN;
        mp.seg = p.seg_cols;
        mp.esz = esz;
    }
    const int smem = (int)sizeof(LinSmem<BN>) + 1024;
    thread_local int cached_dev = -1, sms = 0;  // per host thread: no shared mutable state
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != cached_dev) {
        e = cudaFuncSetAttribute(linear_kernel<T, OutT, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cached_dev = dev;
    }
    const long long tiles = ((p.M + kBM - 1) / kBM) * ((p.Nout + BN - 1) / BN);
    const int grid = (int)(tiles < sms ? tiles : sms);
    linear_kernel<T, OutT, BN><<<grid, kWarpsL * 32, smem, st>>>(p, mp.a, mp.b, mp.o[0], mp.o[1], mp.o[2]);
    return cudaGetLastError();
}

// Tile width: 256 columns where the segments allow it and K is long enough
// for the MMAs to matter (the operand reads of an N = 128 MMA alone fill the
// shared-memory bandwidth), else 128, else 64.
template <typename T, typename OutT>
cudaError_t launch_lin_bn(const LinearParams& p, cudaStream_t st) {
    if (p.seg_cols % 256 == 0 && p.Kin >= 256) return launch_lin<T, OutT, 256>(p, st);
    if (p.seg_cols % 128 == 0) return launch_lin<T, OutT, 128>(p, st);
    return launch_lin<T, OutT, 64>(p, st);
}

bool encode_kmajor(CUtensorMap* m, const void* base, long long rows, int kin, int box_rows) {
    return encode_tile(m, base, rows, kin, 2, box_rows, kBK);
}

}  // namespace

bool linear_supported(int dtype, int out_dtype, int kin, int seg_cols) {
    if (dtype != G3S_F16 && dtype != G3S_BF16) return false;
    if (out_dtype != G3S_F32 && out_dtype != dtype) return false;
    // rows of X and W must be 16-byte multiples for TMA; output segments of whole 64-column tiles
    return kin >= 8 && kin % 8 == 0 && seg_cols >= 64 && seg_cols % 64 == 0;
}

cudaError_t linear_launch(int dtype, int out_dtype, const LinearParams& p, cudaStream_t st) {
    if (p.M <= 0) return cudaSuccess;
    if (!tensor_maps_available()) return cudaErrorNotSupported;
    if (dtype == G3S_BF16) {
        if (out_dtype == G3S_F32) return launch_lin_bn<__nv_bfloat16, float>(p, st);
        return launch_lin_bn<__nv_bfloat16, __nv_bfloat16>(p, st);
    }
    if (out_dtype == G3S_F32) return launch_lin_bn<__half, float>(p, st);
    return launch_lin_bn<__half, __half>(p, st);
}

}  // namespace g3s
