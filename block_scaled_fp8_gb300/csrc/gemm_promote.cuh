// FP8 GEMM with arbitrary FP32 scales: two-level accumulation.
//
// PaperTrace "02 · DeepGEMM 技术解析" §2.1-2.2: the tensor core accumulates one
// 128-wide K block (level 1), then CUDA cores promote it into an FP32
// accumulator as final += sa * sb * accum (level 2); "DeepSeek V4 源码剖析
// 第13章" §13.3 pseudocode.  This kernel is that scheme on sm_103a: the MMA
// issuer accumulates each K block (4 tcgen05.mma kind::f8f6f4, K=32 each,
// no scales) into one of NP TMEM partial buffers; the 8 epilogue warps read the
// partial (tcgen05.ld), release the buffer at once, and apply the row's A scale
// and the column block's B scale in FP32 registers.  It is used when the
// caller passes FP32 scales, which need not be powers of two (UE8M0 could not
// hold them exactly).
//
// Scales: sfa FP32 [M][sf_k] row-major (1x128 groups), sfb FP32
// [ceil(N/128)][sf_k] row-major (128x128 blocks).  BN divides 128, so a
// tile's columns share one B scale per K block.
#pragma once

#include <cuda_bf16.h>

#include "dg_internal.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace dg {

template <int BN>
struct PromoteConfig {
    static_assert(BN == 32 || BN == 64 || BN == 128, "BN must divide the 128-row B scale block");
    static constexpr int kThreads = 320;
    static constexpr int kEpiWarps = 8;
    static constexpr int kABytes = kBlockM * kBlockK;
    static constexpr int kBBytes = BN * kBlockK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTxBytes = kABytes + kBBytes;
    static constexpr int kEpiChunk = 16;
    static constexpr int kNumChunks = BN / kEpiChunk;
    static constexpr int kChunksPerWarp = (kNumChunks + 1) / 2;
    static constexpr int kStagingBytes = kEpiWarps * 2 * 32 * kEpiChunk * 2;
    static constexpr int kSmemLimit = 232448;
    static constexpr int kFixedBytes = 1024 + kStagingBytes + 512;
    static constexpr int kStagesBySmem = (kSmemLimit - kFixedBytes) / kStageBytes;
    static constexpr int kStages = kStagesBySmem > 8 ? 8 : kStagesBySmem;
    static constexpr int kNumPartials = 4;   // TMEM partial-sum buffers (one per K block in flight)
    static constexpr int kTmemCols = 512;
    static_assert(kNumPartials * BN <= kTmemCols, "TMEM budget");
    static constexpr int kSmemBytes = kFixedBytes + kStages * kStageBytes;
    static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
    static_assert(kSmemBytes > 116 * 1024, "one CTA per SM (TMEM is allocated whole)");
};

template <int BN, bool WITH_C>
__global__ void __launch_bounds__(PromoteConfig<BN>::kThreads, 1)
    dg_promote_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                           const __grid_constant__ CUtensorMap tm_b,
                           const __grid_constant__ CUtensorMap tm_d, const GemmParams p) {
    using Cfg = PromoteConfig<BN>;
    constexpr int S = Cfg::kStages;
    constexpr int NP = Cfg::kNumPartials;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *smem_a = smem;
    uint8_t *smem_b = smem_a + S * Cfg::kABytes;
    uint8_t *smem_stage_out = smem_b + S * Cfg::kBBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_stage_out + Cfg::kStagingBytes);
    uint64_t *full_bar = bars;
    uint64_t *empty_bar = bars + S;
    uint64_t *pfull_bar = bars + 2 * S;
    uint64_t *pempty_bar = pfull_bar + NP;
    uint64_t *drain_bar = pempty_bar + NP;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int j = 0; j < NP; ++j) {
            mbar_init(&pfull_bar[j], 1);
            mbar_init(&pempty_bar[j], Cfg::kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_d);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;
    const int num_tiles = p.num_m_blocks * p.num_n_blocks;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
                Tile tile;
                get_tile<BN>(p, nullptr, t, 0, tile, false);
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, ctl, DG_DEV_TIMEOUT)) goto prod_done;
                    mbar_arrive_expect_tx(&full_bar[stage], Cfg::kTxBytes);
                    tma_load_2d(smem_a + stage * Cfg::kABytes, &tm_a, &full_bar[stage],
                                kb * kBlockK, tile.a_row0);
                    tma_load_2d(smem_b + stage * Cfg::kBBytes, &tm_b, &full_bar[stage],
                                kb * kBlockK, tile.b_row0);
                    issued |= 1u << stage;
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
        prod_done:
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s))
                    mbar_wait(&full_bar[s], s < stage ? phase : phase ^ 1, ctl, DG_DEV_TIMEOUT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        int pj = 0;
        uint32_t pphase = 0;
        const uint32_t idesc = make_idesc_f8(kBlockM, BN);
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&pempty_bar[pj], pphase ^ 1, ctl, DG_DEV_TIMEOUT)))
                    goto mma_done;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full_bar[stage], phase, ctl, DG_DEV_TIMEOUT)))
                    goto mma_done;
                // all lanes compute the (warp-uniform) descriptors; one elected lane issues
                tc_fence_after_sync();
                const uint64_t a_desc = make_desc_kmajor_sw128(smem_u32(smem_a + stage * Cfg::kABytes));
                const uint64_t b_desc = make_desc_kmajor_sw128(smem_u32(smem_b + stage * Cfg::kBBytes));
                const uint32_t d_tmem = tmem_base + pj * BN;
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < kBlockK / 32; ++k)
                        tc_mma_f8(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, k != 0);
                    tc_commit(&empty_bar[stage]);
                    tc_commit(&pfull_bar[pj]);
                }
                __syncwarp();
                if (++stage == S) { stage = 0; phase ^= 1; }
                if (++pj == NP) { pj = 0; pphase ^= 1; }
            }
        }
    mma_done:
        if (lane == 0) {
            tc_commit(drain_bar);
            mbar_wait(drain_bar, 0, ctl, DG_DEV_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ promotion + epilogue
        const uint32_t ew = warp - 2;
        const uint32_t quad = warp & 3;
        const uint32_t half = ew >> 2;
        int pj = 0;
        uint32_t pphase = 0;
        uint32_t buf = 0;
        uint8_t *stage_out = smem_stage_out + ew * 2 * (32 * Cfg::kEpiChunk * 2);
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            Tile tile;
            get_tile<BN>(p, nullptr, t, 0, tile, false);
            const int local_row = quad * 32 + lane;
            const int row = tile.a_row0 + local_row;
            const bool row_ok = row < p.rows;
            const float *sa_row = p.sfa_f32 + static_cast<int64_t>(row_ok ? row : 0) * p.sf_k;
            const float *sb_row = p.sfb_f32 + static_cast<int64_t>(tile.n0 / kGran) * p.sf_k;
            float acc[Cfg::kChunksPerWarp][16];
#pragma unroll
            for (int j = 0; j < Cfg::kChunksPerWarp; ++j)
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[j][i] = 0.0f;
            float sa_next = __ldg(sa_row), sb_next = __ldg(sb_row);
            bool ok = true;
            for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                // level 2 scale of this K block: sa[row][kb] * sb[n_block][kb] (FP32)
                const float s = sa_next * sb_next;
                if (kb + 1 < p.num_k_blocks) {
                    sa_next = __ldg(sa_row + kb + 1);
                    sb_next = __ldg(sb_row + kb + 1);
                }
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&pfull_bar[pj], pphase, ctl, DG_DEV_TIMEOUT))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                uint32_t v[Cfg::kChunksPerWarp][16];
#pragma unroll
                for (int j = 0; j < Cfg::kChunksPerWarp; ++j) {
                    const int c = 2 * j + half;
                    if (c < Cfg::kNumChunks)
                        tmem_ld_32x32b_x16(tmem_base + ((quad * 32) << 16) + pj * BN + c * Cfg::kEpiChunk, v[j]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < Cfg::kChunksPerWarp; ++j) reg_fence16(v[j]);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pempty_bar[pj]);
                if (++pj == NP) { pj = 0; pphase ^= 1; }
#pragma unroll
                for (int j = 0; j < Cfg::kChunksPerWarp; ++j)
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[j][i] = fmaf(s, __uint_as_float(v[j][i]), acc[j][i]);
            }
            if (!ok) break;
#pragma unroll
            for (int j = 0; j < Cfg::kChunksPerWarp; ++j) {
                const int c = 2 * j + half;
                if (c >= Cfg::kNumChunks) continue;
                const int col0 = tile.n0 + c * Cfg::kEpiChunk;
                uint32_t out[8];
                uint32_t cw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if constexpr (WITH_C) {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (row_ok && col0 + 8 * h < p.n) {
                            uint4 cv = __ldg(reinterpret_cast<const uint4 *>(
                                p.c + static_cast<int64_t>(row) * p.ldc + col0 + 8 * h));
                            cw[4 * h] = cv.x; cw[4 * h + 1] = cv.y; cw[4 * h + 2] = cv.z; cw[4 * h + 3] = cv.w;
                        }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float lo = acc[j][2 * i], hi = acc[j][2 * i + 1];
                    if constexpr (WITH_C) {
                        lo += __uint_as_float(cw[i] << 16);
                        hi += __uint_as_float(cw[i] & 0xFFFF0000u);
                    }
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                    out[i] = *reinterpret_cast<uint32_t *>(&b2);
                }
                uint8_t *sbuf = stage_out + buf * (32 * Cfg::kEpiChunk * 2);
                if (lane == 0) bulk_wait_group_read<1>();
                __syncwarp();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t off = lane * 32 + ((h ^ ((lane >> 2) & 1)) * 16);
                    *reinterpret_cast<uint4 *>(sbuf + off) =
                        make_uint4(out[4 * h], out[4 * h + 1], out[4 * h + 2], out[4 * h + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tm_d, sbuf, col0, tile.a_row0 + quad * 32);
                    bulk_commit_group();
                }
                buf ^= 1;
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

template <int BN, bool WITH_C>
cudaError_t launch_promote_gemm_impl(const TensorMaps &maps, const GemmParams &p, int grid,
                                     cudaStream_t stream) {
    using Cfg = PromoteConfig<BN>;
    cudaError_t e = cudaFuncSetAttribute(dg_promote_gemm_kernel<BN, WITH_C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    dg_promote_gemm_kernel<BN, WITH_C><<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(
        maps.a, maps.b, maps.d, p);
    return cudaGetLastError();
}

template <int BN>
void fill_promote_info(KernelInfo *info) {
    using Cfg = PromoteConfig<BN>;
    info->block_n = BN;
    info->stages = Cfg::kStages;
    info->smem_bytes = Cfg::kSmemBytes;
    info->threads = Cfg::kThreads;
    info->group_kb = 1;
    info->num_acc = 1;
}

}  // namespace dg
