// Block-scaled FP8 GEMM for sm_103a: D = C + A @ B^T with UE8M0 scales applied
// inside the tensor-core MMA.
//
// Method (sources: "02 · DeepGEMM 技术解析" §2-§4; "DeepSeek V4 源码剖析 第13章"
// §13.3-§13.4): per output tile, accumulate over K-blocks of 128 the products
// sa * sb * (A_kb @ B_kb^T) in FP32 and write bf16.  On this GPU the scale
// multiply happens in the MMA itself: tcgen05.mma kind::mxf8f6f4.block_scale
// reads one UE8M0 exponent per row of A and per row of B for every 32-wide K
// step from tensor memory, so with power-of-two scales the first-level product
// is exact and the FP32 accumulator in TMEM runs over the whole K (the
// Blackwell form of the pages' two-level accumulation, §13.3 point 1).
//
// CTA layout (one CTA per SM, persistent):
//   warp 0      TMA producer: A and B per K-block into a ring of STAGES
//               shared-memory stages (full/empty mbarriers).
//   warp 1      TMEM owner and MMA issuer: 4 MMAs (K=32 each) per stage; the
//               scale byte of K-block kb is selected by the instruction's
//               scale-factor id (kb % 4); signals the accumulator to the epilogue.
//   warps 2..9  epilogue: TMEM -> registers (then the accumulator is released
//               at once), optional + C, bf16 RNE, swizzled staging in shared
//               memory, TMA store (direct stores where masked rows end inside
//               the tile).
//   warps 10-11 scale-factor warps, alternate 4-K-block groups: load the
//               group's packed scale words (one int32 holds 4 K-groups) with
//               cp.async in tcgen05.cp order, then copy them into a ring of
//               TMEM scale slots, off the producer's and MMA issuer's paths.
// Accumulators: NUM_ACC buffers of BLOCK_N TMEM columns each, so the next
// tile's MMAs overlap this tile's stores.
#pragma once

#include <cuda_bf16.h>

#include "dg_internal.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace dg {

template <int BN>
struct BsConfig {
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128 is 16..256, step 16");
    static constexpr int kThreads = 384;
    static constexpr int kEpiWarps = 8;
    static constexpr int kSfWarp = 10;                          // first scale warp
    static constexpr int kSfWarps = 2;                          // they take alternate groups
    static constexpr int kSfbChunks = (BN + 127) / 128;        // 128-word tcgen05.cp chunks
    static constexpr int kSfCols = 4 + 4 * kSfbChunks;          // TMEM columns per scale slot
    // Scale words pass through kSfSlots shared-memory slots (cp.async destination,
    // already in tcgen05.cp order) and kSfTmemSlots TMEM slots (what the MMA
    // reads).  The scale warps load a group up to kSfLookahead groups before
    // they copy it to TMEM: the load takes a global-memory latency and the copy
    // into TMEM queues behind the issued MMAs.
    static constexpr int kSfSlots = 8;
    static constexpr int kSfLookahead = kSfSlots - 3;
    static constexpr int kSfTmemSlots = 4;
    static constexpr int kABytes = kBlockM * kBlockK;           // 16 KB
    static constexpr int kBBytes = BN * kBlockK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSfaBytes = 512;                       // 128 words
    static constexpr int kSfbBytes = 512 * kSfbChunks;
    static constexpr int kSfSlotBytes = kSfaBytes + kSfbBytes;
    static constexpr int kEpiChunk = 16;                        // columns per epilogue chunk
    static constexpr int kNumChunks = BN / kEpiChunk;
    static constexpr int kChunksPerWarp = (kNumChunks + 1) / 2;
    static constexpr int kStagingBytes = kEpiWarps * 2 * 32 * kEpiChunk * 2;  // 16 KB
    static constexpr int kMaskedPrefixBytes = (kMaxGroupsMasked + 1) * 4;
    static constexpr int kSmemLimit = 232448;                   // 227 KB per CTA
    static constexpr int kFixedBytes = 1024 /*align*/ + kStagingBytes + kSfSlots * kSfSlotBytes +
                                       512 /*barriers*/ + kMaskedPrefixBytes;
    static constexpr int kStagesBySmem = (kSmemLimit - kFixedBytes) / kStageBytes;
    static constexpr int kStagesCap = kStagesBySmem > 12 ? 12 : kStagesBySmem;
    // K-blocks per ring slot: the stages of a slot share one full and one empty
    // barrier, so the MMA warp waits and commits once per kGroupKb K-blocks
    // (each wait or commit costs the issuing warp about 100 cycles).  The largest
    // of 4, 2, 1 that still leaves 4 slots in the ring (the load latency needs
    // that depth); it divides 4, so slots never straddle a scale group.
    static constexpr int kGroupKb = kStagesCap >= 16 ? 4 : (kStagesCap >= 8 ? 2 : 1);
    static constexpr int kStages = kStagesCap / kGroupKb * kGroupKb;
    static constexpr int kRing = kStages / kGroupKb;             // barrier slots
    static constexpr int kNumAcc = (2 * BN + kSfTmemSlots * kSfCols <= 512) ? 2 : 1;
    static constexpr int kTmemCols = 512;
    static_assert(kNumAcc * BN + kSfTmemSlots * kSfCols <= kTmemCols, "TMEM budget");
    static_assert(kRing >= 2, "pipeline too shallow");
    static constexpr int kSmemBytes = kFixedBytes + kStages * kStageBytes;
    static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
    static_assert(kSmemBytes > 116 * 1024, "one CTA per SM (TMEM is allocated whole)");
    // full, empty, tfull, tempty, sfree, sf_ready, sf_tfree, drain; then the TMEM
    // holder and abort flag (16 bytes), all inside the 512-byte barrier region
    static constexpr int kNumBars = 2 * kRing + 2 * kNumAcc + kSfSlots + 2 * kSfTmemSlots + 1 + kSfWarps;
    static_assert(kNumBars * 8 + 16 <= 512, "barrier region");
};

// Walks the (tile, 4-K-block group) sequence of one CTA in scheduler order,
// skipping tiles with nothing to compute; the scale warps run one to load and one
// to copy.
template <int BN>
struct GroupCursor {
    const GemmParams *p;
    const int *prefix;
    int t, j, num_tiles, num_ctas, psf_k, groups_per_tile;
    bool valid;
    Tile tile;
    __device__ __forceinline__ void start(const GemmParams &params, const int *pre, int cta, int nctas,
                                          int ntiles, int psf) {
        p = &params; prefix = pre; num_ctas = nctas; num_tiles = ntiles;
        psf_k = psf; groups_per_tile = (params.num_k_blocks + 3) >> 2;
        t = cta - nctas;
        next_tile();
    }
    __device__ __forceinline__ void next_tile() {
        j = 0;
        valid = false;
        for (t += num_ctas; t < num_tiles; t += num_ctas)
            if (get_tile<BN>(*p, prefix, t, psf_k, tile, false)) { valid = true; return; }
    }
    __device__ __forceinline__ void next() {
        if (++j == groups_per_tile) next_tile();
    }
};

template <int BN, bool WITH_C>
__global__ void __launch_bounds__(BsConfig<BN>::kThreads, 1)
    dg_bs_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                      const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_d, const GemmParams p) {
    using Cfg = BsConfig<BN>;
    constexpr int S = Cfg::kStages;
    constexpr int NUM_ACC = Cfg::kNumAcc;
    constexpr int NSF = Cfg::kSfSlots;       // shared-memory scale slots
    constexpr int NTS = Cfg::kSfTmemSlots;   // TMEM scale slots

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *smem_a = smem;
    uint8_t *smem_b = smem_a + S * Cfg::kABytes;
    uint8_t *smem_stage_out = smem_b + S * Cfg::kBBytes;       // 1024-aligned (all sizes are)
    uint8_t *smem_sf = smem_stage_out + Cfg::kStagingBytes;     // NSF slots: [SFA 512 B][SFB]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_sf + NSF * Cfg::kSfSlotBytes);
    constexpr int R = Cfg::kRing;
    constexpr int G = Cfg::kGroupKb;
    uint64_t *full_bar = bars;                        // [R]   a slot's G stages landed
    uint64_t *empty_bar = bars + R;                   // [R]   a slot's stages consumed by the MMAs
    uint64_t *tfull_bar = bars + 2 * R;               // [NUM_ACC] accumulator complete
    uint64_t *tempty_bar = tfull_bar + NUM_ACC;       // [NUM_ACC] accumulator drained
    uint64_t *sf_sfree_bar = tempty_bar + NUM_ACC;    // [NSF] scale words copied out of the slot
    uint64_t *sf_ready_bar = sf_sfree_bar + NSF;      // [NTS] scale words in TMEM
    uint64_t *sf_tfree_bar = sf_ready_bar + NTS;      // [NTS] MMAs done with the TMEM slot
    uint64_t *drain_bar = sf_tfree_bar + NTS;         // [1 + kSfWarps]  MMA warp, scale warps
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain_bar + 1 + Cfg::kSfWarps);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int *prefix = reinterpret_cast<int *>(tmem_holder + 4);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const int psf_k = (p.num_k_blocks + 3) >> 2;
    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    const int cta_id = blockIdx.x;
    const int num_ctas = gridDim.x;

    if (warp == 0) {
        // the barriers are contiguous from full_bar to drain_bar; the lanes of warp 0
        // initialise them, each fencing its own inits.  Both epilogue halves drain an
        // accumulator.
        const int num_bars = static_cast<int>(drain_bar + 1 + Cfg::kSfWarps - bars);  // <= Cfg::kNumBars
        for (int i = static_cast<int>(lane); i < num_bars; i += 32) {
            uint64_t *b = bars + i;
            mbar_init(b, b >= tempty_bar && b < tempty_bar + NUM_ACC ? Cfg::kEpiWarps : 1);
        }
        if (lane == 0) *abort_flag = 0;
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
    // Nothing above reads global memory: it overlaps the previous grid's tail when
    // launched as a programmatic dependent.  From here on every thread may read
    // inputs or write D.
    grid_launch_dependents();
    grid_dependency_wait();
    if (p.mode == kModeMasked) build_masked_prefix(p, prefix);
    // The producer waits for nobody: it signals that the barriers are initialised
    // and starts loading while the others wait for the TMEM allocation (and the
    // masked prefix, which it then waits for too).
    const bool producer_early = p.mode != kModeMasked;
    if (producer_early && warp == 0) {
        named_bar_arrive(1, Cfg::kThreads);
    } else {
        tc_fence_before_sync();
        named_bar_sync(1, Cfg::kThreads);
        tc_fence_after_sync();
    }
    const uint32_t tmem_base = warp != 0 ? *tmem_holder : 0u;
    const uint32_t sf_col0 = NUM_ACC * BN;
    const int num_tiles = total_tiles(p, prefix);

    if (warp == 0) {
        // ------------------------------------------------------------ producer (whole warp)
        int slot = 0;
        uint32_t phase = 0;
        uint32_t issued = 0;
        bool drop = (p.debug_flags & DG_DEBUG_DROP_ONE_LOAD) && blockIdx.x == 0;
        for (int t = cta_id; t < num_tiles; t += num_ctas) {
            Tile tile;
            if (!get_tile<BN>(p, prefix, t, psf_k, tile, lane == 0)) continue;
            for (int kb0 = 0; kb0 < p.num_k_blocks; kb0 += G) {
                const int nk = p.num_k_blocks - kb0 < G ? p.num_k_blocks - kb0 : G;
                if (!mbar_wait_warp(&empty_bar[slot], phase ^ 1, ctl, DG_DEV_TIMEOUT)) goto prod_done;
                if (drop) {
                    drop = false;  // diagnostic: leave this slot empty
                } else {
                    if (p.ab_3d) {
                        // one load per operand fills the slot's G stages; K-blocks past the
                        // end of K are out of bounds (zero-filled) and still count their bytes
                        if (elect_one()) {
                            mbar_arrive_expect_tx(&full_bar[slot], G * Cfg::kStageBytes);
                            tma_load_3d(smem_a + slot * G * Cfg::kABytes, &tm_a, &full_bar[slot], 0,
                                        tile.a_row0, kb0);
                            tma_load_3d(smem_b + slot * G * Cfg::kBBytes, &tm_b, &full_bar[slot], 0,
                                        tile.b_row0, kb0);
                        }
                    } else if (elect_one()) {
                        mbar_arrive_expect_tx(&full_bar[slot], nk * Cfg::kStageBytes);
                        auto load_kb = [&](int j) {
                            const int kb = kb0 + j;
                            const int stage = slot * G + j;
                            tma_load_2d(smem_a + stage * Cfg::kABytes, &tm_a, &full_bar[slot],
                                        kb * kBlockK, tile.a_row0);
                            tma_load_2d(smem_b + stage * Cfg::kBBytes, &tm_b, &full_bar[slot],
                                        kb * kBlockK, tile.b_row0);
                        };
                        if (nk == G) {
#pragma unroll
                            for (int j = 0; j < G; ++j) load_kb(j);
                        } else {
                            for (int j = 0; j < nk; ++j) load_kb(j);
                        }
                    }
                    __syncwarp();
                    issued |= 1u << slot;
                }
                if (++slot == R) { slot = 0; phase ^= 1; }
            }
        }
    prod_done:
        if (lane == 0) {
            // never leave the CTA with loads in flight: wait for the last fill of every buffer
            for (int s = 0; s < R; ++s)
                if (issued & (1u << s))
                    mbar_wait(&full_bar[s], s < slot ? phase : phase ^ 1, ctl, DG_DEV_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (whole warp)
        int slot = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        int g = 0;  // scale groups consumed
        const uint64_t a_desc_base = make_desc_kmajor_sw128(smem_u32(smem_a));
        const uint64_t b_desc_base = make_desc_kmajor_sw128(smem_u32(smem_b));
        constexpr uint32_t idesc_base = make_idesc_mxf8(kBlockM, BN, 0, 0);
        for (int t = cta_id; t < num_tiles; t += num_ctas) {
            Tile tile;
            if (!get_tile<BN>(p, prefix, t, psf_k, tile, false)) continue;
            if (!mbar_wait_warp(&tempty_bar[acc], acc_phase ^ 1, ctl, DG_DEV_TIMEOUT)) goto mma_done;
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb0 = 0; kb0 < p.num_k_blocks; kb0 += G) {
                const int nk = p.num_k_blocks - kb0 < G ? p.num_k_blocks - kb0 : G;
                const int tslot = g % NTS;
                if ((kb0 & 3) == 0) {
                    // scale words of this 4-K-block group are in TMEM slot `tslot`
                    if (!mbar_wait_warp(&sf_ready_bar[tslot], (g / NTS) & 1, ctl, DG_DEV_TIMEOUT))
                        goto mma_done;
                }
                if (!mbar_wait_warp(&full_bar[slot], phase, ctl, DG_DEV_TIMEOUT)) goto mma_done;
                tc_fence_after_sync();
                const uint32_t sfa_tmem = tmem_base + sf_col0 + tslot * Cfg::kSfCols;
                // descriptors of this slot's first stage; a stage further is a fixed
                // address step (>> 4), and the scale byte of K-block kb is kb % 4
                const uint64_t a_desc0 = a_desc_base + static_cast<uint64_t>(slot * G * (Cfg::kABytes >> 4));
                const uint64_t b_desc0 = b_desc_base + static_cast<uint64_t>(slot * G * (Cfg::kBBytes >> 4));
                const int kb_last = kb0 + nk - 1;
                const bool group_end = (kb_last & 3) == 3 || kb_last == p.num_k_blocks - 1;
                if (elect_one()) {
                    auto mma_kb = [&](int j) {
                        const int kb = kb0 + j;
                        const uint32_t sf = static_cast<uint32_t>(kb & 3);
                        const uint32_t idesc = idesc_base | (sf << 4) | (sf << 29);
                        const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(j * (Cfg::kABytes >> 4));
                        const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(j * (Cfg::kBBytes >> 4));
#pragma unroll
                        for (int k = 0; k < kBlockK / 32; ++k)
                            tc_mma_mxf8(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, sfa_tmem,
                                        sfa_tmem + 4, (kb | k) != 0);
                    };
                    if (nk == G) {
#pragma unroll
                        for (int j = 0; j < G; ++j) mma_kb(j);
                    } else {
                        for (int j = 0; j < nk; ++j) mma_kb(j);
                    }
                    tc_commit(&empty_bar[slot]);
                    // last K-block of the scale group: its TMEM slot is free once these MMAs finish
                    if (group_end) tc_commit(&sf_tfree_bar[tslot]);
                }
                __syncwarp();
                if (group_end) ++g;
                if (++slot == R) { slot = 0; phase ^= 1; }
            }
            if (elect_one()) tc_commit(&tfull_bar[acc]);
            __syncwarp();
            if (++acc == NUM_ACC) { acc = 0; acc_phase ^= 1; }
        }
    mma_done:
        // all MMAs this warp issued must finish before TMEM is freed
        if (elect_one()) {
            tc_commit(&drain_bar[0]);
            mbar_wait(&drain_bar[0], 0, ctl, DG_DEV_TIMEOUT);
        }
        __syncwarp();
    } else if (warp >= Cfg::kSfWarp) {
        // ------------------------------------------------------------ scale-factor warps
        // kSfWarps warps take the (tile, 4-K-block group) sequence in turns, so
        // the waits and tcgen05 issues of one group overlap those of the next; a
        // warp reuses only its own slots.  A group's words land in its slot by
        // cp.async, up to kSfLookahead groups ahead of the group being copied to
        // TMEM, each 4-byte copy at the position tcgen05.cp reads it from (source
        // row r holds words r, r+32, r+64, r+96 of a 128-word chunk).  A word
        // past the packed row length reads nothing and lands as zero.
        constexpr int NW = Cfg::kSfWarps;
        static_assert(NSF % NW == 0, "scale slots per warp");
        const int sw = static_cast<int>(warp) - Cfg::kSfWarp;
        GroupCursor<BN> lc, gc;   // next group to load, next group to copy
        lc.start(p, prefix, cta_id, num_ctas, num_tiles, psf_k);
        gc.start(p, prefix, cta_id, num_ctas, num_tiles, psf_k);
        for (int i = 0; i < sw; ++i) { lc.next(); gc.next(); }
        int gl = sw;              // index of lc's group
        // issues the loads of group gl, or an empty commit group past the last one;
        // false if the CTA is aborting
        auto load_group = [&]() -> bool {
            if (lc.valid) {
                const int slot = gl % NSF;
                // the slot's previous words have been copied to TMEM
                if (gl >= NSF &&
                    !mbar_wait_warp(&sf_sfree_bar[slot], ((gl / NSF) & 1) ^ 1, ctl, DG_DEV_TIMEOUT))
                    return false;
                const uint32_t dst0 = smem_u32(smem_sf + slot * Cfg::kSfSlotBytes);
                auto copy_word = [&](const uint32_t *base, int ld, int slices, int x, int y, uint32_t w) {
                    const bool in = x < ld && y < slices;
                    cp_async_4(dst0 + 4u * w, in ? base + static_cast<int64_t>(y) * ld + x : base, in ? 4u : 0u);
                };
                const int ya = lc.tile.sfa_y0 + lc.j, yb = lc.tile.sfb_y0 + lc.j;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    copy_word(p.sfa_words, p.sfa_ld, p.sfa_slices, lc.tile.sfa_x + 32 * q + static_cast<int>(lane),
                              ya, 4 * lane + q);
#pragma unroll
                for (int c = 0; c < Cfg::kSfbChunks; ++c)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        copy_word(p.sfb_words, p.sfb_ld, p.sfb_slices,
                                  lc.tile.n0 + 128 * c + 32 * q + static_cast<int>(lane), yb,
                                  128 + 128 * c + 4 * lane + q);
                for (int i = 0; i < NW; ++i) lc.next();
            }
            cp_async_commit();
            gl += NW;
            return true;
        };
        bool copied = false;
        for (int g = sw; gc.valid; g += NW) {
            const int slot = g % NSF;
            const int tslot = g % NTS;
            // up to two more of this warp's groups, kSfLookahead ahead at most; the
            // first group starts at once
            for (int i = 0; i < 2 && gl <= g + Cfg::kSfLookahead; ++i)
                if (!load_group()) goto sf_done;
            cp_async_wait_dyn((gl - g) / NW - 1);         // this lane's words of group g
            fence_proxy_async_smem();                     // visible to tcgen05.cp
            __syncwarp();
            uint32_t *sfa_buf = reinterpret_cast<uint32_t *>(smem_sf + slot * Cfg::kSfSlotBytes);
            uint32_t *sfb_buf = sfa_buf + 128;
            // the MMAs of the TMEM slot's previous group have completed
            if (!mbar_wait_warp(&sf_tfree_bar[tslot], ((g / NTS) & 1) ^ 1, ctl, DG_DEV_TIMEOUT))
                goto sf_done;
            if (lane == 0) {
                tc_fence_after_sync();
                const uint32_t sfa_tmem = tmem_base + sf_col0 + tslot * Cfg::kSfCols;
                tc_cp_32x128b_warpx4(sfa_tmem, make_desc_sf_32x128b(smem_u32(sfa_buf)));
#pragma unroll
                for (int c = 0; c < Cfg::kSfbChunks; ++c)
                    tc_cp_32x128b_warpx4(sfa_tmem + 4 + 4 * c, make_desc_sf_32x128b(smem_u32(sfb_buf + c * 128)));
                tc_commit(&sf_ready_bar[tslot]);
                tc_commit(&sf_sfree_bar[slot]);   // the slot may be loaded again
                copied = true;
            }
            __syncwarp();
            for (int i = 0; i < NW; ++i) gc.next();
        }
    sf_done:
        cp_async_wait<0>();
        if (lane == 0 && copied) {
            tc_commit(&drain_bar[1 + sw]);
            mbar_wait(&drain_bar[1 + sw], 0, ctl, DG_DEV_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const uint32_t ew = warp - 2;          // 0..7
        const uint32_t quad = warp & 3;        // TMEM lane quadrant this warp may access
        const uint32_t half = ew >> 2;         // which interleaved half of the column chunks
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t buf = 0;
        uint8_t *stage_out = smem_stage_out + ew * 2 * (32 * Cfg::kEpiChunk * 2);
        for (int t = cta_id; t < num_tiles; t += num_ctas) {
            Tile tile;
            if (!get_tile<BN>(p, prefix, t, psf_k, tile, false)) continue;
            const bool tile_has_columns = tile.n0 < p.n;  // false past the last n-block of a group
            const int local_row = quad * 32 + lane;
            const int row = tile.a_row0 + local_row;       // row in the 2-D view of D
            const bool row_ok = local_row < tile.valid_rows && (p.mode == kModeMasked || row < p.rows);
            const bool direct = tile.valid_rows < kBlockM;
            // C does not depend on the accumulator: fetch it before waiting for the MMAs.
            uint32_t cpk[WITH_C ? Cfg::kChunksPerWarp : 1][8];
            constexpr bool has_c = WITH_C;
            if constexpr (WITH_C) {
#pragma unroll
                for (int j = 0; j < Cfg::kChunksPerWarp; ++j) {
                    const int c = 2 * j + half;
                    const int col0 = tile.n0 + c * Cfg::kEpiChunk;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint4 cv = make_uint4(0u, 0u, 0u, 0u);
                        if (c < Cfg::kNumChunks && row_ok && col0 + 8 * h < p.n)
                            cv = __ldg(reinterpret_cast<const uint4 *>(
                                p.c + static_cast<int64_t>(row) * p.ldc + col0 + 8 * h));
                        cpk[j][4 * h + 0] = cv.x;
                        cpk[j][4 * h + 1] = cv.y;
                        cpk[j][4 * h + 2] = cv.z;
                        cpk[j][4 * h + 3] = cv.w;
                    }
                }
            }
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tfull_bar[acc], acc_phase, ctl, DG_DEV_TIMEOUT))) break;
            tc_fence_after_sync();
            // TMEM -> registers, two chunks per wait; + C in FP32; one RNE to bf16.
            uint32_t out[Cfg::kChunksPerWarp][8];
#pragma unroll
            for (int j0 = 0; j0 < Cfg::kChunksPerWarp; j0 += 2) {
                uint32_t v[2][16];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int c = 2 * (j0 + u) + half;
                    if (j0 + u < Cfg::kChunksPerWarp && c < Cfg::kNumChunks)
                        tmem_ld_32x32b_x16(tmem_base + ((quad * 32) << 16) + acc * BN + c * Cfg::kEpiChunk, v[u]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (j0 + u >= Cfg::kChunksPerWarp) continue;
                    reg_fence16(v[u]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float lo = __uint_as_float(v[u][2 * i]);
                        float hi = __uint_as_float(v[u][2 * i + 1]);
                        if constexpr (has_c) {
                            lo += __uint_as_float(cpk[j0 + u][i] << 16);
                            hi += __uint_as_float(cpk[j0 + u][i] & 0xFFFF0000u);
                        }
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                        out[j0 + u][i] = *reinterpret_cast<uint32_t *>(&b2);
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty_bar[acc]);
            if (++acc == NUM_ACC) { acc = 0; acc_phase ^= 1; }

#pragma unroll
            for (int j = 0; j < Cfg::kChunksPerWarp; ++j) {
                const int c = 2 * j + half;
                if (c >= Cfg::kNumChunks || !tile_has_columns) continue;
                const int col0 = tile.n0 + c * Cfg::kEpiChunk;
                if (direct) {
                    if (row_ok) {
                        uint16_t *drow = p.d + static_cast<int64_t>(row) * p.ldd + col0;
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            if (col0 + 8 * h < p.n)
                                *reinterpret_cast<uint4 *>(drow + 8 * h) =
                                    make_uint4(out[j][4 * h], out[j][4 * h + 1], out[j][4 * h + 2],
                                               out[j][4 * h + 3]);
                    }
                } else {
                    uint8_t *sbuf = stage_out + buf * (32 * Cfg::kEpiChunk * 2);
                    if (lane == 0) bulk_wait_group_read<1>();  // this buffer's previous store has read it
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // 32-byte swizzle: 16-byte unit h of row r sits at unit h ^ ((r >> 2) & 1)
                        const uint32_t off = lane * 32 + ((h ^ ((lane >> 2) & 1)) * 16);
                        *reinterpret_cast<uint4 *>(sbuf + off) =
                            make_uint4(out[j][4 * h], out[j][4 * h + 1], out[j][4 * h + 2], out[j][4 * h + 3]);
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
cudaError_t launch_bs_gemm_impl(const TensorMaps &maps, const GemmParams &p, int grid,
                                cudaStream_t stream) {
    using Cfg = BsConfig<BN>;
    // The attribute is per device; setting it on every launch costs ~1 us of
    // host time only, and keeps multi-device processes correct.
    cudaError_t e = cudaFuncSetAttribute(dg_bs_gemm_kernel<BN, WITH_C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    // a programmatic dependent of the stream's previous grid
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dg_bs_gemm_kernel<BN, WITH_C>, maps.a, maps.b, maps.d, p);
}

template <int BN>
void fill_bs_info(KernelInfo *info) {
    using Cfg = BsConfig<BN>;
    info->block_n = BN;
    info->stages = Cfg::kStages;
    info->smem_bytes = Cfg::kSmemBytes;
    info->threads = Cfg::kThreads;
    info->group_kb = Cfg::kGroupKb;
    info->num_acc = Cfg::kNumAcc;
}

}  // namespace dg
