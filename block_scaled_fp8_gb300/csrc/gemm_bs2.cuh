// Block-scaled FP8 GEMM on CTA pairs (tcgen05 cta_group::2): dense, contiguous
// grouped (per-row expert ids or PSUM offsets), masked grouped and K-grouped
// layouts; K-major or M/N-major operands; FP8 or FP4 (E2M1) B; bf16 or FP32 D.
//
// Same method as the single-CTA kernel (gemm_bs.cuh; "02 · DeepGEMM 技术解析"
// §2-§4, "DeepSeek V4 源码剖析 第13章" §13.3): per output tile the block-scaled
// MMA accumulates sa*sb*(A_kb @ B_kb^T) over all K-blocks in FP32 TMEM.  Here a
// cluster of two CTAs on two SMs computes one MP x BN tile with M=MP MMAs
// issued by the leader CTA (MP = 256, or 128 for skinny problems):
//   - each CTA loads its own MP/2 rows of A and half of the tile's B columns
//     (BN/2 rows of B) per 128-K stage; the pair's loads complete on the
//     leader's barrier.  An SM's TMA ingest is capped near 48-60 bytes per cycle,
//     so halving the B bytes each SM loads is what the pair buys;
//   - the MMA reads the leader's A rows and B rows 0..BN/2-1 from the leader's
//     shared memory, the peer's A rows and B rows BN/2..BN-1 from the peer's,
//     and writes each CTA's rows of D into that CTA's TMEM;
//   - each CTA's TMEM holds the A scales of its own rows and the B scales of
//     all BN columns (lane n%32, column n/32; for MP=128 per half of N, see
//     Bs2Config); tcgen05.cp.cta_group::2 copies each CTA's scale words
//     into its own TMEM;
//   - commits reach both CTAs (multicast), and the peer's epilogue and scale
//     warps signal the leader's barriers through their cluster addresses;
//   - tiles wider than 256 columns (MP=256) issue a second MMA per K step for
//     columns [256, BN), from a second B region.
// Ring slots group kGroupKb K-blocks under one barrier pair to keep the MMA
// warp's per-K-block work below the tensor time.  Roles: warp 0 producer,
// warp 1 MMA issuer (leader), warps 2-9 epilogue, warps 10-11 scale words.
// A dense GEMM with bf16 C whose tile is whole 32-column boxes keeps each CTA's
// C tile in shared memory: loaded by TMA a tile ahead, summed with the
// accumulator in place, and stored by TMA from there.
#pragma once

#include <cuda_bf16.h>

#include "dg_internal.h"
#include "gemm_bs.cuh"
#include "ptx.cuh"

namespace dg {

// MP = rows of a pair tile: 256 (each CTA 128 rows; D in TMEM lanes 0-127, BN
// columns) or 128 (each CTA 64 rows; TMEM lanes 0-63 hold D columns [0, BN/2)
// and lanes 64-127 columns [BN/2, BN) of the same 64 rows, so an accumulator is
// BN/2 columns wide).
// B_ATOM: B is MN-major ([K][N]); each CTA's B region per K-block is one whole
// 128-byte swizzle atom wide (128 N-bytes x 128 K-rows) however many of its
// columns (BN/2 <= 128) the MMA reads.
// B4: B is FP4 (E2M1) with one scale per 32 K: its stages take the same shared
// memory as FP8 (the loads leave 8 empty bytes after every 8 bytes of codes),
// and a scale group holds one B word per column for each of its 4 K-blocks.
// SB: output staging buffers per epilogue warp, 0 for as many as fit (up to 4)
// without costing an operand stage.
// S32: A and B scales every 32 K (K-grouped scales at a K granularity of 32): a
// scale group holds one word per row of A and per column of B for each of its 4
// K-blocks, the word's bytes being the K-block's four 32-K scales.
// CT: the bf16 C epilogue of a dense GEMM keeps this CTA's whole C tile in shared
// memory (loaded by TMA a tile ahead, summed in place, stored by TMA from there);
// the region doubles as the output staging of the register C path.
template <int BN, int MP = 256, bool B_ATOM = false, bool B4 = false, int SB = 0, bool S32 = false,
          bool CT = false>
struct Bs2Config {
    // BN/2 rows of B per CTA fill whole 8-row swizzle atoms; pair MMAs take N % 16 == 0, N <= 256;
    // with MP=128 each half of N is whole 16-column epilogue chunks
    static_assert(MP == 256 || MP == 128, "pair tile rows");
    static_assert(MP == 256 ? (BN % 16 == 0 && BN >= 64) : (BN % 32 == 0 && BN >= 32), "tile columns");
    static_assert(BN <= 256 || MP == 256, "wide tiles are 256-row tiles");
    // A pair MMA takes N <= 256: a wider tile issues a second MMA for columns
    // [kBN1, BN).  Each CTA holds kB1Rows + kB2Rows rows of B: its half of each
    // MMA's columns, in two regions (one TMA box each).
    static constexpr int kBN1 = BN > 256 ? 256 : BN;
    static constexpr int kBN2 = BN - kBN1;
    static_assert(kBN2 == 0 || (kBN2 % 16 == 0 && kBN2 <= 256), "second MMA columns");
    static constexpr int kB1Rows = kBN1 / 2;
    static constexpr int kB2Rows = kBN2 / 2;
    static_assert(!B_ATOM || (MP == 256 && kBN2 == 0 && kB1Rows % 16 == 0), "MN-major B: one atom per CTA");
    static constexpr int kThreads = 384;
    static constexpr int kEpiWarps = 8;
    static constexpr int kSfWarp = 10;                           // first scale warp
    static constexpr int kSfWarps = 2;                           // they take alternate groups
    static constexpr int kARows = MP / 2;                        // rows of A (and D) per CTA
    static constexpr int kAccCols = MP == 256 ? BN : BN / 2;     // TMEM columns of one accumulator
    // B scale words: MP=256 copies each 128-column chunk to all four lane quadrants;
    // MP=128 copies the two halves of N to quadrants {0,1} and {2,3} (one 64-row copy)
    static constexpr int kSfbChunks = MP == 256 ? (BN + 127) / 128 : 2;
    static constexpr int kSfbKb = (B4 || S32) ? 4 : 1;           // B words per column per group
    static constexpr int kSfaKb = S32 ? 4 : 1;                   // A words per row per group
    static_assert(!B4 || BN <= 256, "FP4 B: one MMA per K step");
    static_assert(!S32 || (MP == 256 && BN <= 256), "32-K scales: 256-row pairs, one MMA per K step");
    static_assert(!CT || (MP == 256 && BN % 32 == 0 && BN <= 256), "C tile: 32-column boxes of a 256-row pair");
    static constexpr int kSfCols = 4 * kSfaKb + (MP == 256 ? 4 * kSfbChunks : 4) * kSfbKb;
    // Scale words pass through two rings: kSfSlots shared-memory slots (cp.async
    // destination, already in tcgen05.cp order) and kSfTmemSlots TMEM slots (what
    // the MMA reads).  A scale warp loads a group up to kSfLookahead groups before
    // it copies it to TMEM: the load takes a global-memory latency, the peer
    // tells the leader its words have landed, and the copy into TMEM queues
    // behind the issued MMAs.  A shared-memory slot frees when its copy into
    // TMEM completes, which is kSfSlots - kSfLookahead groups before the slot
    // is loaded again.  Four TMEM slots where two accumulators fit beside
    // them; two where that makes room for a second accumulator (BN=240).
    // (32-K scale slots are four times larger; the C tile takes the room of two)
    static constexpr int kSfSlots = S32 ? 4 : (CT ? 6 : 8);
    static constexpr int kSfLookahead = kSfSlots - 3;
    static constexpr int kSfTmemSlots =
        (2 * kAccCols + 4 * kSfCols <= 512 || 2 * kAccCols + 2 * kSfCols > 512) ? 4 : 2;
    static constexpr int kABytes = kARows * kBlockK;            // this CTA's rows of A
    static constexpr int kB1Bytes = (B_ATOM ? 128 : kB1Rows) * kBlockK;
    static constexpr int kB2Bytes = kB2Rows * kBlockK;
    static constexpr int kBBytes = kB1Bytes + kB2Bytes;         // this CTA's half of B
    static constexpr int kStageBytes = kABytes + kBBytes;
    // bytes a K-block's loads deliver (FP4 B: the packed codes, half its stage)
    static constexpr int kTxBytes = kABytes + (B4 ? kBBytes / 2 : kBBytes);
    static constexpr int kSfaBytes = 512 * kSfaKb;
    static constexpr int kSfbBytes = 512 * kSfbChunks * kSfbKb;
    static constexpr int kSfSlotBytes = kSfaBytes + kSfbBytes;
    static constexpr int kEpiChunk = 16;
    static constexpr int kNumChunks = kAccCols / kEpiChunk;      // per TMEM lane quadrant
    static constexpr int kChunksPerWarp = (kNumChunks + 1) / 2;
    static constexpr int kSmemLimit = 232448;
    // grouped-layout unit prefix + info (the 128-row pairs, and the C tile's dense
    // GEMMs, run dense problems only)
    static constexpr int kPrefixBytes = (MP == 256 && !CT) ? (2 * kMaxPairPrefix + 1) * 4 : 0;
    // Operand stages: 256-row pairs keep up to 12, in slots of 4 K-blocks when all
    // 12 fit (the MMA warp waits and commits once per slot), else of one: a slot
    // frees only when all its K-blocks' MMAs are done, so with six stages in slots
    // of two a refill had two slots' MMA time to land, against five K-blocks' with
    // slots of one.  128-row pairs stream B from DRAM at a few bytes per MMA cycle,
    // so what bounds them is the bytes in flight: up to 20 stages in slots of 2
    // K-blocks (a slot frees as soon as its two K-blocks' MMAs complete), 4 at 32
    // columns.
    static constexpr int kMaxStages = MP == 256 ? 12 : 20;
    // Output staging: kStageBufs buffers of one 32-row x 32-byte store box per
    // epilogue warp.  A buffer is rewritten once the TMA store issued from it
    // kStageBufs chunks earlier has read it; the stores queue behind the operand
    // loads in the TMA unit, so more buffers keep more stores in flight.  As many
    // as fit (up to 4) without costing an operand stage.
    static constexpr int kStageBufBytes = 32 * kEpiChunk * 2;
    // C tile: 32-column boxes of this CTA's rows (64-byte rows, 64-byte swizzle); a
    // warp's 32 rows of a box are one TMA box of their own
    static constexpr int kCBoxes = CT ? BN / 32 : 0;
    static constexpr int kCBoxBytes = kARows * 64;
    static constexpr int kCTileBytes = kCBoxes * kCBoxBytes;
    static constexpr int region_bytes(int bufs) {
        return kEpiWarps * bufs * kStageBufBytes > kCTileBytes ? kEpiWarps * bufs * kStageBufBytes : kCTileBytes;
    }
    static constexpr int fixed_bytes(int bufs) {
        return 1024 + region_bytes(bufs) + kSfSlots * kSfSlotBytes + 512 + kPrefixBytes;
    }
    static constexpr int stages_by_smem(int bufs) { return (kSmemLimit - fixed_bytes(bufs)) / kStageBytes; }
    static constexpr int stages_cap(int bufs) {
        return stages_by_smem(bufs) > kMaxStages ? kMaxStages : stages_by_smem(bufs);
    }
    static constexpr int kStageBufs =
        SB > 0 ? SB
        : CT   ? 4
               : (MP == 128 ? 2 : (stages_cap(4) >= stages_cap(2) ? 4 : (stages_cap(3) >= stages_cap(2) ? 3 : 2)));
    static constexpr int kStagingBytes = region_bytes(kStageBufs);
    static constexpr int kFixedBytes = fixed_bytes(kStageBufs);
    static constexpr int kStagesBySmem = (kSmemLimit - kFixedBytes) / kStageBytes;
    static constexpr int kStagesCap = kStagesBySmem > kMaxStages ? kMaxStages : kStagesBySmem;
    // (128-row pairs at 32 columns: four small MMAs per K-block, so the MMA warp's
    // per-slot waits and commits set the pace and slots of 4 K-blocks go faster)
    static constexpr int kGroupKb = MP == 128 ? (BN == 32 ? 4 : 2) : (kStagesCap >= 12 ? 4 : 1);
    // the MMA warp waits for a scale group at slot starts and releases it at the
    // group's last K-block: a slot must not span two 4-K-block scale groups
    static_assert(kGroupKb == 1 || kGroupKb == 2 || kGroupKb == 4, "ring slots divide a scale group");
    static constexpr int kStages = kStagesCap / kGroupKb * kGroupKb;
    static constexpr int kRing = kStages / kGroupKb;
    static constexpr int kNumAcc = (2 * kAccCols + kSfTmemSlots * kSfCols <= 512) ? 2 : 1;
    static constexpr int kTmemCols = 512;
    static_assert(kNumAcc * kAccCols + kSfTmemSlots * kSfCols <= kTmemCols, "TMEM budget");
    static_assert(kRing >= 2, "pipeline too shallow");
    static constexpr int kSmemBytes = kFixedBytes + kStages * kStageBytes;
    static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
    static_assert(kSmemBytes > 116 * 1024, "one CTA per SM (TMEM is allocated whole)");
    // full, empty, tfull, tempty, sf_peer, sfree, sf_ready, sf_tfree, drain, C tile
    // (one per epilogue warp); then the TMEM holder and abort flag, all before the
    // unit prefix 512 bytes on
    static constexpr int kNumBars =
        2 * kRing + 2 * kNumAcc + 2 * kSfSlots + 2 * kSfTmemSlots + 1 + kSfWarps + (CT ? kEpiWarps : 0);
    static_assert(kNumBars * 8 + 8 <= 512, "barrier region");
    static_assert(kSfSlots * kSfSlotBytes >= 2 * (kMaxPsumGroups + 1) * 4, "PSUM segments fit the scale ring");
};

// Output staging of the FP32-output epilogue: four buffers per warp, one operand
// stage fewer where that is their price (that epilogue, not the MMAs, sets the pace
// of the FP32-output GEMMs).
constexpr int kF32StageBufs = 4;
// The bf16 C epilogue keeps its C tile in shared memory where the tile's columns
// are whole 32-column boxes.
template <int BN, int MP, bool WITH_C, bool F32>
constexpr bool kCTile = WITH_C && !F32 && MP == 256 && BN % 32 == 0 && BN <= 256;
template <int BN, int MP, int LAY, bool F32, bool WITH_C = false>
using Bs2Cfg = Bs2Config<BN, MP, (LAY & 2) != 0, (LAY & 4) != 0, F32 ? kF32StageBufs : 0, (LAY & 8) != 0,
                         kCTile<BN, MP, WITH_C, F32>>;

struct PairTile {
    int a_row0;      // this CTA's first row in the 2-D view of A (and D)
    int sfa_x;       // MN index of that row in the packed SFA view
    int sfa_y0;      // row of the packed SFA view for K-slice 0
    int n0;          // first output column of the tile
    int b_row0;      // this CTA's first row of B ([E*N, K] view): its half of the first MMA's columns
    int b2_row0;     // and of the second MMA's (tiles wider than 256 columns)
    int sfb_y0;      // row of the packed SFB view for K-slice 0
    int valid_rows;  // rows of this CTA's MP/2 that are stored (0: none)
    int zero_tail;   // the rest of this CTA's rows are gap rows, written 0 (PSUM layout)
    int d_row0;      // this CTA's first row of D (and C): a_row0 except for the K-grouped layout
    int kb0;         // first 128-K block of the tile's K range
    int nkb;         // 128-K blocks in the tile's K range (K-grouped: 0 for an empty group)
};

// Pair units.  A unit is the row range of one pair tile; the tiles are the
// units crossed with the n-blocks.
//   dense:      unit u = rows [MP u, MP u + MP).
//   contiguous: (MP = 256) m-pair j = rows [256j, 256j + 256): two 128-row
//               blocks, each of one expert or padding.  Both blocks of one
//               expert: one unit.  Otherwise one unit per block that has an
//               expert: the pair still computes 256 rows, but only the CTA
//               holding that block stores.  With PSUM offsets a block's
//               expert comes from the segment starts, and the block's rows
//               past the expert's last row are gap rows, stored as 0.
//   masked:     (MP = 256) expert e gets ceil(masked_m[e] / 256) units of 256
//               of its rows; rows at or past masked_m[e] are not stored.
// For the grouped layouts prefix[i] = units before m-pair (expert) i, built
// once per CTA in shared memory; total units = prefix[count].  info[i] keeps
// what the tile lookup needs without touching global memory: the two blocks'
// experts (contiguous, 16 bits each; PSUM: 8 bits each, 0xFF for none, then
// each block's rows of its expert in 8 bits each) or the clamped masked_m
// (masked).

// Experts of the two blocks of m-pair j (contiguous layout); -1 for padding,
// past the end, or an out-of-range id (reported).
__device__ __forceinline__ void pair_block_experts(const GemmParams &p, int j, int &e0, int &e1) {
    const int r0 = 2 * j * kBlockM, r1 = r0 + kBlockM;
    e0 = __ldg(p.grouped_layout + r0);
    e1 = r1 < p.rows ? __ldg(p.grouped_layout + r1) : -1;
    if (e0 >= p.num_groups) {
        if (p.status) atomicOr(p.status, DG_DEV_BAD_GROUP);
        e0 = -1;
    }
    if (e1 >= p.num_groups) {
        if (p.status) atomicOr(p.status, DG_DEV_BAD_GROUP);
        e1 = -1;
    }
}

__device__ __forceinline__ int clamp_masked_m(const GemmParams &p, int e) {
    int mm = __ldg(p.masked_m + e);
    if (mm < 0 || mm > p.rows) {
        if (p.status) atomicOr(p.status, DG_DEV_BAD_GROUP);
        mm = mm < 0 ? 0 : p.rows;
    }
    return mm;
}

// Largest i with prefix[i] <= u (prefix is non-decreasing, prefix[0] = 0).
__device__ __forceinline__ int prefix_find(const int *prefix, int count, int u) {
    int lo = 0, hi = count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Prefix sums by warp 0 (call with all 32 lanes): on entry x[1..count] hold
// counts; on exit x[i] = x[1] + ... + x[i] and x[0] = 0.
__device__ __forceinline__ void warp0_prefix_sums(int *x, int count, uint32_t lane) {
    const int per = (count + 31) / 32;
    const int lo = static_cast<int>(lane) * per, hi = lo + per < count ? lo + per : count;
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += x[i + 1];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (static_cast<int>(lane) >= o) incl += v;
    }
    int run = incl - sum;
    if (lane == 0) x[0] = 0;
    for (int i = lo; i < hi; ++i) {
        run += x[i + 1];
        x[i + 1] = run;
    }
}

// PSUM contiguous layout: the segment of expert e starts at S_e, S_0 = 0 and
// S_{e+1} = align128(S_e + m_e) = S_e + align128(m_e) (m_e = psum[e] -
// psum[e-1]); rows [S_e + m_e, S_{e+1}) are gap rows.  Fills seg[0..E] and
// cnt[0..E) with the whole CTA; ends with __syncthreads.  A decreasing psum
// (the count is taken as 0) or segments ending past the rows set
// DG_DEV_BAD_GROUP.
__device__ __forceinline__ void build_psum_segments(const GemmParams &p, int *seg, int *cnt) {
    const int E = p.num_groups;
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
        int m = __ldg(p.psum + i) - (i > 0 ? __ldg(p.psum + i - 1) : 0);
        if (m < 0) {
            if (p.status) atomicOr(p.status, DG_DEV_BAD_GROUP);
            m = 0;
        }
        cnt[i] = m;
        seg[i + 1] = (m + kBlockM - 1) / kBlockM * kBlockM;
    }
    __syncthreads();
    if (threadIdx.x < 32) warp0_prefix_sums(seg, E, threadIdx.x);
    __syncthreads();
    if (threadIdx.x == 0 && seg[E] > p.rows && p.status) atomicOr(p.status, DG_DEV_BAD_GROUP);
}

// Builds prefix[0..count] and info[0..count) (count = m-pairs or experts)
// with the whole CTA: unit counts in parallel, then one warp scans them.
// scratch (2 * (kMaxPsumGroups + 1) ints, dead afterwards) holds the PSUM
// segments.  Ends with __syncthreads.
__device__ __forceinline__ void build_pair_prefix(const GemmParams &p, int *prefix, int *info, int *scratch) {
    if (p.mode == kModeKGrouped) {
        // prefix[e]: first 128-K block of group e; info[e]: its first packed scale row
        // (each group's scale rows are packed on their own, 4 per word)
        const int E = p.num_groups;
        for (int i = threadIdx.x; i < E; i += blockDim.x) {
            int k = __ldg(p.ks + i);
            if (k < 0 || k % kBlockK != 0) {
                if (p.status) atomicOr(p.status, DG_DEV_BAD_GROUP);
                k = 0;
            }
            prefix[i + 1] = k / kBlockK;
            info[i + 1] = (k / kBlockK + 3) / 4;
        }
        __syncthreads();
        if (threadIdx.x < 32) warp0_prefix_sums(prefix, E, threadIdx.x);
        else if (threadIdx.x < 64) warp0_prefix_sums(info, E, threadIdx.x - 32);
        __syncthreads();
        // more K than the operands hold: the loads past the end read zeros, the words nothing
        if (threadIdx.x == 0 && p.status &&
            (prefix[E] > p.num_k_blocks || ((p.layout & 8) ? prefix[E] : info[E]) > p.sfa_slices))
            atomicOr(p.status, DG_DEV_BAD_GROUP);
        return;
    }
    const bool psum = p.mode == kModeContiguous && p.psum != nullptr;
    int *seg = scratch, *cnt = scratch + kMaxPsumGroups + 1;
    if (psum) build_psum_segments(p, seg, cnt);
    const int count = p.mode == kModeMasked ? p.num_groups : p.num_m_blocks;
    for (int i = threadIdx.x; i < count; i += blockDim.x) {
        int units;
        if (p.mode == kModeMasked) {
            const int mm = clamp_masked_m(p, i);
            info[i] = mm;
            units = (mm + 2 * kBlockM - 1) / (2 * kBlockM);
        } else if (psum) {
            // each block's expert (0xFF: none) and the rows of it that are the expert's
            uint32_t word = 0;
            int e[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row0 = (2 * i + h) * kBlockM;
                int s = -1, v = 0;
                if (row0 < p.rows) {
                    s = prefix_find(seg, p.num_groups + 1, row0);
                    if (s >= p.num_groups) {
                        s = -1;
                    } else {
                        v = seg[s] + cnt[s] - row0;
                        v = v < kBlockM ? v : kBlockM;
                        v = v < p.rows - row0 ? v : p.rows - row0;
                    }
                }
                e[h] = s;
                word |= (static_cast<uint32_t>(s & 0xFF) << (8 * h)) | (static_cast<uint32_t>(v) << (16 + 8 * h));
            }
            info[i] = static_cast<int>(word);
            units = (e[0] >= 0 && e[0] == e[1]) ? 1 : (e[0] >= 0) + (e[1] >= 0);
        } else {
            int e0, e1;
            pair_block_experts(p, i, e0, e1);
            info[i] = (e0 & 0xFFFF) | (e1 << 16);
            units = (e0 >= 0 && e0 == e1) ? 1 : (e0 >= 0) + (e1 >= 0);
        }
        prefix[i + 1] = units;
    }
    __syncthreads();
    if (threadIdx.x < 32) warp0_prefix_sums(prefix, count, threadIdx.x);
    __syncthreads();
}

__device__ __forceinline__ int pair_units(const GemmParams &p, const int *prefix) {
    if (p.mode == kModeDense) return p.num_m_blocks;
    if (p.mode == kModeKGrouped) return p.num_groups * p.num_m_blocks;   // m-units per group
    return prefix[p.mode == kModeMasked ? p.num_groups : p.num_m_blocks];
}

// Pair tile t (< units * n-blocks) for cluster rank `rank`; units are grouped
// along M in runs of group_m so that pairs running at the same time share B.
template <int BN, int MP>
__device__ __forceinline__ void get_pair_tile(const GemmParams &p, const int *prefix, const int *info,
                                              int num_units, int psf_k, int t, int rank, PairTile &tile) {
    const int per_group = p.group_m * p.num_n_blocks;
    const int g = t / per_group;
    const int first = g * p.group_m;
    const int rem = num_units - first;
    const int gsize = rem < p.group_m ? rem : p.group_m;
    const int r = t - g * per_group;
    const int u = first + r % gsize;
    const int nb = r / gsize;
    tile.n0 = nb * BN;
    int group = 0;
    tile.zero_tail = 0;
    tile.kb0 = 0;
    tile.nkb = p.num_k_blocks;
    if (MP == 128 || p.mode == kModeDense) {
        tile.a_row0 = u * MP + rank * (MP / 2);
        tile.sfa_x = tile.a_row0;
        tile.sfa_y0 = 0;
        tile.valid_rows = MP / 2;
    } else if (p.mode == kModeKGrouped) {
        // unit u = (group e, m-unit): A and B are [K][M] / [K][N], so the tile's
        // coordinates along M and N are those of a dense tile; D is [E * M][N]
        const int e = u / p.num_m_blocks;
        const int m0 = (u - e * p.num_m_blocks) * MP + rank * (MP / 2);
        tile.a_row0 = m0;
        tile.sfa_x = m0;
        // packed scale rows: per group 4 K-blocks a row; 32-K scales: one row a K-block
        tile.sfa_y0 = (p.layout & 8) ? prefix[e] : info[e];
        tile.d_row0 = e * p.group_rows + m0;
        const int v = p.group_rows - m0;
        tile.valid_rows = v <= 0 ? 0 : (v < MP / 2 ? v : MP / 2);
        tile.kb0 = prefix[e];
        tile.nkb = prefix[e + 1] - prefix[e];
    } else if (p.mode == kModeContiguous) {
        const int j = prefix_find(prefix, p.num_m_blocks, u);
        int e0, e1, v0 = kBlockM, v1 = kBlockM;
        if (p.psum != nullptr) {
            const uint32_t w = static_cast<uint32_t>(info[j]);
            e0 = (w & 0xFFu) == 0xFFu ? -1 : static_cast<int>(w & 0xFFu);
            e1 = ((w >> 8) & 0xFFu) == 0xFFu ? -1 : static_cast<int>((w >> 8) & 0xFFu);
            v0 = static_cast<int>((w >> 16) & 0xFFu);
            v1 = static_cast<int>(w >> 24);
        } else {
            e0 = static_cast<int16_t>(info[j] & 0xFFFF);
            e1 = info[j] >> 16;
        }
        tile.a_row0 = j * 2 * kBlockM + rank * kBlockM;
        tile.sfa_x = tile.a_row0;
        tile.sfa_y0 = 0;
        if (e0 >= 0 && e0 == e1) {
            group = e0;
            tile.valid_rows = rank == 0 ? v0 : v1;
        } else {
            // the unit's block: the first valid one, or the second if this is the pair's second unit
            const int h = (e0 >= 0 && u > prefix[j]) || e0 < 0 ? 1 : 0;
            group = h == 0 ? e0 : e1;
            tile.valid_rows = rank == h ? (h == 0 ? v0 : v1) : 0;
        }
        tile.zero_tail = p.psum != nullptr && tile.valid_rows > 0;
    } else {
        const int e = prefix_find(prefix, p.num_groups, u);
        const int local0 = (u - prefix[e]) * 2 * kBlockM + rank * kBlockM;
        const int v = info[e] - local0;
        group = e;
        tile.a_row0 = e * p.rows + local0;
        tile.sfa_x = local0;
        tile.sfa_y0 = e * psf_k;
        tile.valid_rows = v <= 0 ? 0 : (v < kBlockM ? v : kBlockM);
    }
    tile.b_row0 = group * p.n + tile.n0 + rank * Bs2Config<BN, MP>::kB1Rows;
    tile.b2_row0 = group * p.n + tile.n0 + Bs2Config<BN, MP>::kBN1 + rank * Bs2Config<BN, MP>::kB2Rows;
    // (FP4 B: one packed scale row per K-block, so an expert's rows start at e * K-blocks)
    tile.sfb_y0 = p.mode == kModeKGrouped ? tile.sfa_y0 : group * ((p.layout & 4) ? p.num_k_blocks : psf_k);
    if (p.mode != kModeKGrouped) tile.d_row0 = tile.a_row0;
}

// LAY: operand layouts, bit 0 = A MN-major (stored [K][M]), bit 1 = B MN-major
// (stored [K][N]), bit 2 = B is FP4 (E2M1, K-major, one scale per 32 K); 0 is
// the NT layout (both K-major FP8).  An MN-major operand's
// stage is a TMA box of 128 MN-bytes x 128 K-rows with 128-byte swizzle: one
// swizzle atom along MN (MP=256; an MN-major B half of BN/2 <= 128 columns,
// the rest of the atom unread), 8-row groups 1024 bytes apart, and a 32-K step
// of the MMA 4096 bytes on; the instruction descriptor's transpose bits (15:
// A, 16: B) select the layout.
template <int BN, bool WITH_C, int MP, bool F32 = false, int LAY = 0>
__global__ void __launch_bounds__(Bs2Config<BN, MP>::kThreads, 1) __cluster_dims__(2, 1, 1)
    dg_bs2_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                       const __grid_constant__ CUtensorMap tm_b,
                       const __grid_constant__ CUtensorMap tm_b2,
                       const __grid_constant__ CUtensorMap tm_d,
                       const __grid_constant__ CUtensorMap tm_c, const GemmParams p) {
    constexpr bool A_MN = (LAY & 1) != 0, B_MN = (LAY & 2) != 0, B4 = (LAY & 4) != 0, S32 = (LAY & 8) != 0;
    static_assert(!B4 || (!A_MN && !B_MN && !F32), "FP4 B: K-major operands, bf16 D");
    using Cfg = Bs2Cfg<BN, MP, LAY, F32, WITH_C>;
    static_assert(!(A_MN || B_MN) || (MP == 256 && BN <= 256), "MN-major operands: 256-row pair tiles, one MMA");
    constexpr int S = Cfg::kStages;
    constexpr int R = Cfg::kRing;
    constexpr int G = Cfg::kGroupKb;
    static_assert(!(A_MN || B_MN) || G * kBlockK <= 256, "an MN-major box holds at most 256 K rows");
    constexpr int NUM_ACC = Cfg::kNumAcc;
    constexpr int NSF = Cfg::kSfSlots;       // shared-memory scale slots
    constexpr int NTS = Cfg::kSfTmemSlots;   // TMEM scale slots
    constexpr int MMA_M = MP;
    constexpr int ACC = Cfg::kAccCols;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *smem_a = smem;
    uint8_t *smem_b = smem_a + S * Cfg::kABytes;
    uint8_t *smem_stage_out = smem_b + S * Cfg::kBBytes;
    uint8_t *smem_sf = smem_stage_out + Cfg::kStagingBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_sf + NSF * Cfg::kSfSlotBytes);
    uint64_t *full_bar = bars;                        // [R] leader: both CTAs' stages landed
    uint64_t *empty_bar = full_bar + R;               // [R] both: MMAs done with the slot
    uint64_t *tfull_bar = empty_bar + R;              // [NUM_ACC] both: accumulator complete
    uint64_t *tempty_bar = tfull_bar + NUM_ACC;       // [NUM_ACC] leader: both epilogues drained
    uint64_t *sf_peer_bar = tempty_bar + NUM_ACC;     // [NSF] leader: peer's words landed
    uint64_t *sf_sfree_bar = sf_peer_bar + NSF;       // [NSF] both: words copied out of the slot
    uint64_t *sf_ready_bar = sf_sfree_bar + NSF;      // [NTS] leader: words in both TMEMs
    uint64_t *sf_tfree_bar = sf_ready_bar + NTS;      // [NTS] leader: MMAs done with the slot
    uint64_t *drain_bar = sf_tfree_bar + NTS;         // [1 + kSfWarps] MMA warp, scale warps
    uint64_t *cfull_bar = drain_bar + 1 + Cfg::kSfWarps;   // [kEpiWarps, C tile] a warp's C boxes landed
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(cfull_bar + (Cfg::kCBoxes > 0 ? Cfg::kEpiWarps : 0));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int *prefix = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(bars) + 512);  // grouped layouts
    int *pinfo = prefix + kMaxPairPrefix + 1;

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    const int rank = static_cast<int>(cluster_ctarank());   // 0 = leader
    const bool leader = rank == 0;
    const int pair_id = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;
    const int groups_per_tile = (p.num_k_blocks + 3) >> 2;
    const int psf_k = groups_per_tile;

    if (warp == 0) {
        // the barriers are contiguous from full_bar to the TMEM holder; the lanes of
        // warp 0 initialise them, each fencing its own inits
        const int num_bars = static_cast<int>(reinterpret_cast<uint64_t *>(tmem_holder) - bars);  // <= kNumBars
        for (int i = static_cast<int>(lane); i < num_bars; i += 32) {
            uint64_t *b = bars + i;
            mbar_init(b, b >= tempty_bar && b < tempty_bar + NUM_ACC ? 2 * Cfg::kEpiWarps : 1);
        }
        if (lane == 0) *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
        if constexpr (Cfg::kBN2 > 0) tma_prefetch_desc(&tm_b2);
        tma_prefetch_desc(&tm_d);
        if (Cfg::kCBoxes > 0 && p.c_tma) tma_prefetch_desc(&tm_c);
    }
    // Nothing above reads global memory: it overlaps the previous grid's tail when
    // launched as a programmatic dependent.  From here on every thread may read
    // inputs or write D.
    grid_launch_dependents();
    grid_dependency_wait();
    // (the scale ring is free until the roles start: PSUM segments go there)
    if (MP == 256 && p.mode != kModeDense) build_pair_prefix(p, prefix, pinfo, reinterpret_cast<int *>(smem_sf));
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, Cfg::kTmemCols);
        tmem_relinquish_pair();
    }
    // the producer needs no TMEM: it starts loading while the others wait for the allocation
    if (warp != 0) {
        tc_fence_before_sync();
        named_bar_sync(1, Cfg::kThreads - 32);
        tc_fence_after_sync();
    }
    const uint32_t tmem_base = warp != 0 ? *tmem_holder : 0u;
    const uint32_t sf_col0 = NUM_ACC * ACC;
    const int num_units = MP == 128 ? p.num_m_blocks : pair_units(p, prefix);
    const int num_tiles = num_units * p.num_n_blocks;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs, whole warp)
        const uint32_t leader_full = mapa_shared(smem_u32(full_bar), 0);
        int slot = 0;
        uint32_t phase = 0;
        uint32_t issued = 0;
        bool drop = (p.debug_flags & DG_DEBUG_DROP_ONE_LOAD) && pair_id == 0;
        for (int t = pair_id; t < num_tiles; t += num_pairs) {
            PairTile tile;
            get_pair_tile<BN, MP>(p, prefix, pinfo, num_units, psf_k, t, rank, tile);
            for (int kb0 = 0; kb0 < tile.nkb; kb0 += G) {
                const int nk = tile.nkb - kb0 < G ? tile.nkb - kb0 : G;
                const int kg0 = tile.kb0 + kb0;   // the slot's first 128-K block in the operands
                if (!mbar_wait_warp(&empty_bar[slot], phase ^ 1, ctl, DG_DEV_TIMEOUT)) goto prod_done;
                if (drop) {
                    drop = false;  // diagnostic: leave this slot empty
                } else {
                    const uint32_t fb = leader_full + slot * 8;
                    if constexpr (A_MN || B_MN) {
                        // an MN-major operand: one box of 128 MN-bytes x G*128 K-rows fills the
                        // slot; the K-major one: G boxes (K-blocks past K are out of bounds,
                        // zero-filled, and still count their bytes)
                        if (elect_one()) {
                            if (leader) mbar_arrive_expect_tx(&full_bar[slot], 2 * G * Cfg::kStageBytes);
                            uint8_t *a_slot = smem_a + slot * G * Cfg::kABytes;
                            uint8_t *b_slot = smem_b + slot * G * Cfg::kBBytes;
                            if constexpr (A_MN) {
                                tma_load_2d_pair(a_slot, &tm_a, fb, tile.a_row0, kg0 * kBlockK);
                            } else {
#pragma unroll
                                for (int j = 0; j < G; ++j)
                                    tma_load_2d_pair(a_slot + j * Cfg::kABytes, &tm_a, fb, (kg0 + j) * kBlockK,
                                                     tile.a_row0);
                            }
                            if constexpr (B_MN) {
                                tma_load_2d_pair(b_slot, &tm_b, fb, tile.b_row0, kg0 * kBlockK);
                            } else {
#pragma unroll
                                for (int j = 0; j < G; ++j)
                                    tma_load_2d_pair(b_slot + j * Cfg::kB1Bytes, &tm_b, fb, (kg0 + j) * kBlockK,
                                                     tile.b_row0);
                            }
                        }
                    } else if (p.ab_3d) {
                        // one load per operand fills the slot's G stages; K-blocks past the
                        // end of K are out of bounds (zero-filled) and still count their bytes
                        if (elect_one()) {
                            if (leader) mbar_arrive_expect_tx(&full_bar[slot], 2 * G * Cfg::kStageBytes);
                            uint8_t *b_slot = smem_b + slot * G * Cfg::kBBytes;
                            tma_load_3d_pair(smem_a + slot * G * Cfg::kABytes, &tm_a, fb, 0, tile.a_row0, kg0);
                            tma_load_3d_pair(b_slot, &tm_b, fb, 0, tile.b_row0, kg0);
                            if constexpr (Cfg::kBN2 > 0)
                                tma_load_3d_pair(b_slot + G * Cfg::kB1Bytes, &tm_b2, fb, 0, tile.b2_row0, kg0);
                        }
                    } else if (elect_one()) {
                        // the leader expects both CTAs' bytes; each CTA's loads count there
                        if (leader) mbar_arrive_expect_tx(&full_bar[slot], 2 * nk * Cfg::kTxBytes);
                        // a slot's B: the G K-blocks of the first MMA's rows, then the G
                        // K-blocks of the second's
                        auto load_kb = [&](int j) {
                            const int kb = kg0 + j;
                            uint8_t *b_slot = smem_b + slot * G * Cfg::kBBytes;
                            tma_load_2d_pair(smem_a + (slot * G + j) * Cfg::kABytes, &tm_a, fb, kb * kBlockK,
                                             tile.a_row0);
                            tma_load_2d_pair(b_slot + j * Cfg::kB1Bytes, &tm_b, fb, kb * kBlockK, tile.b_row0);
                            if constexpr (Cfg::kBN2 > 0)
                                tma_load_2d_pair(b_slot + G * Cfg::kB1Bytes + j * Cfg::kB2Bytes, &tm_b2, fb,
                                                 kb * kBlockK, tile.b2_row0);
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
        // the leader waits for the last fill of every slot (both CTAs' bytes count there)
        if (lane == 0 && leader)
            for (int s = 0; s < R; ++s)
                if (issued & (1u << s)) mbar_wait_drain(&full_bar[s], s < slot ? phase : phase ^ 1, ctl);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader, whole warp)
        if (leader) {
            int slot = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int g = 0;
            const uint64_t a_desc_base = A_MN ? make_smem_desc(smem_u32(smem_a), 16384, 1024, kSwizzle128B)
                                              : make_desc_kmajor_sw128(smem_u32(smem_a));
            const uint64_t b_desc_base = B_MN ? make_smem_desc(smem_u32(smem_b), 16384, 1024, kSwizzle128B)
                                              : make_desc_kmajor_sw128(smem_u32(smem_b));
            // a 32-K step: 32 bytes along a K-major row, 32 rows (4096 bytes) of an MN-major tile
            constexpr uint64_t kStepA = A_MN ? (4096 >> 4) : 2, kStepB = B_MN ? (4096 >> 4) : 2;
            // (B format 5: E2M1)
            constexpr uint32_t idesc_base = make_idesc_mxf8(MMA_M, Cfg::kBN1, 0, 0) | (A_MN ? 1u << 15 : 0u) |
                                            (B_MN ? 1u << 16 : 0u) | (B4 ? 5u << 10 : 0u);
            constexpr uint32_t idesc2_base = make_idesc_mxf8(MMA_M, Cfg::kBN2 > 0 ? Cfg::kBN2 : 16, 0, 0);
            for (int t = pair_id; t < num_tiles; t += num_pairs) {
                // the tile's 128-K blocks (K-grouped: its group's; none for an empty group,
                // whose accumulator is then handed over unwritten and read as zero)
                int nkb = p.num_k_blocks;
                if (p.mode == kModeKGrouped) {
                    PairTile tl;
                    get_pair_tile<BN, MP>(p, prefix, pinfo, num_units, psf_k, t, rank, tl);
                    nkb = tl.nkb;
                }
                if (!mbar_wait_cluster_warp(&tempty_bar[acc], acc_phase ^ 1, ctl, DG_DEV_TIMEOUT)) goto mma_done;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * ACC;
                for (int kb0 = 0; kb0 < nkb; kb0 += G) {
                    const int nk = nkb - kb0 < G ? nkb - kb0 : G;
                    const int sslot = g % NTS;
                    if ((kb0 & 3) == 0) {
                        if (!mbar_wait_warp(&sf_ready_bar[sslot], (g / NTS) & 1, ctl, DG_DEV_TIMEOUT))
                            goto mma_done;
                    }
                    if (!mbar_wait_warp(&full_bar[slot], phase, ctl, DG_DEV_TIMEOUT)) goto mma_done;
                    tc_fence_after_sync();
                    const uint32_t sfa_tmem = tmem_base + sf_col0 + sslot * Cfg::kSfCols;
                    const uint64_t a_desc0 = a_desc_base + static_cast<uint64_t>(slot * G * (Cfg::kABytes >> 4));
                    const uint64_t b_desc0 = b_desc_base + static_cast<uint64_t>(slot * G * (Cfg::kBBytes >> 4));
                    const int kb_last = kb0 + nk - 1;
                    const bool group_end = (kb_last & 3) == 3 || kb_last == nkb - 1;
                    if (elect_one()) {
                        auto mma_kb = [&](int j) {
                            const int kb = kb0 + j;
                            const uint32_t sf = static_cast<uint32_t>(kb & 3);
                            const uint32_t idesc = idesc_base | (sf << 4) | (sf << 29);
                            const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(j * (Cfg::kABytes >> 4));
                            const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(j * (Cfg::kB1Bytes >> 4));
                            // FP4 B (and 32-K scales): this K-block's B cells, whose byte k
                            // scales the k-th 32 K; 32-K scales: the same for A's cells
                            constexpr int kSfbRegionCols = MP == 256 ? 4 * Cfg::kSfbChunks : 4;
                            const uint32_t sfb_tmem = sfa_tmem + 4 * Cfg::kSfaKb +
                                                      ((B4 || S32) ? static_cast<uint32_t>((kb & 3) * kSfbRegionCols) : 0u);
                            const uint32_t sfa_cells = sfa_tmem + (S32 ? static_cast<uint32_t>(4 * (kb & 3)) : 0u);
#pragma unroll
                            for (int k = 0; k < kBlockK / 32; ++k) {
                                // instruction descriptor: B's scale-factor id in bits 4-5, A's in 29-30
                                const uint32_t sfk = static_cast<uint32_t>(k);
                                const uint32_t idesc_k = S32  ? (idesc_base | (sfk << 4) | (sfk << 29))
                                                         : B4 ? (idesc_base | (sfk << 4) | (sf << 29))
                                                              : idesc;
                                tc_mma_mxf8_pair(d_tmem, a_desc + kStepA * k, b_desc + kStepB * k, idesc_k, sfa_cells,
                                                 sfb_tmem, (kb | k) != 0);
                                if constexpr (Cfg::kBN2 > 0) {
                                    // columns [kBN1, BN): their accumulator columns, B rows and
                                    // B scale cells (column x at lane x % 32, cell x / 32)
                                    const uint64_t b2_desc =
                                        b_desc0 + static_cast<uint64_t>((G * Cfg::kB1Bytes + j * Cfg::kB2Bytes) >> 4);
                                    tc_mma_mxf8_pair(d_tmem + Cfg::kBN1, a_desc + 2 * k, b2_desc + 2 * k,
                                                     idesc2_base | (sf << 4) | (sf << 29), sfa_tmem,
                                                     sfa_tmem + 4 + Cfg::kBN1 / 32, (kb | k) != 0);
                                }
                            }
                        };
                        if (nk == G) {
#pragma unroll
                            for (int j = 0; j < G; ++j) mma_kb(j);
                        } else {
                            for (int j = 0; j < nk; ++j) mma_kb(j);
                        }
                        tc_commit_pair(&empty_bar[slot], 0x3);
                        if (group_end) tc_commit_pair(&sf_tfree_bar[sslot], 0x1);
                    }
                    __syncwarp();
                    if (group_end) ++g;
                    if (++slot == R) { slot = 0; phase ^= 1; }
                }
                if (elect_one()) tc_commit_pair(&tfull_bar[acc], 0x3);
                __syncwarp();
                if (++acc == NUM_ACC) { acc = 0; acc_phase ^= 1; }
            }
        mma_done:
            if (elect_one()) {
                tc_commit_pair(&drain_bar[0], 0x1);
                mbar_wait(&drain_bar[0], 0, ctl, DG_DEV_TIMEOUT);
            }
            __syncwarp();
        }
    } else if (warp >= Cfg::kSfWarp) {
        // ------------------------------------------------------------ scale-factor warps (both CTAs)
        // kSfWarps warps take the (tile, 4-K-block group) sequence in turns, so
        // the waits and tcgen05 issues of one group overlap those of the next.
        // A warp reuses only its own slots (kSfSlots is a multiple of kSfWarps).
        // This CTA's words of a group (its A rows, all BN columns of B) land in a
        // slot by cp.async, up to kSfLookahead groups ahead of the group being
        // copied to TMEM: plain loads keep the TMA unit to the operand tiles and
        // the producer's loop to A and B.  Each 4-byte copy puts its word where
        // tcgen05.cp wants it (source row r holds words r, r+32, r+64, r+96 of a
        // 128-word chunk; for MP=128 the two halves of N are rows 0-31 and
        // 32-63), so the words need no reordering.  A word past the packed row
        // length reads nothing and lands as zero.
        constexpr int NW = Cfg::kSfWarps;
        static_assert(NSF % NW == 0, "scale slots per warp");
        const int sw = static_cast<int>(warp) - Cfg::kSfWarp;
        const uint32_t leader_peer = mapa_shared(smem_u32(sf_peer_bar), 0);
        // groups of 4 K-blocks in tile t: the same for every tile, except in the
        // K-grouped layout, where a tile has its group's K-blocks (maybe none)
        auto tile_groups = [&](int t) -> int {
            if (p.mode != kModeKGrouped) return groups_per_tile;
            PairTile tl;
            get_pair_tile<BN, MP>(p, prefix, pinfo, num_units, psf_k, t, rank, tl);
            return (tl.nkb + 3) >> 2;
        };
        // this pair's groups: those of tiles pair_id, pair_id + num_pairs, ...
        int num_groups_here = 0;
        if (p.mode != kModeKGrouped)
            num_groups_here =
                pair_id < num_tiles ? (num_tiles - pair_id + num_pairs - 1) / num_pairs * groups_per_tile : 0;
        else
            for (int t = pair_id; t < num_tiles; t += num_pairs) num_groups_here += tile_groups(t);
        int lt = pair_id, lj = sw;  // tile and group of the next load
        int lt_groups = lt < num_tiles ? tile_groups(lt) : 0;
        // moves (lt, lj) past the end of tile lt's groups
        auto settle = [&]() {
            while (lt < num_tiles && lj >= lt_groups) {
                lj -= lt_groups;
                lt += num_pairs;
                lt_groups = lt < num_tiles ? tile_groups(lt) : 0;
            }
        };
        settle();
        int gl = sw;                // next group to load (this warp's: sw, sw + NW, ...)
        int st_t = -1;              // tile whose coordinates st holds
        PairTile st;
        // issues the loads of group gl, or an empty commit group past the last one;
        // false if the CTA is aborting
        auto load_group = [&]() -> bool {
            if (gl < num_groups_here) {
                const int slot = gl % NSF;
                // the slot's previous words have been copied to TMEM
                if (gl >= NSF &&
                    !mbar_wait_warp(&sf_sfree_bar[slot], ((gl / NSF) & 1) ^ 1, ctl, DG_DEV_TIMEOUT))
                    return false;
                if (st_t != lt) {
                    get_pair_tile<BN, MP>(p, prefix, pinfo, num_units, psf_k, lt, rank, st);
                    st_t = lt;
                }
                const uint32_t dst0 = smem_u32(smem_sf + slot * Cfg::kSfSlotBytes);
                // word x of packed row y of one scale tensor -> word w of the slot
                auto copy_word = [&](const uint32_t *base, int ld, int slices, int x, int y, uint32_t w) {
                    const bool in = x < ld && y < slices;
                    cp_async_4(dst0 + 4u * w, in ? base + static_cast<int64_t>(y) * ld + x : base, in ? 4u : 0u);
                };
                const int ya = st.sfa_y0 + lj, yb = st.sfb_y0 + lj;
                // 32-K scales: one packed row per K-block, the group's 4 rows in 4 regions
#pragma unroll
                for (int ja = 0; ja < Cfg::kSfaKb; ++ja)
#pragma unroll
                    for (int q = 0; q < Cfg::kARows / 32; ++q)
                        copy_word(p.sfa_words, p.sfa_ld, p.sfa_slices, st.sfa_x + 32 * q + static_cast<int>(lane),
                                  S32 ? st.sfa_y0 + 4 * lj + ja : ya, 128 * ja + 4 * lane + q);
                if constexpr (MP == 256) {
                    // FP4 B: one packed row per K-block, the group's 4 rows in 4 regions
#pragma unroll
                    for (int jj = 0; jj < Cfg::kSfbKb; ++jj)
#pragma unroll
                        for (int c = 0; c < Cfg::kSfbChunks; ++c)
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                copy_word(p.sfb_words, p.sfb_ld, p.sfb_slices,
                                          st.n0 + 128 * c + 32 * q + static_cast<int>(lane),
                                          (B4 || S32) ? st.sfb_y0 + 4 * lj + jj : yb,
                                          128 * Cfg::kSfaKb + 128 * (jj * Cfg::kSfbChunks + c) + 4 * lane + q);
                } else {
                    constexpr int kHalf = BN / 2;
#pragma unroll
                    for (int jj = 0; jj < Cfg::kSfbKb; ++jj)
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int q = 0; q < (kHalf + 31) / 32; ++q)
                                if (32 * q + static_cast<int>(lane) < kHalf)
                                    copy_word(p.sfb_words, p.sfb_ld, p.sfb_slices,
                                              st.n0 + h * kHalf + 32 * q + static_cast<int>(lane),
                                              B4 ? st.sfb_y0 + 4 * lj + jj : yb, 128 + 256 * jj + 4 * (32 * h + lane) + q);
                }
                lj += NW;
                settle();
            }
            cp_async_commit();
            gl += NW;
            return true;
        };
        bool copied = false;
        for (int g = sw; g < num_groups_here; g += NW) {
            const int slot = g % NSF;
            // up to two more of this warp's groups, kSfLookahead ahead at most;
            // the first group starts at once
            for (int i = 0; i < 2 && gl <= g + Cfg::kSfLookahead; ++i)
                if (!load_group()) goto sf_done;
            cp_async_wait_dyn((gl - g) / NW - 1);         // this lane's words of group g
            fence_proxy_async_smem();                     // visible to tcgen05.cp
            __syncwarp();
            uint32_t *sfa_buf = reinterpret_cast<uint32_t *>(smem_sf + slot * Cfg::kSfSlotBytes);
            uint32_t *sfb_buf = sfa_buf + 128 * Cfg::kSfaKb;
            if (!leader) {
                // tell the leader this CTA's words for the group are in place
                if (lane == 0) mbar_arrive_remote(leader_peer + slot * 8);
            } else {
                const int tslot = g % NTS;
                if (!mbar_wait_cluster_warp(&sf_peer_bar[slot], (g / NSF) & 1, ctl, DG_DEV_TIMEOUT))
                    goto sf_done;
                if (!mbar_wait_warp(&sf_tfree_bar[tslot], ((g / NTS) & 1) ^ 1, ctl, DG_DEV_TIMEOUT))
                    goto sf_done;
                if (lane == 0) {
                    tc_fence_after_sync();
                    const uint32_t sfa_tmem = tmem_base + sf_col0 + tslot * Cfg::kSfCols;
#pragma unroll
                    for (int ja = 0; ja < Cfg::kSfaKb; ++ja)
                        tc_cp_32x128b_warpx4_pair(sfa_tmem + 4 * ja, make_desc_sf_32x128b(smem_u32(sfa_buf + 128 * ja)));
                    if constexpr (MP == 256) {
#pragma unroll
                        for (int c = 0; c < Cfg::kSfbKb * Cfg::kSfbChunks; ++c)
                            tc_cp_32x128b_warpx4_pair(sfa_tmem + 4 * Cfg::kSfaKb + 4 * c,
                                                      make_desc_sf_32x128b(smem_u32(sfb_buf + c * 128)));
                    } else {
#pragma unroll
                        for (int jj = 0; jj < Cfg::kSfbKb; ++jj)
                            tc_cp_64x128b_warpx2_01_23_pair(sfa_tmem + 4 + 4 * jj,
                                                            make_desc_sf_32x128b(smem_u32(sfb_buf + 256 * jj)));
                    }
                    tc_commit_pair(&sf_ready_bar[tslot], 0x1);
                    tc_commit_pair(&sf_sfree_bar[slot], 0x3);   // both CTAs may refill the slot
                    copied = true;
                }
            }
            __syncwarp();
        }
    sf_done:
        cp_async_wait<0>();
        if (lane == 0 && leader && copied) {
            tc_commit_pair(&drain_bar[1 + sw], 0x1);
            mbar_wait(&drain_bar[1 + sw], 0, ctl, DG_DEV_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const uint32_t ew = warp - 2;
        const uint32_t quad = warp & 3;       // TMEM lane quadrant this warp may access
        const uint32_t half = ew >> 2;        // which interleaved half of the quadrant's column chunks
        // the quadrant's 32 rows (offset in this CTA's rows) and D-column offset of its TMEM columns
        const int row_off = MP == 256 ? static_cast<int>(quad) * 32 : static_cast<int>(quad & 1) * 32;
        const int col_off = MP == 256 ? 0 : static_cast<int>(quad >> 1) * (BN / 2);
        const uint32_t leader_tempty = mapa_shared(smem_u32(tempty_bar), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t buf = 0;
        uint8_t *stage_out = smem_stage_out + ew * Cfg::kStageBufs * Cfg::kStageBufBytes;
        // C (bf16) of one chunk of this thread's row; zero outside [rows, n)
        // (the bf16 C epilogue gives each warp of a quadrant a contiguous half of the
        // chunks, so that two adjacent chunks go out in one store box)
        auto load_c = [&](const PairTile &tl, int j, uint32_t (&dst)[8]) {
            const int c = j + static_cast<int>(half) * Cfg::kChunksPerWarp;
            const int row = tl.d_row0 + row_off + lane;
            const int col0 = tl.n0 + col_off + c * Cfg::kEpiChunk;
            if (p.c_v8 && c < Cfg::kNumChunks && row < p.rows && col0 + 16 <= p.n) {
                ld_global_cg_v8(p.c + static_cast<int64_t>(row) * p.ldc + col0, dst);
                return;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint4 cv = make_uint4(0u, 0u, 0u, 0u);
                if (c < Cfg::kNumChunks && row < p.rows && col0 + 8 * h < p.n)
                    cv = __ldg(reinterpret_cast<const uint4 *>(p.c + static_cast<int64_t>(row) * p.ldc +
                                                               col0 + 8 * h));
                dst[4 * h + 0] = cv.x;
                dst[4 * h + 1] = cv.y;
                dst[4 * h + 2] = cv.z;
                dst[4 * h + 3] = cv.w;
            }
        };
        // bf16 C: a tile's C rows are fetched into L2 a tile ahead, one bulk prefetch
        // of the whole row segment per row (long, contiguous DRAM reads), and loaded
        // into registers from L2 just before the tile's epilogue.  Loading a whole
        // tile ahead into registers instead kept thousands of scattered row loads in
        // flight during the stores, which then queued behind them.
        uint32_t cpk[(WITH_C && !F32) ? Cfg::kChunksPerWarp : 1][8];
        auto prefetch_c = [&](const PairTile &tl) {
            if (half != 0 || tl.valid_rows == 0) return;
            const int row = tl.d_row0 + row_off + static_cast<int>(lane);
            const int cols = p.n - (tl.n0 + col_off) < (MP == 256 ? BN : BN / 2) ? p.n - (tl.n0 + col_off)
                                                                                  : (MP == 256 ? BN : BN / 2);
            if (row < p.rows && cols > 0)
                prefetch_l2_bulk(p.c + static_cast<int64_t>(row) * p.ldc + tl.n0 + col_off,
                                 static_cast<uint32_t>(cols) * 2u);
        };
        // FP32 C: a ring of kCDepth chunks of this thread's row; chunk j of every tile
        // lives in slot j % kCDepth.  Once chunk j is added, its slot is refilled with
        // chunk j + kCDepth of the tile, or, past the tile's last chunk, with chunk
        // j % kCDepth of the next tile, so the loads run up to kCDepth chunks ahead
        // and overlap the TMEM reads and stores of the chunks before.
        constexpr int kCDepth = Cfg::kChunksPerWarp < 4 ? Cfg::kChunksPerWarp : 4;
        static_assert(!F32 || Cfg::kNumChunks % 2 == 0, "FP32 epilogue: both halves have every chunk");
        float4 cring[(WITH_C && F32) ? kCDepth : 1][4];
        // FP32 C that is D itself: no C is loaded; each chunk is added to D at L2 by a
        // TMA reduce, and the tile's D rows are prefetched into L2 a tile ahead (one
        // bulk request per row) so that those additions find their lines there
        // (C in a buffer of its own: its rows are prefetched the same way, then loaded
        // chunk by chunk through the ring below)
        auto prefetch_d32 = [&](const PairTile &tl) {
            if (half != 0 || tl.valid_rows == 0 || (p.c_in_place && tl.nkb == 0)) return;
            const int row = tl.d_row0 + row_off + static_cast<int>(lane);
            const int cols = p.n - (tl.n0 + col_off) < (MP == 256 ? BN : BN / 2) ? p.n - (tl.n0 + col_off)
                                                                                  : (MP == 256 ? BN : BN / 2);
            const float *src = p.c_in_place ? p.d_f32 : p.c_f32;
            const int64_t ld = p.c_in_place ? p.ldd : p.ldc;
            if (row < p.rows && cols > 0) {
                const float *r0 = src + static_cast<int64_t>(row) * ld + tl.n0 + col_off;
                if (p.c_in_place) {
                    prefetch_l2_bulk(r0, static_cast<uint32_t>(cols) * 4u);
                } else {
                    // a C of its own: one L2 prefetch per 128-byte line from this thread
                    // (measured faster here than the bulk request, which is faster in place)
                    for (int c = 0; c < cols; c += 32) prefetch_l2_line(r0 + c);
                }
            }
        };
        auto load_c32 = [&](const PairTile &tl, int j, float4 (&dst)[4]) {
            const int row = tl.d_row0 + row_off + static_cast<int>(lane);
            const int col0 = tl.n0 + col_off + (2 * j + static_cast<int>(half)) * Cfg::kEpiChunk;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                dst[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (tl.valid_rows > 0 && row < p.rows && col0 + 4 * q < p.n)
                    dst[q] = __ldg(reinterpret_cast<const float4 *>(p.c_f32 + static_cast<int64_t>(row) * p.ldc +
                                                                    col0 + 4 * q));
            }
        };
        // C tile (dense bf16 C, TMA-aligned): this warp's 32 rows of every other
        // 32-column box of the tile (boxes half, half + 2, ...) land in shared memory by
        // TMA, are summed in place and go out by TMA from there; the next tile's boxes
        // are loaded as soon as the stores have read them, a tile ahead of their use
        const bool c_tma = Cfg::kCBoxes > 0 && p.c_tma;
        constexpr int kMyBoxes = (Cfg::kCBoxes + 1) / 2;
        uint8_t *const ctile = smem_stage_out + quad * 32 * 64;
        uint32_t c_phase = 0;
        bool c_pending = false;
        auto load_ctile = [&](const PairTile &tl) {
            if (lane == 0) {
                const int nb = (Cfg::kCBoxes - static_cast<int>(half) + 1) / 2;
                mbar_arrive_expect_tx(&cfull_bar[ew], static_cast<uint32_t>(nb) * 32u * 64u);
#pragma unroll
                for (int q = 0; q < kMyBoxes; ++q) {
                    const int j = 2 * q + static_cast<int>(half);
                    if (j < Cfg::kCBoxes)
                        tma_load_2d(ctile + j * Cfg::kCBoxBytes, &tm_c, &cfull_bar[ew], tl.n0 + 32 * j,
                                    tl.d_row0 + row_off);
                }
            }
            __syncwarp();
            c_pending = true;
        };
        PairTile tile;
        if (pair_id < num_tiles) {
            get_pair_tile<BN, MP>(p, prefix, pinfo, num_units, psf_k, pair_id, rank, tile);
            if constexpr (WITH_C && !F32) prefetch_c(tile);
            if (c_tma) load_ctile(tile);
            if constexpr (WITH_C && F32) {
                prefetch_d32(tile);
                if (!p.c_in_place) {
#pragma unroll
                    for (int j = 0; j < kCDepth; ++j) load_c32(tile, j, cring[j]);
                }
            }
        }
        for (int t = pair_id; t < num_tiles; t += num_pairs) {
            const bool has_next = t + num_pairs < num_tiles;
            PairTile next_tile = tile;
            if (has_next) get_pair_tile<BN, MP>(p, prefix, pinfo, num_units, psf_k, t + num_pairs, rank, next_tile);
            // bf16 chunk (16 columns of this thread's row) -> swizzled staging -> TMA store
            // valid_rows: all (MP/2) -> TMA store (clipped at the tensor's edge); 0 -> this
            // CTA's rows belong to no unit of the tile; otherwise (masked edge) direct stores
            // of the valid rows only
            auto store_chunk = [&](const uint32_t (&o)[8], int c) {
                const int col0 = tile.n0 + col_off + c * Cfg::kEpiChunk;
                if (tile.valid_rows == 0 || col0 >= p.n) return;
                if (tile.valid_rows < MP / 2) {
                    // the valid rows; with zero_tail the block's other rows get 0
                    const int local_row = row_off + static_cast<int>(lane);
                    const bool value = local_row < tile.valid_rows;
                    if (value || (tile.zero_tail && tile.d_row0 + local_row < p.rows)) {
                        uint16_t *drow = p.d + static_cast<int64_t>(tile.d_row0 + local_row) * p.ldd + col0;
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            if (col0 + 8 * h < p.n)
                                *reinterpret_cast<uint4 *>(drow + 8 * h) =
                                    value ? make_uint4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3])
                                          : make_uint4(0u, 0u, 0u, 0u);
                    }
                    return;
                }
                if constexpr (WITH_C && !F32) {
                    // the C epilogue's store map is 32 columns wide: a lone chunk goes out
                    // directly (it lies inside the tile, and columns past n are skipped)
                    const int drow = tile.d_row0 + row_off + static_cast<int>(lane);
                    if (drow < p.rows) {
                        uint16_t *dp = p.d + static_cast<int64_t>(drow) * p.ldd + col0;
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            if (col0 + 8 * h < p.n)
                                *reinterpret_cast<uint4 *>(dp + 8 * h) =
                                    make_uint4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]);
                    }
                    return;
                }
                uint8_t *sbuf = stage_out + buf * Cfg::kStageBufBytes;
                if (lane == 0) bulk_wait_group_read<Cfg::kStageBufs - 1>();
                __syncwarp();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t off = lane * 32 + ((h ^ ((lane >> 2) & 1)) * 16);
                    *reinterpret_cast<uint4 *>(sbuf + off) = make_uint4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tm_d, sbuf, col0, tile.d_row0 + row_off);
                    bulk_commit_group();
                }
                buf = buf + 1 == Cfg::kStageBufs ? 0 : buf + 1;
            };
            // bf16 C of this tile into registers (the first tile's once its accumulator is
            // complete, so that its loads do not compete with the first operand loads)
            if constexpr (WITH_C && !F32) {
                if (t != pair_id && !c_tma) {
#pragma unroll
                    for (int j = 0; j < Cfg::kChunksPerWarp; ++j) load_c(tile, j, cpk[j]);
                }
            }
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&tfull_bar[acc], acc_phase, ctl, DG_DEV_TIMEOUT))) break;
            tc_fence_after_sync();
            if constexpr (WITH_C && !F32) {
                if (t == pair_id && !c_tma) {
#pragma unroll
                    for (int j = 0; j < Cfg::kChunksPerWarp; ++j) load_c(tile, j, cpk[j]);
                }
                if (has_next) prefetch_c(next_tile);
            }
            if constexpr (Cfg::kCBoxes > 0) {
                if (c_tma) {
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&cfull_bar[ew], c_phase, ctl, DG_DEV_TIMEOUT))) break;
                    c_phase ^= 1;
                    c_pending = false;
                    // bf16(acc + C) over each box's two 16-column chunks, back into the box
#pragma unroll
                    for (int q = 0; q < kMyBoxes; ++q) {
                        const int j = 2 * q + static_cast<int>(half);
                        if (j >= Cfg::kCBoxes) break;
                        uint32_t v[2][16];
                        const uint32_t tcol = tmem_base + ((quad * 32) << 16) + acc * ACC + j * 32;
                        tmem_ld_32x32b_x16(tcol, v[0]);
                        tmem_ld_32x32b_x16(tcol + 16, v[1]);
                        tmem_ld_wait();
                        reg_fence16(v[0]);
                        reg_fence16(v[1]);
                        uint8_t *rowp = ctile + j * Cfg::kCBoxBytes + lane * 64;
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            // 64-byte swizzle: 16-byte unit h (columns 8h..8h+7) of row r at h ^ ((r >> 1) & 3)
                            uint4 *up = reinterpret_cast<uint4 *>(rowp + ((h ^ ((lane >> 1) & 3)) * 16));
                            const uint4 cv = *up;
                            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
                            const uint32_t *x = v[h >> 1] + 8 * (h & 1);
                            uint32_t ow[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float lo = __uint_as_float(x[2 * i]) + __uint_as_float(cw[i] << 16);
                                const float hi = __uint_as_float(x[2 * i + 1]) + __uint_as_float(cw[i] & 0xFFFF0000u);
                                __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                                ow[i] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                            *up = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                        }
                    }
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(leader_tempty + acc * 8);
                    if (++acc == NUM_ACC) { acc = 0; acc_phase ^= 1; }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        // boxes wholly past the last row or column store nothing
#pragma unroll
                        for (int q = 0; q < kMyBoxes; ++q) {
                            const int j = 2 * q + static_cast<int>(half);
                            if (j < Cfg::kCBoxes && tile.n0 + 32 * j < p.n && tile.d_row0 + row_off < p.rows)
                                tma_store_2d(&tm_d, ctile + j * Cfg::kCBoxBytes, tile.n0 + 32 * j,
                                             tile.d_row0 + row_off);
                        }
                        bulk_commit_group();
                        if (has_next) bulk_wait_group_read<0>();   // the boxes may be refilled
                    }
                    __syncwarp();
                    if (has_next) load_ctile(next_tile);
                    tile = next_tile;
                    continue;
                }
            }
            if constexpr (F32) {
                // FP32 D (and FP32 C): each chunk goes TMEM -> registers (+ C) -> one
                // 16-column FP32 box through a pair of staging buffers; the accumulator is
                // released after its last chunk is read
                const int row = tile.d_row0 + row_off + static_cast<int>(lane);
                // D = C in place: an empty group leaves D as it is; the next tile's rows go to L2
                const bool in_place = WITH_C && p.c_in_place;
                if (WITH_C && has_next) prefetch_d32(next_tile);
                const bool skip_tile = in_place && tile.nkb == 0;
                // chunks in runs of kCDepth, so that a chunk's ring slot is a constant
#pragma unroll 1
                for (int j0 = 0; j0 < Cfg::kChunksPerWarp; j0 += kCDepth)
#pragma unroll
                for (int u = 0; u < kCDepth; ++u) {
                    const int j = j0 + u;
                    if (j >= Cfg::kChunksPerWarp || skip_tile) break;
                    const int c = 2 * j + half;
                    const int col0 = tile.n0 + col_off + c * Cfg::kEpiChunk;
                    float f[16];
                    if (tile.nkb > 0) {
                        uint32_t v[16];
                        tmem_ld_32x32b_x16(tmem_base + ((quad * 32) << 16) + acc * ACC + c * Cfg::kEpiChunk, v);
                        tmem_ld_wait();
                        reg_fence16(v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
                    } else {
                        // no K-blocks (an empty group): the accumulator was never written
#pragma unroll
                        for (int i = 0; i < 16; ++i) f[i] = 0.f;
                    }
                    if constexpr (WITH_C) {
                        if (!in_place) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                f[4 * q + 0] += cring[u][q].x;
                                f[4 * q + 1] += cring[u][q].y;
                                f[4 * q + 2] += cring[u][q].z;
                                f[4 * q + 3] += cring[u][q].w;
                            }
                            // refill the slot: chunk j + kCDepth of this tile, or chunk u of the next
                            if (j + kCDepth < Cfg::kChunksPerWarp)
                                load_c32(tile, j + kCDepth, cring[u]);
                            else if (has_next)
                                load_c32(next_tile, u, cring[u]);
                        }
                    }
                    if (tile.valid_rows == 0 || col0 >= p.n) continue;
                    if (tile.valid_rows < MP / 2) {
                        const int local_row = row_off + static_cast<int>(lane);
                        const bool value = local_row < tile.valid_rows;
                        if (value || (tile.zero_tail && row < p.rows)) {
                            float *drow = p.d_f32 + static_cast<int64_t>(row) * p.ldd + col0;
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (col0 + 4 * q < p.n) {
                                    float4 o4 = value ? make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3])
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                                    if (in_place && value) {
                                        // this thread owns these elements: D += sum, one FP32 add each
                                        const float4 d4 = *reinterpret_cast<const float4 *>(drow + 4 * q);
                                        o4 = make_float4(d4.x + o4.x, d4.y + o4.y, d4.z + o4.z, d4.w + o4.w);
                                    }
                                    *reinterpret_cast<float4 *>(drow + 4 * q) = o4;
                                }
                        }
                        continue;
                    }
                    {
                        // one 16-column FP32 box (32 rows of 64 bytes) per chunk, through
                        // staging buffer pairs: a TMA store or reduce costs the SM's TMA unit
                        // per operation, so fewer, larger boxes drain the tile sooner
                        constexpr int NB2 = Cfg::kStageBufs / 2;
                        static_assert(NB2 >= 1, "FP32 staging: pairs of buffers");
                        uint8_t *sbuf = stage_out + buf * 2 * Cfg::kStageBufBytes;
                        if (lane == 0) bulk_wait_group_read<NB2 - 1>();
                        __syncwarp();
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            // 64-byte swizzle: 16-byte unit h of row r sits at unit h ^ ((r >> 1) & 3)
                            const uint32_t off = lane * 64 + ((h ^ ((lane >> 1) & 3)) * 16);
                            const float *x = f + 4 * h;
                            *reinterpret_cast<float4 *>(sbuf + off) = make_float4(x[0], x[1], x[2], x[3]);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (in_place) tma_reduce_add_2d(&tm_d, sbuf, col0, tile.d_row0 + row_off);
                            else tma_store_2d(&tm_d, sbuf, col0, tile.d_row0 + row_off);
                            bulk_commit_group();
                        }
                        buf = buf + 1 == NB2 ? 0 : buf + 1;
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(leader_tempty + acc * 8);
                if (++acc == NUM_ACC) { acc = 0; acc_phase ^= 1; }
            } else if constexpr (WITH_C) {
                // each chunk's bf16(acc + C) overwrites that chunk's C registers; the
                // accumulator is released once every chunk is read (the MMAs of the tile
                // after next need it), and only then are the chunks stored, two adjacent
                // chunks (32 columns, 64-byte rows) per TMA store: the SM's TMA unit, where
                // the stores queue behind the operand loads, costs per operation
#pragma unroll
                for (int j0 = 0; j0 < Cfg::kChunksPerWarp; j0 += 2) {
                    uint32_t v[2][16];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int c = (j0 + u) + static_cast<int>(half) * Cfg::kChunksPerWarp;
                        if (j0 + u < Cfg::kChunksPerWarp && c < Cfg::kNumChunks)
                            tmem_ld_32x32b_x16(tmem_base + ((quad * 32) << 16) + acc * ACC + c * Cfg::kEpiChunk, v[u]);
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int j = j0 + u;
                        const int c = j + static_cast<int>(half) * Cfg::kChunksPerWarp;
                        if (j >= Cfg::kChunksPerWarp || c >= Cfg::kNumChunks) continue;
                        reg_fence16(v[u]);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float lo = __uint_as_float(v[u][2 * i]) + __uint_as_float(cpk[j][i] << 16);
                            const float hi = __uint_as_float(v[u][2 * i + 1]) + __uint_as_float(cpk[j][i] & 0xFFFF0000u);
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                            cpk[j][i] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(leader_tempty + acc * 8);
                if (++acc == NUM_ACC) { acc = 0; acc_phase ^= 1; }
#pragma unroll
                for (int j = 0; j < Cfg::kChunksPerWarp; j += 2) {
                    const int c = j + static_cast<int>(half) * Cfg::kChunksPerWarp;
                    if (c >= Cfg::kNumChunks) continue;
                    const bool pair = j + 1 < Cfg::kChunksPerWarp && c + 1 < Cfg::kNumChunks;
                    const int col0 = tile.n0 + col_off + c * Cfg::kEpiChunk;
                    if (!pair || tile.valid_rows < MP / 2) {
                        // a lone chunk, or rows ending inside the tile: chunk by chunk
                        store_chunk(cpk[j], c);
                        if (pair) store_chunk(cpk[j + 1], c + 1);
                        continue;
                    }
                    if (tile.valid_rows == 0 || col0 >= p.n) continue;
                    constexpr int NB2 = Cfg::kStageBufs / 2;
                    static_assert(NB2 >= 1, "bf16 C staging: pairs of buffers");
                    uint8_t *sbuf = stage_out + (buf % NB2) * 2 * Cfg::kStageBufBytes;
                    if (lane == 0) bulk_wait_group_read<NB2 - 1>();
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        // 64-byte swizzle: 16-byte unit h of row r sits at unit h ^ ((r >> 1) & 3)
                        const uint32_t off = lane * 64 + ((h ^ ((lane >> 1) & 3)) * 16);
                        const uint32_t *x = (h < 2 ? cpk[j] : cpk[j + 1]) + 4 * (h & 1);
                        *reinterpret_cast<uint4 *>(sbuf + off) = make_uint4(x[0], x[1], x[2], x[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_d, sbuf, col0, tile.d_row0 + row_off);
                        bulk_commit_group();
                    }
                    ++buf;
                }
            } else {
                // the whole row segment to registers, release the accumulator, then store
                uint32_t out[Cfg::kChunksPerWarp][8];
#pragma unroll
                for (int j0 = 0; j0 < Cfg::kChunksPerWarp; j0 += 2) {
                    uint32_t v[2][16];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int c = 2 * (j0 + u) + half;
                        if (j0 + u < Cfg::kChunksPerWarp && c < Cfg::kNumChunks)
                            tmem_ld_32x32b_x16(tmem_base + ((quad * 32) << 16) + acc * ACC + c * Cfg::kEpiChunk, v[u]);
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        if (j0 + u >= Cfg::kChunksPerWarp) continue;
                        reg_fence16(v[u]);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[u][2 * i]),
                                                                      __uint_as_float(v[u][2 * i + 1]));
                            out[j0 + u][i] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(leader_tempty + acc * 8);
                if (++acc == NUM_ACC) { acc = 0; acc_phase ^= 1; }
#pragma unroll
                for (int j = 0; j < Cfg::kChunksPerWarp; ++j) {
                    const int c = 2 * j + half;
                    if (c < Cfg::kNumChunks) store_chunk(out[j], c);
                }
            }
            tile = next_tile;
        }
        // (an aborted loop leaves no C load landing in shared memory after the CTA is gone)
        if (c_pending && lane == 0) mbar_wait_drain(&cfull_bar[ew], c_phase, ctl);
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    // neither CTA leaves while its peer may still signal its barriers or read its shared memory
    cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    }
}

template <int BN, bool WITH_C, int MP, bool F32, int LAY>
cudaError_t launch_bs2_gemm_impl(const TensorMaps &maps, const GemmParams &p, int grid,
                                 cudaStream_t stream) {
    using Cfg = Bs2Cfg<BN, MP, LAY, F32, WITH_C>;
    cudaError_t e = cudaFuncSetAttribute(dg_bs2_gemm_kernel<BN, WITH_C, MP, F32, LAY>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    // a programmatic dependent of the stream's previous grid (the cluster shape is
    // the kernel's own)
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
    return cudaLaunchKernelEx(&cfg, dg_bs2_gemm_kernel<BN, WITH_C, MP, F32, LAY>, maps.a, maps.b, maps.b2, maps.d,
                              maps.c, p);
}

template <int BN, bool WITH_C, int MP, bool F32, int LAY>
int max_active_pairs_impl() {
    using Cfg = Bs2Cfg<BN, MP, LAY, F32, WITH_C>;
    if (cudaFuncSetAttribute(dg_bs2_gemm_kernel<BN, WITH_C, MP, F32, LAY>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, dg_bs2_gemm_kernel<BN, WITH_C, MP, F32, LAY>, &cfg) != cudaSuccess) return 0;
    return n;
}

template <int BN, int MP, int LAY = 0, bool F32 = false, bool WITH_C = false>
void fill_bs2_info(KernelInfo *info) {
    using Cfg = Bs2Cfg<BN, MP, LAY, F32, WITH_C>;
    info->block_n = BN;
    info->stages = Cfg::kStages;
    info->smem_bytes = Cfg::kSmemBytes;
    info->threads = Cfg::kThreads;
    info->group_kb = Cfg::kGroupKb;
    info->num_acc = Cfg::kNumAcc;
}

}  // namespace dg
