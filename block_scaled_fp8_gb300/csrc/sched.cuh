// Persistent tile scheduler of the single-CTA GEMM kernels.
//
// Every CTA walks tile ids t = blockIdx.x, blockIdx.x + gridDim.x, ... (the
// persistent loop of PaperTrace "02 · DeepGEMM 技术解析" §4.3).  A tile is one
// 128-row m-block and one n-block.  Tiles map to (m-block, n-block) in groups of
// `group_m` m-blocks so that CTAs running at the same time share A and B tiles
// through L2.  There is no split-K: one CTA owns every K-block of its tile.  All
// roles of a CTA call the scheduler with the same ids and reach the same
// decisions, including skips, so they stay in step without talking to each
// other.
#pragma once

#include "dg_internal.h"

namespace dg {

struct Tile {
    int a_row0;      // first row of this tile in the 2-D view of A (and D)
    int sfa_x;       // column of the packed SFA view (MN index of the tile's first row)
    int sfa_y0;      // row of the packed SFA view for K-slice 0
    int b_row0;      // first row of this tile in the 2-D view of B ([E*N, K])
    int sfb_y0;      // row of the packed SFB view for K-slice 0
    int n0;          // first output column
    int valid_rows;  // rows of the tile that may be written (128 unless at a masked edge)
    int group;       // expert (0 for dense)
};

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// Prefix sums of per-expert tile counts (masked mode), built once per CTA in
// shared memory.  prefix[e] = tiles of experts < e; prefix[E] = total.
__device__ __forceinline__ void build_masked_prefix(const GemmParams &p, int *prefix) {
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int e = 0; e < p.num_groups; ++e) {
            prefix[e] = acc;
            int mm = p.masked_m[e];
            if (mm > p.rows || mm < 0) {
                if (p.status) atomicOr(p.status, DG_DEV_BAD_GROUP);
                mm = mm < 0 ? 0 : p.rows;
            }
            acc += ceil_div_i(mm, kBlockM) * p.num_n_blocks;
        }
        prefix[p.num_groups] = acc;
    }
}

__device__ __forceinline__ int total_tiles(const GemmParams &p, const int *prefix) {
    if (p.mode == kModeMasked) return prefix[p.num_groups];
    return p.num_m_blocks * p.num_n_blocks;
}

// Fills `tile` for tile id t (< total).  Returns false when the tile is skipped
// (contiguous layout: a padding block or an out-of-range expert).
template <int BN>
__device__ __forceinline__ bool get_tile(const GemmParams &p, const int *prefix, int t, int psf_k,
                                         Tile &tile, bool report) {
    int mb, ng, group = 0;
    if (p.mode == kModeMasked) {
        // find the expert: largest e with prefix[e] <= t
        int lo = 0, hi = p.num_groups - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
        }
        group = lo;
        int mm = p.masked_m[group];
        mm = mm < 0 ? 0 : (mm > p.rows ? p.rows : mm);
        int mbe = ceil_div_i(mm, kBlockM);
        int local = t - prefix[group];
        mb = local % mbe;
        ng = local / mbe;
        tile.a_row0 = group * p.rows + mb * kBlockM;
        tile.sfa_x = mb * kBlockM;
        tile.sfa_y0 = group * psf_k;
        int v = mm - mb * kBlockM;
        tile.valid_rows = v < kBlockM ? v : kBlockM;
    } else {
        const int per_group = p.group_m * p.num_n_blocks;
        const int g = t / per_group;
        const int first_m = g * p.group_m;
        const int rem_m = p.num_m_blocks - first_m;
        const int gsize = rem_m < p.group_m ? rem_m : p.group_m;
        const int r = t - g * per_group;
        mb = first_m + r % gsize;
        ng = r / gsize;
        tile.a_row0 = mb * kBlockM;
        tile.sfa_x = mb * kBlockM;
        tile.sfa_y0 = 0;
        tile.valid_rows = kBlockM;
        if (p.mode == kModeContiguous) {
            group = __ldg(p.grouped_layout + mb * kBlockM);
            if (group < 0) return false;
            if (group >= p.num_groups) {
                if (report && p.status) atomicOr(p.status, DG_DEV_BAD_GROUP);
                return false;
            }
        }
    }
    const int nb = ng;
    tile.group = group;
    tile.n0 = nb * BN;
    tile.b_row0 = group * p.n + nb * BN;
    tile.sfb_y0 = group * psf_k;
    return true;
}

}  // namespace dg
