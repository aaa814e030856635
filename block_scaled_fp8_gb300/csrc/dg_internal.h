// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg.h"  // include/ is on the include path

namespace dg {

constexpr int kBlockM = 128;   // rows per tile (one UMMA M=128, TMEM lanes)
constexpr int kBlockK = 128;   // K per pipeline stage (= scale granularity)
constexpr int kGran = 128;     // scale granularity along K (and N for FP32 B scales)
constexpr int kMaxGroupsMasked = 1024;
// Grouped layouts on CTA pairs: at most this many m-pairs (contiguous) or experts (masked).
constexpr int kMaxPairPrefix = 512;
// Experts of the PSUM contiguous layout (8-bit ids in the pair kernel's unit info).
constexpr int kMaxPsumGroups = 255;

enum GemmMode : int { kModeDense = 0, kModeContiguous = 1, kModeMasked = 2, kModeKGrouped = 3 };

// Runtime parameters of one GEMM launch (passed by value).
struct GemmParams {
    int mode;
    int rows;            // dense: M; contiguous: M_total; masked: max_m (rows per expert)
    int n, k;
    int num_m_blocks;    // blocks of 128 rows (dense/contiguous: over all rows; masked: per expert, max)
    int num_n_blocks;
    int num_k_blocks;
    int num_groups;
    int group_m;         // tile-order group size along M (L2 reuse)
    const int32_t *grouped_layout;  // contiguous: expert id per row
    const int32_t *psum;            // contiguous with PSUM offsets instead: [num_groups]
    const int32_t *masked_m;        // masked
    const int32_t *ks;              // K-grouped: rows of K per group [num_groups], multiples of 128
    int group_rows;                 // K-grouped: M, the rows of each group's D
    const uint16_t *c;   // dense: bf16 C or nullptr
    int64_t ldc;
    uint16_t *d;         // bf16 D (used for direct stores)
    float *d_f32;        // FP32 D (FP32-output GEMMs; then c_f32 is the FP32 C or null)
    const float *c_f32;
    int64_t ldd;
    int32_t *status;
    uint64_t timeout_ns;
    uint32_t debug_flags;
    int ab_3d;           // A/B tensor maps are the 3-D K-blocked views: one load per ring slot
    int c_v8;            // bf16 C rows are 32-byte aligned (base and ldc): 16 columns in one load
    int c_in_place;      // FP32 C is D itself (same pointer and stride): D is accumulated into at L2
    int c_tma;           // bf16 C goes through shared memory by TMA (dense pair GEMMs, 16-byte aligned rows)
    int layout;          // operand layouts: bit 0 A MN-major ([K][M]), bit 1 B MN-major ([K][N]),
                         // bit 2 B FP4 (E2M1, one scale per 32 K)
    // packed UE8M0 scale words, [slices][ld] int32 with ld = align4(mn); the
    // block-scaled kernels' scale warps read them with cp.async
    const uint32_t *sfa_words;
    const uint32_t *sfb_words;
    int sfa_ld, sfb_ld;
    int sfa_slices, sfb_slices;
    // FP32-promotion kernel only
    const float *sfa_f32;   // [rows][sf_k]
    const float *sfb_f32;   // [ceil(n/128)][sf_k]
    int sf_k;
};

struct TensorMaps {
    CUtensorMap a, b, d;
    CUtensorMap b2;   // pair tiles wider than 256 columns: the second MMA's rows of B
    CUtensorMap c;    // the pair kernel's bf16 C boxes (C tile in shared memory)
};

// Per-instantiation launch information.
struct KernelInfo {
    int block_n;
    int stages;
    int smem_bytes;
    int threads;
    int group_kb;   // K-blocks per ring slot (the depth of a 3-D A/B load)
    int num_acc;    // TMEM accumulators (1: the next tile's MMAs wait for the epilogue's reads)
};

// Block-scaled (UE8M0) tcgen05 kernel family: returns false if block_n is not
// compiled in.
bool get_bs_kernel_info(int block_n, bool with_c, KernelInfo *info);
cudaError_t launch_bs_gemm(int block_n, const TensorMaps &maps, const GemmParams &p, int grid,
                           cudaStream_t stream);

// CTA-pair (cta_group::2) block-scaled kernel family (the instantiations are
// listed in gemm_bs2_list.h).  mp = rows of a pair tile: 256 or 128; f32 picks
// the FP32-output (and FP32-C) epilogue; launch_bs2_gemm takes C and f32 from p.
bool get_bs2_kernel_info(int block_n, bool with_c, int mp, KernelInfo *info, bool f32 = false, int lay = 0);
cudaError_t launch_bs2_gemm(int block_n, int mp, const TensorMaps &maps, const GemmParams &p, int grid,
                            cudaStream_t stream);
int bs2_max_active_pairs(int block_n, bool with_c, int mp, bool f32 = false, int lay = 0);

// FP32-scale promotion kernel family.
bool get_promote_kernel_info(int block_n, KernelInfo *info);
cudaError_t launch_promote_gemm(int block_n, const TensorMaps &maps, const GemmParams &p, int grid,
                                cudaStream_t stream);

// Scale-factor transform.
// Scale rows of the K-grouped layout, per group: srow[e] = first 128-K block
// (FP32 scale row), prow[e] = first packed row; entries 0..num_groups.
struct KGroupRows {
    int num_groups;
    int srow[kMaxPsumGroups + 2];
    int prow[kMaxPsumGroups + 2];
};
cudaError_t launch_transform_sf_k_grouped(const float *sf, int mn, const KGroupRows &t, int packed_rows,
                                          void *out, int32_t *status, cudaStream_t stream);
cudaError_t launch_transform_sf(const float *sf, int batch, int mn_rows, int sf_k, int gran_mn,
                                int mn, int out_fmt, void *out, int32_t *status,
                                cudaStream_t stream);

}  // namespace dg
