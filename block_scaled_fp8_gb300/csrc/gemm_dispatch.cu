// Maps a runtime BLOCK_N to the compiled block-scaled kernel instantiations
// (which live in the gemm_bs_inst_*.cu units).
#include "gemm_bs.cuh"
#include "gemm_promote.cuh"
#include "gemm_bs2.cuh"
#include "gemm_bs2_list.h"

namespace dg {

// BLOCK_N values compiled without C, and the subset also compiled with C
// (the C-accumulate epilogue holds C in registers, which caps BLOCK_N).
#define DG_BS_BLOCK_N_LIST(X) X(16) X(32) X(48) X(64) X(96) X(128) X(160) X(176) X(192) X(224) X(256)
#define DG_BS_BLOCK_N_LIST_C(X) X(16) X(32) X(48) X(64) X(96) X(128) X(160)

#define DG_EXTERN(BN) \
    extern template cudaError_t launch_bs_gemm_impl<BN, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
DG_BS_BLOCK_N_LIST(DG_EXTERN)
#undef DG_EXTERN
#define DG_EXTERN(BN) \
    extern template cudaError_t launch_bs_gemm_impl<BN, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
DG_BS_BLOCK_N_LIST_C(DG_EXTERN)
#undef DG_EXTERN

#define DG_EXTERN2(BN, C, MP, F32, LAY)                                                                 \
    extern template cudaError_t launch_bs2_gemm_impl<BN, C, MP, F32, LAY>(const TensorMaps &,             \
                                                                     const GemmParams &, int, cudaStream_t); \
    extern template int max_active_pairs_impl<BN, C, MP, F32, LAY>();
DG_BS2_LIST(DG_EXTERN2)
#undef DG_EXTERN2

bool get_bs2_kernel_info(int block_n, bool with_c, int mp, KernelInfo *info, bool f32, int lay) {
#define DG_CASE2(BN, C, MP, F32, LAY) \
    if (block_n == BN && with_c == C && mp == MP && f32 == F32 && lay == LAY) { fill_bs2_info<BN, MP, LAY, F32, C>(info); return true; }
    DG_BS2_LIST(DG_CASE2)
#undef DG_CASE2
    return false;
}

cudaError_t launch_bs2_gemm(int block_n, int mp, const TensorMaps &maps, const GemmParams &p, int grid,
                            cudaStream_t stream) {
    const bool f32 = p.d_f32 != nullptr;
    const bool with_c = f32 ? p.c_f32 != nullptr : p.c != nullptr;
#define DG_CASE2(BN, C, MP, F32, LAY)                                       \
    if (block_n == BN && with_c == C && mp == MP && f32 == F32 && p.layout == LAY) \
        return launch_bs2_gemm_impl<BN, C, MP, F32, LAY>(maps, p, grid, stream);
    DG_BS2_LIST(DG_CASE2)
#undef DG_CASE2
    return cudaErrorInvalidValue;
}

int bs2_max_active_pairs(int block_n, bool with_c, int mp, bool f32, int lay) {
#define DG_CASE2(BN, C, MP, F32, LAY) \
    if (block_n == BN && with_c == C && mp == MP && f32 == F32 && lay == LAY) \
        return max_active_pairs_impl<BN, C, MP, F32, LAY>();
    DG_BS2_LIST(DG_CASE2)
#undef DG_CASE2
    return 0;
}

bool get_bs_kernel_info(int block_n, bool with_c, KernelInfo *info) {
    if (with_c) {
        switch (block_n) {
#define DG_CASE(BN) case BN: fill_bs_info<BN>(info); return true;
            DG_BS_BLOCK_N_LIST_C(DG_CASE)
#undef DG_CASE
            default: return false;
        }
    }
    switch (block_n) {
#define DG_CASE(BN) case BN: fill_bs_info<BN>(info); return true;
        DG_BS_BLOCK_N_LIST(DG_CASE)
#undef DG_CASE
        default: return false;
    }
}

cudaError_t launch_bs_gemm(int block_n, const TensorMaps &maps, const GemmParams &p, int grid,
                           cudaStream_t stream) {
    if (p.c != nullptr) {
        switch (block_n) {
#define DG_CASE(BN) case BN: return launch_bs_gemm_impl<BN, true>(maps, p, grid, stream);
            DG_BS_BLOCK_N_LIST_C(DG_CASE)
#undef DG_CASE
            default: return cudaErrorInvalidValue;
        }
    }
    switch (block_n) {
#define DG_CASE(BN) case BN: return launch_bs_gemm_impl<BN, false>(maps, p, grid, stream);
        DG_BS_BLOCK_N_LIST(DG_CASE)
#undef DG_CASE
        default: return cudaErrorInvalidValue;
    }
}

#define DG_PROMOTE_BLOCK_N_LIST(X) X(32) X(64) X(128)
#define DG_EXTERN(BN)                                                                              \
    extern template cudaError_t launch_promote_gemm_impl<BN, false>(const TensorMaps &,             \
                                                                    const GemmParams &, int,         \
                                                                    cudaStream_t);                   \
    extern template cudaError_t launch_promote_gemm_impl<BN, true>(const TensorMaps &,              \
                                                                   const GemmParams &, int,          \
                                                                   cudaStream_t);
DG_PROMOTE_BLOCK_N_LIST(DG_EXTERN)
#undef DG_EXTERN

bool get_promote_kernel_info(int block_n, KernelInfo *info) {
    switch (block_n) {
#define DG_CASE(BN) case BN: fill_promote_info<BN>(info); return true;
        DG_PROMOTE_BLOCK_N_LIST(DG_CASE)
#undef DG_CASE
        default: return false;
    }
}

cudaError_t launch_promote_gemm(int block_n, const TensorMaps &maps, const GemmParams &p, int grid,
                                cudaStream_t stream) {
    const bool with_c = p.c != nullptr;
    switch (block_n) {
#define DG_CASE(BN)                                                                    \
    case BN:                                                                           \
        return with_c ? launch_promote_gemm_impl<BN, true>(maps, p, grid, stream)      \
                      : launch_promote_gemm_impl<BN, false>(maps, p, grid, stream);
        DG_PROMOTE_BLOCK_N_LIST(DG_CASE)
#undef DG_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dg
