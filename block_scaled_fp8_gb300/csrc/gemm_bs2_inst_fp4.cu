// Instantiations of the CTA-pair block-scaled GEMM kernel with FP4 (E2M1) B operands
// (the FP8 x FP4 GEMM).
#include "gemm_bs2.cuh"
#include "gemm_bs2_list.h"

namespace dg {
#define DG_INST2(BN, C, MP, F32, LAY)                                                                   \
    template cudaError_t launch_bs2_gemm_impl<BN, C, MP, F32, LAY>(const TensorMaps &, const GemmParams &, \
                                                              int, cudaStream_t);                      \
    template int max_active_pairs_impl<BN, C, MP, F32, LAY>();
DG_BS2_LIST_FP4(DG_INST2)
#undef DG_INST2
}  // namespace dg
