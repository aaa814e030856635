// Instantiations of the CTA-pair block-scaled GEMM kernel.
#include "gemm_bs2.cuh"

namespace dg {
template cudaError_t launch_bs2_gemm_impl<128, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<128, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<192, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<224, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<240, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<192, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<224, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<240, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<256, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template int max_active_pairs_impl<128, false>();
template int max_active_pairs_impl<128, true>();
template int max_active_pairs_impl<192, true>();
template int max_active_pairs_impl<224, true>();
template int max_active_pairs_impl<240, true>();
template int max_active_pairs_impl<192, false>();
template int max_active_pairs_impl<224, false>();
template int max_active_pairs_impl<240, false>();
template int max_active_pairs_impl<256, false>();
}  // namespace dg
