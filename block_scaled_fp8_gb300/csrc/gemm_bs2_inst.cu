// Instantiations of the CTA-pair block-scaled GEMM kernel: (BLOCK_N, with C, rows per pair).
#include "gemm_bs2.cuh"

namespace dg {
template cudaError_t launch_bs2_gemm_impl<128, false, 256>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<128, true, 256>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<192, false, 256>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<192, true, 256>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<224, false, 256>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<224, true, 256>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<240, false, 256>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<240, true, 256>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<256, false, 256>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<32, false, 128>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<64, false, 128>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<96, false, 128>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<128, false, 128>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs2_gemm_impl<384, false, 256>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template int max_active_pairs_impl<128, false, 256>();
template int max_active_pairs_impl<128, true, 256>();
template int max_active_pairs_impl<192, false, 256>();
template int max_active_pairs_impl<192, true, 256>();
template int max_active_pairs_impl<224, false, 256>();
template int max_active_pairs_impl<224, true, 256>();
template int max_active_pairs_impl<240, false, 256>();
template int max_active_pairs_impl<240, true, 256>();
template int max_active_pairs_impl<256, false, 256>();
template int max_active_pairs_impl<32, false, 128>();
template int max_active_pairs_impl<64, false, 128>();
template int max_active_pairs_impl<96, false, 128>();
template int max_active_pairs_impl<128, false, 128>();
template int max_active_pairs_impl<384, false, 256>();
}  // namespace dg
