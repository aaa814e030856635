// Instantiations of the block-scaled GEMM kernel (compiled in parallel, one group per file).
#include "gemm_bs.cuh"

namespace dg {
template cudaError_t launch_bs_gemm_impl<16, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs_gemm_impl<16, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs_gemm_impl<32, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs_gemm_impl<32, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs_gemm_impl<48, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs_gemm_impl<48, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs_gemm_impl<64, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs_gemm_impl<64, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
}  // namespace dg
