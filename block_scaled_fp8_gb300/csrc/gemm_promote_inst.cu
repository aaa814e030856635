// Instantiations of the FP32-scale promotion GEMM kernel.
#include "gemm_promote.cuh"

namespace dg {
template cudaError_t launch_promote_gemm_impl<32, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_promote_gemm_impl<32, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_promote_gemm_impl<64, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_promote_gemm_impl<64, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_promote_gemm_impl<128, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_promote_gemm_impl<128, true>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
}  // namespace dg
