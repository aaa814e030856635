// Instantiations of the block-scaled GEMM kernel (compiled in parallel, one group per file).
#include "gemm_bs.cuh"

namespace dg {
template cudaError_t launch_bs_gemm_impl<176, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
template cudaError_t launch_bs_gemm_impl<192, false>(const TensorMaps &, const GemmParams &, int, cudaStream_t);
}  // namespace dg
