// Backward GEMMs 5 and 6: dA = X^T*dH and dB = G^T*dY (both operands MN-major).
#include "umma_gemm.cuh"

namespace mlp {
template cudaError_t launch_umma_gemm<128, true, true, EPI_PLAIN, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, true, true, EPI_PLAIN, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, true, true, EPI_PLAIN, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<512, true, true, EPI_PLAIN, 2>(const GemmArgs&, int, cudaStream_t);
template int umma_gemm_max_clusters<512, true, true, EPI_PLAIN, 2>(int, int);
}  // namespace mlp
