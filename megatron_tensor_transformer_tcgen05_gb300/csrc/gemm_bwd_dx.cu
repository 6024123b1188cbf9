// Backward GEMM 4: dX = dH*A^T, K loop over all shards (both operands K-major).
#include "umma_gemm.cuh"

namespace mlp {
template cudaError_t launch_umma_gemm<128, false, false, EPI_PLAIN, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, false, EPI_PLAIN, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, false, EPI_PLAIN, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<512, false, false, EPI_PLAIN, 2>(const GemmArgs&, int, cudaStream_t);
template int umma_gemm_max_clusters<512, false, false, EPI_PLAIN, 2>(int, int);
}  // namespace mlp
