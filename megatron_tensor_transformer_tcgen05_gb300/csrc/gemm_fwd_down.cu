// Forward GEMM 2: Y = G*B + b, K loop over all shards (A operand G K-major, B operand B MN-major),
// and its variant with the bias + dropout + residual-add epilogue (Z = R + dropout(G*B + b)).
#include "umma_gemm.cuh"

namespace mlp {
template cudaError_t launch_umma_gemm<128, false, true, EPI_BIAS, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_BIAS, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_BIAS, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<512, false, true, EPI_BIAS, 2>(const GemmArgs&, int, cudaStream_t);
template int umma_gemm_max_clusters<512, false, true, EPI_BIAS, 2>(int, int);
template cudaError_t launch_umma_gemm<128, false, true, EPI_BIAS_DROPOUT_RES, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_BIAS_DROPOUT_RES, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_BIAS_DROPOUT_RES, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<512, false, true, EPI_BIAS_DROPOUT_RES, 2>(const GemmArgs&, int, cudaStream_t);
template int umma_gemm_max_clusters<512, false, true, EPI_BIAS_DROPOUT_RES, 2>(int, int);
}  // namespace mlp
