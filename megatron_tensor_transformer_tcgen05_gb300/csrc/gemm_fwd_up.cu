// Forward GEMM 1: H = X*A + a, G = GELU(H) (A operand X K-major, B operand A MN-major).
#include "umma_gemm.cuh"

namespace mlp {
template cudaError_t launch_umma_gemm<128, false, true, EPI_BIAS_GELU, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_BIAS_GELU, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_BIAS_GELU, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<512, false, true, EPI_BIAS_GELU, 2>(const GemmArgs&, int, cudaStream_t);
template int umma_gemm_max_clusters<512, false, true, EPI_BIAS_GELU, 2>(int, int);
}  // namespace mlp
