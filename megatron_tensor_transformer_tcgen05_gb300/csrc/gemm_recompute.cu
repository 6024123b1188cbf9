// The GELU-recompute GEMMs: their A operand is read as H and turned into G = GELU(H) in
// shared memory before the MMAs (operand-transform warps), so G never goes to HBM.
//   forward GEMM 2:  Y = GELU(H)*B + b   (A operand H K-major, B operand B MN-major)
//   backward GEMM 6: dB = GELU(H)^T*dY   (both operands MN-major)
#include "umma_gemm.cuh"

namespace mlp {
template cudaError_t launch_umma_gemm<128, false, true, EPI_BIAS_GA, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_BIAS_GA, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_BIAS_GA, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<512, false, true, EPI_BIAS_GA, 2>(const GemmArgs&, int, cudaStream_t);
template int umma_gemm_max_clusters<512, false, true, EPI_BIAS_GA, 2>(int, int);
template cudaError_t launch_umma_gemm<128, true, true, EPI_PLAIN_GA, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, true, true, EPI_PLAIN_GA, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, true, true, EPI_PLAIN_GA, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<512, true, true, EPI_PLAIN_GA, 2>(const GemmArgs&, int, cudaStream_t);
template int umma_gemm_max_clusters<512, true, true, EPI_PLAIN_GA, 2>(int, int);
}  // namespace mlp
