// Backward GEMM 3: dH = (dY*B^T) (.) GELU'(H) (both operands K-major), with da's per-32-row
// column sums.
#include "umma_gemm.cuh"

namespace mlp {
template cudaError_t launch_umma_gemm<128, false, false, EPI_DGELU, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, false, EPI_DGELU, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, false, EPI_DGELU, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<512, false, false, EPI_DGELU, 2>(const GemmArgs&, int, cudaStream_t);
template int umma_gemm_max_clusters<512, false, false, EPI_DGELU, 2>(int, int);
}  // namespace mlp
