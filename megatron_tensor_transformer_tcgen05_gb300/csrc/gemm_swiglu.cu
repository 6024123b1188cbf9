// SwiGLU variant of the block: the dual up-projection (Ha = X A, Hg = X Wg, U = SiLU(Ha) Hg)
// and the dU GEMM with the SwiGLU derivative in its epilogue.
#include "umma_gemm.cuh"

namespace mlp {
template cudaError_t launch_umma_gemm<256, false, true, EPI_SWIGLU, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_SWIGLU, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<128, false, false, EPI_DSWIGLU, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, false, EPI_DSWIGLU, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, false, EPI_DSWIGLU, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<128, false, true, EPI_PLAIN, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_PLAIN, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_PLAIN, 2>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<512, false, true, EPI_PLAIN, 2>(const GemmArgs&, int, cudaStream_t);
template int umma_gemm_max_clusters<512, false, true, EPI_PLAIN, 2>(int, int);
}  // namespace mlp
