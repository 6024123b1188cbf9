// Forward GEMM 2: Y = G*B + b, K loop over all shards (A operand G K-major, B operand B MN-major).
#include "umma_gemm.cuh"

namespace mlp {
template cudaError_t launch_umma_gemm<128, false, true, EPI_BIAS, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_BIAS, 1>(const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_umma_gemm<256, false, true, EPI_BIAS, 2>(const GemmArgs&, int, cudaStream_t);
}  // namespace mlp
