// gemm_args.h -- launch arguments of the tcgen05 GEMM family (host and device view).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "philox.cuh"

namespace mlp {

enum Epi : int { EPI_PLAIN = 0, EPI_BIAS = 1, EPI_BIAS_GELU = 2, EPI_DGELU = 3, EPI_BIAS_DROPOUT_RES = 4 };

struct GemmArgs {
    CUtensorMap tmA;    // A operand (K-major box 64x128, or MN-major box 64x64)
    CUtensorMap tmB;    // B operand (K-major box 64xBN, or MN-major box 64x64)
    CUtensorMap tmD0;   // first output, store box 32x32, 64B swizzle
    CUtensorMap tmD1;   // second output (G of EPI_BIAS_GELU), same box
    int M, N, K;
    int n_fastest;               // tile order: 0 = M index fastest, 1 = N index fastest
    int raster_group;            // tiles of the fast index per group (<= 0: all of them)
    const __nv_bfloat16* bias;   // [N] for EPI_BIAS / EPI_BIAS_GELU
    const __nv_bfloat16* aux;    // H [M, ld_aux] for EPI_DGELU; residual R for EPI_BIAS_DROPOUT_RES
    float* colsum_rows;          // EPI_DGELU, optional: per-32-row column sums of D (fp32),
                                 // [ceil(M/32), N] row-major; NULL = not wanted
    long long ld_aux;
    int* status;                 // device status word (first error code wins)
    DropoutParams drop;          // EPI_BIAS_DROPOUT_RES
    unsigned long long timeout_ns;
};

// Defined in umma_gemm.cuh; explicitly instantiated once per flavour (gemm_*.cu).
template <int BN, bool A_MN, bool B_MN, int EPI, int CG>
cudaError_t launch_umma_gemm(const GemmArgs& args, int grid, cudaStream_t stream);

}  // namespace mlp
