// gemm_args.h -- launch arguments of the tcgen05 GEMM family (host and device view).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "philox.cuh"

namespace mlp {

enum Epi : int {
    EPI_PLAIN = 0,
    EPI_BIAS = 1,
    EPI_BIAS_GELU = 2,
    EPI_DGELU = 3,
    EPI_BIAS_DROPOUT_RES = 4,
    EPI_SWIGLU = 5,   // dual B operand: D = [X A | X Wg] per 128 output columns -> Ha, Hg, U
    EPI_DSWIGLU = 6,  // dU = acc; dHa = dU Hg SiLU'(Ha), dHg = dU SiLU(Ha) -> dHa, dHg
    // The A operand is H, turned into G = GELU(H) in shared memory before the MMAs read it
    // (operand-transform warps); the epilogue is that of EPI_PLAIN / EPI_BIAS.
    EPI_PLAIN_GA = 8,
    EPI_BIAS_GA = 9,
};

struct GemmArgs {
    CUtensorMap tmA;    // A operand (K-major box 64x128, or MN-major box 64x64)
    CUtensorMap tmB;    // B operand (K-major box 64xBN, or MN-major box 64x64)
    CUtensorMap tmD0;   // first output, store box 32x32, 64B swizzle
    CUtensorMap tmD1;   // second output (G of EPI_BIAS_GELU), same box
    CUtensorMap tmD2;   // third output (U of EPI_SWIGLU), same box
    CUtensorMap tmA2;   // A operand of the second K segment (kb_split > 0)
    CUtensorMap tmB2;   // B operand of the second K segment, or the gate weight of EPI_SWIGLU
    int M, N, K;
    int n_fastest;               // tile order: 0 = M index fastest, 1 = N index fastest
    int raster_group;            // tiles of the fast index per group (<= 0: all of them)
    const __nv_bfloat16* bias;   // [N] for EPI_BIAS / EPI_BIAS_GELU
    const __nv_bfloat16* aux;    // H [M, ld_aux] for EPI_DGELU(_G); residual R for EPI_BIAS_DROPOUT_RES
    float* colsum_rows;          // EPI_DGELU, optional: per-32-row column sums of D (fp32),
                                 // [ceil(M/32), N] row-major; NULL = not wanted
    const __nv_bfloat16* aux2;   // Hg [M, ld_aux] for EPI_DSWIGLU (aux is Ha)
    long long ld_aux;
    // K concatenation: k blocks [0, kb_split) read (tmA, tmB), the rest read (tmA2, tmB2)
    // from their own k = 0, so D = A1 B1^T + A2 B2^T in one accumulator (0 = one segment).
    int kb_split;
    // Split tail (EPI_PLAIN, EPI_BIAS, EPI_BIAS_GELU, EPI_DGELU): the last split_tiles tiles of the tile order each
    // run as split_k parts over consecutive ranges of k blocks; part p writes its fp32
    // accumulator to split_ws[p * TM * OBN ...] and splitk_fixup_kernel sums them in order.
    int split_tiles;             // 0 = every tile whole
    // CTA pairs per cluster for 512-wide pair tiles: 2 = a work tile is 512 x 512, the two
    // pairs' rows, and each stage's B is fetched once and multicast to both pairs; else 1.
    int cluster_pairs;
    int split_k;
    float* split_ws;
    int* status;                 // device status word (first error code wins)
    DropoutParams drop;          // EPI_BIAS_DROPOUT_RES
    unsigned long long timeout_ns;
};

// Defined in umma_gemm.cuh; explicitly instantiated once per flavour (gemm_*.cu).
template <int BN, bool A_MN, bool B_MN, int EPI, int CG>
cudaError_t launch_umma_gemm(const GemmArgs& args, int grid, cudaStream_t stream);

// Clusters of `cluster` CTAs of that flavour that can be resident at once (0 on error).
template <int BN, bool A_MN, bool B_MN, int EPI, int CG>
int umma_gemm_max_clusters(int cluster, int num_sms);

// After a GEMM launched with split_tiles > 0: for the split tiles, the sum of each tile's
// parts in order, then the epilogue `epi` (EPI_PLAIN, EPI_BIAS, EPI_BIAS_GELU: out0 = H,
// out1 = G; EPI_DGELU: out0 = dH, and args.colsum_rows when set). TM x BN is the GEMM's work
// tile (rows x output columns); outputs are row-major with leading dimension ld_out. One launch.
cudaError_t launch_splitk_fixup(const GemmArgs& args, int epi, int TM, int BN, __nv_bfloat16* out0,
                                __nv_bfloat16* out1, long long ld_out, cudaStream_t stream);

}  // namespace mlp
