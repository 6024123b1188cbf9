// Split-tail fixup: the bf16 output tiles of a GEMM whose last tiles ran as K-range parts.
#include "umma_gemm.cuh"

namespace mlp {

// Block (r, c): split tile r, output columns [32c, 32c + 32) of it; thread = row of the
// tile (up to 512 rows: a cluster's two CTA pairs). Each thread reads its row's 32 fp32
// values from each part (128 contiguous bytes; consecutive rows are consecutive), adds the
// parts in index order, then the bias, and writes 32 bf16 with round-to-nearest-even.
__global__ void __launch_bounds__(512) splitk_fixup_kernel(const float* __restrict__ ws, int split_k, int n_whole,
                                                           int tiles_m, int tiles_n, int n_fastest, int group,
                                                           int TM, int BN, int M, int N,
                                                           const __nv_bfloat16* __restrict__ bias,
                                                           __nv_bfloat16* __restrict__ out, long long ld_out)
{
    const int r = blockIdx.x, c = blockIdx.y, row = threadIdx.x;
    int m0, n0;
    tile_origin(n_whole + r, tiles_m, tiles_n, n_fastest, group, TM, BN, m0, n0);
    const int gm = m0 + row, gn = n0 + 32 * c;
    if (row >= TM || gm >= M || gn >= N) return;
    const size_t part = static_cast<size_t>(TM) * BN;
    const float4* p = reinterpret_cast<const float4*>(ws + static_cast<size_t>(r) * split_k * part +
                                                      (static_cast<size_t>(c) * TM + row) * 32);
    float v[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 x = p[j];
        v[4 * j] = x.x;
        v[4 * j + 1] = x.y;
        v[4 * j + 2] = x.z;
        v[4 * j + 3] = x.w;
    }
    for (int sk = 1; sk < split_k; ++sk) {
        p += part / 4;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 x = p[j];
            v[4 * j] += x.x;
            v[4 * j + 1] += x.y;
            v[4 * j + 2] += x.z;
            v[4 * j + 3] += x.w;
        }
    }
    // N is a multiple of 8: whole groups of 8 columns are in or out
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int n = gn + 8 * i;
        if (n >= N) break;
        float w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = v[8 * i + j];
        if (bias) {
            float bv[8];
            unpack_bf16x8(*reinterpret_cast<const uint4*>(bias + n), bv);
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] += bv[j];
        }
        uint4 o;
        o.x = pack_bf16x2(w[0], w[1]);
        o.y = pack_bf16x2(w[2], w[3]);
        o.z = pack_bf16x2(w[4], w[5]);
        o.w = pack_bf16x2(w[6], w[7]);
        *reinterpret_cast<uint4*>(out + static_cast<size_t>(gm) * ld_out + n) = o;
    }
}

cudaError_t launch_splitk_fixup(const GemmArgs& args, int TM, int BN, __nv_bfloat16* out, long long ld_out,
                                cudaStream_t stream)
{
    if (args.split_tiles <= 0) return cudaSuccess;
    const int tiles_m = (args.M + TM - 1) / TM, tiles_n = (args.N + BN - 1) / BN;
    const int n_whole = tiles_m * tiles_n - args.split_tiles;
    splitk_fixup_kernel<<<dim3(args.split_tiles, BN / 32), TM, 0, stream>>>(
        args.split_ws, args.split_k, n_whole, tiles_m, tiles_n, args.n_fastest, args.raster_group, TM, BN, args.M,
        args.N, args.bias, out, ld_out);
    return cudaGetLastError();
}

}  // namespace mlp
