// Split-tail fixup: the output tiles of a GEMM whose last tiles ran as K-range parts, with
// the epilogue those tiles skipped.
#include "umma_gemm.cuh"

namespace mlp {

// Block (r, c): split tile r, output columns [32c, 32c + 32) of it; thread = row of the
// tile (up to 512 rows: a cluster's two CTA pairs). Each thread reads its row's 32 fp32
// values from each part (128 contiguous bytes; consecutive rows are consecutive) and adds the
// parts in index order. Then, as the GEMM's own epilogue would:
//   EPI_PLAIN / EPI_BIAS  out0 = bf16(sum (+ bias))
//   EPI_BIAS_GELU         out0 = H = bf16(sum + bias), out1 = G = bf16(GELU(H))
//   EPI_DGELU             out0 = dH = bf16(sum * GELU'(H)) with H = aux; and, when wanted, the
//                         column sums of the fp32 dH over each 32-row block (a warp's rows)
// all with round-to-nearest-even.
template <int EPI>
__global__ void __launch_bounds__(512) splitk_fixup_kernel(const GemmArgs args, int TM, int BN, int n_whole,
                                                           int tiles_m, int tiles_n, __nv_bfloat16* __restrict__ out0,
                                                           __nv_bfloat16* __restrict__ out1, long long ld_out)
{
    const int r = blockIdx.x, c = blockIdx.y, row = threadIdx.x, lane = threadIdx.x & 31;
    const int M = args.M, N = args.N;
    int m0, n0;
    tile_origin(n_whole + r, tiles_m, tiles_n, args.n_fastest, args.raster_group, TM, BN, m0, n0);
    const int gm = m0 + row, gn = n0 + 32 * c;
    if (gn >= N) return;  // block-uniform
    // rows past M: no output; in the dH flavour they still take part in the warp's column
    // sums, with zeros, as the GEMM's epilogue's out-of-range rows do
    const bool in_row = gm < M;
    if (EPI != EPI_DGELU && !in_row) return;
    const size_t part = static_cast<size_t>(TM) * BN;
    const float4* p = reinterpret_cast<const float4*>(args.split_ws + static_cast<size_t>(r) * args.split_k * part +
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
    for (int sk = 1; sk < args.split_k; ++sk) {
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
    if (EPI == EPI_BIAS || EPI == EPI_BIAS_GELU) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = gn + 8 * i;
            float bv[8];
            unpack_bf16x8(n < N ? *reinterpret_cast<const uint4*>(args.bias + n) : make_uint4(0, 0, 0, 0), bv);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[8 * i + j] += bv[j];
        }
    }
    if (EPI == EPI_DGELU) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = gn + 8 * i;
            float hv[8];
            unpack_bf16x8(in_row && n < N ? ldg_nc_v4(args.aux + static_cast<size_t>(gm) * args.ld_aux + n)
                                          : make_uint4(0, 0, 0, 0),
                          hv);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[8 * i + j] = in_row ? v[8 * i + j] * gelu_tanh_grad_f(hv[j]) : 0.0f;
        }
        if (args.colsum_rows) {  // this warp's 32 rows, summed per column
            float cs[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) cs[j] = v[j];
            warp_column_sums(cs, lane);
            if (gm - lane < M && gn + lane < N)
                args.colsum_rows[static_cast<size_t>((gm - lane) >> 5) * N + gn + lane] = cs[0];
        }
        if (!in_row) return;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int n = gn + 8 * i;
        if (n >= N) break;
        uint4 o;
        o.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
        o.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
        o.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
        o.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
        *reinterpret_cast<uint4*>(out0 + static_cast<size_t>(gm) * ld_out + n) = o;
        if (EPI == EPI_BIAS_GELU) {  // G = GELU(H) of the rounded H
            const uint32_t w[4] = {o.x, o.y, o.z, o.w};
            uint32_t g[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                g[k] = pack_bf16x2(gelu_tanh_f(__uint_as_float(w[k] << 16)),
                                   gelu_tanh_f(__uint_as_float(w[k] & 0xFFFF0000u)));
            *reinterpret_cast<uint4*>(out1 + static_cast<size_t>(gm) * ld_out + n) = make_uint4(g[0], g[1], g[2], g[3]);
        }
    }
}

cudaError_t launch_splitk_fixup(const GemmArgs& args, int epi, int TM, int BN, __nv_bfloat16* out0,
                                __nv_bfloat16* out1, long long ld_out, cudaStream_t stream)
{
    if (args.split_tiles <= 0) return cudaSuccess;
    const int tiles_m = (args.M + TM - 1) / TM, tiles_n = (args.N + BN - 1) / BN;
    const int n_whole = tiles_m * tiles_n - args.split_tiles;
    const dim3 grid(args.split_tiles, BN / 32);
    switch (epi) {
    case EPI_PLAIN:
        splitk_fixup_kernel<EPI_PLAIN><<<grid, TM, 0, stream>>>(args, TM, BN, n_whole, tiles_m, tiles_n, out0, out1,
                                                                ld_out);
        break;
    case EPI_BIAS:
        splitk_fixup_kernel<EPI_BIAS><<<grid, TM, 0, stream>>>(args, TM, BN, n_whole, tiles_m, tiles_n, out0, out1,
                                                               ld_out);
        break;
    case EPI_BIAS_GELU:
        splitk_fixup_kernel<EPI_BIAS_GELU><<<grid, TM, 0, stream>>>(args, TM, BN, n_whole, tiles_m, tiles_n, out0,
                                                                    out1, ld_out);
        break;
    case EPI_DGELU:
        splitk_fixup_kernel<EPI_DGELU><<<grid, TM, 0, stream>>>(args, TM, BN, n_whole, tiles_m, tiles_n, out0, out1,
                                                                ld_out);
        break;
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace mlp
