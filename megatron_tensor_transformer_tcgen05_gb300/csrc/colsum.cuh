// colsum.cuh -- bias-gradient column reductions da[j] = sum_r dH[r,j], db[j] = sum_r dY[r,j].
// In the backward pass the dH GEMM's epilogue already sums dH over each 32-row block, so
// only dY goes through the partial pass here; the entry point without a workspace reduces
// both matrices with these kernels.
//
// Memory-bound. Each warp reads 4 rows x 64 columns per step with 16-byte vector loads
// (lane = 8 columns of one row; 8 lanes cover one 128-byte row segment), keeps 8 fp32
// running sums per lane, folds the 4 row-lanes together with warp shuffles, then the 8
// warps of the block combine in shared memory in a fixed order. Rows are split into a
// fixed number of slices whose partial sums go to a workspace; a second kernel adds the
// slices in slice order. No atomics: results are bitwise reproducible run to run.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace mlp {

constexpr int kColsumThreads = 256;
constexpr int kColsumStrip = 64;  // columns per block

__device__ __forceinline__ uint4 colsum_ldg(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void colsum_acc8(float* s, const uint4& u)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        s[2 * i] += __uint_as_float(w[i] << 16);
        s[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Two matrices share one launch: column strips [0, strips1) belong to P1 (cols1 wide), the
// rest to P2. blockIdx.y is the row slice. partial is [nsplit][cols1 + cols2].
__global__ void __launch_bounds__(kColsumThreads)
colsum_partial_kernel(const __nv_bfloat16* __restrict__ P1, int cols1, const __nv_bfloat16* __restrict__ P2,
                      int cols2, long long rows, int nsplit, float* __restrict__ partial)
{
    __shared__ float red[kColsumThreads / 32][kColsumStrip];
    const int strips1 = (cols1 + kColsumStrip - 1) / kColsumStrip;
    const bool second = static_cast<int>(blockIdx.x) >= strips1;
    const __nv_bfloat16* P = second ? P2 : P1;
    const int cols = second ? cols2 : cols1;
    const int strip = second ? static_cast<int>(blockIdx.x) - strips1 : static_cast<int>(blockIdx.x);
    const int out_off = second ? cols1 : 0;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cg = lane & 7, ro = lane >> 3;
    const int col = strip * kColsumStrip + cg * 8;
    const long long per = (rows + nsplit - 1) / nsplit;
    const long long r_begin = per * blockIdx.y;
    const long long r_end = r_begin + per < rows ? r_begin + per : rows;

    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (col < cols) {
        const long long step = 4LL * (kColsumThreads / 32);  // rows per block step
        long long r = r_begin + 4 * warp + ro;
        for (; r + 3 * step < r_end; r += 4 * step) {
            const uint4 u0 = colsum_ldg(P + r * cols + col);
            const uint4 u1 = colsum_ldg(P + (r + step) * cols + col);
            const uint4 u2 = colsum_ldg(P + (r + 2 * step) * cols + col);
            const uint4 u3 = colsum_ldg(P + (r + 3 * step) * cols + col);
            colsum_acc8(s, u0);
            colsum_acc8(s, u1);
            colsum_acc8(s, u2);
            colsum_acc8(s, u3);
        }
        for (; r < r_end; r += step) colsum_acc8(s, colsum_ldg(P + r * cols + col));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        s[j] += __shfl_xor_sync(0xffffffffu, s[j], 8);
        s[j] += __shfl_xor_sync(0xffffffffu, s[j], 16);
    }
    if (ro == 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) red[warp][cg * 8 + j] = s[j];
    }
    __syncthreads();
    if (threadIdx.x < kColsumStrip) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kColsumThreads / 32; ++w) t += red[w][threadIdx.x];
        const int c = strip * kColsumStrip + static_cast<int>(threadIdx.x);
        if (c < cols) partial[static_cast<long long>(blockIdx.y) * (cols1 + cols2) + out_off + c] = t;
    }
}

// out1[c] = sum_s partial[s][c] for c < cols1, out2[c] = sum_s partial[s][cols1 + c].
__global__ void colsum_finalize_kernel(const float* __restrict__ partial, int nsplit, int cols1,
                                       int cols2, float* __restrict__ out1, float* __restrict__ out2)
{
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const int total = cols1 + cols2;
    if (c >= total) return;
    float t = 0.f;
    for (int s = 0; s < nsplit; ++s) t += partial[static_cast<long long>(s) * total + c];
    if (c < cols1)
        out1[c] = t;
    else
        out2[c - cols1] = t;
}

// da[c] = sum over 32-row blocks rb of rows[rb][c] (written by the dH GEMM's epilogue);
// db[c] = sum over slices s of partial[s][c] (from colsum_partial_kernel over dY alone).
// Both sums run in index order, so the results are bitwise reproducible.
__global__ void bias_grad_finalize_kernel(const float* __restrict__ rows, int nrb, int f,
                                          const float* __restrict__ partial, int nsplit, int h,
                                          float* __restrict__ da, float* __restrict__ db)
{
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c < f) {
        float t = 0.f;
        for (int rb = 0; rb < nrb; ++rb) t += rows[static_cast<long long>(rb) * f + c];
        da[c] = t;
    } else if (c < f + h) {
        const int j = c - f;
        float t = 0.f;
        for (int s = 0; s < nsplit; ++s) t += partial[static_cast<long long>(s) * h + j];
        db[j] = t;
    }
}

}  // namespace mlp
