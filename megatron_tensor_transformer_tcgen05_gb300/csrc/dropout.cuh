// dropout.cuh -- backward of the block's output step: dY = dZ (.) keep / (1 - p), with the
// keep mask regenerated from the same Philox counters the forward epilogue used. HBM-bound:
// each thread streams 16-byte vectors (8 bf16 = two Philox draws), grid-stride.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "philox.cuh"

namespace mlp {

__global__ void __launch_bounds__(256) dropout_backward_kernel(const __nv_bfloat16* __restrict__ dZ, long long n8,
                                                               DropoutParams d, __nv_bfloat16* __restrict__ dY)
{
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
        uint4 u;
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                     : "l"(dZ + 8 * i));
        const uint32_t keep = dropout_keep4(d, 2 * static_cast<unsigned long long>(i)) |
                              (dropout_keep4(d, 2 * static_cast<unsigned long long>(i) + 1) << 4);
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = (keep >> (2 * j)) & 1u ? __uint_as_float(w[j] << 16) * d.scale : 0.0f;
            const float hi = (keep >> (2 * j + 1)) & 1u ? __uint_as_float(w[j] & 0xFFFF0000u) * d.scale : 0.0f;
            __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
            w[j] = *reinterpret_cast<uint32_t*>(&v);
        }
        asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(dY + 8 * i), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                     "r"(w[3])
                     : "memory");
    }
}

}  // namespace mlp
