// philox.cuh -- Philox4x32-10 counter-based random numbers (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC 2011) and the dropout keep rule of the
// block's output step: element e of a row-major [T, h] tensor uses word e % 4 of Philox on
// counter (lo32(e/4), hi32(e/4), lo32(offset), hi32(offset)) with key (lo32(seed),
// hi32(seed)), and is kept when its top 24 bits are >= p24 = floor(p * 2^24).
#pragma once
#include <cstdint>

namespace mlp {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;  // key schedule: Weyl increments
        k1 += 0xBB67AE85u;
    }
    return c;
}

struct DropoutParams {
    unsigned long long seed, offset;
    uint32_t p24;  // floor(p * 2^24): keep when the word's top 24 bits are >= p24
    float scale;   // 1 / (1 - p)
};

// Keep bits of the 4 elements 4q .. 4q+3 (bit w = element 4q + w).
__device__ __forceinline__ uint32_t dropout_keep4(const DropoutParams& d, unsigned long long q)
{
    const uint4 r = philox4x32_10(make_uint4(static_cast<uint32_t>(q), static_cast<uint32_t>(q >> 32),
                                             static_cast<uint32_t>(d.offset), static_cast<uint32_t>(d.offset >> 32)),
                                  static_cast<uint32_t>(d.seed), static_cast<uint32_t>(d.seed >> 32));
    return static_cast<uint32_t>((r.x >> 8) >= d.p24) | (static_cast<uint32_t>((r.y >> 8) >= d.p24) << 1) |
           (static_cast<uint32_t>((r.z >> 8) >= d.p24) << 2) | (static_cast<uint32_t>((r.w >> 8) >= d.p24) << 3);
}

}  // namespace mlp
