// attention.cu -- fused causal self-attention for the head-parallel attention block, on
// tcgen05 tensor cores with TMEM accumulators, for sm_103a.
//
// Per head h of width d = 128, with Q, K, V the head's columns of the QKV projection:
//   S = Q K^T / sqrt(d),  key j > query i masked when causal,  P = softmax_rows(S),  C = P V
// ("Efficient Large-Scale Language Model Training on GPU Clusters Using Megatron-LM",
// section 3, Figure 5b: each tensor-parallel shard runs whole heads, so the softmax never
// crosses a shard; and its "Computation Optimizations: Fused Kernels and Data Layout" fuses
// scale, mask and softmax into one kernel with the causal mask implicit). Here the whole of
// S -> P -> C also stays on chip: S is never written to HBM.
//
// Forward (attn_fwd_kernel): one CTA per (sequence, head, 128-query block), 192 threads, two
// CTAs per SM (one's softmax overlaps the other's MMAs).
//   warp 0     TMA: the Q block once, then K and V blocks of 64 keys through two 2-slot rings
//   warp 1     TMEM allocation and every tcgen05.mma: S_j = Q K_j^T into one of two TMEM
//              S buffers, O += P_j V_j into the TMEM output accumulator
//   warps 2-5  softmax, thread r <-> query row r (TMEM lane r): read S_j from TMEM, mask,
//              running row max and sum (base 2), P_j (bf16) back into TMEM over S_j, where
//              the P_j V_j MMA reads it as its A operand; rescale O in TMEM only when the row max has grown by more
//              than 2^16 since the last rescale (the final division by the row sum makes the
//              result exact whatever reference the exponentials used). Finally C = O / l and
//              the row's base-2 log-sum-exp L for the backward pass.
// Backward, deterministic (no atomics), two kernels that each recompute P from Q, K and L:
//   attn_bwd_dkdv_kernel: one CTA per (sequence, head, 128-key block), looping over 64-query
//     blocks: S^T = K Q^T, dP^T = V dC^T, P^T = exp2(S^T c - L), dS^T = P^T (dP^T - D) (both
//     back into TMEM over S^T and dP^T), dV += P^T dC, dK += dS^T Q.
//   attn_bwd_dq_kernel: one CTA per (sequence, head, 128-query block), looping over 128-key
//     blocks: S = Q K^T, dP = dC V^T, dS = P (dP - D) (into a TMEM double buffer), dQ += dS K;
//     the next block's S and dP products start as soon as this block's are in registers.
//   with D = rowsum(dC * C) from attn_bwd_dot_kernel.
// A tile of Q, K, V or dC is loaded once, row-major with a 128-byte swizzle, and read by
// the tensor core both as a K-major operand (contraction over d) and as an MN-major one
// (contraction over tokens): only the shared-memory descriptor differs, nothing is
// transposed in memory.
#include <cuda_bf16.h>
#include <cstdint>

#include "attn_args.h"
#include "sm103_ptx.cuh"

namespace mlp {

namespace {

constexpr unsigned long long kAttnDrainNs = 2000000000ull;
// Rescale O only once the row max has grown by more than 2^16 since the last rescale: P (bf16)
// and the fp32 row sum and O then stay within 2^16 x their normalised size (2^27 for the sum
// at s = 2048), far inside fp32, and rows whose max keeps creeping up rescale rarely.
constexpr int kLazyRescaleLog2 = 16;

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float4 lds128f(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// 2^x on the special-function unit (hand-written wrapper of the PTX instruction;
// ex2 of -inf is +0, which is what a masked score needs).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Pairs of fp32 values in one 64-bit register, for the sm_100-family f32x2 instructions: two
// IEEE round-to-nearest operations each, so the same bits as the scalar forms at half the issue.
typedef unsigned long long f2_t;
__device__ __forceinline__ f2_t f2(float lo, float hi)
{
    f2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(f2_t v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_fma_(f2_t a, f2_t b, f2_t c)
{
    f2_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2_t f2_add_(f2_t a, f2_t b)
{
    f2_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2_t f2_mul_(f2_t a, f2_t b)
{
    f2_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// x[c] = 2^(x[c] a + b) for N values, the fma on pairs
template <int N>
__device__ __forceinline__ void exp2_affine(float (&x)[N], float a, float b)
{
    const f2_t av = f2(a, a), bv = f2(b, b);
#pragma unroll
    for (int c = 0; c < N; c += 2) {
        float lo, hi;
        f2_split(f2_fma_(f2(x[c], x[c + 1]), av, bv), lo, hi);
        x[c] = ex2(lo);
        x[c + 1] = ex2(hi);
    }
}

__device__ __forceinline__ void sts_f32(uint32_t addr, float v)
{
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// 32 fp32 values * mul -> 32 bf16 at dst (64 bytes, 16-byte aligned).
__device__ __forceinline__ void store32_global(__nv_bfloat16* dst, const uint32_t (&r)[32], float mul)
{
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 w;
        w.x = pack2_bf16(__uint_as_float(r[8 * i + 0]) * mul, __uint_as_float(r[8 * i + 1]) * mul);
        w.y = pack2_bf16(__uint_as_float(r[8 * i + 2]) * mul, __uint_as_float(r[8 * i + 3]) * mul);
        w.z = pack2_bf16(__uint_as_float(r[8 * i + 4]) * mul, __uint_as_float(r[8 * i + 5]) * mul);
        w.w = pack2_bf16(__uint_as_float(r[8 * i + 6]) * mul, __uint_as_float(r[8 * i + 7]) * mul);
        d4[i] = w;
    }
}

__device__ __forceinline__ uint64_t desc_k(uint32_t addr) { return smem_desc_sw128(addr, 16u, 1024u); }

// The descriptor of a tile `off` bytes further on: the start-address field (bits 0-13) holds
// addr >> 4 and every shared address here is below 2^18, so the field never carries and a
// 64-bit add equals a fresh encoding. Building each buffer's descriptor once and adding
// constants keeps the MMA-issuing thread to a few instructions per MMA (it shares its
// SM sub-partition with two busy softmax warps, and the MMAs here are short).
__device__ __forceinline__ uint64_t desc_at(uint64_t base_desc, uint32_t off) { return base_desc + (off >> 4); }
__device__ __forceinline__ uint64_t desc_mn(uint32_t addr, uint32_t chunk_stride)
{
    return smem_desc_sw128(addr, chunk_stride, 1024u);
}

// One lane waits; the warp follows its verdict (TMEM loads are warp-collective).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status,
                                          unsigned long long limit, int code, int wa, int wb)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, abort, status, limit, code, wa, wb);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Producer-side drain after an abort: wait (bounded, ignoring the abort flag) for every
// copy this CTA started, so that none lands after the CTA has exited.
__device__ __forceinline__ void drain_loads(uint32_t bars, int nbars, uint32_t issued, uint32_t par, int* status)
{
    volatile int never = 0;
    for (int i = 0; i < nbars; ++i)
        if (issued & (1u << i))
            mbar_wait_bounded(bars + 8u * i, (par >> i) & 1u, &never, status, kAttnDrainNs, DEV_TIMEOUT_DRAIN);
}

__device__ __forceinline__ void drain_mma(uint32_t bar, int* status)
{
    volatile int never = 0;
    umma_commit(bar);
    mbar_wait_bounded(bar, 0, &never, status, kAttnDrainNs, DEV_TIMEOUT_DRAIN);
}

// ---- forward -------------------------------------------------------------------------------

// Max and sum of N values through 8 independent partial results (short dependency chains).
template <int N>
__device__ __forceinline__ float max_tree(const float (&x)[N])
{
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = x[i];
#pragma unroll
    for (int c = 8; c < N; ++c) m[c & 7] = fmaxf(m[c & 7], x[c]);
    return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}

template <int N>
__device__ __forceinline__ float sum_tree(const float (&x)[N])
{
    // m[i] = x[i] + x[i + 8] + x[i + 16] + ... in that order, four pairs at a time
    f2_t m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = f2(x[2 * i], x[2 * i + 1]);
#pragma unroll
    for (int c = 8; c < N; c += 8)
#pragma unroll
        for (int i = 0; i < 4; ++i) m[i] = f2_add_(m[i], f2(x[c + 2 * i], x[c + 2 * i + 1]));
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) f2_split(m[i], v[2 * i], v[2 * i + 1]);
    return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

struct FwdCfg {
    static constexpr int BQ = 128, BKV = 64;
    // producer, MMA, 4 softmax warps (one thread per query row); two CTAs share an SM, so one
    // CTA's softmax runs while the other's MMAs keep the tensor pipe busy
    static constexpr int THREADS = 192;
    static constexpr uint32_t QTILE = 128 * kHeadDim * 2;  // Q block: 32 KB
    static constexpr uint32_t KVTILE = 64 * kHeadDim * 2;  // K or V block: 16 KB
    // K and V blocks have a ring of two slots each (slots 0-1 hold K, 2-3 hold V). A K slot is
    // freed as soon as its S MMA completes and a V slot when its PV MMA completes; the
    // producer issues K_0 K_1 and then V_j, K_{j+2} for each j, so a K load never queues
    // behind a V load that waits for a later PV.
    static constexpr uint32_t OFF_Q = 0, OFF_KV = QTILE, OFF_BAR = QTILE + 4 * KVTILE;
    // barriers: q | full[4] | empty[4] | sfull[2] | pfull[2] | pvdone[2] | drain. Everything that
    // alternates between the two score buffers has a barrier per buffer (P_j V_j completes
    // pvdone[j % 2]): a softmax warp may run one block ahead of another, and a parity wait is
    // only sound while its barrier is at most one phase from the phase waited for.
    static constexpr int NUM_BARS = 1 + 8 + 2 + 2 + 2 + 1;
    // No alignment slack (two CTAs must fit in one SM's shared memory): the kernel checks
    // that its dynamic shared memory starts on a 1 KB boundary and otherwise does nothing.
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 8 * NUM_BARS + 16;
    static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 64, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 128, false, true);
    // S[0] 0..63 | S[1] 64..127 | O 128..255. P_j (bf16 pairs) overwrites the first 32 columns
    // of S_j's buffer once the softmax has read S_j, and is the A operand of P_j V_j from there.
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr uint32_t O_COL = 128;
    static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs per SM");
};

__global__ void __launch_bounds__(192, 2) attn_fwd_kernel(const __grid_constant__ AttnArgs args)
{
    using C = FwdCfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    if ((base & 1023u) != 0) {  // uniform: every thread leaves before any barrier or TMEM use
        if (threadIdx.x == 0) atomicCAS(args.status, 0, DEV_SMEM_MISALIGNED);
        return;
    }
    uint8_t* gbase = smem_raw;
    const uint32_t sQ = base + C::OFF_Q, sKV = base + C::OFF_KV;
    const uint32_t bar = base + C::OFF_BAR;
    const uint32_t b_q = bar, b_full = bar + 8, b_empty = b_full + 32, b_sf = b_empty + 32, b_pf = b_sf + 16,
                   b_pv = b_pf + 16, b_drain = b_pv + 16;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_BAR + 8 * C::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_BAR + 8 * C::NUM_BARS + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = args.s, a = args.a;
    // Head-major order: the query blocks of one head run side by side and share its K and V
    // blocks through L2; within a head the longest rows start first.
    const int nqb = (s + C::BQ - 1) / C::BQ;
    const int bh = static_cast<int>(blockIdx.x) / nqb, bi = bh / a, head = bh % a;
    const int qb = nqb - 1 - static_cast<int>(blockIdx.x) % nqb;
    const int q0 = qb * C::BQ;
    const int nkb_all = (s + C::BKV - 1) / C::BKV;
    const int nkb = args.causal ? min(nkb_all, (q0 + C::BQ - 1) / C::BKV + 1) : nkb_all;
    const int row0 = bi * s;
    const int hd = a * kHeadDim;
    const int colQ = head * kHeadDim, colK = hd + colQ, colV = 2 * hd + colQ;
    const unsigned long long limit = args.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(b_q, 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(b_full + 8 * i, 1);
            mbar_init(b_empty + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(b_sf + 8 * i, 1);
            mbar_init(b_pf + 8 * i, 4);
            mbar_init(b_pv + 8 * i, 1);
        }
        mbar_init(b_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&args.tmQ);
        tma_prefetch_desc(&args.tmKV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            // drain indices: 0 = q, 1 + i = full[i]
            uint32_t issued = 1u, par = 0u;
            bool ok = true;
            mbar_arrive_expect_tx(b_q, C::QTILE);
            tma_load_2d(sQ, &args.tmQ, colQ, row0 + q0, b_q);
            tma_load_2d(sQ + C::QTILE / 2, &args.tmQ, colQ + 64, row0 + q0, b_q);
            // load order K_0 K_1 V_0 K_2 V_1 K_3 ...: step n < 2 is K_n; then V_j, K_{j+2}
            for (int n = 0; n < 2 * nkb + 2; ++n) {
                const bool isv = n >= 2 && (n & 1) == 0;
                const int j = n < 2 ? n : (isv ? (n - 2) >> 1 : ((n - 3) >> 1) + 2);
                if (j >= nkb) continue;  // K_{j+2} past the last block
                const int slot = (isv ? 2 : 0) + (j & 1);
                const uint32_t ph = static_cast<uint32_t>(j >> 1) & 1u;
                if (j >= 2 && !mbar_wait_bounded(b_empty + 8 * slot, ph ^ 1u, abort_flag, args.status, limit,
                                                 DEV_TIMEOUT_PRODUCER, 1000, n)) {
                    ok = false;
                    break;
                }
                const int y = row0 + j * C::BKV;
                const int x = isv ? colV : colK;
                const uint32_t dst = sKV + slot * C::KVTILE, fb = b_full + 8 * slot;
                mbar_arrive_expect_tx(fb, C::KVTILE);
                tma_load_2d(dst, &args.tmKV, x, y, fb);
                tma_load_2d(dst + C::KVTILE / 2, &args.tmKV, x + 64, y, fb);
                issued |= 1u << (1 + slot);
                par = (par & ~(1u << (1 + slot))) | (ph << (1 + slot));
            }
            if (!ok) drain_loads(bar, 5, issued, par, args.status);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer --------------------------------
        if (lane == 0) {
            bool ok = mbar_wait_bounded(b_q, 0, abort_flag, args.status, limit, DEV_TIMEOUT_MMA_FULL, 1001, -1);
            bool any = false;
            const uint64_t dQ = desc_k(sQ), dKV = desc_k(sKV), dV = desc_mn(sKV, C::KVTILE / 2);
            // S_j = Q K_j^T into TMEM score buffer j % 2. For j >= 2 that buffer held P_{j-2}, the
            // A operand of PV_{j-2}: that product must have completed first.
            auto issue_s = [&](int j) -> bool {
                const int st = j & 1;
                if (!mbar_wait_bounded(b_full + 8 * st, (j >> 1) & 1, abort_flag, args.status, limit,
                                       DEV_TIMEOUT_MMA_FULL, 1002, j) ||
                    (j >= 2 && !mbar_wait_bounded(b_pv + 8 * st, ((j - 2) >> 1) & 1, abort_flag, args.status, limit,
                                                  DEV_TIMEOUT_MMA_ACC, 1003, j)))
                    return false;
                tc_fence_after();
                const uint64_t dK = desc_at(dKV, st * C::KVTILE);
#pragma unroll
                for (int k = 0; k < kHeadDim / 16; ++k) {
                    const uint32_t oq = (C::QTILE / 2) * (k >> 2) + 32u * (k & 3);
                    const uint32_t ok2 = (C::KVTILE / 2) * (k >> 2) + 32u * (k & 3);
                    umma_bf16(tmem + 64u * st, desc_at(dQ, oq), desc_at(dK, ok2), C::IDESC_S, k > 0);
                }
                any = true;
                umma_commit(b_sf + 8 * st);
                umma_commit(b_empty + 8 * st);
                return true;
            };
            // Scores run two blocks ahead: S_0, S_1, then after each P_j: PV_j and S_{j+2}.
            for (int j = 0; ok && j < 2 && j < nkb; ++j) ok = issue_s(j);
            for (int j = 0; ok && j < nkb; ++j) {  // O += P_j V_j
                const int vs = 2 + (j & 1);
                if (!mbar_wait_bounded(b_pf + 8 * (j & 1), (j >> 1) & 1, abort_flag, args.status, limit,
                                       DEV_TIMEOUT_MMA_ACC, 1004, j) ||
                    !mbar_wait_bounded(b_full + 8 * vs, (j >> 1) & 1, abort_flag, args.status, limit,
                                       DEV_TIMEOUT_MMA_FULL, 1005, j)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dVs = desc_at(dV, vs * C::KVTILE);
                // A = P_j in TMEM: 16 keys per MMA are 8 columns of bf16 pairs
#pragma unroll
                for (int k = 0; k < C::BKV / 16; ++k)
                    umma_bf16_tmem_a(tmem + C::O_COL, tmem + 64u * (j & 1) + 8u * k, desc_at(dVs, 2048u * k),
                                     C::IDESC_PV, (j > 0 || k > 0) ? 1u : 0u);
                umma_commit(b_pv + 8 * (j & 1));
                umma_commit(b_empty + 8 * vs);
                if (j + 2 < nkb) ok = issue_s(j + 2);
            }
            if (!ok && any) drain_mma(b_drain, args.status);
        }
    } else {
        // ------------------------------ softmax -----------------------------------
        const int q = warp & 3;  // TMEM lanes [32q, 32q + 32) are the ones this warp may read
        const int r = 32 * q + lane;
        const int qi = q0 + r;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q) << 16);
        const float NEG_INF = -__int_as_float(0x7f800000);
        const float c2 = args.scale_log2;
        float m_used = NEG_INF, l = 0.0f;  // m_used in base-2 units of the scaled scores
        bool ok = true;
        for (int j = 0; j < nkb; ++j) {
            const int st = j & 1;
            if (!warp_wait(b_sf + 8 * st, (j >> 1) & 1, abort_flag, args.status, limit, DEV_TIMEOUT_EPILOGUE, 1006, j)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float x[64];
            {
                uint32_t u0[32], u1[32];
                tmem_ld_32x32b_x32(t_lane + 64u * st, u0);
                tmem_ld_32x32b_x32(t_lane + 64u * st + 32u, u1);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    x[i] = __uint_as_float(u0[i]);
                    x[32 + i] = __uint_as_float(u1[i]);
                }
            }
            const int k0 = j * C::BKV;
            if ((args.causal && k0 + C::BKV - 1 > q0) || k0 + C::BKV > s) {  // CTA-uniform
                // keys after min(s - 1, query) are masked: one compare per column
                const int lim = min(s - 1, args.causal ? qi : 0x7fffffff) - k0;
#pragma unroll
                for (int c = 0; c < 64; ++c) x[c] = c > lim ? NEG_INF : x[c];
            }
            const float mx = max_tree(x) * c2;  // the scale is positive: max commutes with it
            const bool resc = mx > m_used + static_cast<float>(kLazyRescaleLog2);
            float alpha = 1.0f;
            if (resc) {
                alpha = ex2(m_used - mx);  // 0 when m_used is -inf
                m_used = mx;
                l *= alpha;
            }
            const float nref = (m_used == NEG_INF) ? 0.0f : -m_used;
            exp2_affine(x, c2, nref);
            l += sum_tree(x);
            // O may be rescaled once PV_{j-1} has completed (only when some row's max grew)
            if (j >= 1 && __any_sync(0xffffffffu, resc)) {
                if (!warp_wait(b_pv + 8 * (st ^ 1), ((j - 1) >> 1) & 1, abort_flag, args.status, limit,
                               DEV_TIMEOUT_EPILOGUE, 1007, j)) {
                    ok = false;
                    break;
                }
                {
                    tc_fence_after();
                    uint32_t o[32];
#pragma unroll 1
                    for (int c = 0; c < kHeadDim / 32; ++c) {
                        const uint32_t ta = t_lane + C::O_COL + 32u * c;
                        tmem_ld_32x32b_x32(ta, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st_32x32b_x32(ta, o);
                    }
                    tmem_st_wait();
                }
            }
            {  // P_j as bf16 pairs over the first 32 columns of S_j's buffer (read above)
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = pack2_bf16(x[2 * i], x[2 * i + 1]);
                tmem_st_32x32b_x32(t_lane + 64u * st, pk);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_pf + 8 * st);
        }
        // O is final once PV_{nkb-2} and PV_{nkb-1} have completed (a warp's last S implies only
        // PV_{nkb-3}); each waits on its own buffer's barrier, whose next phase never comes.
        const int l1 = nkb - 1, l2 = nkb - 2;
        if (ok && l2 >= 0 &&
            !warp_wait(b_pv + 8 * (l2 & 1), (l2 >> 1) & 1, abort_flag, args.status, limit, DEV_TIMEOUT_EPILOGUE, 1008,
                       nkb))
            ok = false;
        if (ok && l1 >= 0 &&
            warp_wait(b_pv + 8 * (l1 & 1), (l1 >> 1) & 1, abort_flag, args.status, limit, DEV_TIMEOUT_EPILOGUE, 1009,
                      nkb)) {
            tc_fence_after();
            const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
            __nv_bfloat16* dst = args.out + static_cast<size_t>(row0 + qi) * hd + colQ;
            uint32_t o[32];
#pragma unroll 1
            for (int c = 0; c < kHeadDim / 32; ++c) {
                tmem_ld_32x32b_x32(t_lane + C::O_COL + 32u * c, o);
                tmem_ld_wait();
                if (qi < s) store32_global(dst + 32 * c, o, inv_l);
            }
            if (qi < s) args.lse[static_cast<size_t>(bh) * s + qi] = m_used + log2f(l);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---- backward: dK and dV ---------------------------------------------------------------------

struct DkdvCfg {
    static constexpr int BKV = 128, BQ = 64;
    // producer, MMA, 16 element-wise warps (four threads per key, 16 queries each)
    static constexpr int THREADS = 576;
    static constexpr int EW_WARPS = 16;
    static constexpr int STAGES = 4;                    // Q / dC blocks in flight
    static constexpr uint32_t KT = 128 * kHeadDim * 2;  // K or V block: 32 KB
    static constexpr uint32_t QT = 64 * kHeadDim * 2;   // Q or dC block: 16 KB
    // per element-wise warp: its 16 queries' L and D (fp32), 128 bytes
    static constexpr uint32_t OFF_K = 0, OFF_V = KT, OFF_QD = 2 * KT, OFF_LD = 2 * KT + STAGES * 2 * QT,
                              OFF_BAR = OFF_LD + EW_WARPS * 2 * 16 * 4;
    // barriers: kv | qdofull[4] | qdoempty[4] | stfull[2] | pdfull[2] | dvdkdone[2] | accfull | drain
    static constexpr int NUM_BARS = 1 + 2 * STAGES + 6 + 2;
    static constexpr uint32_t SMEM_BYTES = 1024 + OFF_BAR + 8 * NUM_BARS + 16;
    static constexpr uint32_t IDESC_ST = idesc_bf16_f32(128, 64, false, false);
    static constexpr uint32_t IDESC_ACC = idesc_bf16_f32(128, 128, false, true);
    // S^T[x] at 128x, dP^T[x] at 128x + 64; dV 256; dK 384. P^T and dS^T (bf16 pairs) are
    // written back over the S^T and dP^T columns each thread has read (queries [16g, 16g+16) as
    // 8 columns at +16g) and are the A operands of dV += P^T dC and dK += dS^T Q from there.
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t DV_COL = 256, DK_COL = 384;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(DkdvCfg::THREADS, 1) attn_bwd_dkdv_kernel(const __grid_constant__ AttnArgs args)
{
    using C = DkdvCfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sQD = base + C::OFF_QD, sLD = base + C::OFF_LD;
    const uint32_t bar = base + C::OFF_BAR;
    const uint32_t b_kv = bar, b_qf = bar + 8, b_qe = b_qf + 8 * C::STAGES, b_stf = b_qe + 8 * C::STAGES,
                   b_pdf = b_stf + 16, b_dvd = b_pdf + 16, b_acc = b_dvd + 16, b_drain = b_acc + 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_BAR + 8 * C::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_BAR + 8 * C::NUM_BARS + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = args.s, a = args.a;
    // Head-major order (the key blocks of one head share its Q and dC blocks through L2);
    // with a causal mask, low key blocks have the most queries and start first.
    const int nkbk = (s + C::BKV - 1) / C::BKV;
    const int bh = static_cast<int>(blockIdx.x) / nkbk, bi = bh / a, head = bh % a;
    const int kb = static_cast<int>(blockIdx.x) % nkbk;
    const int k0 = kb * C::BKV;
    const int nqb_all = (s + C::BQ - 1) / C::BQ;
    const int qb_first = args.causal ? k0 / C::BQ : 0;
    const int nq = nqb_all - qb_first;
    const int row0 = bi * s;
    const int hd = a * kHeadDim;
    const int colQ = head * kHeadDim, colK = hd + colQ, colV = 2 * hd + colQ;
    const unsigned long long limit = args.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(b_kv, 1);
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(b_qf + 8 * i, 1);
            mbar_init(b_qe + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(b_stf + 8 * i, 1);
            mbar_init(b_pdf + 8 * i, C::EW_WARPS);
            mbar_init(b_dvd + 8 * i, 1);
        }
        mbar_init(b_acc, 1);
        mbar_init(b_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&args.tmQ);
        tma_prefetch_desc(&args.tmKV);
        tma_prefetch_desc(&args.tmdO);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // drain indices: 0 = kv, 1 + i = qdofull[i]
            uint32_t issued = 1u, par = 0u;
            bool ok = true;
            mbar_arrive_expect_tx(b_kv, 2 * C::KT);
            tma_load_2d(sK, &args.tmKV, colK, row0 + k0, b_kv);
            tma_load_2d(sK + C::KT / 2, &args.tmKV, colK + 64, row0 + k0, b_kv);
            tma_load_2d(sV, &args.tmKV, colV, row0 + k0, b_kv);
            tma_load_2d(sV + C::KT / 2, &args.tmKV, colV + 64, row0 + k0, b_kv);
            for (int i = 0; i < nq; ++i) {
                const int st = i % C::STAGES;
                const uint32_t ph = static_cast<uint32_t>(i / C::STAGES) & 1u;
                if (i >= C::STAGES && !mbar_wait_bounded(b_qe + 8 * st, ph ^ 1u, abort_flag, args.status, limit,
                                                         DEV_TIMEOUT_PRODUCER, 3000, i)) {
                    ok = false;
                    break;
                }
                const int y = row0 + (qb_first + i) * C::BQ;
                const uint32_t dq = sQD + st * 2 * C::QT, dd = dq + C::QT, fb = b_qf + 8 * st;
                mbar_arrive_expect_tx(fb, 2 * C::QT);
                tma_load_2d(dq, &args.tmQ, colQ, y, fb);
                tma_load_2d(dq + C::QT / 2, &args.tmQ, colQ + 64, y, fb);
                tma_load_2d(dd, &args.tmdO, colQ, y, fb);
                tma_load_2d(dd + C::QT / 2, &args.tmdO, colQ + 64, y, fb);
                issued |= 1u << (1 + st);
                par = (par & ~(1u << (1 + st))) | (ph << (1 + st));
            }
            if (!ok) drain_loads(bar, 1 + C::STAGES, issued, par, args.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = mbar_wait_bounded(b_kv, 0, abort_flag, args.status, limit, DEV_TIMEOUT_MMA_FULL, 3001, -1);
            bool any = false;
            const uint64_t dK = desc_k(sK), dV = desc_k(sV), dQD = desc_k(sQD), dQDmn = desc_mn(sQD, C::QT / 2);
            for (int i = 0; ok && i <= nq; ++i) {
                if (i < nq) {  // S^T_i = K Q_i^T, dP^T_i = V dC_i^T
                    const int st = i & 1, qs = i % C::STAGES;
                    if (!mbar_wait_bounded(b_qf + 8 * qs, (i / C::STAGES) & 1, abort_flag, args.status, limit,
                                           DEV_TIMEOUT_MMA_FULL, 3002, i) ||
                        // the buffer held P^T_{i-2} and dS^T_{i-2}, the A operands of dV / dK of block i-2
                        (i >= 2 && !mbar_wait_bounded(b_dvd + 8 * st, ((i - 2) >> 1) & 1, abort_flag, args.status,
                                                      limit, DEV_TIMEOUT_MMA_ACC, 3003, i))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t qoff = qs * 2 * C::QT, dooff = qoff + C::QT;
#pragma unroll
                    for (int k = 0; k < kHeadDim / 16; ++k) {
                        const uint32_t ka = (C::KT / 2) * (k >> 2) + 32u * (k & 3);
                        const uint32_t kq = (C::QT / 2) * (k >> 2) + 32u * (k & 3);
                        umma_bf16(tmem + 128u * st, desc_at(dK, ka), desc_at(dQD, qoff + kq), C::IDESC_ST, k > 0);
                        umma_bf16(tmem + 128u * st + 64u, desc_at(dV, ka), desc_at(dQD, dooff + kq), C::IDESC_ST,
                                  k > 0);
                    }
                    any = true;
                    umma_commit(b_stf + 8 * st);
                }
                if (i >= 1) {  // dV += P^T_{i-1} dC_{i-1}, dK += dS^T_{i-1} Q_{i-1}
                    const int pi = i - 1, qs = pi % C::STAGES, pst = pi & 1;
                    if (!mbar_wait_bounded(b_pdf + 8 * pst, (pi >> 1) & 1, abort_flag, args.status, limit,
                                           DEV_TIMEOUT_MMA_ACC, 3004, pi)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t qoff = qs * 2 * C::QT, dooff = qoff + C::QT;
                    // A = P^T and dS^T in TMEM: queries [16k, 16k+16) are 8 columns at +16k
#pragma unroll
                    for (int k = 0; k < C::BQ / 16; ++k) {
                        const uint32_t acc = (pi > 0 || k > 0) ? 1u : 0u;
                        const uint32_t pa = tmem + 128u * pst + 16u * k;
                        umma_bf16_tmem_a(tmem + C::DV_COL, pa, desc_at(dQDmn, dooff + 2048u * k), C::IDESC_ACC, acc);
                        umma_bf16_tmem_a(tmem + C::DK_COL, pa + 64u, desc_at(dQDmn, qoff + 2048u * k), C::IDESC_ACC,
                                         acc);
                    }
                    umma_commit(b_qe + 8 * qs);
                    umma_commit(b_dvd + 8 * pst);
                }
            }
            if (ok && any) umma_commit(b_acc);
            if (!ok && any) drain_mma(b_drain, args.status);
        }
    } else {
        // Four threads per key row: warp w (2..17) takes TMEM lane quadrant w % 4 and query
        // columns [16g, 16g + 16) of each 64-query block, g = (w - 2) / 4.
        const int q = warp & 3, grp = (warp - 2) >> 2;
        const int r = 32 * q + lane;
        const int kj = k0 + r;
        const int cb = 16 * grp;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q) << 16);
        const uint32_t sL = sLD + static_cast<uint32_t>(warp - 2) * 128u, sD = sL + 64u;
        const size_t lbase = static_cast<size_t>(bh) * s;
        bool ok = true;
        for (int i = 0; i < nq; ++i) {
            const int st = i & 1;
            const int qq0 = (qb_first + i) * C::BQ + cb;  // this thread's first query column
            // this warp's 16 values of L and D into its own staging slots
            {
                const int qa = qq0 + lane;
                const bool in = lane < 16 && qa < s;
                const float la = in ? args.lse[lbase + qa] : 0.0f;
                const float da = in ? args.delta[lbase + qa] : 0.0f;
                __syncwarp();
                if (lane < 16) {
                    sts_f32(sL + 4u * lane, la);
                    sts_f32(sD + 4u * lane, da);
                }
                __syncwarp();
            }
            if (!warp_wait(b_stf + 8 * st, (i >> 1) & 1, abort_flag, args.status, limit, DEV_TIMEOUT_EPILOGUE, 3005, i)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float p[16], dp[16];
            {
                uint32_t u0[16], u1[16];
                tmem_ld_32x32b_x16(t_lane + 128u * st + cb, u0);
                tmem_ld_32x32b_x16(t_lane + 128u * st + 64u + cb, u1);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    p[e] = __uint_as_float(u0[e]);
                    dp[e] = __uint_as_float(u1[e]);
                }
            }
            const int blk0 = (qb_first + i) * C::BQ;
            const bool need_mask = (args.causal && blk0 < k0 + C::BKV - 1) || blk0 + C::BQ > s || k0 + C::BKV > s;
            float Dv[16];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const float4 L4 = lds128f(sL + 16u * c4), D4 = lds128f(sD + 16u * c4);
                const float Lv[4] = {L4.x, L4.y, L4.z, L4.w};
                Dv[4 * c4] = D4.x;
                Dv[4 * c4 + 1] = D4.y;
                Dv[4 * c4 + 2] = D4.z;
                Dv[4 * c4 + 3] = D4.w;
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    float lo, hi;
                    f2_split(f2_fma_(f2(p[4 * c4 + e], p[4 * c4 + e + 1]), f2(args.scale_log2, args.scale_log2),
                                     f2(-Lv[e], -Lv[e + 1])),
                             lo, hi);
                    p[4 * c4 + e] = ex2(lo);
                    p[4 * c4 + e + 1] = ex2(hi);
                }
            }
            // Masked pairs (query past the sequence, key past it, or key after query) are zeroed
            // by one compare per column against this thread's valid range of c: a test on
            // need_mask per column would cost a branch each.
            if (need_mask) {
                const int c_lo = args.causal ? kj - qq0 : -(1 << 30);  // query >= key
                const int c_hi = kj < s ? s - qq0 : -(1 << 30);        // query < s, key < s
#pragma unroll
                for (int c = 0; c < 16; ++c) p[c] = (c >= c_lo && c < c_hi) ? p[c] : 0.0f;
            }
#pragma unroll
            for (int c = 0; c < 16; c += 2)  // dS^T = P^T (dP^T - D), on pairs
                f2_split(f2_mul_(f2(p[c], p[c + 1]), f2_add_(f2(dp[c], dp[c + 1]), f2(-Dv[c], -Dv[c + 1]))), dp[c],
                         dp[c + 1]);
            {  // P^T and dS^T over the first 8 of the 16 S^T / dP^T columns this thread has read
                uint32_t pk[8], dk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    pk[e] = pack2_bf16(p[2 * e], p[2 * e + 1]);
                    dk[e] = pack2_bf16(dp[2 * e], dp[2 * e + 1]);
                }
                tmem_st_32x32b_x8(t_lane + 128u * st + cb, pk);
                tmem_st_32x32b_x8(t_lane + 128u * st + 64u + cb, dk);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_pdf + 8 * st);
        }
        if (ok && nq > 0 && warp_wait(b_acc, 0, abort_flag, args.status, limit, DEV_TIMEOUT_EPILOGUE, 3007, -1)) {
            tc_fence_after();
            __nv_bfloat16* rowp = args.out + static_cast<size_t>(row0 + kj) * (3 * hd);
            const int db = 32 * grp;  // this thread's quarter of the d columns of dV and dK
            uint32_t o[32];
            tmem_ld_32x32b_x32(t_lane + C::DV_COL + db, o);
            tmem_ld_wait();
            if (kj < s) store32_global(rowp + colV + db, o, 1.0f);
            tmem_ld_32x32b_x32(t_lane + C::DK_COL + db, o);
            tmem_ld_wait();
            if (kj < s) store32_global(rowp + colK + db, o, args.scale);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---- backward: dQ ----------------------------------------------------------------------------

struct DqCfg {
    static constexpr int BQ = 128, BKV = 128;  // N = 128 score products
    // producer, MMA, 16 element-wise warps (four threads per query, 32 keys each)
    static constexpr int THREADS = 576;
    static constexpr int EW_WARPS = 16;
    // K blocks are read by S_j and dQ_j, V blocks by dP_j only: three K slots, freed when
    // dQ_j completes, and two V slots, freed when dP_j completes, keep the next loads ahead of
    // the products that wait for them.
    static constexpr int KSLOTS = 3, VSLOTS = 2;
    static constexpr uint32_t QT = 128 * kHeadDim * 2;  // Q or dC block: 32 KB
    static constexpr uint32_t KT = 128 * kHeadDim * 2;  // K or V block: 32 KB
    static constexpr uint32_t OFF_Q = 0, OFF_DO = QT, OFF_K = 2 * QT, OFF_V = OFF_K + KSLOTS * KT,
                              OFF_BAR = OFF_V + VSLOTS * KT;
    // barriers: qdo | kfull[3] | vfull[2] | kempty[3] | vempty[2] | spfull | spread | dsfull[2] |
    // dqdone[2] | dqfull | drain (the loads' barriers first, for the abort drain)
    static constexpr int NUM_LOAD_BARS = 1 + KSLOTS + VSLOTS;
    static constexpr int NUM_BARS = NUM_LOAD_BARS + KSLOTS + VSLOTS + 8;
    static constexpr uint32_t SMEM_BYTES = 1024 + OFF_BAR + 8 * NUM_BARS + 16;
    static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, false, false);
    static constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, 128, false, true);
    // S at 0, dP at 128, dQ at 256; dS_j (bf16 pairs, keys [16k, 16k+16) as 8 columns at
    // DS_COL + 64 (j % 2) + 8k) double-buffered at 384, the A operand of dQ += dS_j K_j. The
    // next block's S and dP overwrite this one's as soon as every element-wise warp has loaded
    // them, so those products run while dS is computed.
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t DP_COL = 128, DQ_COL = 256, DS_COL = 384;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(DqCfg::THREADS, 1) attn_bwd_dq_kernel(const __grid_constant__ AttnArgs args)
{
    using C = DqCfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + C::OFF_Q, sdO = base + C::OFF_DO, sK = base + C::OFF_K, sV = base + C::OFF_V;
    const uint32_t bar = base + C::OFF_BAR;
    const uint32_t b_qdo = bar, b_kf = bar + 8, b_vf = b_kf + 8 * C::KSLOTS, b_ke = b_vf + 8 * C::VSLOTS,
                   b_ve = b_ke + 8 * C::KSLOTS, b_spf = b_ve + 8 * C::VSLOTS, b_spr = b_spf + 8, b_dsf = b_spr + 8,
                   b_dqd = b_dsf + 16, b_dq = b_dqd + 16, b_drain = b_dq + 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + C::OFF_BAR + 8 * C::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_BAR + 8 * C::NUM_BARS + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = args.s, a = args.a;
    // Head-major order, longest rows first within a head (as in the forward kernel).
    const int nqb = (s + C::BQ - 1) / C::BQ;
    const int bh = static_cast<int>(blockIdx.x) / nqb, bi = bh / a, head = bh % a;
    const int qb = nqb - 1 - static_cast<int>(blockIdx.x) % nqb;
    const int q0 = qb * C::BQ;
    const int nkb_all = (s + C::BKV - 1) / C::BKV;
    const int nkb = args.causal ? min(nkb_all, (q0 + C::BQ - 1) / C::BKV + 1) : nkb_all;
    const int row0 = bi * s;
    const int hd = a * kHeadDim;
    const int colQ = head * kHeadDim, colK = hd + colQ, colV = 2 * hd + colQ;
    const unsigned long long limit = args.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(b_qdo, 1);
        for (int i = 0; i < C::KSLOTS; ++i) {
            mbar_init(b_kf + 8 * i, 1);
            mbar_init(b_ke + 8 * i, 1);
        }
        for (int i = 0; i < C::VSLOTS; ++i) {
            mbar_init(b_vf + 8 * i, 1);
            mbar_init(b_ve + 8 * i, 1);
        }
        mbar_init(b_spf, 1);
        mbar_init(b_spr, C::EW_WARPS);
        for (int i = 0; i < 2; ++i) {
            mbar_init(b_dsf + 8 * i, C::EW_WARPS);
            mbar_init(b_dqd + 8 * i, 1);
        }
        mbar_init(b_dq, 1);
        mbar_init(b_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&args.tmQ);
        tma_prefetch_desc(&args.tmKV);
        tma_prefetch_desc(&args.tmdO);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // drain indices: 0 = qdo, 1 + i = kfull[i], 1 + KSLOTS + i = vfull[i]
            uint32_t issued = 1u, par = 0u;
            bool ok = true;
            mbar_arrive_expect_tx(b_qdo, 2 * C::QT);
            tma_load_2d(sQ, &args.tmQ, colQ, row0 + q0, b_qdo);
            tma_load_2d(sQ + C::QT / 2, &args.tmQ, colQ + 64, row0 + q0, b_qdo);
            tma_load_2d(sdO, &args.tmdO, colQ, row0 + q0, b_qdo);
            tma_load_2d(sdO + C::QT / 2, &args.tmdO, colQ + 64, row0 + q0, b_qdo);
            for (int j = 0; j < nkb; ++j) {
                const int y = row0 + j * C::BKV;
                // V_j into slot j % 2, free once dP_{j-2} has completed
                const int vs = j % C::VSLOTS;
                const uint32_t vph = static_cast<uint32_t>(j / C::VSLOTS) & 1u;
                if (j >= C::VSLOTS && !mbar_wait_bounded(b_ve + 8 * vs, vph ^ 1u, abort_flag, args.status, limit,
                                                         DEV_TIMEOUT_PRODUCER, 2000, j)) {
                    ok = false;
                    break;
                }
                const uint32_t dv = sV + vs * C::KT, vb = b_vf + 8 * vs;
                mbar_arrive_expect_tx(vb, C::KT);
                tma_load_2d(dv, &args.tmKV, colV, y, vb);
                tma_load_2d(dv + C::KT / 2, &args.tmKV, colV + 64, y, vb);
                issued |= 1u << (1 + C::KSLOTS + vs);
                par = (par & ~(1u << (1 + C::KSLOTS + vs))) | (vph << (1 + C::KSLOTS + vs));
                // K_j into slot j % 3, free once dQ_{j-3} has completed
                const int ks = j % C::KSLOTS;
                const uint32_t kph = static_cast<uint32_t>(j / C::KSLOTS) & 1u;
                if (j >= C::KSLOTS && !mbar_wait_bounded(b_ke + 8 * ks, kph ^ 1u, abort_flag, args.status, limit,
                                                         DEV_TIMEOUT_PRODUCER, 2008, j)) {
                    ok = false;
                    break;
                }
                const uint32_t dk = sK + ks * C::KT, kb = b_kf + 8 * ks;
                mbar_arrive_expect_tx(kb, C::KT);
                tma_load_2d(dk, &args.tmKV, colK, y, kb);
                tma_load_2d(dk + C::KT / 2, &args.tmKV, colK + 64, y, kb);
                issued |= 1u << (1 + ks);
                par = (par & ~(1u << (1 + ks))) | (kph << (1 + ks));
            }
            if (!ok) drain_loads(bar, C::NUM_LOAD_BARS, issued, par, args.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = mbar_wait_bounded(b_qdo, 0, abort_flag, args.status, limit, DEV_TIMEOUT_MMA_FULL, 2001, -1);
            bool any = false;
            const uint64_t dQ = desc_k(sQ), dO = desc_k(sdO), dK = desc_k(sK), dV = desc_k(sV),
                           dKmn = desc_mn(sK, C::KT / 2);
            for (int j = 0; ok && j <= nkb; ++j) {
                if (j < nkb) {  // S_j = Q K_j^T, dP_j = dC V_j^T
                    const int ks = j % C::KSLOTS, vs = j % C::VSLOTS;
                    if (!mbar_wait_bounded(b_kf + 8 * ks, (j / C::KSLOTS) & 1, abort_flag, args.status, limit,
                                           DEV_TIMEOUT_MMA_FULL, 2002, j) ||
                        // every element-wise warp has loaded S_{j-1} and dP_{j-1}
                        (j >= 1 && !mbar_wait_bounded(b_spr, (j - 1) & 1, abort_flag, args.status, limit,
                                                      DEV_TIMEOUT_MMA_ACC, 2003, j)) ||
                        !mbar_wait_bounded(b_vf + 8 * vs, (j / C::VSLOTS) & 1, abort_flag, args.status, limit,
                                           DEV_TIMEOUT_MMA_FULL, 2006, j)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t koff = ks * C::KT, voff = vs * C::KT;
#pragma unroll
                    for (int k = 0; k < kHeadDim / 16; ++k) {
                        const uint32_t aq = (C::QT / 2) * (k >> 2) + 32u * (k & 3);
                        const uint32_t bk = (C::KT / 2) * (k >> 2) + 32u * (k & 3);
                        umma_bf16(tmem, desc_at(dQ, aq), desc_at(dK, koff + bk), C::IDESC_S, k > 0);
                    }
#pragma unroll
                    for (int k = 0; k < kHeadDim / 16; ++k) {
                        const uint32_t aq = (C::QT / 2) * (k >> 2) + 32u * (k & 3);
                        const uint32_t bk = (C::KT / 2) * (k >> 2) + 32u * (k & 3);
                        umma_bf16(tmem + C::DP_COL, desc_at(dO, aq), desc_at(dV, voff + bk), C::IDESC_S, k > 0);
                    }
                    any = true;
                    umma_commit(b_spf);
                    umma_commit(b_ve + 8 * vs);
                }
                if (j >= 1) {  // dQ += dS_{j-1} K_{j-1}
                    const int pj = j - 1, pst = pj & 1, ks = pj % C::KSLOTS;
                    if (!mbar_wait_bounded(b_dsf + 8 * pst, (pj >> 1) & 1, abort_flag, args.status, limit,
                                           DEV_TIMEOUT_MMA_ACC, 2004, pj)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t koff = ks * C::KT;
#pragma unroll
                    for (int k = 0; k < C::BKV / 16; ++k)
                        umma_bf16_tmem_a(tmem + C::DQ_COL, tmem + C::DS_COL + 64u * pst + 8u * k,
                                         desc_at(dKmn, koff + 2048u * k), C::IDESC_DQ, (pj > 0 || k > 0) ? 1u : 0u);
                    umma_commit(b_ke + 8 * ks);
                    umma_commit(b_dqd + 8 * pst);
                }
            }
            if (ok && any) umma_commit(b_dq);
            if (!ok && any) drain_mma(b_drain, args.status);
        }
    } else {
        // Four threads per query row: warp w (2..17) takes TMEM lane quadrant w % 4 and key
        // columns [32g, 32g + 32) of each 128-key block, g = (w - 2) / 4.
        const int q = warp & 3, grp = (warp - 2) >> 2;
        const int r = 32 * q + lane;
        const int qi = q0 + r;
        const int cb = 32 * grp;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q) << 16);
        const size_t li = static_cast<size_t>(bh) * s + qi;
        const float nLq = qi < s ? -args.lse[li] : 0.0f;
        const float Dq = qi < s ? args.delta[li] : 0.0f;
        bool ok = true;
        for (int j = 0; j < nkb; ++j) {
            const int pst = j & 1;
            if (!warp_wait(b_spf, j & 1, abort_flag, args.status, limit, DEV_TIMEOUT_EPILOGUE, 2005, j)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float p[32], dp[32];
            {
                uint32_t u0[32], u1[32];
                tmem_ld_32x32b_x32(t_lane + cb, u0);
                tmem_ld_32x32b_x32(t_lane + C::DP_COL + cb, u1);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    p[e] = __uint_as_float(u0[e]);
                    dp[e] = __uint_as_float(u1[e]);
                }
            }
            // S and dP of this block are in registers: the next block's products may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_spr);
            const int kk0 = j * C::BKV;
            const bool need_mask = (args.causal && kk0 + C::BKV - 1 > q0) || kk0 + C::BKV > s || q0 + C::BQ > s;
            exp2_affine(p, args.scale_log2, nLq);
            if (need_mask) {  // columns past lim are masked (key past the sequence or after the query)
                const int lim = (qi >= s ? -1 : min(s - 1, args.causal ? qi : 0x7fffffff)) - (kk0 + cb);
#pragma unroll
                for (int c = 0; c < 32; ++c) p[c] = c > lim ? 0.0f : p[c];
            }
            {  // dS = P (dP - D), on pairs
                const f2_t nd = f2(-Dq, -Dq);
#pragma unroll
                for (int c = 0; c < 32; c += 2)
                    f2_split(f2_mul_(f2(p[c], p[c + 1]), f2_add_(f2(dp[c], dp[c + 1]), nd)), dp[c], dp[c + 1]);
            }
            // dS_j goes where dS_{j-2} was: dQ_{j-2} must have read it
            if (j >= 2 && !warp_wait(b_dqd + 8 * pst, ((j - 2) >> 1) & 1, abort_flag, args.status, limit,
                                     DEV_TIMEOUT_EPILOGUE, 2006, j)) {
                ok = false;
                break;
            }
            tc_fence_after();
            {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pk[i] = pack2_bf16(dp[2 * i], dp[2 * i + 1]);
                tmem_st_32x32b_x16(t_lane + C::DS_COL + 64u * pst + 16u * grp, pk);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_dsf + 8 * pst);
        }
        if (ok && nkb > 0 && warp_wait(b_dq, 0, abort_flag, args.status, limit, DEV_TIMEOUT_EPILOGUE, 2007, -1)) {
            tc_fence_after();
            const int db = 32 * grp;  // this thread's quarter of the d columns
            uint32_t o[32];
            tmem_ld_32x32b_x32(t_lane + C::DQ_COL + db, o);
            tmem_ld_wait();
            if (qi < s) store32_global(args.out + static_cast<size_t>(row0 + qi) * (3 * hd) + colQ + db, o, args.scale);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---- D = rowsum(dC * C) per (token, head) ----------------------------------------------------

__global__ void __launch_bounds__(256) attn_bwd_dot_kernel(const __nv_bfloat16* __restrict__ dC,
                                                          const __nv_bfloat16* __restrict__ Cc, int T, int s, int a,
                                                          float* __restrict__ D)
{
    // Rows are (token, head) pairs of 128 contiguous elements, consecutive in memory. A warp
    // takes 4 consecutive rows per step (1 KB of each tensor, fully coalesced): 8 lanes per
    // row, 16 elements (two 16-byte loads of each tensor) per lane, then a 3-step shuffle sum.
    // Two steps in flight per warp keep enough bytes outstanding to run at HBM speed.
    const int lane = threadIdx.x & 31, sub = lane & 7;
    const long long rows = static_cast<long long>(T) * a;
    const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    for (long long g = 4 * w0; g < rows; g += 8 * nwarps) {
        float acc[2] = {0.0f, 0.0f};
        uint4 u[2][2], v[2][2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const long long w = g + 4 * nwarps * k + (lane >> 3);
            if (w < rows) {
                const size_t off = static_cast<size_t>(w) * kHeadDim + 16 * sub;
                u[k][0] = __ldg(reinterpret_cast<const uint4*>(dC + off));
                u[k][1] = __ldg(reinterpret_cast<const uint4*>(dC + off + 8));
                v[k][0] = __ldg(reinterpret_cast<const uint4*>(Cc + off));
                v[k][1] = __ldg(reinterpret_cast<const uint4*>(Cc + off + 8));
            } else {
                u[k][0] = u[k][1] = v[k][0] = v[k][1] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t uu[4] = {u[k][h].x, u[k][h].y, u[k][h].z, u[k][h].w};
                const uint32_t vv[4] = {v[k][h].x, v[k][h].y, v[k][h].z, v[k][h].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[k] = fmaf(__uint_as_float(uu[i] << 16), __uint_as_float(vv[i] << 16), acc[k]);
                    acc[k] = fmaf(__uint_as_float(uu[i] & 0xFFFF0000u), __uint_as_float(vv[i] & 0xFFFF0000u), acc[k]);
                }
            }
#pragma unroll
            for (int o = 4; o >= 1; o >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
            const long long w = g + 4 * nwarps * k + (lane >> 3);
            if (sub == 0 && w < rows) {
                const long long t = w / a, bi = t / s, p = t % s;
                const int head = static_cast<int>(w % a);
                D[(bi * a + head) * s + p] = acc[k];
            }
        }
    }
}

template <typename Cfg, typename K>
cudaError_t launch_tile_kernel(K kern, const AttnArgs& args, int blocks_y, cudaStream_t stream)
{
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    // all of the SM's unified L1 / shared memory as shared memory (the forward kernel needs it
    // for two CTAs per SM)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    const long long grid = static_cast<long long>(args.b) * args.a * blocks_y;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(grid), Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnArgs& args, cudaStream_t stream)
{
    return launch_tile_kernel<FwdCfg>(attn_fwd_kernel, args, (args.s + FwdCfg::BQ - 1) / FwdCfg::BQ, stream);
}

cudaError_t launch_attn_bwd_dq(const AttnArgs& args, cudaStream_t stream)
{
    return launch_tile_kernel<DqCfg>(attn_bwd_dq_kernel, args, (args.s + DqCfg::BQ - 1) / DqCfg::BQ, stream);
}

cudaError_t launch_attn_bwd_dkdv(const AttnArgs& args, cudaStream_t stream)
{
    return launch_tile_kernel<DkdvCfg>(attn_bwd_dkdv_kernel, args, (args.s + DkdvCfg::BKV - 1) / DkdvCfg::BKV, stream);
}

cudaError_t launch_attn_bwd_dot(const __nv_bfloat16* dC, const __nv_bfloat16* Cc, int T, int s, int a, float* D,
                                int num_sms, cudaStream_t stream)
{
    const long long rows = static_cast<long long>(T) * a;
    if (rows <= 0) return cudaSuccess;
    long long blocks = (rows + 63) / 64;  // 8 warps of 8 rows (two steps of 4) per block pass
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    attn_bwd_dot_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(dC, Cc, T, s, a, D);
    return cudaGetLastError();
}

}  // namespace mlp
