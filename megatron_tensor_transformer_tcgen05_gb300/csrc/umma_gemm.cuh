// umma_gemm.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a with fused
// epilogues for the tensor-parallel MLP block.
//
//   D[M,N] = sum_k  Aop[m,k] * Bop[n,k]      (bf16 operands, fp32 accumulation in TMEM)
//
// Aop and Bop are read from row-major global tensors through TMA tensor maps, either
// K-contiguous ("K-major") or M/N-contiguous ("MN-major", i.e. the transposed use of a
// row-major tensor); the tcgen05 instruction descriptor carries the major-ness, so no
// operand is ever transposed in memory.
//
// Roles in one CTA (one CTA per SM, persistent over work tiles; 192 threads, or 320 with
// eight epilogue warps):
//   warp 0     TMA producer: fills a ring of {A 128 x 64, B (its share) x 64} stages (128B
//              swizzle)
//   warp 1     allocates TMEM and issues tcgen05.mma (in a CTA pair, the even CTA's alone)
//   warps 2-5 (2-9)  epilogue: tcgen05.ld of the accumulator, fused element-wise math, bf16
//              RNE, swizzled staging in shared memory, TMA store of 32x32 boxes
// Tile shapes (GemmCfg): one CTA, 128 x BN (BN = 128, 256), two accumulators; a CTA pair
// (cta_group::2), 256 x 256, two accumulators; a CTA pair, 256 x 512, one accumulator of all
// 512 TMEM columns, released in two halves. With two accumulators the epilogue of tile i
// overlaps the main loop of tile i+1; with one, the next tile's first MMAs wait for half 0 to
// be read out, and its first half-1 MMA for half 1. A 512-wide pair tile may also run as one
// of the two pairs of a cluster of four (args.cluster_pairs = 2): the pairs compute the two
// 256-row halves of a 512 x 512 work tile, and CTA (p, r) fetches only B half p of each
// stage and multicasts it to CTA r of both pairs.
//
// Split tail (EPI_PLAIN, EPI_BIAS, EPI_BIAS_GELU, EPI_DGELU): when the tile count leaves the
// last round of tiles short (tiles % units of them), those last tiles may each be cut into
// split_k ranges of K, so the short round becomes up to one part per unit. A part writes its
// fp32 partial accumulator to split_ws; splitk_fixup_kernel then adds the parts of each tile
// in order and applies the epilogue, so the result is the same on every run.
//
// Epilogues (the step of the MLP block each one implements):
//   EPI_BIAS_GELU  H = acc + a[n]; G = GELU(H) of H rounded to bf16 (so a backward that
//                  recomputes G from the stored H gets the same bits)  -> stores H and G
//   EPI_BIAS       Y = acc + b[n]                          -> stores Y
//   EPI_BIAS_DROPOUT_RES  Z = R[m,n] + keep(m,n) (acc + b[n]) / (1 - p)   -> stores Z
//                  (keep from Philox4x32-10 on the element's index; philox.cuh)
//   EPI_DGELU      dH = acc * GELU'(H[m,n])                -> stores dH (and, optionally,
//                  its column sums over each 32-row block in fp32, for the bias gradient)
//                  (the backward that recomputes G instead of keeping it from the forward)
//   EPI_PLAIN      D = acc                                 -> stores D
//   EPI_SWIGLU     acc = [X A | X Wg] over 128 columns: Ha, Hg, U = SiLU(Ha) Hg -> stores all three
//   EPI_DSWIGLU    dU = acc: dHa = dU Hg SiLU'(Ha), dHg = dU SiLU(Ha)            -> stores both
//   EPI_PLAIN_GA, EPI_BIAS_GA   as EPI_PLAIN, EPI_BIAS, with the A operand read as H and
//                  turned into G = GELU(H) in shared memory by eight operand-transform
//                  warps before the MMAs read it (the GELU recompute: G never goes to HBM)
// GELU is the tanh form 0.5 x (1 + tanh u), u = sqrt(2/pi) (x + 0.044715 x^3), evaluated
// through the identity 1 + tanh u = 2 / (1 + exp(-2u)), which stays accurate where
// 1 + tanh u is small.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "gemm_args.h"
#include "philox.cuh"
#include "sm103_ptx.cuh"

namespace mlp {

template <int BN_, bool A_MN_, bool B_MN_, int EPI_, int CG_>
struct GemmCfg {
    // CG = 1: one CTA computes a 128 x BN tile. CG = 2: a CTA pair (cluster of 2) computes a
    // 256 x BN tile with cta_group::2 MMAs; each CTA holds 128 rows of A, BN/2 rows of B and
    // its 128 x BN half of the accumulator. A 512-wide pair tile is two MMA halves of N = 256
    // (CTA r holds B rows [256h + 128r, +128) of half h) into all 512 TMEM columns: one
    // accumulator instead of two, for 25% fewer operand bytes per FLOP than 256 x 256.
    static constexpr int CG = CG_;
    static constexpr int BM = 128, BN = BN_, BK = 64, UMMA_K = 16;
    static constexpr int BN_CTA = BN / CG;  // rows of the B operand one CTA loads
    static constexpr bool A_MN = A_MN_, B_MN = B_MN_;
    static constexpr int EPI = EPI_;
    // Operand transform: the A tiles hold H and become G = GELU(H) in shared memory before
    // the MMAs read them; the epilogue is then EPI_B's (plain or + bias).
    static constexpr bool XFORM = (EPI == EPI_PLAIN_GA || EPI == EPI_BIAS_GA);
    static constexpr int EPI_B = (EPI == EPI_PLAIN_GA) ? EPI_PLAIN : (EPI == EPI_BIAS_GA) ? EPI_BIAS : EPI;
    // Dual B operand (SwiGLU up-projection): each tile covers OBN = BN/2 output columns,
    // its MMA N = BN spans [A's columns | Wg's columns] of that range.
    static constexpr bool DUAL = (EPI_B == EPI_SWIGLU);
    static constexpr int OBN = DUAL ? BN / 2 : BN;
    static constexpr int HALVES = (BN == 512) ? 2 : 1;  // MMAs per k step, each N = MMA_N
    static constexpr int MMA_N = BN / HALVES;
    // accumulators in TMEM: two (the epilogue of tile i overlaps the main loop of tile i+1),
    // or one 512-column accumulator whose halves are released one after the other
    static constexpr int NACC = (BN == 512) ? 1 : 2;
    // epilogues the split-tail fixup can finish: their last tiles may be split
    static constexpr bool SPLITTABLE =
        (EPI_B == EPI_PLAIN || EPI_B == EPI_BIAS || EPI_B == EPI_BIAS_GELU || EPI_B == EPI_DGELU);
    static constexpr uint32_t A_BYTES = BM * BK * 2;
    static constexpr uint32_t B_BYTES = BN_CTA * BK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int NOUT = (EPI_B == EPI_SWIGLU) ? 3 : (EPI_B == EPI_BIAS_GELU || EPI_B == EPI_DSWIGLU) ? 2 : 1;
    static constexpr uint32_t STG_BYTES = 32 * 32 * 2;              // one 32x32 bf16 box
    // Epilogue warps: 8 (two per TMEM lane quadrant, taking alternate 32-column chunks) for the
    // one-accumulator 512-wide tiles, whose epilogue holds up the next tile's MMAs until each
    // half is read out; else 4. With 8, each warp stages through one buffer instead of two.
    static constexpr int EPI_WARPS = (NACC == 1) ? 8 : 4;
    static constexpr int EPI_SETS = EPI_WARPS / 4;
    // Operand-transform warps: 8 GELUs per clock per SM keep pace with a 512-wide tile's MMAs
    // (one A value per 512 MACs).
    static constexpr int XF_WARPS = XFORM ? 16 : 0;
    static constexpr int STG_BUFS = EPI_WARPS == 8 ? 1 : 2;
    static constexpr uint32_t EPI_BYTES = EPI_WARPS * STG_BUFS * NOUT * STG_BYTES;
    // Epilogues whose first output is the accumulator (+ bias) rounded to bf16 read each
    // half of a one-accumulator tile out of TMEM (packed, 16 words a chunk) and release it
    // before staging and storing anything; the bias + GELU epilogue then computes G from
    // the rounded H.
    static constexpr bool DRAIN_FIRST =
        NACC == 1 && EPI_WARPS == 8 && !XFORM && (EPI_B == EPI_PLAIN || EPI_B == EPI_BIAS || EPI_B == EPI_BIAS_GELU);
    static constexpr uint32_t TMEM_COLS = NACC * BN;                 // fp32 accumulators
    // 32-column chunks one epilogue warp handles per tile: chunks eset + EPI_SETS * k
    static constexpr int NCH = OBN / 32 / EPI_SETS;
    static constexpr bool HAS_BIAS = (EPI_B == EPI_BIAS || EPI_B == EPI_BIAS_GELU || EPI_B == EPI_BIAS_DROPOUT_RES);
    // as many stages as fit beside the epilogue staging (at most 6 for pairs, 4 alone)
    static constexpr int STAGES_FIT = static_cast<int>((232448u - 1024u - 256u - EPI_BYTES) / STAGE_BYTES);
    static constexpr int STAGES = STAGES_FIT < ((CG == 2) ? 6 : 4) ? STAGES_FIT : ((CG == 2) ? 6 : 4);
    // The transform warps work in XF_GROUPS groups; group g owns the ring slots s with
    // s % XF_GROUPS == g and transforms every fill of them, whole, in order. Fills then move
    // through several groups at once (each fill's chain of waits, shared-memory round trip
    // and proxy fence overlaps the others'), and a group never waits on a slot's barrier more
    // than one phase ahead of its last completed phase.
    static constexpr int XF_GROUPS = (STAGES % 4 == 0) ? 4 : 2;
    static constexpr int XF_GROUP_WARPS = XFORM ? XF_WARPS / XF_GROUPS : 1;
    static_assert(!XFORM || (STAGES % XF_GROUPS == 0 && (A_BYTES / 16) % (32 * XF_GROUP_WARPS) == 0),
                  "transform groups own whole ring slots and whole 16-byte columns of the A tile");
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 1 + (XFORM ? 2 * STAGES : 0);
    static constexpr uint32_t BAR_BYTES = 8 * NUM_BARS + 16;
    static constexpr uint32_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
    static constexpr int THREADS = 64 + 32 * (EPI_WARPS + XF_WARPS);  // producer, MMA issuer, epilogue, transform
    static constexpr uint32_t IDESC = idesc_bf16_f32(BM * CG, MMA_N, A_MN, B_MN);
    static_assert(BN == 128 || BN == 256 || BN == 512, "tile width");
    static_assert(CG == 1 ? BN <= 256 : (BN == 256 || (BN == 512 && !DUAL)), "CTA pairs use 256- or 512-wide tiles");
    static_assert(TMEM_COLS <= 512, "tensor memory columns");
    static_assert(!HAS_BIAS || (NCH >= 1 && NCH <= 8), "a warp's bias values fit one 16-byte load per lane");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(STAGES >= 3, "pipeline depth");
    static_assert(!DUAL || (B_MN && BN == 256), "dual B operand: MN-major, 256-wide MMA");
};

// In-flight copies get this long to land after an abort before the CTA exits.
constexpr unsigned long long kDrainLimitNs = 2000000000ull;

// ---- packed fp32 pairs --------------------------------------------------------------------
// The sm_100-family f32x2 fma / mul / add do two IEEE round-to-nearest operations in one
// instruction; a pair lives in one 64-bit register.
typedef unsigned long long f32x2_t;

__device__ __forceinline__ f32x2_t f2_pack(float lo, float hi)
{
    f32x2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(f32x2_t v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2_t f2_splat(float k) { return f2_pack(k, k); }
__device__ __forceinline__ f32x2_t f2_fma(f32x2_t a, f32x2_t b, f32x2_t c)
{
    f32x2_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2_t f2_mul(f32x2_t a, f32x2_t b)
{
    f32x2_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float ex2_approx(float z)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(z));
    return r;
}

__device__ __forceinline__ float rcp_approx_f(float d)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// GELU, tanh form, on a pair of values. With u = sqrt(2/pi) (x + 0.044715 x^3):
//   1 + tanh u = 2 s,  s = sigmoid(2u) = 1 / (1 + e),  e = exp(-2u),
//   GELU(x) = x s,     GELU'(x) = s + 2 x s (1 - s) u'(x),  u'(x) = sqrt(2/pi) (1 + 3 0.044715 x^2).
// e = 2^z with z = -2 log2(e) u = x (c0 + c1 x^2), and s = 1 / (1 + e) from the hardware's
// approximate reciprocal (<= 1 ulp): two special-function ops per value. The epilogues and
// the operand transform that evaluate it are bound by their instruction counts, not by that
// pipe (a reciprocal by three Newton steps on the FMA pipe measured slower in both). Since
// 1 - s = e s, s (1 - s) = s^2 e has no cancellation.
// x is first raised to at least -kGeluFloor (z <= 117.9 there, so e and 1 + e stay normal
// numbers): below it GELU(x) and GELU'(x) are below 3.1e-35 in magnitude, which is what the
// clamped x gives, and a huge negative x can no longer meet a tiny s in x s. GELU' also caps
// x at +kGeluFloor (GELU' = 1 in fp32 from there on), so that x^2 stays finite where e = 0.
constexpr float kGeluFloor = 9.75f;
struct GeluPair {
    f32x2_t x, x2, e, s;
};

// x0, x1 already clamped as the caller needs
__device__ __forceinline__ GeluPair gelu_sigmoid_clamped(float x0, float x1)
{
    constexpr float kC0 = static_cast<float>(-2.0 * 1.4426950408889634 * 0.7978845608028654);
    constexpr float kC1 = static_cast<float>(-2.0 * 1.4426950408889634 * 0.7978845608028654 * 0.044715);
    GeluPair g;
    g.x = f2_pack(x0, x1);
    g.x2 = f2_mul(g.x, g.x);
    float z0, z1;
    f2_unpack(f2_mul(g.x, f2_fma(g.x2, f2_splat(kC1), f2_splat(kC0))), z0, z1);
    const float e0 = ex2_approx(z0), e1 = ex2_approx(z1);
    g.e = f2_pack(e0, e1);
    g.s = f2_pack(rcp_approx_f(1.0f + e0), rcp_approx_f(1.0f + e1));
    return g;
}

// for GELU: x raised to at least -kGeluFloor
__device__ __forceinline__ GeluPair gelu_sigmoid_pair(f32x2_t x)
{
    float x0, x1;
    f2_unpack(x, x0, x1);
    return gelu_sigmoid_clamped(fmaxf(x0, -kGeluFloor), fmaxf(x1, -kGeluFloor));
}

__device__ __forceinline__ f32x2_t gelu_value_pair(const GeluPair& g) { return f2_mul(g.x, g.s); }

__device__ __forceinline__ f32x2_t gelu_grad_pair(const GeluPair& g)
{
    constexpr float kD0 = static_cast<float>(2.0 * 0.7978845608028654);
    constexpr float kD1 = static_cast<float>(2.0 * 0.7978845608028654 * 3.0 * 0.044715);
    const f32x2_t w = f2_mul(g.x, f2_fma(g.x2, f2_splat(kD1), f2_splat(kD0)));  // 2 x u'(x)
    const f32x2_t q = f2_mul(f2_mul(g.s, g.s), g.e);                            // s (1 - s)
    return f2_fma(q, w, g.s);
}

// GELU'(x) on a pair: x clamped to [-kGeluFloor, kGeluFloor]
__device__ __forceinline__ f32x2_t gelu_grad_fast_pair(f32x2_t x)
{
    float x0, x1;
    f2_unpack(x, x0, x1);
    return gelu_grad_pair(gelu_sigmoid_clamped(fminf(fmaxf(x0, -kGeluFloor), kGeluFloor),
                                               fminf(fmaxf(x1, -kGeluFloor), kGeluFloor)));
}

// Scalar forms (the split-tail fixup): the pair code on (x, x), so every path gets the same bits.
__device__ __forceinline__ float gelu_tanh_f(float x)
{
    float lo, hi;
    f2_unpack(gelu_value_pair(gelu_sigmoid_pair(f2_pack(x, x))), lo, hi);
    return lo;
}
__device__ __forceinline__ float gelu_tanh_grad_f(float x)
{
    float lo, hi;
    f2_unpack(gelu_grad_fast_pair(f2_pack(x, x)), lo, hi);
    return lo;
}

// G = GELU of the bf16 pair packed in w (low half first), rounded to a bf16 pair.
__device__ __forceinline__ uint32_t gelu_bf16x2(uint32_t w);

__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// SiLU(x) = x sigma(x); SiLU'(x) = sigma(x) (1 + x (1 - sigma(x))).
__device__ __forceinline__ float silu_f(float x) { return x * sigmoid_f(x); }
__device__ __forceinline__ float silu_grad_f(float x)
{
    const float s = sigmoid_f(x);
    return s * fmaf(x, 1.0f - s, 1.0f);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t gelu_bf16x2(uint32_t w)
{
    float g0, g1;
    f2_unpack(gelu_value_pair(gelu_sigmoid_pair(f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)))), g0,
              g1);
    return pack_bf16x2(g0, g1);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* out)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Column sums over the 32 lanes of a warp: lane l holds v[0..31] (its row, 32 columns);
// afterwards v[0] of lane l is the sum over all lanes of column l. Five halving stages,
// 31 shuffles: at stage s each lane keeps the half of its columns selected by bit s of
// its lane index and adds the partner's copy of that half.
__device__ __forceinline__ void warp_column_sums(float (&v)[32], int lane)
{
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int j = 0; j < s; ++j) {
            const float send = upper ? v[j] : v[j + s];
            const float keep = upper ? v[j + s] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
}

// Write one thread's 32 bf16 (16 packed words) as row `lane` of a 32x32 box laid out the
// way a 64-byte-swizzled TMA store reads it: 16-byte chunk j of row r sits at chunk
// j ^ ((r >> 1) & 3).
__device__ __forceinline__ void stage_row_sw64(uint32_t buf, int lane, const uint32_t (&p)[16])
{
    const uint32_t row = buf + static_cast<uint32_t>(lane) * 64u;
    const uint32_t x = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
    for (uint32_t j = 0; j < 4; ++j)
        sts_v4(row + ((j ^ x) << 4), p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
}

// Bias of chunk wc of this warp: before the tile's accumulator is ready, lane l loads the 8
// bias values of columns [8 (l % 4), +8) of chunk l / 4 as one 16-byte word (bw); here each
// lane takes the 32 values of chunk wc from lanes 4 wc .. 4 wc + 3 by shuffles and adds
// them to its row. Shuffles instead of a load per chunk: the loads' latency would otherwise
// sit between reading the accumulator out of TMEM and releasing it.
__device__ __forceinline__ void add_bias_chunk(float (&v)[32], const uint4& bw, int wc)
{
#pragma unroll
    for (int jp = 0; jp < 16; ++jp) {
        const uint32_t w = (jp & 3) == 0 ? bw.x : (jp & 3) == 1 ? bw.y : (jp & 3) == 2 ? bw.z : bw.w;
        const uint32_t x = __shfl_sync(0xffffffffu, w, 4 * wc + (jp >> 2));
        v[2 * jp] += __uint_as_float(x << 16);
        v[2 * jp + 1] += __uint_as_float(x & 0xFFFF0000u);
    }
}

// Output tile `tile` -> its first row and column. Tiles that run at the same time (about
// one per unit, consecutive indices) share operand blocks through L2 while their k loops
// run in step; with large K nothing survives in L2 from one wave to the next, so a wave
// reads every distinct A and B block it touches from DRAM. Tiles are therefore ordered
// in groups of `group` consecutive indices along the fast dimension (M, or N when
// n_fastest), sweeping the other dimension within a group: a wave covers about
// group x (units / group) tiles and reads group + units / group blocks instead of
// (all of the fast dimension) + (units / that).
__device__ __forceinline__ void tile_origin(int tile, int tiles_m, int tiles_n, int n_fastest, int group, int TM,
                                            int BN, int& m0, int& n0)
{
    const int fast_n = n_fastest ? tiles_n : tiles_m;  // extent of the grouped index
    const int slow_n = n_fastest ? tiles_m : tiles_n;
    const int gsz = (group > 0 && group < fast_n) ? group : fast_n;
    const int per_group = gsz * slow_n;
    const int g = tile / per_group, r = tile % per_group;
    const int glen = min(gsz, fast_n - g * gsz);
    const int fast = g * gsz + r % glen, slow = r / glen;
    if (n_fastest) {
        m0 = slow * TM;
        n0 = fast * BN;
    } else {
        m0 = fast * TM;
        n0 = slow * BN;
    }
}

// Work unit u -> its tile, its range of k blocks [kb_lo, kb_hi) and, for a part of a split
// tile, its index among all parts (part = -1 for a whole tile). Units [0, n_whole) are the
// whole tiles in tile order; then each of the last split_tiles tiles comes as split_k parts.
__device__ __forceinline__ void work_unit(int u, int n_whole, int split_k, int num_kb, int& tile, int& kb_lo,
                                          int& kb_hi, int& part)
{
    if (u < n_whole) {
        tile = u;
        kb_lo = 0;
        kb_hi = num_kb;
        part = -1;
        return;
    }
    const int v = u - n_whole, r = v / split_k, sk = v - r * split_k;
    tile = n_whole + r;
    part = v;
    kb_lo = static_cast<int>(static_cast<long long>(sk) * num_kb / split_k);
    kb_hi = static_cast<int>(static_cast<long long>(sk + 1) * num_kb / split_k);
}

template <int BN, bool A_MN, bool B_MN, int EPI, int CG>
__global__ void __launch_bounds__(GemmCfg<BN, A_MN, B_MN, EPI, CG>::THREADS, 1) umma_gemm_kernel(const __grid_constant__ GemmArgs args)
{
    using C = GemmCfg<BN, A_MN, B_MN, EPI, CG>;
    constexpr int E = C::EPI_B;  // the epilogue (the transform flavours use the plain or bias one)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t s_stages = base;
    const uint32_t s_epi = base + C::STAGES * C::STAGE_BYTES;
    const uint32_t s_bar = s_epi + C::EPI_BYTES;
    // barrier map: full[S] | empty[S] | acc_full[2] | acc_empty[2] | drain | (transform
    // flavours: a_full[S] | xf[S]) | tmem slot | abort. With the transform, each CTA's A tile
    // lands on its own a_full barrier, its transform warps turn it into G, and xf (in the
    // pair's even CTA, which issues the MMAs) completes once both CTAs' warps are done.
    const uint32_t b_full = s_bar, b_empty = s_bar + 8u * C::STAGES;
    const uint32_t b_accf = s_bar + 16u * C::STAGES, b_acce = b_accf + 16u;
    const uint32_t b_drain = b_acce + 16u;
    const uint32_t b_afull = b_drain + 8u, b_xf = b_afull + 8u * C::STAGES;
    const uint32_t s_slot = b_drain + 8u + (C::XFORM ? 16u * C::STAGES : 0u);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + (s_slot - base));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (s_slot + 4u - base));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Pair mode: rank 0 (the even CTA) of a pair issues every MMA; rank r owns rows
    // [128r, 128r+128) of each 256-row tile and B rows [r*BN/2, (r+1)*BN/2) of each stage.
    // With two pairs per cluster (512-wide tiles only), pair p computes rows [256p, 256p+256)
    // of a 512-row work tile, and the pairs share each stage's B: CTA (p, r) fetches B half p
    // and multicasts it to CTA r of both pairs.
    const int npc = (CG == 2 && C::HALVES == 2 && args.cluster_pairs == 2) ? 2 : 1;  // pairs per cluster
    const uint32_t crank = (CG == 2) ? cluster_ctarank() : 0u;
    const uint32_t rank = crank & 1u, pidx = crank >> 1, lead = crank & ~1u;
    const int unit = static_cast<int>(blockIdx.x) / (CG * npc);
    const int num_units = static_cast<int>(gridDim.x) / (CG * npc);
    const int M = args.M, N = args.N, K = args.K;
    const int TM = C::BM * CG * npc;  // rows per work tile
    const int prow = C::BM * CG * static_cast<int>(pidx);  // this pair's first row in it
    const int tiles_m = (M + TM - 1) / TM;
    const int tiles_n = (N + C::OBN - 1) / C::OBN;
    const int num_tiles = tiles_m * tiles_n;
    const int num_kb = (K + C::BK - 1) / C::BK;
    const int split_tiles = C::SPLITTABLE ? args.split_tiles : 0;
    const int split_k = split_tiles > 0 ? args.split_k : 1;
    const int n_whole = num_tiles - split_tiles;
    const int num_work = n_whole + split_tiles * split_k;
    const unsigned long long limit = args.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(b_full + 8u * s, 1);
            mbar_init(b_empty + 8u * s, npc);  // each pair's MMAs release the stage
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(b_accf + 8u * a, 1);
            mbar_init(b_acce + 8u * a, C::EPI_WARPS * CG);  // one arrive per epilogue warp of the pair
        }
        mbar_init(b_drain, 1);
        if (C::XFORM)
            for (int s = 0; s < C::STAGES; ++s) {
                mbar_init(b_afull + 8u * s, 1);
                mbar_init(b_xf + 8u * s, C::XF_GROUP_WARPS * CG);  // one transform group, in each CTA of the pair
            }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&args.tmA);
        tma_prefetch_desc(&args.tmB);
        tma_prefetch_desc(&args.tmD0);
        if (C::NOUT >= 2) tma_prefetch_desc(&args.tmD1);
        if (C::NOUT >= 3) tma_prefetch_desc(&args.tmD2);
        if (C::DUAL || args.kb_split > 0) tma_prefetch_desc(&args.tmB2);
        if (args.kb_split > 0) tma_prefetch_desc(&args.tmA2);
    }
    if (CG == 2) cluster_sync();  // the peer CTA is running before the collective allocation
    if (warp == 1) {
        if (CG == 2) {
            tmem_alloc_pair(s_slot, C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(s_slot, C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if (CG == 2)
        cluster_sync();  // both CTAs' barriers and TMEM exist before either signals the other
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued = 0, par = 0;
            bool ok = true;
            for (int u = unit; ok && u < num_work; u += num_units) {
                int tile, kb_lo, kb_hi, part;
                work_unit(u, n_whole, split_k, num_kb, tile, kb_lo, kb_hi, part);
                int m0, n0;
                tile_origin(tile, tiles_m, tiles_n, args.n_fastest, args.raster_group, TM, C::OBN, m0, n0);
                const int m_cta = m0 + prow + C::BM * static_cast<int>(rank);
                const int n_cta = n0 + C::BN_CTA * static_cast<int>(rank);
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait_bounded(b_empty + 8u * stage, phase ^ 1u, abort_flag, args.status,
                                           limit, DEV_TIMEOUT_PRODUCER, tile, kb)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = s_stages + stage * C::STAGE_BYTES;
                    const uint32_t sb = sa + C::A_BYTES;
                    const uint32_t fb = b_full + 8u * stage;
                    // second K segment (kb_split > 0): its own operands, from their k = 0
                    const bool seg2 = args.kb_split > 0 && kb >= args.kb_split;
                    const int k0 = (seg2 ? kb - args.kb_split : kb) * C::BK;
                    const CUtensorMap* tA = seg2 ? &args.tmA2 : &args.tmA;
                    const CUtensorMap* tB = seg2 ? &args.tmB2 : &args.tmB;
                    // transform flavours: this CTA's A tile lands on its own a_full barrier
                    const uint32_t fa = C::XFORM ? b_afull + 8u * stage : fb;
                    if (CG == 1) {
                        if (C::XFORM) mbar_arrive_expect_tx(fa, C::A_BYTES);
                        mbar_arrive_expect_tx(fb, C::XFORM ? C::B_BYTES : C::STAGE_BYTES);
                        if (A_MN) {
                            tma_load_2d(sa, tA, m_cta, k0, fa);
                            tma_load_2d(sa + 8192u, tA, m_cta + 64, k0, fa);
                        } else {
                            tma_load_2d(sa, tA, k0, m_cta, fa);
                        }
                        if (C::DUAL) {  // rows [0, BN/2): A's columns; [BN/2, BN): Wg's, same range
#pragma unroll
                            for (int i = 0; i < C::BN_CTA / 64; ++i)
                                tma_load_2d(sb + 8192u * i, i < C::BN_CTA / 128 ? &args.tmB : &args.tmB2,
                                            n0 + 64 * (i % (C::BN_CTA / 128)), k0, fb);
                        } else if (B_MN) {
#pragma unroll
                            for (int i = 0; i < C::BN_CTA / 64; ++i)
                                tma_load_2d(sb + 8192u * i, tB, n_cta + 64 * i, k0, fb);
                        } else {
                            tma_load_2d(sb, tB, k0, n_cta, fb);
                        }
                    } else {
                        // Both CTAs' bytes complete on the pair's even CTA's barrier, which that
                        // CTA alone arms with the pair's total (with two pairs, the B half the
                        // other pair multicasts into this pair completes there too).
                        const uint32_t fb0 = mapa_shared(fb, lead);
                        if (rank == 0) mbar_arrive_expect_tx(fb, 2 * (C::XFORM ? C::B_BYTES : C::STAGE_BYTES));
                        if (C::XFORM) {
                            mbar_arrive_expect_tx(fa, C::A_BYTES);
                            if (A_MN) {
                                tma_load_2d(sa, tA, m_cta, k0, fa);
                                tma_load_2d(sa + 8192u, tA, m_cta + 64, k0, fa);
                            } else {
                                tma_load_2d(sa, tA, k0, m_cta, fa);
                            }
                        } else if (A_MN) {
                            tma_load_2d_pair(sa, tA, m_cta, k0, fb0);
                            tma_load_2d_pair(sa + 8192u, tA, m_cta + 64, k0, fb0);
                        } else {
                            tma_load_2d_pair(sa, tA, k0, m_cta, fb0);
                        }
                        if (C::DUAL) {  // the even CTA holds A's columns, the odd one Wg's
#pragma unroll
                            for (int i = 0; i < C::BN_CTA / 64; ++i)
                                tma_load_2d_pair(sb + 8192u * i, rank == 0 ? &args.tmB : &args.tmB2, n0 + 64 * i,
                                                 k0, fb0);
                        } else if (npc == 2) {  // B half `pidx` to CTA `rank` of both pairs
                            const uint16_t mask = static_cast<uint16_t>((1u << rank) | (1u << (2u + rank)));
                            const int nb = n0 + C::MMA_N * static_cast<int>(pidx) + 128 * static_cast<int>(rank);
                            const uint32_t sbh = sb + 16384u * pidx;
                            if (B_MN) {
                                tma_load_2d_pair_mc(sbh, tB, nb, k0, fb0, mask);
                                tma_load_2d_pair_mc(sbh + 8192u, tB, nb + 64, k0, fb0, mask);
                            } else {
                                tma_load_2d_pair_mc(sbh, tB, k0, nb, fb0, mask);
                            }
                        } else if (B_MN) {  // half h: 128 rows at sb + 16 KB h, in 64-wide boxes
#pragma unroll
                            for (int h = 0; h < C::HALVES; ++h)
#pragma unroll
                                for (int i = 0; i < 2; ++i)
                                    tma_load_2d_pair(sb + 16384u * h + 8192u * i, tB,
                                                     n0 + C::MMA_N * h + 128 * static_cast<int>(rank) + 64 * i, k0,
                                                     fb0);
                        } else {
#pragma unroll
                            for (int h = 0; h < C::HALVES; ++h)
                                tma_load_2d_pair(sb + 16384u * h, tB, k0,
                                                 n0 + C::MMA_N * h + 128 * static_cast<int>(rank), fb0);
                        }
                    }
                    // Transform flavours: a fill waits for its load, its transform and its MMAs in
                    // series, and with four stages that round trip nearly sets the rate. The A and B
                    // blocks one ring ahead are pulled into L2 now, so their loads do not wait on DRAM.
                    if (C::XFORM && kb + C::STAGES < kb_hi) {
                        const int k1 = (kb + C::STAGES) * C::BK;
                        if (A_MN) {
                            tma_prefetch_l2_2d(tA, m_cta, k1);
                            tma_prefetch_l2_2d(tA, m_cta + 64, k1);
                        } else {
                            tma_prefetch_l2_2d(tA, k1, m_cta);
                        }
#pragma unroll
                        for (int h = 0; h < C::HALVES; ++h) {
                            if (npc == 2 && h != static_cast<int>(pidx)) continue;  // the other pair's half
                            const int nb = n0 + C::MMA_N * h + 128 * static_cast<int>(rank);
                            if (B_MN) {
                                tma_prefetch_l2_2d(tB, nb, k1);
                                tma_prefetch_l2_2d(tB, nb + 64, k1);
                            } else {
                                tma_prefetch_l2_2d(tB, k1, nb);
                            }
                        }
                    }
                    issued |= 1u << stage;
                    par = (par & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let every copy this CTA started land before the CTA may exit.
                if (C::XFORM) {  // its A tiles, on its own barriers
                    volatile int never = 0;
                    for (int s = 0; s < C::STAGES; ++s)
                        if (issued & (1u << s))
                            mbar_wait_bounded(b_afull + 8u * s, (par >> s) & 1u, &never, args.status, kDrainLimitNs,
                                              DEV_TIMEOUT_DRAIN);
                }
                if (rank == 0) {
                    volatile int never = 0;
                    for (int s = 0; s < C::STAGES; ++s)
                        if (issued & (1u << s))
                            mbar_wait_bounded(b_full + 8u * s, (par >> s) & 1u, &never, args.status,
                                              kDrainLimitNs, DEV_TIMEOUT_DRAIN);
                } else if (issued) {
                    spin_ns(2000000ull);  // its barrier lives in the even CTA: give them 2 ms
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer --------------------------------
        if (lane == 0 && rank == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true, any = false;
            for (int u = unit; ok && u < num_work; u += num_units) {
                int tile, kb_lo, kb_hi, part;
                work_unit(u, n_whole, split_k, num_kb, tile, kb_lo, kb_hi, part);
                if (!mbar_wait_bounded(b_acce + 8u * acc, acc_phase ^ 1u, abort_flag, args.status,
                                       limit, DEV_TIMEOUT_MMA_ACC, tile, -1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                // One accumulator: half 1 may still be draining when the tile starts. Until the
                // epilogue releases it, each k block's half-0 MMAs are issued and its stage is
                // held with its half-1 MMAs deferred (at most STAGES - 1 stages, so the producer
                // never waits on a stage this loop needs next); once half 1 is free the deferred
                // half-1 MMAs go out in k order, so each half accumulates in the same order as
                // without deferral and the results are the same bits.
                bool half1_free = C::NACC == 2;
                int ndef = 0, def_kb = 0;  // deferred k blocks: def_kb, def_kb + 1, ...
                uint32_t def_stage = 0;    // the first one's stage
                auto issue_half = [&](uint32_t st, int kbi, int h) {
                    const uint32_t sa = s_stages + st * C::STAGE_BYTES;
                    const uint32_t sbh = sa + C::A_BYTES + 16384u * h;
#pragma unroll
                    for (int k = 0; k < C::BK / C::UMMA_K; ++k) {
                        // K-major: next 16 elements are 32 bytes further along the swizzled
                        // row. MN-major: next 16 k-rows are two 8-row (1024-byte) groups on.
                        const uint64_t ad = A_MN ? smem_desc_sw128(sa + 2048u * k, 8192u, 1024u)
                                                 : smem_desc_sw128(sa + 32u * k, 16u, 1024u);
                        const uint64_t bd = B_MN ? smem_desc_sw128(sbh + 2048u * k, 8192u, 1024u)
                                                 : smem_desc_sw128(sbh + 32u * k, 16u, 1024u);
                        const uint32_t accum = (kbi != kb_lo || k != 0) ? 1u : 0u;
                        if (CG == 2)
                            umma_bf16_pair(d_tmem + C::MMA_N * h, ad, bd, C::IDESC, accum);
                        else
                            umma_bf16(d_tmem + C::MMA_N * h, ad, bd, C::IDESC, accum);
                    }
                };
                // the stage is free, in both CTAs (and, with two pairs, in the other pair's,
                // which multicast into it), once the MMAs issued so far finish
                auto release = [&](uint32_t st) {
                    if (CG == 2) {
                        umma_commit_pair_both(b_empty + 8u * st, lead + 1u);
                        if (npc == 2) {
                            const uint32_t other = lead ^ 2u;
                            umma_commit_pair(mapa_shared(b_empty + 8u * st, other));
                            umma_commit_pair(mapa_shared(b_empty + 8u * st, other + 1u));
                        }
                    } else {
                        umma_commit(b_empty + 8u * st);
                    }
                };
                // half 1 released: the deferred k blocks' half-1 MMAs, then their stages
                auto flush = [&]() {
                    tc_fence_after();
                    half1_free = true;
                    uint32_t st = def_stage;
                    for (int i = 0; i < ndef; ++i) {
                        issue_half(st, def_kb + i, 1);
                        release(st);
                        if (++st == C::STAGES) st = 0;
                    }
                    ndef = 0;
                };
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait_bounded(b_full + 8u * stage, phase, abort_flag, args.status, limit,
                                           DEV_TIMEOUT_MMA_FULL, tile, kb) ||
                        (C::XFORM && !mbar_wait_bounded<CG == 2>(b_xf + 8u * stage, phase, abort_flag, args.status,
                                                                 limit, DEV_TIMEOUT_MMA_FULL, tile, kb))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    any = true;
                    issue_half(stage, kb, 0);
                    if (C::HALVES == 2) {
                        if (!half1_free) {
                            bool freed = mbar_test_wait(b_acce + 8u, acc_phase ^ 1u);
                            if (!freed && ndef + 1 >= C::STAGES) {  // no stage left to hold: wait
                                if (!mbar_wait_bounded(b_acce + 8u, acc_phase ^ 1u, abort_flag, args.status, limit,
                                                       DEV_TIMEOUT_MMA_ACC, tile, -2)) {
                                    ok = false;
                                    break;
                                }
                                freed = true;
                            }
                            if (freed) {
                                flush();
                            } else {  // hold this stage; its half 1 comes later
                                if (ndef == 0) {
                                    def_stage = stage;
                                    def_kb = kb;
                                }
                                ++ndef;
                                if (++stage == C::STAGES) {
                                    stage = 0;
                                    phase ^= 1u;
                                }
                                continue;
                            }
                        }
                        issue_half(stage, kb, 1);
                    }
                    release(stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok && ndef > 0) {  // the tile's k blocks ran out before half 1 was released
                    if (!mbar_wait_bounded(b_acce + 8u, acc_phase ^ 1u, abort_flag, args.status, limit,
                                           DEV_TIMEOUT_MMA_ACC, tile, -2))
                        ok = false;
                    else
                        flush();
                }
                if (!ok) break;
                // accumulator ready for the epilogue warps of both CTAs
                if (CG == 2)
                    umma_commit_pair_both(b_accf + 8u * acc, lead + 1u);
                else
                    umma_commit(b_accf + 8u * acc);
                if (C::NACC == 2) {
                    acc ^= 1u;
                    if (acc == 0) acc_phase ^= 1u;
                } else {
                    acc_phase ^= 1u;
                }
            }
            if (!ok && any) {
                // Let the MMAs already issued finish before TMEM is released.
                volatile int never = 0;
                if (CG == 2)
                    umma_commit_pair(b_drain);
                else
                    umma_commit(b_drain);
                mbar_wait_bounded(b_drain, 0, &never, args.status, kDrainLimitNs, DEV_TIMEOUT_DRAIN);
            }
        }
    } else if (C::XFORM && warp >= 2 + C::EPI_WARPS) {
        // --------------------------- operand transform ----------------------------
        // Each landed A tile of H (16 KB: 128 rows x 64 k) becomes G = GELU(H) in place, 16
        // bytes (8 values) per thread and step, with the same arithmetic as the forward's
        // bias + GELU epilogue (gelu_bf16x2), so G matches the stored G bit for bit. The
        // values are elementwise, so the tile's layout (K- or MN-major, swizzled) does not
        // matter; zero fill past the matrix edges stays zero (GELU(0) = 0).
        const int xw = warp - (2 + C::EPI_WARPS);
        const int group = xw / C::XF_GROUP_WARPS;
        const int xt = 32 * (xw % C::XF_GROUP_WARPS) + lane;  // thread within its group
        const uint32_t xf0 = (CG == 2) ? mapa_shared(b_xf, lead) : b_xf;
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int u = unit; ok && u < num_work; u += num_units) {
            int tile, kb_lo, kb_hi, part;
            work_unit(u, n_whole, split_k, num_kb, tile, kb_lo, kb_hi, part);
            for (int kb = kb_lo; kb < kb_hi; ++kb) {
                const uint32_t st = stage, ph = phase;
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (static_cast<int>(st) % C::XF_GROUPS != group) continue;  // another group's ring slot
                // every lane waits, as each reads bytes the copy wrote; the warp acts on all
                const bool got = mbar_wait_bounded(b_afull + 8u * st, ph, abort_flag, args.status, limit,
                                                   DEV_TIMEOUT_XFORM, tile, kb);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = s_stages + st * C::STAGE_BYTES;
#pragma unroll 4
                for (int i = 0; i < static_cast<int>(C::A_BYTES / 16) / (32 * C::XF_GROUP_WARPS); ++i) {
                    const uint32_t ad = sa + 16u * static_cast<uint32_t>(xt + 32 * C::XF_GROUP_WARPS * i);
                    const uint4 hv = lds_v4(ad);
                    sts_v4(ad, gelu_bf16x2(hv.x), gelu_bf16x2(hv.y), gelu_bf16x2(hv.z), gelu_bf16x2(hv.w));
                }
                fence_proxy_async_smem();  // the MMAs read the tile through the async proxy
                __syncwarp();
                if (lane == 0) {
                    if (CG == 2)
                        mbar_arrive_cluster(xf0 + 8u * st);
                    else
                        mbar_arrive(b_xf + 8u * st);
                }
            }
        }
    } else {
        // ------------------------------ epilogue ----------------------------------
        const int q = warp & 3;  // TMEM lanes [32q, 32q+32) are the ones this warp may read
        const int ewarp = warp - 2, eset = ewarp >> 2;  // chunks eset, eset + EPI_SETS, ...
        // accumulator release goes to the even CTA, which issues the MMAs
        const uint32_t acce0 = (CG == 2) ? mapa_shared(b_acce, lead) : b_acce;
        uint32_t acc = 0, acc_phase = 0, sel = 0;
        for (int u = unit; u < num_work; u += num_units) {
            int tile, kb_lo, kb_hi, part;
            work_unit(u, n_whole, split_k, num_kb, tile, kb_lo, kb_hi, part);
            int m0, n0;
            tile_origin(tile, tiles_m, tiles_n, args.n_fastest, args.raster_group, TM, C::OBN, m0, n0);
            const int row_blk = m0 + prow + C::BM * static_cast<int>(rank) + 32 * q;
            const int row = row_blk + lane;
            // While the tile's main loop still runs: this warp's bias values (add_bias_chunk)
            // and, for the GELU' epilogues, this lane's row of H for its first three chunks
            // pulled into L2 (then each chunk pulls in the one three ahead).
            uint4 bias_w = make_uint4(0, 0, 0, 0);
            if (C::HAS_BIAS && part < 0) {
                const int wc = lane >> 2;
                const int n = n0 + 32 * (eset + C::EPI_SETS * wc) + 8 * (lane & 3);
                if (wc < C::NCH && n < N) bias_w = ldg_nc_v4(args.bias + n);
            }
            if (E == EPI_DGELU && part < 0 && row < M) {
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const int n = n0 + 32 * (eset + C::EPI_SETS * k);
                    if (k < C::NCH && n < N) prefetch_l2(args.aux + static_cast<size_t>(row) * args.ld_aux + n);
                }
            }
            // 512-wide GELU' epilogue: GELU'(H) of this warp's first chunk, computed while the
            // tile's main loop still runs (the same function on the same H, so the same bits), so
            // that accumulator half 0 is read out and released sooner. (Two chunks exceed the
            // register budget of ten warps and spill.)
            constexpr int PRE_N = (E == EPI_DGELU && C::NACC == 1) ? 1 : 0;
            f32x2_t gpre[PRE_N > 0 ? PRE_N : 1][16];
            if (PRE_N > 0 && part < 0) {
#pragma unroll
                for (int k = 0; k < PRE_N; ++k) {
                    float hv[32];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int n = n0 + 32 * (eset + C::EPI_SETS * k) + 8 * i;
                        const uint4 hw = (row < M && n < N)
                                             ? ldg_nc_v4(args.aux + static_cast<size_t>(row) * args.ld_aux + n)
                                             : make_uint4(0, 0, 0, 0);
                        unpack_bf16x8(hw, hv + 8 * i);
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) gpre[k][j] = gelu_grad_fast_pair(f2_pack(hv[2 * j], hv[2 * j + 1]));
                }
            }
            // One lane waits; the warp follows its verdict so the .sync.aligned TMEM loads
            // below always run with all 32 lanes.
            int ready = 0;
            if (lane == 0)
                ready = mbar_wait_bounded(b_accf + 8u * acc, acc_phase, abort_flag, args.status, limit,
                                          DEV_TIMEOUT_EPILOGUE, tile, -1);
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * BN;
            // a part of a split tile: its fp32 accumulator, chunk c of 32 columns at
            // [c][row within the tile][32] of this part's TM x OBN block of split_ws
            float* part_out = nullptr;
            if (C::SPLITTABLE && part >= 0)
                part_out = args.split_ws + static_cast<size_t>(part) * TM * C::OBN +
                           static_cast<size_t>(prow + C::BM * static_cast<int>(rank) + 32 * q + lane) * 32;

            // hnext: the aux row segment of this warp's next chunk (H, the residual, Ha);
            // gnext: Hg.
            uint4 hnext[4], gnext[4];
            if (E == EPI_DGELU || E == EPI_BIAS_DROPOUT_RES || E == EPI_DSWIGLU) {
                const int c_first = eset + C::EPI_SETS * (part < 0 ? PRE_N : 0);  // past the precomputed chunks
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int n = n0 + 32 * c_first + 8 * i;
                    const bool in = row < M && n < N;
                    hnext[i] = in ? ldg_nc_v4(args.aux + static_cast<size_t>(row) * args.ld_aux + n) : make_uint4(0, 0, 0, 0);
                    if (E == EPI_DSWIGLU)
                        gnext[i] = in ? ldg_nc_v4(args.aux2 + static_cast<size_t>(row) * args.ld_aux + n)
                                      : make_uint4(0, 0, 0, 0);
                }
            }
            if (C::DRAIN_FIRST && part_out == nullptr) {
                constexpr int KPH = C::OBN / 64 / C::EPI_SETS;  // this warp's chunks per half
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t pk[KPH][16];
#pragma unroll
                    for (int k = 0; k < KPH; ++k) {
                        const int c = hh * (C::OBN / 64) + eset + k * C::EPI_SETS;
                        const int nc = n0 + 32 * c;
                        uint32_t r[32];
                        if (nc < N) {  // warp-uniform
                            tmem_ld_32x32b_x32(t_row + 32u * c, r);
                            tmem_ld_wait();
                        }
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                        if (E == EPI_BIAS || E == EPI_BIAS_GELU) add_bias_chunk(v, bias_w, hh * KPH + k);
#pragma unroll
                        for (int j = 0; j < 16; ++j) pk[k][j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {  // this half of the accumulator may be reused
                        if (CG == 2)
                            mbar_arrive_cluster(acce0 + 8u * hh);
                        else
                            mbar_arrive(b_acce + 8u * hh);
                    }
#pragma unroll
                    for (int k = 0; k < KPH; ++k) {
                        const int c = hh * (C::OBN / 64) + eset + k * C::EPI_SETS;
                        const int nc = n0 + 32 * c;
                        if (nc >= N || row_blk >= M) continue;
                        uint32_t p1[16];
                        if (E == EPI_BIAS_GELU) {  // G = GELU(H) of the rounded H
#pragma unroll
                            for (int j = 0; j < 16; ++j) p1[j] = gelu_bf16x2(pk[k][j]);
                        }
                        const uint32_t buf0 = s_epi + ((ewarp * C::STG_BUFS + sel) * C::NOUT) * C::STG_BYTES;
                        if (lane == 0) bulk_wait_group_read<C::STG_BUFS - 1>();  // its last store has read it
                        __syncwarp();
                        stage_row_sw64(buf0, lane, pk[k]);
                        if (C::NOUT >= 2) stage_row_sw64(buf0 + C::STG_BYTES, lane, p1);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&args.tmD0, nc, row_blk, buf0);
                            if (C::NOUT >= 2) tma_store_2d(&args.tmD1, nc, row_blk, buf0 + C::STG_BYTES);
                            bulk_commit_group();
                        }
                        if (C::STG_BUFS == 2) sel ^= 1u;
                    }
                }
            } else
#pragma unroll 1
            for (int c = eset, wc = 0; c < C::OBN / 32; c += C::EPI_SETS, ++wc) {
                const int nc = n0 + 32 * c;
                const bool active = nc < N;  // warp-uniform
                uint32_t r[32], r2[32];
                if (active) {
                    tmem_ld_32x32b_x32(t_row + 32u * c, r);
                    if (C::DUAL) tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(C::OBN) + 32u * c, r2);  // X Wg
                    tmem_ld_wait();
                }
                // release: the whole accumulator after its last chunk, or (one 512-column
                // accumulator) each 256-column half after its last chunk
                const bool last_mine = c + C::EPI_SETS >= C::OBN / 32;
                const bool release =
                    C::NACC == 2 ? last_mine : (last_mine || (c < C::OBN / 64 && c + C::EPI_SETS >= C::OBN / 64));
                if (release) {
                    const uint32_t rel = C::NACC == 2 ? acc : (c >= C::OBN / 64 ? 1u : 0u);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {  // accumulator (half) may be reused
                        if (CG == 2)
                            mbar_arrive_cluster(acce0 + 8u * rel);
                        else
                            mbar_arrive(b_acce + 8u * rel);
                    }
                }
                if (C::SPLITTABLE && part_out) {
                    if (active) {
                        float4* dst = reinterpret_cast<float4*>(part_out + static_cast<size_t>(c) * TM * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                    }
                    continue;
                }
                if (!active || row_blk >= M) continue;

                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                uint32_t p0[16], p1[16], p2[16];
                if (E == EPI_SWIGLU) {  // v = Ha = X A, r2 = Hg = X Wg: keep both, U = SiLU(Ha) Hg
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float ga = __uint_as_float(r2[2 * j]), gb = __uint_as_float(r2[2 * j + 1]);
                        p1[j] = pack_bf16x2(ga, gb);
                        p2[j] = pack_bf16x2(silu_f(v[2 * j]) * ga, silu_f(v[2 * j + 1]) * gb);
                    }
                }
                if (E == EPI_DSWIGLU) {  // v = dU; dHa = dU Hg SiLU'(Ha) (in v), dHg = dU SiLU(Ha)
                    float ha[32], hg[32];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        unpack_bf16x8(hnext[i], ha + 8 * i);
                        unpack_bf16x8(gnext[i], hg + 8 * i);
                    }
                    if (c + C::EPI_SETS < C::OBN / 32) {  // prefetch the next chunk of Ha and Hg
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int n = nc + 32 * C::EPI_SETS + 8 * i;
                            const bool in = row < M && n < N;
                            const size_t o = static_cast<size_t>(row) * args.ld_aux + n;
                            hnext[i] = in ? ldg_nc_v4(args.aux + o) : make_uint4(0, 0, 0, 0);
                            gnext[i] = in ? ldg_nc_v4(args.aux2 + o) : make_uint4(0, 0, 0, 0);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float d0 = v[2 * j], d1 = v[2 * j + 1];
                        p1[j] = pack_bf16x2(d0 * silu_f(ha[2 * j]), d1 * silu_f(ha[2 * j + 1]));
                        v[2 * j] = d0 * hg[2 * j] * silu_grad_f(ha[2 * j]);
                        v[2 * j + 1] = d1 * hg[2 * j + 1] * silu_grad_f(ha[2 * j + 1]);
                    }
                }
                if (C::HAS_BIAS) add_bias_chunk(v, bias_w, wc);
                if (E == EPI_BIAS_DROPOUT_RES) {
                    float rv[32];
#pragma unroll
                    for (int i = 0; i < 4; ++i) unpack_bf16x8(hnext[i], rv + 8 * i);
                    if (c + C::EPI_SETS < C::OBN / 32) {  // prefetch the next chunk of the residual
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int n = nc + 32 * C::EPI_SETS + 8 * i;
                            hnext[i] = (row < M && n < N)
                                           ? ldg_nc_v4(args.aux + static_cast<size_t>(row) * args.ld_aux + n)
                                           : make_uint4(0, 0, 0, 0);
                        }
                    }
                    // element index of column nc of this row; a multiple of 4 (N % 8 == 0)
                    const unsigned long long q0 = (static_cast<unsigned long long>(row) * N + nc) >> 2;
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        const uint32_t kb = dropout_keep4(args.drop, q0 + g);
#pragma unroll
                        for (int w = 0; w < 4; ++w)
                            v[4 * g + w] = rv[4 * g + w] + (((kb >> w) & 1u) ? v[4 * g + w] * args.drop.scale : 0.0f);
                    }
                }
                float cs0 = 0.0f;  // GELU' epilogues: column sum of this warp's 32 rows, column nc + lane
                if (E == EPI_DGELU) {
                    if (c + 3 * C::EPI_SETS < C::OBN / 32 && row < M && nc + 96 * C::EPI_SETS < N)  // three ahead into L2
                        prefetch_l2(args.aux + static_cast<size_t>(row) * args.ld_aux + nc + 96 * C::EPI_SETS);
                    // dH = dG GELU'(H), two columns at a time (constant indices into gpre only)
                    auto apply = [&](const f32x2_t (&g)[16]) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            f2_unpack(f2_mul(f2_pack(v[2 * j], v[2 * j + 1]), g[j]), v[2 * j], v[2 * j + 1]);
                    };
                    if (PRE_N > 0 && wc == 0) {
                        apply(gpre[0]);
                    } else if (PRE_N > 1 && wc == 1) {
                        apply(gpre[PRE_N > 1 ? 1 : 0]);
                    } else {
                        float hv[32];
#pragma unroll
                        for (int i = 0; i < 4; ++i) unpack_bf16x8(hnext[i], hv + 8 * i);
                        if (c + C::EPI_SETS < C::OBN / 32) {  // the next chunk of H into registers
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int n = nc + 32 * C::EPI_SETS + 8 * i;
                                hnext[i] = (row < M && n < N)
                                               ? ldg_nc_v4(args.aux + static_cast<size_t>(row) * args.ld_aux + n)
                                               : make_uint4(0, 0, 0, 0);
                            }
                        }
                        f32x2_t g[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) g[j] = gelu_grad_fast_pair(f2_pack(hv[2 * j], hv[2 * j + 1]));
                        apply(g);
                    }
                    if (args.colsum_rows) {  // this warp's 32 rows of dH, summed per column
                        float cs[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) cs[j] = v[j];
                        warp_column_sums(cs, lane);
                        cs0 = cs[0];
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) p0[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                if (E == EPI_BIAS_GELU) {  // G = GELU(H) of the rounded H, as in every path
#pragma unroll
                    for (int j = 0; j < 16; ++j) p1[j] = gelu_bf16x2(p0[j]);
                }

                const uint32_t buf0 = s_epi + ((ewarp * C::STG_BUFS + sel) * C::NOUT) * C::STG_BYTES;
                if (lane == 0) bulk_wait_group_read<C::STG_BUFS - 1>();  // the store that last used it has read it
                __syncwarp();
                stage_row_sw64(buf0, lane, p0);
                if (C::NOUT >= 2) stage_row_sw64(buf0 + C::STG_BYTES, lane, p1);
                if (C::NOUT >= 3) stage_row_sw64(buf0 + 2 * C::STG_BYTES, lane, p2);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&args.tmD0, nc, row_blk, buf0);
                    if (C::NOUT >= 2) tma_store_2d(&args.tmD1, nc, row_blk, buf0 + C::STG_BYTES);
                    if (C::NOUT >= 3) tma_store_2d(&args.tmD2, nc, row_blk, buf0 + 2 * C::STG_BYTES);
                    bulk_commit_group();
                }
                if (C::STG_BUFS == 2) sel ^= 1u;
                // the column sums go out after the staging fence and the store
                if (E == EPI_DGELU && args.colsum_rows && nc + lane < N)
                    args.colsum_rows[static_cast<size_t>(row_blk >> 5) * N + nc + lane] = cs0;
            }
            if (C::NACC == 2) {
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            } else {
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_group<0>();
    }

    tc_fence_before();
    if (CG == 2)
        cluster_sync();  // the even CTA's MMAs touch both CTAs' TMEM and shared memory
    else
        __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        if (CG == 2)
            tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// Host-side launcher, instantiated once per GEMM flavour in its own translation unit.
// `grid` counts CTAs (a multiple of CG).
template <int BN, bool A_MN, bool B_MN, int EPI, int CG>
cudaError_t launch_umma_gemm(const GemmArgs& args, int grid, cudaStream_t stream)
{
    using C = GemmCfg<BN, A_MN, B_MN, EPI, CG>;
    auto kern = umma_gemm_kernel<BN, A_MN, B_MN, EPI, CG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (CG == 2 && C::HALVES == 2 && args.cluster_pairs == 2) ? 4 : CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int BN, bool A_MN, bool B_MN, int EPI, int CG>
int umma_gemm_max_clusters(int cluster, int num_sms)
{
    using C = GemmCfg<BN, A_MN, B_MN, EPI, CG>;
    auto kern = umma_gemm_kernel<BN, A_MN, B_MN, EPI, CG>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM_BYTES)) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms / cluster * cluster), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace mlp
