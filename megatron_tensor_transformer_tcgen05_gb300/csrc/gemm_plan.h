// gemm_plan.h -- how one GEMM of the family runs: tile shape, CTAs per MMA, pairs per
// cluster, work tiles, split tail and grid. Pure host arithmetic (no CUDA calls), shared by
// the library's launcher and its CPU tests.
#pragma once
#include <algorithm>
#include <cmath>
#include <cstddef>

namespace mlp {

// What an epilogue does per output element, for the tile-width rule: round the accumulator
// (+ bias); math on it (GELU, GELU', dropout and residual); or read two saved activations and
// write two outputs (the SwiGLU derivative).
enum EpiWeight : int { kEpiRound = 0, kEpiMath = 1, kEpiTwoAux = 2 };
// CTA pairs take 512-wide tiles (25% fewer operand bytes per FLOP than 256-wide; one
// accumulator, so each tile's epilogue delays the next tile's MMAs by about half an
// epilogue) when N allows and the K loop is long enough to hide that delay: K >= 2048 for
// the epilogues that only round the accumulator (+ bias), K >= 4096 for those with math.
// The two-input, two-output epilogue keeps 256-wide tiles with two accumulators at any K
// (its read-out on one 512-column accumulator measured 10% slower at K = 12288).
constexpr int kWideMinK = 2048, kWideMinKMath = 4096;
// Each part of a split tile runs at least this many 64-deep k blocks.
constexpr int kMinSplitKb = 16;

struct GemmPlan {
    int bn = 128;             // output columns per work tile (the kernel's BN)
    int cg = 1;               // CTAs per MMA: 1, or 2 (a pair, cta_group::2)
    int cluster_pairs = 1;    // pairs per cluster: 2 = 512 x 512 work tiles, B multicast
    int tm = 128;             // rows per work tile
    int units = 0;            // work units that run at once: CTAs, pairs or clusters
    long long tiles = 0;      // work tiles
    int split_tiles = 0;      // the last split_tiles tiles run as split_k K ranges each
    int split_k = 1;
    int grid = 0;             // CTAs launched
    int n_fastest = 0;        // tile order: 0 = M index fastest, 1 = N index fastest
    int raster_group = 1;     // tiles of the fast index per group
};

// Whether a GEMM of these sizes would take 512-wide pair tiles, so that clusters of four
// (whose residency the caller looks up) are worth considering.
inline bool plan_wants_wide(int M, int N, int K, int bn, int weight)
{
    return bn >= 256 && M > 128 && N % 512 == 0 && weight != kEpiTwoAux &&
           K >= (weight == kEpiMath ? kWideMinKMath : kWideMinK);
}

// The plan for D[M,N] = sum_k A[m,k] B[n,k] on num_sms SMs.
//   bn: 256 when the N extent the entry point tiles by is a multiple of 256, else 128.
//   weight: the epilogue's EpiWeight.
//   splittable: the split-tail fixup can finish this epilogue.
//   quads: clusters of four CTAs that fit at once (0: unknown or none).
//   split_ws_bytes: room for split parts (0: no split).
inline GemmPlan plan_gemm(int M, int N, int K, int bn, int weight, bool splittable, int num_sms, int quads,
                          size_t split_ws_bytes)
{
    GemmPlan p;
    // Keep the smaller operand resident in L2 and stream the larger one once: with A (M*K)
    // no larger than B (N*K), sweep M fastest so every concurrent tile shares one B block;
    // otherwise sweep N fastest so they share one A block.
    p.n_fastest = M > N ? 1 : 0;
    const bool pairs = bn >= 256 && M > 128;
    if (pairs && plan_wants_wide(M, N, K, bn, weight)) bn = 512;
    p.bn = bn;
    p.cg = pairs ? 2 : 1;
    p.tm = pairs ? 256 : 128;
    p.units = pairs ? num_sms / 2 : num_sms;
    // Two pairs per cluster when the rows make whole 512-row tiles and clusters of four
    // cover at least 90% of the SMs (36 of 38 on a GB300: the multicast saves enough
    // operand traffic that the power-capped clock rises ~5%, more than the idle SMs cost).
    const int q = std::min(quads, num_sms / 4);
    if (bn == 512 && ((M + 255) / 256) % 2 == 0 && q > 0 && 4 * q * 10 >= 9 * num_sms) {
        p.cluster_pairs = 2;
        p.tm = 512;
        p.units = q;
    }
    // Group ~sqrt(units) tiles of the fast dimension: a wave then touches the fewest distinct
    // operand blocks.
    p.raster_group = static_cast<int>(std::lround(std::sqrt(static_cast<double>(p.units > 1 ? p.units : 1))));
    p.tiles = static_cast<long long>((M + p.tm - 1) / p.tm) * ((N + bn - 1) / bn);
    // Split tail: the tiles % units tiles of the short last round (all tiles when there are
    // fewer than units) are cut into as many K ranges as keep the parts within one round of
    // units, each of at least kMinSplitKb k blocks, within the workspace; fewer than two
    // parts: no split.
    if (splittable && split_ws_bytes > 0 && p.tiles > 0 && p.units > 1) {
        const long long rem = p.tiles % p.units;
        if (rem > 0) {
            const int num_kb = (K + 63) / 64;
            long long sk = p.units / rem;
            sk = std::min<long long>(sk, num_kb / kMinSplitKb);
            const size_t part_bytes = static_cast<size_t>(p.tm) * bn * 4;
            sk = std::min<long long>(sk, static_cast<long long>(split_ws_bytes / (part_bytes * static_cast<size_t>(rem))));
            if (sk >= 2) {
                p.split_tiles = static_cast<int>(rem);
                p.split_k = static_cast<int>(sk);
            }
        }
    }
    const long long work = p.tiles - p.split_tiles + static_cast<long long>(p.split_tiles) * p.split_k;
    const long long active = std::min<long long>(work, p.units);
    p.grid = static_cast<int>(active * p.cg * p.cluster_pairs);
    return p;
}

}  // namespace mlp
