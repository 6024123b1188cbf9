// mlp_tp_api.cu -- the C ABI of include/mlp_tp.h: argument checks, TMA tensor maps, launch
// sequencing of the MLP block's forward (2 kernels) and backward (6 kernels), of its dropout,
// SwiGLU and GELU-recompute variants and of the attention block (3 + 7 kernels), and the
// device status word that bounded waits report into.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "attn_args.h"
#include "colsum.cuh"
#include "dropout.cuh"
#include "gemm_args.h"
#include "gemm_plan.h"
#include "mlp_tp.h"
#include "sm103_ptx.cuh"

namespace mlp {

// Device status words: [0] = code of the first bounded wait that gave up (0 = none);
// [1..4] = where: block index, thread index, tile, k block (or stage) of that wait.
constexpr int kStatusWords = 8;
__device__ int g_device_status[kStatusWords];

// Limit for every bounded wait inside the GEMMs: one wait never lasts longer than one
// tile's main loop (well under a millisecond), so two seconds only trips on a real stall.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Kernel launches issued by the library since it was loaded (all devices and streams).
static std::atomic<long long> g_launches{0};
static void note_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// Split tail workspace: room for one fp32 part per unit of up to 160 SMs (a part is a
// 512 x 512 tile for a cluster of four, 256 x 512 for a CTA pair, at most 128 x 256 for one
// CTA: at most 256 KB per SM).
constexpr size_t kSplitWsBytes = size_t(160) * 256 * 1024;
// 512-wide pair tiles run two pairs per cluster (512 x 512 work tiles, each stage's B fetched
// once and multicast to both pairs) when gemm_plan.h's rule allows; off, every GEMM uses pairs.
constexpr bool kClusterPairs = true;

// Clusters of four CTAs of this 512-wide flavour that fit at once, looked up once per SM count.
template <bool A_MN, bool B_MN, int EPI>
static int quad_clusters(int num_sms)
{
    static std::mutex mu;
    static int for_sms = -1, clusters = 0;
    std::lock_guard<std::mutex> lk(mu);
    if (for_sms != num_sms) {
        clusters = umma_gemm_max_clusters<512, A_MN, B_MN, EPI, 2>(4, num_sms);
        for_sms = num_sms;
    }
    return clusters;
}
// The split region of a workspace: none when there are no tokens (no GEMM runs then).
static size_t split_ws_bytes(long long tokens) { return tokens > 0 ? kSplitWsBytes : 0; }

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    int* status = nullptr;
};

constexpr int kMaxDevices = 64;
static DeviceInfo g_dev[kMaxDevices];
static std::mutex g_dev_mu;
static int g_last_status[kStatusWords] = {0};

static mlp_status device_info(DeviceInfo** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLP_ECUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MLP_ECUDA;
        d.supported = (major == 10 && minor == 3);
        d.num_sms = sms;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return MLP_ECUDA;
        d.status = static_cast<int*>(p);  // the first of kStatusWords words
        d.ready = true;
    }
    if (!d.supported) return MLP_EUNSUPPORTED;
    *out = &d;
    return MLP_OK;
}

// ---- TMA tensor maps -------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major bf16 matrix [outer, inner]; a box of box_inner x box_outer elements.
static bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                     uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand maps: K-major [rows, K] -> box 64 (K) x rows_box; MN-major [K, MN] -> box 64 x 64.
static bool map_kmajor(CUtensorMap* m, const void* p, uint64_t K, uint64_t rows, uint32_t rows_box)
{
    return make_map(m, p, K, rows, 64, rows_box, CU_TENSOR_MAP_SWIZZLE_128B);
}
static bool map_mnmajor(CUtensorMap* m, const void* p, uint64_t MN, uint64_t K)
{
    return make_map(m, p, MN, K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
}
static bool map_store(CUtensorMap* m, const void* p, uint64_t cols, uint64_t rows)
{
    return make_map(m, p, cols, rows, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Tile width along N: 256 when the N extent splits into whole 256-wide tiles, else 128.
static int tile_n(int n) { return (n % 256 == 0) ? 256 : 128; }

// CTA pairs (256-row tiles, cta_group::2) for 256- and 512-wide tiles over more than 128 rows.
static bool use_pairs(int M, int BN) { return BN >= 256 && M > 128; }

// Rows of a K-major B operand one CTA loads per stage: half the tile width for a pair.
static uint32_t kmajor_b_box(int M, int BN) { return use_pairs(M, BN) ? 128 : BN; }

// Where a GEMM may put the parts of split tiles, and the output the fixup then writes
// (row-major [M, N], the GEMM's only output).
struct SplitOut {
    float* ws = nullptr;
    size_t ws_bytes = 0;
    void* out = nullptr;
    void* out1 = nullptr;  // G of the bias + GELU epilogue
};

// tiles_as_math: plan the tile shapes as for an epilogue with math (-1: by EPI). The GELU
// recompute's up-projection (bias only) takes the bias + GELU GEMM's plan, so that its H is
// bitwise the H of the forward that keeps G.
template <bool A_MN, bool B_MN, int EPI>
static cudaError_t gemm(GemmArgs& g, int BN, int num_sms, cudaStream_t s, const SplitOut* so = nullptr,
                        int tiles_as_math = -1)
{
    // the transform flavours finish like their plain / bias epilogue
    constexpr int kEpiB = (EPI == EPI_PLAIN_GA) ? EPI_PLAIN : (EPI == EPI_BIAS_GA) ? EPI_BIAS : EPI;
    constexpr bool kSplittable =
        (kEpiB == EPI_PLAIN || kEpiB == EPI_BIAS || kEpiB == EPI_BIAS_GELU || kEpiB == EPI_DGELU);
    // the SwiGLU derivative never takes 512-wide tiles (gemm_plan.h), so none is built for it
    constexpr bool kMayWide = kEpiB != EPI_DSWIGLU;
    const int weight = tiles_as_math >= 0 ? (tiles_as_math != 0 ? kEpiMath : kEpiRound)
                       : (kEpiB == EPI_PLAIN || kEpiB == EPI_BIAS) ? kEpiRound
                       : kMayWide                                   ? kEpiMath
                                                                    : kEpiTwoAux;
    if (!kSplittable || !so || !so->ws || !so->out) so = nullptr;
    int quads = 0;  // looked up only when two-pair clusters are possible
    if constexpr (kMayWide)
        if (kClusterPairs && plan_wants_wide(g.M, g.N, g.K, BN, weight) && ((g.M + 255) / 256) % 2 == 0)
            quads = quad_clusters<A_MN, B_MN, EPI>(num_sms);
    const GemmPlan p = plan_gemm(g.M, g.N, g.K, BN, weight, kSplittable, num_sms, quads, so ? so->ws_bytes : 0);
    g.n_fastest = p.n_fastest;
    g.raster_group = p.raster_group;
    g.cluster_pairs = p.cluster_pairs;
    g.split_tiles = p.split_tiles;
    g.split_k = p.split_k;
    g.split_ws = p.split_tiles > 0 ? so->ws : nullptr;
    if (p.grid <= 0) return cudaSuccess;
    cudaError_t e;
    if (p.cg == 2) {
        if constexpr (kMayWide)
            e = p.bn == 512 ? launch_umma_gemm<512, A_MN, B_MN, EPI, 2>(g, p.grid, s)
                            : launch_umma_gemm<256, A_MN, B_MN, EPI, 2>(g, p.grid, s);
        else
            e = launch_umma_gemm<256, A_MN, B_MN, EPI, 2>(g, p.grid, s);
    } else
        e = p.bn == 256 ? launch_umma_gemm<256, A_MN, B_MN, EPI, 1>(g, p.grid, s)
                        : launch_umma_gemm<128, A_MN, B_MN, EPI, 1>(g, p.grid, s);
    if (e != cudaSuccess) return e;
    note_launches(1);
    if (p.split_tiles > 0) {
        e = launch_splitk_fixup(g, kEpiB, p.tm, p.bn, static_cast<__nv_bfloat16*>(so->out),
                                static_cast<__nv_bfloat16*>(so->out1), g.N, s);
        if (e != cudaSuccess) return e;
        note_launches(1);
    }
    return cudaSuccess;
}

// The SwiGLU up-projection: one 256-wide MMA per 128 output columns ([X A | X Wg]).
static cudaError_t gemm_dual(GemmArgs& g, int num_sms, cudaStream_t s)
{
    g.n_fastest = g.M > g.N ? 1 : 0;
    const bool pair = g.M > 128;
    const int units = pair ? num_sms / 2 : num_sms;
    g.raster_group = static_cast<int>(std::lround(std::sqrt(static_cast<double>(units > 1 ? units : 1))));
    const long long tiles = static_cast<long long>((g.M + (pair ? 255 : 127)) / (pair ? 256 : 128)) * ((g.N + 127) / 128);
    const int grid_units = static_cast<int>(tiles < units ? tiles : units);
    if (grid_units <= 0) return cudaSuccess;
    const cudaError_t e = pair ? launch_umma_gemm<256, false, true, EPI_SWIGLU, 2>(g, 2 * grid_units, s)
                               : launch_umma_gemm<256, false, true, EPI_SWIGLU, 1>(g, grid_units, s);
    if (e == cudaSuccess) note_launches(1);
    return e;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static mlp_status check_shape(int T, int h, int f, int t)
{
    if (T < 0 || h < 8 || f < 8 || t < 1) return MLP_EINVAL;
    if (h % 8 != 0 || f % 8 != 0 || f % t != 0 || (f / t) % 8 != 0) return MLP_ESHAPE;
    return MLP_OK;
}

static int colsum_splits(int T)
{
    int s = T / 512;
    return s < 1 ? 1 : (s > 16 ? 16 : s);
}

static size_t round256(size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); }

// ---- optional per-kernel timing (benchmarks) ---------------------------------------------
// When enabled, each call records a CUDA event on its stream before its first launch and
// after every launch; mlp_tp_timing_collect() turns the pairs into per-kernel milliseconds.

struct TimingMark {
    int kernel;
    cudaEvent_t start, stop;
};
static std::mutex g_tm_mu;
static bool g_timing = false;
static std::vector<TimingMark> g_marks;
static std::vector<cudaEvent_t> g_event_pool;

static cudaEvent_t take_event()
{
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

class CallTimer {
  public:
    explicit CallTimer(cudaStream_t s) : s_(s)
    {
        std::lock_guard<std::mutex> lk(g_tm_mu);
        on_ = g_timing;
        if (on_) {
            prev_ = take_event();
            on_ = prev_ != nullptr && cudaEventRecord(prev_, s_) == cudaSuccess;
        }
    }
    void mark(int kernel)
    {
        if (!on_) return;
        std::lock_guard<std::mutex> lk(g_tm_mu);
        cudaEvent_t e = take_event();
        if (!e || cudaEventRecord(e, s_) != cudaSuccess) {
            on_ = false;
            return;
        }
        g_marks.push_back({kernel, prev_, e});
        prev_ = e;
    }

  private:
    cudaStream_t s_;
    bool on_ = false;
    cudaEvent_t prev_ = nullptr;
};

}  // namespace mlp

using namespace mlp;

extern "C" {

const char* mlp_tp_status_string(mlp_status s)
{
    switch (s) {
    case MLP_OK: return "MLP_OK";
    case MLP_EINVAL: return "MLP_EINVAL: null pointer or non-positive size";
    case MLP_ESHAPE: return "MLP_ESHAPE: a size breaks the call's shape rules (f % t, multiples of 8, a % t, d)";
    case MLP_EALIGN: return "MLP_EALIGN: pointer not 16-byte aligned";
    case MLP_ECUDA: return "MLP_ECUDA: CUDA runtime error";
    case MLP_ETIMEOUT: return "MLP_ETIMEOUT: a device-side check failed (a bounded wait ran out, or see mlp_tp_last_device_code)";
    case MLP_EUNSUPPORTED: return "MLP_EUNSUPPORTED: current device is not sm_103";
    case MLP_EWORKSPACE: return "MLP_EWORKSPACE: workspace too small";
    }
    return "unknown mlp_status";
}

// Backward workspace: dH [T,f] bf16 | dH column sums per 32-row block [ceil(T/32), f] fp32 |
// dY column sums per row slice [slices, h] fp32 | split-tail parts (kSplitWsBytes), each
// region 256-byte aligned. The recompute backward uses the same layout (G is never stored).
static size_t ws_dh_bytes(int T, int f) { return round256(static_cast<size_t>(T) * f * 2); }
static size_t ws_rows_bytes(int T, int f) { return round256(static_cast<size_t>((T + 31) / 32) * f * 4); }
static size_t ws_dy_bytes(int T, int h) { return round256(static_cast<size_t>(colsum_splits(T)) * h * 4); }
static size_t bwd_ws_before_split(int T, int h, int f)
{
    return ws_dh_bytes(T, f) + ws_rows_bytes(T, f) + ws_dy_bytes(T, h);
}

size_t mlp_tp_workspace_bytes(int T, int h, int f, int t)
{
    if (check_shape(T, h, f, t) != MLP_OK) return 0;
    return bwd_ws_before_split(T, h, f) + split_ws_bytes(T);
}

size_t mlp_tp_forward_workspace_bytes(void) { return kSplitWsBytes; }

long long mlp_tp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"

namespace mlp {

// The forward pass; with `drop` set, GEMM 2's epilogue also applies dropout and adds the
// residual R, writing Z instead of Y. With G == NULL (the GELU recompute), GEMM 1 stores H
// alone and GEMM 2 reads H, turning each A tile into G = GELU(H) in shared memory.
static mlp_status forward_impl(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a, const mlp_bf16* B,
                               const mlp_bf16* b, const mlp_bf16* R, const DropoutParams* drop, int T, int h,
                               int f, int t, mlp_bf16* H, mlp_bf16* G, mlp_bf16* Y, void* workspace,
                               size_t workspace_bytes, void* cuda_stream)
{
    const bool recompute = (G == nullptr);
    mlp_status st = check_shape(T, h, f, t);
    if (st != MLP_OK) return st;
    // Token-indexed buffers may be NULL only when there are no tokens.
    if (!A || !a || !B || !b || (T > 0 && (!X || !H || !Y || (drop && !R)))) return MLP_EINVAL;
    const void* ptrs[] = {X, A, a, B, b, H, G, Y, R};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MLP_EALIGN;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MLP_EALIGN;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != MLP_OK) return st;
    if (T == 0) return MLP_OK;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const SplitOut so{static_cast<float*>(workspace), workspace ? workspace_bytes : 0, Y, nullptr};
    const int fs = f / t;
    const int bn_f = tile_n(fs), bn_h = tile_n(h);
    CallTimer timer(s);

    // GEMM 1: H = X*A + a, G = GELU(H) (H alone when recomputing). N-tiles never straddle a
    // shard when f/t % BN == 0.
    GemmArgs g1{};
    if (!map_kmajor(&g1.tmA, X, h, T, 128) || !map_mnmajor(&g1.tmB, A, f, h) ||
        !map_store(&g1.tmD0, H, f, T) || (!recompute && !map_store(&g1.tmD1, G, f, T)))
        return MLP_ECUDA;
    if (recompute) g1.tmD1 = g1.tmD0;
    g1.M = T; g1.N = f; g1.K = h;
    g1.bias = reinterpret_cast<const __nv_bfloat16*>(a);
    g1.status = dev->status;
    g1.timeout_ns = kWaitLimitNs;
    const SplitOut so1{static_cast<float*>(workspace), workspace ? workspace_bytes : 0, H, G};
    const cudaError_t e1 = recompute ? gemm<false, true, EPI_BIAS>(g1, bn_f, dev->num_sms, s, &so1, 1)
                                     : gemm<false, true, EPI_BIAS_GELU>(g1, bn_f, dev->num_sms, s, &so1);
    if (e1 != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_FWD_UP);

    // GEMM 2: Y = sum over shards of G_i*B_i, + b (then dropout and + R). One accumulator
    // over K = f. Recomputing: the A operand is H, and G = GELU(H) is formed on chip.
    GemmArgs g2{};
    if (!map_kmajor(&g2.tmA, recompute ? H : G, f, T, 128) || !map_mnmajor(&g2.tmB, B, h, f) ||
        !map_store(&g2.tmD0, Y, h, T))
        return MLP_ECUDA;
    g2.tmD1 = g2.tmD0;
    g2.M = T; g2.N = h; g2.K = f;
    g2.bias = reinterpret_cast<const __nv_bfloat16*>(b);
    g2.status = dev->status;
    g2.timeout_ns = kWaitLimitNs;
    cudaError_t e;
    if (drop) {
        g2.aux = reinterpret_cast<const __nv_bfloat16*>(R);
        g2.ld_aux = h;
        g2.drop = *drop;
        e = gemm<false, true, EPI_BIAS_DROPOUT_RES>(g2, bn_h, dev->num_sms, s);
    } else if (recompute) {
        e = gemm<false, true, EPI_BIAS_GA>(g2, bn_h, dev->num_sms, s, &so);
    } else {
        e = gemm<false, true, EPI_BIAS>(g2, bn_h, dev->num_sms, s, &so);
    }
    if (e != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_FWD_DOWN);
    return MLP_OK;
}

// Dropout parameters from p in [0, 1): keep when the top 24 bits of the element's Philox
// word are >= floor(p * 2^24); kept values are scaled by 1 / (1 - p).
static bool make_dropout(double p, unsigned long long seed, unsigned long long offset, DropoutParams* d)
{
    if (!(p >= 0.0 && p < 1.0)) return false;
    d->seed = seed;
    d->offset = offset;
    d->p24 = static_cast<uint32_t>(std::floor(p * 16777216.0));
    d->scale = static_cast<float>(1.0 / (1.0 - p));
    return true;
}

}  // namespace mlp

extern "C" {

mlp_status mlp_tp_forward(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a, const mlp_bf16* B,
                          const mlp_bf16* b, int T, int h, int f, int t, mlp_bf16* H, mlp_bf16* G,
                          mlp_bf16* Y, void* workspace, size_t workspace_bytes, void* cuda_stream)
{
    if (T > 0 && !G) return MLP_EINVAL;
    return forward_impl(X, A, a, B, b, nullptr, nullptr, T, h, f, t, H, G, Y, workspace, workspace_bytes,
                        cuda_stream);
}

mlp_status mlp_tp_forward_recompute(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a, const mlp_bf16* B,
                                    const mlp_bf16* b, int T, int h, int f, int t, mlp_bf16* H, mlp_bf16* Y,
                                    void* workspace, size_t workspace_bytes, void* cuda_stream)
{
    return forward_impl(X, A, a, B, b, nullptr, nullptr, T, h, f, t, H, nullptr, Y, workspace, workspace_bytes,
                        cuda_stream);
}

mlp_status mlp_tp_forward_residual_dropout(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a,
                                           const mlp_bf16* B, const mlp_bf16* b, const mlp_bf16* R, int T, int h,
                                           int f, int t, double p, unsigned long long seed,
                                           unsigned long long offset, mlp_bf16* H, mlp_bf16* G, mlp_bf16* Z,
                                           void* cuda_stream)
{
    DropoutParams d;
    if (!make_dropout(p, seed, offset, &d)) return MLP_EINVAL;
    if (T > 0 && !G) return MLP_EINVAL;
    return forward_impl(X, A, a, B, b, R, &d, T, h, f, t, H, G, Z, nullptr, 0, cuda_stream);
}

mlp_status mlp_tp_dropout_backward(const mlp_bf16* dZ, int T, int h, double p, unsigned long long seed,
                                   unsigned long long offset, mlp_bf16* dY, void* cuda_stream)
{
    DropoutParams d;
    if (!make_dropout(p, seed, offset, &d) || T < 0 || h < 8) return MLP_EINVAL;
    if (h % 8 != 0) return MLP_ESHAPE;
    if (T > 0 && (!dZ || !dY)) return MLP_EINVAL;
    if (!aligned16(dZ) || !aligned16(dY)) return MLP_EALIGN;
    DeviceInfo* dev = nullptr;
    mlp_status st = device_info(&dev);
    if (st != MLP_OK) return st;
    if (T == 0) return MLP_OK;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    CallTimer timer(s);
    const long long n8 = static_cast<long long>(T) * h / 8;
    long long blocks = (n8 + 255) / 256;
    const long long cap = static_cast<long long>(dev->num_sms) * 8;
    if (blocks > cap) blocks = cap;
    dropout_backward_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(dZ), n8, d,
                                                                      reinterpret_cast<__nv_bfloat16*>(dY));
    if (cudaGetLastError() != cudaSuccess) return MLP_ECUDA;
    note_launches(1);
    timer.mark(MLP_K_DROPOUT_BWD);
    return MLP_OK;
}

}  // extern "C"

namespace mlp {

// The backward pass. With G == NULL (the GELU recompute) GEMM 6 reads H, turning each A tile
// into G = GELU(H) in shared memory: G is neither kept from the forward nor stored here.
static mlp_status backward_impl(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* B, const mlp_bf16* H,
                                const mlp_bf16* G, const mlp_bf16* dY, int T, int h, int f, int t, mlp_bf16* dX,
                                mlp_bf16* dA, mlp_bf16* dB, float* da, float* db, void* workspace,
                                size_t workspace_bytes, void* cuda_stream)
{
    const bool recompute = (G == nullptr);
    mlp_status st = check_shape(T, h, f, t);
    if (st != MLP_OK) return st;
    // Token-indexed buffers may be NULL only when there are no tokens.
    if (!A || !B || !dA || !dB || !da || !db || !workspace || (T > 0 && (!X || !H || !dY || !dX)))
        return MLP_EINVAL;
    const void* ptrs[] = {X, A, B, H, G, dY, dX, dA, dB, da, db};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MLP_EALIGN;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MLP_EALIGN;
    if (workspace_bytes < mlp_tp_workspace_bytes(T, h, f, t)) return MLP_EWORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != MLP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

    if (T == 0) {  // no tokens: every gradient is an empty sum
        if (cudaMemsetAsync(dA, 0, static_cast<size_t>(h) * f * 2, s) != cudaSuccess ||
            cudaMemsetAsync(dB, 0, static_cast<size_t>(f) * h * 2, s) != cudaSuccess ||
            cudaMemsetAsync(da, 0, static_cast<size_t>(f) * 4, s) != cudaSuccess ||
            cudaMemsetAsync(db, 0, static_cast<size_t>(h) * 4, s) != cudaSuccess)
            return MLP_ECUDA;
        return MLP_OK;
    }
    const int fs = f / t;
    const int bn_f = tile_n(fs), bn_h = tile_n(h);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    mlp_bf16* dH = reinterpret_cast<mlp_bf16*>(ws);
    float* split_ws = reinterpret_cast<float*>(ws + bwd_ws_before_split(T, h, f));
    float* dh_rows = reinterpret_cast<float*>(ws + ws_dh_bytes(T, f));
    float* dy_part = reinterpret_cast<float*>(ws + ws_dh_bytes(T, f) + ws_rows_bytes(T, f));
    const int nsplit = colsum_splits(T);
    CallTimer timer(s);

    // GEMM 3: dH = (dY*B^T) (.) GELU'(H); B [f,h] is K-major for N = f, K = h.
    GemmArgs g3{};
    if (!map_kmajor(&g3.tmA, dY, h, T, 128) || !map_kmajor(&g3.tmB, B, h, f, kmajor_b_box(T, bn_f)) ||
        !map_store(&g3.tmD0, dH, f, T))
        return MLP_ECUDA;
    g3.tmD1 = g3.tmD0;
    g3.M = T; g3.N = f; g3.K = h;
    g3.aux = reinterpret_cast<const __nv_bfloat16*>(H);
    g3.ld_aux = f;
    g3.colsum_rows = dh_rows;  // da's per-32-row partial sums come out of this epilogue
    g3.status = dev->status;
    g3.timeout_ns = kWaitLimitNs;
    const SplitOut so3{split_ws, kSplitWsBytes, dH, nullptr};
    if (gemm<false, false, EPI_DGELU>(g3, bn_f, dev->num_sms, s, &so3) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_BWD_DH);

    // GEMM 4: dX = sum over shards of dH_i*A_i^T; A [h,f] is K-major for N = h, K = f.
    GemmArgs g4{};
    if (!map_kmajor(&g4.tmA, dH, f, T, 128) || !map_kmajor(&g4.tmB, A, f, h, kmajor_b_box(T, bn_h)) ||
        !map_store(&g4.tmD0, dX, h, T))
        return MLP_ECUDA;
    g4.tmD1 = g4.tmD0;
    g4.M = T; g4.N = h; g4.K = f;
    g4.status = dev->status;
    g4.timeout_ns = kWaitLimitNs;
    const SplitOut so4{split_ws, kSplitWsBytes, dX};
    if (gemm<false, false, EPI_PLAIN>(g4, bn_h, dev->num_sms, s, &so4) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_BWD_DX);

    // GEMM 5: dA = X^T*dH (M = h, N = f, K = T), both operands MN-major.
    GemmArgs g5{};
    if (!map_mnmajor(&g5.tmA, X, h, T) || !map_mnmajor(&g5.tmB, dH, f, T) ||
        !map_store(&g5.tmD0, dA, f, h))
        return MLP_ECUDA;
    g5.tmD1 = g5.tmD0;
    g5.M = h; g5.N = f; g5.K = T;
    g5.status = dev->status;
    g5.timeout_ns = kWaitLimitNs;
    const SplitOut so5{split_ws, kSplitWsBytes, dA};
    if (gemm<true, true, EPI_PLAIN>(g5, bn_f, dev->num_sms, s, &so5) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_BWD_DA);

    // GEMM 6: dB = G^T*dY (M = f, N = h, K = T), both operands MN-major; recomputing, the A
    // operand is H and G = GELU(H) is formed on chip.
    GemmArgs g6{};
    if (!map_mnmajor(&g6.tmA, recompute ? H : G, f, T) || !map_mnmajor(&g6.tmB, dY, h, T) ||
        !map_store(&g6.tmD0, dB, h, f))
        return MLP_ECUDA;
    g6.tmD1 = g6.tmD0;
    g6.M = f; g6.N = h; g6.K = T;
    g6.status = dev->status;
    g6.timeout_ns = kWaitLimitNs;
    const SplitOut so6{split_ws, kSplitWsBytes, dB};
    const cudaError_t e6 = recompute ? gemm<true, true, EPI_PLAIN_GA>(g6, bn_h, dev->num_sms, s, &so6)
                                     : gemm<true, true, EPI_PLAIN>(g6, bn_h, dev->num_sms, s, &so6);
    if (e6 != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_BWD_DB);

    // Bias gradients: db's partial column sums over row slices of dY (da's came out of the
    // dH GEMM), then one pass adding both sets of partials in a fixed order.
    const int strips_h = (h + kColsumStrip - 1) / kColsumStrip;
    colsum_partial_kernel<<<dim3(strips_h, nsplit), kColsumThreads, 0, s>>>(
        nullptr, 0, reinterpret_cast<const __nv_bfloat16*>(dY), h, T, nsplit, dy_part);
    if (cudaGetLastError() != cudaSuccess) return MLP_ECUDA;
    note_launches(1);
    timer.mark(MLP_K_COLSUM_PARTIAL);
    bias_grad_finalize_kernel<<<(f + h + 255) / 256, 256, 0, s>>>(dh_rows, (T + 31) / 32, f, dy_part, nsplit, h,
                                                                  da, db);
    if (cudaGetLastError() != cudaSuccess) return MLP_ECUDA;
    note_launches(1);
    timer.mark(MLP_K_COLSUM_FINAL);
    return MLP_OK;
}

}  // namespace mlp

extern "C" {

mlp_status mlp_tp_backward(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* B, const mlp_bf16* H,
                           const mlp_bf16* G, const mlp_bf16* dY, int T, int h, int f, int t,
                           mlp_bf16* dX, mlp_bf16* dA, mlp_bf16* dB, float* da, float* db,
                           void* workspace, size_t workspace_bytes, void* cuda_stream)
{
    if (T > 0 && !G) return MLP_EINVAL;
    return backward_impl(X, A, B, H, G, dY, T, h, f, t, dX, dA, dB, da, db, workspace, workspace_bytes, cuda_stream);
}

size_t mlp_tp_recompute_workspace_bytes(int T, int h, int f, int t) { return mlp_tp_workspace_bytes(T, h, f, t); }

mlp_status mlp_tp_backward_recompute(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* B, const mlp_bf16* H,
                                     const mlp_bf16* dY, int T, int h, int f, int t, mlp_bf16* dX, mlp_bf16* dA,
                                     mlp_bf16* dB, float* da, float* db, void* workspace, size_t workspace_bytes,
                                     void* cuda_stream)
{
    return backward_impl(X, A, B, H, nullptr, dY, T, h, f, t, dX, dA, dB, da, db, workspace, workspace_bytes,
                         cuda_stream);
}

mlp_status mlp_tp_query_device_status(void* cuda_stream)
{
    DeviceInfo* dev = nullptr;
    mlp_status st = device_info(&dev);
    if (st != MLP_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return MLP_ECUDA;
    int v[kStatusWords] = {0};
    if (cudaMemcpy(v, dev->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MLP_ECUDA;
    if (v[0] != 0) {
        for (int i = 0; i < kStatusWords; ++i) g_last_status[i] = v[i];
        const int zero[kStatusWords] = {0};
        if (cudaMemcpy(dev->status, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return MLP_ECUDA;
        return MLP_ETIMEOUT;
    }
    return MLP_OK;
}

int mlp_tp_last_device_code(void) { return g_last_status[0]; }

int mlp_tp_last_device_where(int* block, int* thread, int* tile, int* kblock)
{
    if (block) *block = g_last_status[1];
    if (thread) *thread = g_last_status[2];
    if (tile) *tile = g_last_status[3];
    if (kblock) *kblock = g_last_status[4];
    return g_last_status[0];
}

mlp_status mlp_tp_timing_enable(int on)
{
    std::lock_guard<std::mutex> lk(g_tm_mu);
    g_timing = on != 0;
    return MLP_OK;
}

mlp_status mlp_tp_timing_collect(double* ms, int* counts)
{
    if (!ms || !counts) return MLP_EINVAL;
    std::lock_guard<std::mutex> lk(g_tm_mu);
    for (int k = 0; k < MLP_NUM_KERNELS; ++k) {
        ms[k] = 0.0;
        counts[k] = 0;
    }
    mlp_status st = MLP_OK;
    for (const TimingMark& m : g_marks) {
        float t = 0.f;
        if (cudaEventSynchronize(m.stop) != cudaSuccess || cudaEventElapsedTime(&t, m.start, m.stop) != cudaSuccess)
            st = MLP_ECUDA;
        if (m.kernel >= 0 && m.kernel < MLP_NUM_KERNELS) {
            ms[m.kernel] += t;
            counts[m.kernel] += 1;
        }
    }
    // Every event appears once as a stop; starts are either a previous stop or a call's
    // first event, which is never a stop. Return each exactly once to the pool.
    std::vector<cudaEvent_t> seen;
    for (const TimingMark& m : g_marks) {
        seen.push_back(m.start);
        seen.push_back(m.stop);
    }
    std::sort(seen.begin(), seen.end());
    seen.erase(std::unique(seen.begin(), seen.end()), seen.end());
    for (cudaEvent_t e : seen) g_event_pool.push_back(e);
    g_marks.clear();
    return st;
}

const char* mlp_tp_kernel_name(int kernel)
{
    static const char* names[MLP_NUM_KERNELS] = {
        "gemm_fwd_up (H=XA+a, G=GELU(H))", "gemm_fwd_down (Y=GB+b)", "gemm_bwd_dh (dH=dY B^T * GELU'(H))",
        "gemm_bwd_dx (dX=dH A^T)",          "gemm_bwd_da (dA=X^T dH)", "gemm_bwd_db (dB=G^T dY)",
        "colsum_partial (db)",              "bias_grad_finalize (da, db)", "dropout_backward (dY)",
        "attn gemm_qkv (QKV=X Wqkv)",       "attn_fwd (C, L per head)",    "attn gemm_out (Y=C Wo)",
        "attn gemm_dc (dC=dY Wo^T)",        "attn gemm_dwo (dWo=C^T dY)",  "attn_bwd_dot (D=rowsum dC*C)",
        "attn_bwd_dq (dQ)",                 "attn_bwd_dkdv (dK, dV)",      "attn gemm_dx (dX=dQKV Wqkv^T)",
        "attn gemm_dwqkv (dWqkv=X^T dQKV)"};
    return (kernel >= 0 && kernel < MLP_NUM_KERNELS) ? names[kernel] : "unknown";
}

}  // extern "C"

namespace mlp {

// Waits on a barrier whose phase nothing completes; the bounded wait must give up.
__global__ void selftest_wait_kernel(int* status, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, status, limit_ns, DEV_TIMEOUT_SELFTEST);
}

}  // namespace mlp

extern "C" mlp_status mlp_tp_selftest_wait_timeout(unsigned long long limit_ns, void* cuda_stream)
{
    DeviceInfo* dev = nullptr;
    mlp_status st = device_info(&dev);
    if (st != MLP_OK) return st;
    if (limit_ns > 10000000000ull) return MLP_EINVAL;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(cuda_stream)>>>(dev->status, limit_ns);
    if (cudaGetLastError() != cudaSuccess) return MLP_ECUDA;
    note_launches(1);
    return MLP_OK;
}

// ---- SwiGLU variant of the block ----------------------------------------------------------

extern "C" size_t mlp_tp_swiglu_workspace_bytes(int T, int h, int f, int t)
{
    if (check_shape(T, h, f, t) != MLP_OK) return 0;
    return 2 * round256(static_cast<size_t>(T) * f * 2) + split_ws_bytes(T);  // dHa, dHg, split-tail parts
}

extern "C" mlp_status mlp_tp_swiglu_forward(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* Wg,
                                            const mlp_bf16* B, int T, int h, int f, int t, mlp_bf16* Ha,
                                            mlp_bf16* Hg, mlp_bf16* U, mlp_bf16* Y, void* workspace,
                                            size_t workspace_bytes, void* cuda_stream)
{
    mlp_status st = check_shape(T, h, f, t);
    if (st != MLP_OK) return st;
    if (!A || !Wg || !B || (T > 0 && (!X || !Ha || !Hg || !U || !Y))) return MLP_EINVAL;
    const void* ptrs[] = {X, A, Wg, B, Ha, Hg, U, Y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MLP_EALIGN;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MLP_EALIGN;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != MLP_OK) return st;
    if (T == 0) return MLP_OK;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    CallTimer timer(s);

    // Up-projection, both halves at once: Ha = X A, Hg = X Wg, U = SiLU(Ha) Hg.
    GemmArgs g1{};
    if (!map_kmajor(&g1.tmA, X, h, T, 128) || !map_mnmajor(&g1.tmB, A, f, h) || !map_mnmajor(&g1.tmB2, Wg, f, h) ||
        !map_store(&g1.tmD0, Ha, f, T) || !map_store(&g1.tmD1, Hg, f, T) || !map_store(&g1.tmD2, U, f, T))
        return MLP_ECUDA;
    g1.M = T; g1.N = f; g1.K = h;
    g1.status = dev->status;
    g1.timeout_ns = kWaitLimitNs;
    if (gemm_dual(g1, dev->num_sms, s) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_FWD_UP);

    // Down-projection: Y = U B, the shard sum in one accumulator over K = f.
    GemmArgs g2{};
    if (!map_kmajor(&g2.tmA, U, f, T, 128) || !map_mnmajor(&g2.tmB, B, h, f) || !map_store(&g2.tmD0, Y, h, T))
        return MLP_ECUDA;
    g2.M = T; g2.N = h; g2.K = f;
    g2.status = dev->status;
    g2.timeout_ns = kWaitLimitNs;
    const SplitOut so{static_cast<float*>(workspace), workspace ? workspace_bytes : 0, Y};
    if (gemm<false, true, EPI_PLAIN>(g2, tile_n(h), dev->num_sms, s, &so) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_FWD_DOWN);
    return MLP_OK;
}

extern "C" mlp_status mlp_tp_swiglu_backward(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* Wg,
                                             const mlp_bf16* B, const mlp_bf16* Ha, const mlp_bf16* Hg,
                                             const mlp_bf16* U, const mlp_bf16* dY, int T, int h, int f, int t,
                                             mlp_bf16* dX, mlp_bf16* dA, mlp_bf16* dWg, mlp_bf16* dB,
                                             void* workspace, size_t workspace_bytes, void* cuda_stream)
{
    mlp_status st = check_shape(T, h, f, t);
    if (st != MLP_OK) return st;
    if (!A || !Wg || !B || !dA || !dWg || !dB || !workspace ||
        (T > 0 && (!X || !Ha || !Hg || !U || !dY || !dX)))
        return MLP_EINVAL;
    const void* ptrs[] = {X, A, Wg, B, Ha, Hg, U, dY, dX, dA, dWg, dB};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MLP_EALIGN;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MLP_EALIGN;
    if (workspace_bytes < mlp_tp_swiglu_workspace_bytes(T, h, f, t)) return MLP_EWORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != MLP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (T == 0) {
        const size_t w = static_cast<size_t>(h) * f * 2;
        if (cudaMemsetAsync(dA, 0, w, s) != cudaSuccess || cudaMemsetAsync(dWg, 0, w, s) != cudaSuccess ||
            cudaMemsetAsync(dB, 0, w, s) != cudaSuccess)
            return MLP_ECUDA;
        return MLP_OK;
    }
    const int bn_f = tile_n(f / t), bn_h = tile_n(h);
    mlp_bf16* dHa = static_cast<mlp_bf16*>(workspace);
    mlp_bf16* dHg = reinterpret_cast<mlp_bf16*>(static_cast<uint8_t*>(workspace) + round256(static_cast<size_t>(T) * f * 2));
    float* split_ws =
        reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 2 * round256(static_cast<size_t>(T) * f * 2));
    CallTimer timer(s);

    // dU = dY B^T, and in the epilogue dHa = dU Hg SiLU'(Ha), dHg = dU SiLU(Ha).
    GemmArgs g3{};
    if (!map_kmajor(&g3.tmA, dY, h, T, 128) || !map_kmajor(&g3.tmB, B, h, f, kmajor_b_box(T, bn_f)) ||
        !map_store(&g3.tmD0, dHa, f, T) || !map_store(&g3.tmD1, dHg, f, T))
        return MLP_ECUDA;
    g3.M = T; g3.N = f; g3.K = h;
    g3.aux = reinterpret_cast<const __nv_bfloat16*>(Ha);
    g3.aux2 = reinterpret_cast<const __nv_bfloat16*>(Hg);
    g3.ld_aux = f;
    g3.status = dev->status;
    g3.timeout_ns = kWaitLimitNs;
    if (gemm<false, false, EPI_DSWIGLU>(g3, bn_f, dev->num_sms, s) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_BWD_DH);

    // dX = dHa A^T + dHg Wg^T: one accumulator over the two K segments (the shard sum of
    // both column-split weights at once).
    GemmArgs g4{};
    if (!map_kmajor(&g4.tmA, dHa, f, T, 128) || !map_kmajor(&g4.tmB, A, f, h, kmajor_b_box(T, bn_h)) ||
        !map_kmajor(&g4.tmA2, dHg, f, T, 128) || !map_kmajor(&g4.tmB2, Wg, f, h, kmajor_b_box(T, bn_h)) ||
        !map_store(&g4.tmD0, dX, h, T))
        return MLP_ECUDA;
    const int kb_f = (f + 63) / 64;
    g4.M = T; g4.N = h; g4.K = 2 * 64 * kb_f;
    g4.kb_split = kb_f;
    g4.status = dev->status;
    g4.timeout_ns = kWaitLimitNs;
    const SplitOut so4{split_ws, kSplitWsBytes, dX};
    if (gemm<false, false, EPI_PLAIN>(g4, bn_h, dev->num_sms, s, &so4) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_BWD_DX);

    // dA = X^T dHa and dWg = X^T dHg.
    const mlp_bf16* dHs[2] = {dHa, dHg};
    mlp_bf16* dWs[2] = {dA, dWg};
    for (int i = 0; i < 2; ++i) {
        GemmArgs g5{};
        if (!map_mnmajor(&g5.tmA, X, h, T) || !map_mnmajor(&g5.tmB, dHs[i], f, T) || !map_store(&g5.tmD0, dWs[i], f, h))
            return MLP_ECUDA;
        g5.M = h; g5.N = f; g5.K = T;
        g5.status = dev->status;
        g5.timeout_ns = kWaitLimitNs;
        const SplitOut so5{split_ws, kSplitWsBytes, dWs[i]};
        if (gemm<true, true, EPI_PLAIN>(g5, bn_f, dev->num_sms, s, &so5) != cudaSuccess) return MLP_ECUDA;
        timer.mark(MLP_K_BWD_DA);
    }

    // dB = U^T dY.
    GemmArgs g6{};
    if (!map_mnmajor(&g6.tmA, U, f, T) || !map_mnmajor(&g6.tmB, dY, h, T) || !map_store(&g6.tmD0, dB, h, f))
        return MLP_ECUDA;
    g6.M = f; g6.N = h; g6.K = T;
    g6.status = dev->status;
    g6.timeout_ns = kWaitLimitNs;
    const SplitOut so6{split_ws, kSplitWsBytes, dB};
    if (gemm<true, true, EPI_PLAIN>(g6, bn_h, dev->num_sms, s, &so6) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_BWD_DB);
    return MLP_OK;
}

// ---- bias gradients with no device allocation --------------------------------------------
//
// Some callers cannot allocate device memory at the point where they need the bias
// gradients: code embedded in another runtime that owns all device memory (a framework's
// caching allocator or a fixed arena with no room to lend a workspace), and latency-bound
// loops where a cudaMalloc would synchronise the device. For them this entry point keeps
// the reduction's partial sums in a fixed, file-scope device array instead of a caller
// workspace. The array is loaded with the library and stays resident on every GPU that
// loads it until the process exits.

namespace mlp {

// Room for the partial sums of slices x (f + h) columns: 2^20 floats = 4 MiB per GPU.
constexpr size_t kNoAllocScratchFloats = size_t(1) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

static float* g_noalloc_ptr[kMaxDevices];
static std::mutex g_noalloc_mu;

// Device address of g_noalloc_scratch on the current device, looked up once per device.
// (In host code the array's name is only a host-side stand-in, never a device address.)
static mlp_status noalloc_scratch(float** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLP_ECUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MLP_ECUDA;
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return MLP_OK;
}

}  // namespace mlp

extern "C" mlp_status mlp_tp_bias_grads_noalloc(const mlp_bf16* dH, const mlp_bf16* dY, int T, int h, int f,
                                                float* da, float* db, void* cuda_stream)
{
    mlp_status st = check_shape(T, h, f, 1);
    if (st != MLP_OK) return st;
    if (!da || !db || (T > 0 && (!dH || !dY))) return MLP_EINVAL;
    const void* ptrs[] = {dH, dY, da, db};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MLP_EALIGN;
    const int nsplit = colsum_splits(T);
    if (static_cast<size_t>(nsplit) * (static_cast<size_t>(f) + h) > kNoAllocScratchFloats)
        return MLP_EWORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != MLP_OK) return st;
    float* partial = nullptr;
    if ((st = noalloc_scratch(&partial)) != MLP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    // Every slice row of the partial array is written by the first kernel before the second
    // reads it, so nothing left from an earlier call is ever read and no clearing is needed.
    const int strips = (f + kColsumStrip - 1) / kColsumStrip + (h + kColsumStrip - 1) / kColsumStrip;
    colsum_partial_kernel<<<dim3(strips, nsplit), kColsumThreads, 0, s>>>(
        reinterpret_cast<const __nv_bfloat16*>(dH), f, reinterpret_cast<const __nv_bfloat16*>(dY), h, T,
        nsplit, partial);
    if (cudaGetLastError() != cudaSuccess) return MLP_ECUDA;
    colsum_finalize_kernel<<<(f + h + 255) / 256, 256, 0, s>>>(partial, nsplit, f, h, da, db);
    if (cudaGetLastError() != cudaSuccess) return MLP_ECUDA;
    note_launches(2);
    return MLP_OK;
}

// ---- head-parallel self-attention block ---------------------------------------------------

namespace mlp {

static mlp_status check_attn(int b, int s, int h, int a, int d, int t)
{
    if (b < 0 || s < 1 || h < 8 || a < 1 || d < 1 || t < 1) return MLP_EINVAL;
    if (h % 8 != 0 || d != kHeadDim || a % t != 0) return MLP_ESHAPE;
    if (static_cast<long long>(b) * s > 0x7fffffffLL || static_cast<long long>(a) * d * 3 > 0x7fffffffLL)
        return MLP_EINVAL;
    return MLP_OK;
}

static AttnArgs attn_args(const DeviceInfo* dev, int b, int s, int a, int causal)
{
    AttnArgs at{};
    at.b = b;
    at.s = s;
    at.a = a;
    at.causal = causal ? 1 : 0;
    at.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(kHeadDim)));
    at.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHeadDim)));
    at.status = dev->status;
    at.timeout_ns = kWaitLimitNs;
    return at;
}

static size_t attn_ws_dc(int T, int hd) { return round256(static_cast<size_t>(T) * hd * 2); }
static size_t attn_ws_d(int b, int a, int s) { return round256(static_cast<size_t>(b) * a * s * 4); }

}  // namespace mlp

extern "C" mlp_status mlp_tp_attn_forward(const mlp_bf16* X, const mlp_bf16* Wqkv, const mlp_bf16* Wo, int b, int s,
                                          int h, int a, int d, int t, int causal, mlp_bf16* QKV, mlp_bf16* Cctx,
                                          float* L, mlp_bf16* Y, void* workspace, size_t workspace_bytes,
                                          void* cuda_stream)
{
    mlp_status st = check_attn(b, s, h, a, d, t);
    if (st != MLP_OK) return st;
    if (!Wqkv || !Wo || (b > 0 && (!X || !QKV || !Cctx || !L || !Y))) return MLP_EINVAL;
    const void* ptrs[] = {X, Wqkv, Wo, QKV, Cctx, L, Y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MLP_EALIGN;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MLP_EALIGN;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != MLP_OK) return st;
    if (b == 0) return MLP_OK;
    float* split_ws = static_cast<float*>(workspace);
    const size_t split_bytes = workspace ? workspace_bytes : 0;
    cudaStream_t strm = static_cast<cudaStream_t>(cuda_stream);
    const int T = b * s, hd = a * d;
    CallTimer timer(strm);

    // QKV = X Wqkv: every head of every shard in one GEMM (N = 3 a d).
    GemmArgs g1{};
    if (!map_kmajor(&g1.tmA, X, h, T, 128) || !map_mnmajor(&g1.tmB, Wqkv, 3 * hd, h) ||
        !map_store(&g1.tmD0, QKV, 3 * hd, T))
        return MLP_ECUDA;
    g1.M = T; g1.N = 3 * hd; g1.K = h;
    g1.status = dev->status;
    g1.timeout_ns = kWaitLimitNs;
    const SplitOut so1{split_ws, split_bytes, QKV};
    if (gemm<false, true, EPI_PLAIN>(g1, tile_n(3 * hd), dev->num_sms, strm, &so1) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_ATTN_QKV);

    // Per head: scores, mask, softmax and P V on chip; C and L to HBM.
    AttnArgs at = attn_args(dev, b, s, a, causal);
    if (!make_map(&at.tmQ, QKV, 3 * hd, T, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&at.tmKV, QKV, 3 * hd, T, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return MLP_ECUDA;
    at.out = reinterpret_cast<__nv_bfloat16*>(Cctx);
    at.lse = L;
    if (launch_attn_fwd(at, strm) != cudaSuccess) return MLP_ECUDA;
    note_launches(1);
    timer.mark(MLP_K_ATTN_FWD);

    // Y = C Wo: the sum over the t head shards is the K loop of one accumulator (K = a d).
    GemmArgs g2{};
    if (!map_kmajor(&g2.tmA, Cctx, hd, T, 128) || !map_mnmajor(&g2.tmB, Wo, h, hd) || !map_store(&g2.tmD0, Y, h, T))
        return MLP_ECUDA;
    g2.M = T; g2.N = h; g2.K = hd;
    g2.status = dev->status;
    g2.timeout_ns = kWaitLimitNs;
    const SplitOut so2{split_ws, split_bytes, Y};
    if (gemm<false, true, EPI_PLAIN>(g2, tile_n(h), dev->num_sms, strm, &so2) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_ATTN_OUT);
    return MLP_OK;
}

extern "C" size_t mlp_tp_attn_workspace_bytes(int b, int s, int h, int a, int d, int t)
{
    if (check_attn(b, s, h, a, d, t) != MLP_OK) return 0;
    const int T = b * s, hd = a * d;
    return attn_ws_dc(T, hd) + attn_ws_d(b, a, s) + round256(static_cast<size_t>(T) * 3 * hd * 2) + split_ws_bytes(T);
}

extern "C" mlp_status mlp_tp_attn_backward(const mlp_bf16* X, const mlp_bf16* Wqkv, const mlp_bf16* Wo,
                                           const mlp_bf16* QKV, const mlp_bf16* Cctx, const float* L,
                                           const mlp_bf16* dY, int b, int s, int h, int a, int d, int t, int causal,
                                           mlp_bf16* dX, mlp_bf16* dWqkv, mlp_bf16* dWo, void* workspace,
                                           size_t workspace_bytes, void* cuda_stream)
{
    mlp_status st = check_attn(b, s, h, a, d, t);
    if (st != MLP_OK) return st;
    if (!Wqkv || !Wo || !dWqkv || !dWo || !workspace || (b > 0 && (!X || !QKV || !Cctx || !L || !dY || !dX)))
        return MLP_EINVAL;
    const void* ptrs[] = {X, Wqkv, Wo, QKV, Cctx, L, dY, dX, dWqkv, dWo};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MLP_EALIGN;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MLP_EALIGN;
    if (workspace_bytes < mlp_tp_attn_workspace_bytes(b, s, h, a, d, t)) return MLP_EWORKSPACE;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != MLP_OK) return st;
    cudaStream_t strm = static_cast<cudaStream_t>(cuda_stream);
    const int T = b * s, hd = a * d;
    if (T == 0) {
        if (cudaMemsetAsync(dWqkv, 0, static_cast<size_t>(h) * 3 * hd * 2, strm) != cudaSuccess ||
            cudaMemsetAsync(dWo, 0, static_cast<size_t>(hd) * h * 2, strm) != cudaSuccess)
            return MLP_ECUDA;
        return MLP_OK;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    mlp_bf16* dC = reinterpret_cast<mlp_bf16*>(ws);
    float* D = reinterpret_cast<float*>(ws + attn_ws_dc(T, hd));
    mlp_bf16* dQKV = reinterpret_cast<mlp_bf16*>(ws + attn_ws_dc(T, hd) + attn_ws_d(b, a, s));
    float* split_ws = reinterpret_cast<float*>(ws + attn_ws_dc(T, hd) + attn_ws_d(b, a, s) +
                                               round256(static_cast<size_t>(T) * 3 * hd * 2));
    CallTimer timer(strm);

    // dC = dY Wo^T (each head shard's rows of Wo).
    GemmArgs g3{};
    const int bn_hd = tile_n(hd);
    if (!map_kmajor(&g3.tmA, dY, h, T, 128) || !map_kmajor(&g3.tmB, Wo, h, hd, kmajor_b_box(T, bn_hd)) ||
        !map_store(&g3.tmD0, dC, hd, T))
        return MLP_ECUDA;
    g3.M = T; g3.N = hd; g3.K = h;
    g3.status = dev->status;
    g3.timeout_ns = kWaitLimitNs;
    const SplitOut so3{split_ws, kSplitWsBytes, dC};
    if (gemm<false, false, EPI_PLAIN>(g3, bn_hd, dev->num_sms, strm, &so3) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_ATTN_DC);

    // dWo = C^T dY.
    GemmArgs g4{};
    if (!map_mnmajor(&g4.tmA, Cctx, hd, T) || !map_mnmajor(&g4.tmB, dY, h, T) || !map_store(&g4.tmD0, dWo, h, hd))
        return MLP_ECUDA;
    g4.M = hd; g4.N = h; g4.K = T;
    g4.status = dev->status;
    g4.timeout_ns = kWaitLimitNs;
    const SplitOut so4{split_ws, kSplitWsBytes, dWo};
    if (gemm<true, true, EPI_PLAIN>(g4, tile_n(h), dev->num_sms, strm, &so4) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_ATTN_DWO);

    // D = rowsum(dC (.) C) per (token, head).
    if (launch_attn_bwd_dot(reinterpret_cast<const __nv_bfloat16*>(dC), reinterpret_cast<const __nv_bfloat16*>(Cctx),
                            T, s, a, D, dev->num_sms, strm) != cudaSuccess)
        return MLP_ECUDA;
    note_launches(1);
    timer.mark(MLP_K_ATTN_DOT);

    // dQ: per 128-query block over 128-key blocks.
    AttnArgs aq = attn_args(dev, b, s, a, causal);
    if (!make_map(&aq.tmQ, QKV, 3 * hd, T, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&aq.tmKV, QKV, 3 * hd, T, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&aq.tmdO, dC, hd, T, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return MLP_ECUDA;
    aq.out = reinterpret_cast<__nv_bfloat16*>(dQKV);
    aq.lse = const_cast<float*>(L);
    aq.delta = D;
    if (launch_attn_bwd_dq(aq, strm) != cudaSuccess) return MLP_ECUDA;
    note_launches(1);
    timer.mark(MLP_K_ATTN_DQ);

    // dK, dV: per 128-key block over 64-query blocks.
    AttnArgs ak = aq;
    if (!make_map(&ak.tmKV, QKV, 3 * hd, T, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&ak.tmQ, QKV, 3 * hd, T, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&ak.tmdO, dC, hd, T, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return MLP_ECUDA;
    if (launch_attn_bwd_dkdv(ak, strm) != cudaSuccess) return MLP_ECUDA;
    note_launches(1);
    timer.mark(MLP_K_ATTN_DKDV);

    // dX = dQKV Wqkv^T: one accumulator over K = 3 a d sums Q, K, V and all head shards.
    GemmArgs g6{};
    const int bn_h = tile_n(h);
    if (!map_kmajor(&g6.tmA, dQKV, 3 * hd, T, 128) || !map_kmajor(&g6.tmB, Wqkv, 3 * hd, h, kmajor_b_box(T, bn_h)) ||
        !map_store(&g6.tmD0, dX, h, T))
        return MLP_ECUDA;
    g6.M = T; g6.N = h; g6.K = 3 * hd;
    g6.status = dev->status;
    g6.timeout_ns = kWaitLimitNs;
    const SplitOut so6{split_ws, kSplitWsBytes, dX};
    if (gemm<false, false, EPI_PLAIN>(g6, bn_h, dev->num_sms, strm, &so6) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_ATTN_DX);

    // dWqkv = X^T dQKV.
    GemmArgs g7{};
    if (!map_mnmajor(&g7.tmA, X, h, T) || !map_mnmajor(&g7.tmB, dQKV, 3 * hd, T) ||
        !map_store(&g7.tmD0, dWqkv, 3 * hd, h))
        return MLP_ECUDA;
    g7.M = h; g7.N = 3 * hd; g7.K = T;
    g7.status = dev->status;
    g7.timeout_ns = kWaitLimitNs;
    const SplitOut so7{split_ws, kSplitWsBytes, dWqkv};
    if (gemm<true, true, EPI_PLAIN>(g7, tile_n(3 * hd), dev->num_sms, strm, &so7) != cudaSuccess) return MLP_ECUDA;
    timer.mark(MLP_K_ATTN_DWQKV);
    return MLP_OK;
}
