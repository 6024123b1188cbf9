// attn_args.h -- launch arguments of the fused causal-attention kernels (host and device view).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mlp {

// Width of one attention head; the kernels are written for this one value.
constexpr int kHeadDim = 128;

// Token rows are batch-major: row bi*s + p is position p of sequence bi. QKV is
// [T, 3*a*d] with Q in columns [0, a*d), K in [a*d, 2*a*d), V in [2*a*d, 3*a*d); head j
// of each occupies its d columns starting at j*d.
struct AttnArgs {
    CUtensorMap tmQ;    // Q blocks: QKV, box 64 x (query block rows), 128B swizzle
    CUtensorMap tmKV;   // K and V blocks: QKV, box 64 x (key block rows)
    CUtensorMap tmdO;   // dC blocks (backward): [T, a*d], box 64 x (query block rows)
    __nv_bfloat16* out;      // forward: C [T, a*d]; backward: dQKV [T, 3*a*d]
    float* lse;              // [b*a, s]: base-2 log-sum-exp of each query's scaled scores
    const float* delta;      // [b*a, s]: rowsum(dC * C) per head (backward)
    int b, s, a;             // sequences, their length, heads
    int causal;              // 1: key j > query i is masked
    float scale;             // 1 / sqrt(d)
    float scale_log2;        // log2(e) / sqrt(d)
    int* status;             // device status word (first error code wins)
    unsigned long long timeout_ns;
};

cudaError_t launch_attn_fwd(const AttnArgs& args, cudaStream_t stream);
cudaError_t launch_attn_bwd_dq(const AttnArgs& args, cudaStream_t stream);
cudaError_t launch_attn_bwd_dkdv(const AttnArgs& args, cudaStream_t stream);
cudaError_t launch_attn_bwd_dot(const __nv_bfloat16* dC, const __nv_bfloat16* Cc, int T, int s, int a, float* D,
                                int num_sms, cudaStream_t stream);

}  // namespace mlp
