/*
 * mlp_tp.h -- C ABI of the tensor-parallel Transformer MLP block on one sm_103a GPU.
 *
 * The block (Megatron partitioning, "Efficient Large-Scale Language Model Training on GPU
 * Clusters Using Megatron-LM", section 3 "Tensor Model Parallelism: The Megatron
 * Partitioning", Figure 5a; with the biases of the fused bias+GeLU kernel of the same
 * section):
 *
 *     H = X*A + a,    G = GELU(H),    Y = G*B + b
 *
 * with A = [A_1 | ... | A_t] split by columns and B = [B_1; ...; B_t] split by rows into
 * t equal contiguous shards ("Distributed training", ml-interview-book, section 2.6 and
 * section 3.2, torch.chunk blocks). Every shard's GELU is shard-local and
 * Y = sum_i GELU(X A_i + a_i) B_i + b; here all t shards live on one GPU and the sum over
 * shards is the K loop of one tensor-core accumulator (the all-reduce g of the pages
 * becomes an on-chip sum). Backward, likewise, dX = sum_i dH_i A_i^T (the all-reduce f:
 * "the backward of a copy is a sum", "Parallelism", xuewyang.github.io, "The backward
 * pass").
 *
 * GELU is the tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 *
 * Layout: every matrix is row-major and dense (row stride = number of columns).
 *   X [T,h]  A [h,f]  a [f]  B [f,h]  b [h]  H, G [T,f]  Y [T,h]
 *   dY [T,h] dX [T,h] dA [h,f] dB [f,h] da [f] db [h]
 * mlp_bf16 is the raw bit pattern of a bfloat16; da and db are fp32.
 *
 * Ownership: the caller allocates every buffer (device memory) and owns the stream; the
 * library allocates no device memory and keeps no pointer after a call returns.
 *
 * Split tails (all GEMMs whose output is the accumulator, or the accumulator plus a bias):
 * a GEMM of tiles tiles on u units (CTA pairs, or CTAs) runs them in rounds of u; when
 * tiles % u leaves the last round short, the call may cut each of those last tiles into
 * S >= 2 ranges of K (each at least 16 k blocks of 64, S * (tiles % u) <= u) that run side
 * by side. Each range writes its fp32 partial tile to the workspace, and one more launch
 * adds a tile's S partials in range order (then the bias) and rounds once to bf16. This
 * needs workspace room (at most mlp_tp_forward_workspace_bytes(), which every backward
 * workspace size below includes); the forward entry points take it as an optional
 * argument and, without it, run every tile whole. The sum order is fixed by the sizes and
 * the device's SM count, so results stay bitwise reproducible run to run.
 *
 * Execution: calls are asynchronous on `cuda_stream` (a cudaStream_t; NULL = the legacy
 * default stream) of the current device. All arguments are checked before anything is
 * launched; a failing check returns its status and launches nothing. Launch failures
 * return MLP_ECUDA. Device-side waits are bounded; a wait that runs out records an error
 * that mlp_tp_query_device_status() reports as MLP_ETIMEOUT.
 *
 * Shapes: T >= 0; h, f >= 8 and multiples of 8; t >= 1 with f % t == 0 and (f/t) % 8 == 0.
 * Pointers: 16-byte aligned and non-NULL, except that buffers indexed by tokens (X, H, G,
 * Y, dY, dX) may be NULL when T == 0. Results agree, within bf16 rounding, for every
 * admissible t (the shard-sum identity), and are bitwise reproducible run to run.
 */
#ifndef MLP_TP_H
#define MLP_TP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLP_OK = 0,
    MLP_EINVAL = 1,       /* NULL pointer, t < 1, T < 0, h or f < 8 */
    MLP_ESHAPE = 2,       /* a size breaks the call's shape rules (MLP: f % t != 0, or h, f,
                             f/t not multiples of 8; attention: a % t != 0, d != 128) */
    MLP_EALIGN = 3,       /* a pointer is not 16-byte aligned */
    MLP_ECUDA = 4,        /* a CUDA runtime call or launch failed */
    MLP_ETIMEOUT = 5,     /* a device-side check failed, reported by query: a bounded wait ran
                             out, or (device code 7) a kernel found its dynamic shared memory
                             off its 1 KB alignment and did nothing */
    MLP_EUNSUPPORTED = 6, /* no sm_100-family tensor cores on the current device */
    MLP_EWORKSPACE = 7    /* workspace smaller than mlp_tp_workspace_bytes() */
} mlp_status;

typedef uint16_t mlp_bf16;

/* Forward pass: H = X*A + a and G = GELU(H) (first GEMM, bias and GELU in its epilogue; G is
 * computed from H as stored, rounded to bf16),
 * then Y = G*B + b (second GEMM; its K loop runs over the t shards' row blocks of B into
 * one accumulator, so the shard sum never leaves the chip). H and G are the activations
 * the backward needs ("Distributed training", section 2.2: the MLP keeps the GELU input
 * and the down-projection input). Two kernel launches, plus one when the second GEMM's
 * tail is split. `workspace` is optional (NULL, or device memory 256-byte aligned, else
 * MLP_EALIGN): room for the split tail's partial tiles, used up to workspace_bytes
 * (mlp_tp_forward_workspace_bytes() is always enough); its contents on entry do not
 * matter. */
mlp_status mlp_tp_forward(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a,
                          const mlp_bf16* B, const mlp_bf16* b, int T, int h, int f, int t,
                          mlp_bf16* H, mlp_bf16* G, mlp_bf16* Y, void* workspace,
                          size_t workspace_bytes, void* cuda_stream);

/* Workspace bytes with which every forward entry point (mlp_tp_forward,
 * mlp_tp_swiglu_forward, mlp_tp_attn_forward) splits every tail it can: 40 MiB. */
size_t mlp_tp_forward_workspace_bytes(void);

/* Forward pass followed by the block's fused output step ("Efficient Large-Scale Language
 * Model Training on GPU Clusters Using Megatron-LM", section 3, "Fused element-wise
 * kernels": bias + dropout + residual add, on the output of Figure 5a, Z = Dropout(Y B)):
 *     Z = R + keep (.) (G*B + b) / (1 - p)
 * R [T,h] is the residual stream (bf16). keep is drawn per element with Philox4x32-10
 * (Salmon et al., SC 2011): element e = r*h + c uses word e % 4 of Philox on counter
 * (lo32(e/4), hi32(e/4), lo32(offset), hi32(offset)) with key (lo32(seed), hi32(seed)) and
 * is kept when that word's top 24 bits are >= floor(p * 2^24); 0 <= p < 1 (else
 * MLP_EINVAL). H and G are written as by mlp_tp_forward; Y itself is not, Z takes its
 * place (both in the epilogue of the second GEMM). Same launches as mlp_tp_forward. */
mlp_status mlp_tp_forward_residual_dropout(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a,
                                           const mlp_bf16* B, const mlp_bf16* b, const mlp_bf16* R,
                                           int T, int h, int f, int t, double p,
                                           unsigned long long seed, unsigned long long offset,
                                           mlp_bf16* H, mlp_bf16* G, mlp_bf16* Z, void* cuda_stream);

/* Backward of that output step: dY = dZ (.) keep / (1 - p) with the same (p, seed, offset),
 * so the mask is regenerated, never stored. dL/dR is dZ itself. Feed dY to
 * mlp_tp_backward. dZ, dY [T,h] bf16; h >= 8 and a multiple of 8. One launch. */
mlp_status mlp_tp_dropout_backward(const mlp_bf16* dZ, int T, int h, double p, unsigned long long seed,
                                   unsigned long long offset, mlp_bf16* dY, void* cuda_stream);

/* Backward pass given dY = dL/dY ("Parallelism", "The backward pass"; chain rule):
 *   dH = (dY*B^T) (.) GELU'(H)        per shard, GELU' in the GEMM epilogue
 *   dX = dH*A^T = sum_i dH_i A_i^T    shard sum in one accumulator
 *   dA = X^T*dH,  dB = G^T*dY         local weight gradients
 *   da = colsum(dH) (fp32; the dH GEMM sums its fp32 dH over 32-row blocks in the
 *        epilogue),  db = colsum(dY) (fp32)
 * `workspace` (device, >= mlp_tp_workspace_bytes(T,h,f,t) bytes, 256-byte aligned) holds
 * dH, the reduction partials and the split tails' parts; its contents on entry do not
 * matter. On return its first
 * T*f*2 bytes hold dH = dL/dH (row-major bf16 [T,f]). Six launches, plus one for each of
 * the dX, dA and dB GEMMs whose tail is split. */
mlp_status mlp_tp_backward(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* B,
                           const mlp_bf16* H, const mlp_bf16* G, const mlp_bf16* dY,
                           int T, int h, int f, int t,
                           mlp_bf16* dX, mlp_bf16* dA, mlp_bf16* dB, float* da, float* db,
                           void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Bias gradients da = colsum(dH), db = colsum(dY) (fp32) with no workspace and no device
 * allocation of any kind. db is bit for bit mlp_tp_backward's (the same reduction over dY
 * in the same order). da sums the bf16 dH given here, while mlp_tp_backward's da sums the
 * dH GEMM's fp32 values before they are rounded, so the two agree to within the bf16
 * rounding of dH, not bitwise. The paper has
 * no counterpart to this entry point; it exists for callers that cannot allocate device
 * memory when they need these sums: code running inside another runtime that owns all
 * device memory (a framework allocator or fixed arena with nothing to lend), and
 * latency-bound loops where a cudaMalloc would synchronise the device.
 * The partial sums live in one fixed device array inside the library (4 MiB per GPU, held
 * from library load until process exit): sizes with clamp(T/512, 1, 16) * (f + h) > 2^20
 * are rejected with MLP_EWORKSPACE before anything is launched. The first call on a device
 * looks up that array's device address (one cudaGetSymbolAddress, with the device
 * current); make that first call outside any stream capture. Every call on a device
 * shares the one array: calls that can overlap on the GPU (different streams without
 * ordering between them) race and give wrong sums, so order them. Each call rewrites every
 * partial it later reads, so stale contents from an earlier call are harmless.
 * dH [T,f], dY [T,h] row-major bf16 (may be NULL when T == 0); da [f], db [h] fp32; all
 * 16-byte aligned; h, f >= 8 and multiples of 8. Asynchronous on cuda_stream. */
mlp_status mlp_tp_bias_grads_noalloc(const mlp_bf16* dH, const mlp_bf16* dY, int T, int h, int f,
                                     float* da, float* db, void* cuda_stream);

/* SwiGLU variant of the block ("Distributed training", ml-interview-book, section 7,
 * exercise 3): Y = (SiLU(X A) (.) X Wg) B, with A and Wg both split by columns and B by
 * rows into t shards (each shard's SiLU and product are shard-local; one sum remains, the
 * K loop of the down-projection). No biases. SiLU(x) = x sigma(x).
 *   X [T,h]  A, Wg [h,f]  B [f,h]  Ha, Hg, U [T,f]  Y [T,h]
 * Forward: Ha = X A and Hg = X Wg come out of one GEMM (both halves of one 256-wide MMA per
 * 128 output columns, sharing the X tiles) whose epilogue also writes U = SiLU(Ha) Hg; then
 * Y = U B. Ha, Hg, U are kept for the backward. Two launches (plus one when Y's GEMM tail
 * is split; `workspace` is optional, as for mlp_tp_forward). */
mlp_status mlp_tp_swiglu_forward(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* Wg,
                                 const mlp_bf16* B, int T, int h, int f, int t, mlp_bf16* Ha,
                                 mlp_bf16* Hg, mlp_bf16* U, mlp_bf16* Y, void* workspace,
                                 size_t workspace_bytes, void* cuda_stream);

/* SwiGLU backward given dY: dU = dY B^T; dHa = dU Hg SiLU'(Ha), dHg = dU SiLU(Ha) (in the
 * dU GEMM's epilogue); dX = dHa A^T + dHg Wg^T (one accumulator over both K segments);
 * dA = X^T dHa; dWg = X^T dHg; dB = U^T dY. `workspace` (>= mlp_tp_swiglu_workspace_bytes(),
 * 256-byte aligned) holds dHa and dHg, then the split tails' parts. Five launches, plus
 * one per split tail. */
mlp_status mlp_tp_swiglu_backward(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* Wg,
                                  const mlp_bf16* B, const mlp_bf16* Ha, const mlp_bf16* Hg,
                                  const mlp_bf16* U, const mlp_bf16* dY, int T, int h, int f, int t,
                                  mlp_bf16* dX, mlp_bf16* dA, mlp_bf16* dWg, mlp_bf16* dB,
                                  void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Device bytes mlp_tp_swiglu_backward needs as workspace (0 on invalid sizes). */
size_t mlp_tp_swiglu_workspace_bytes(int T, int h, int f, int t);

/* Device bytes mlp_tp_backward needs as workspace for these sizes (0 on invalid sizes). */
size_t mlp_tp_workspace_bytes(int T, int h, int f, int t);

/* GELU recompute ("Efficient Large-Scale Language Model Training ... Megatron-LM", section 3
 * "Activation Recomputation": keep fewer activations, recompute them in the backward; and
 * "Distributed training", section 2.2: the MLP's saved activations are the GELU input and
 * the down-projection input). G = GELU(H) is never stored:
 *   mlp_tp_forward_recompute  writes H = X*A + a (first GEMM, bias epilogue) and
 *       Y = GELU(H)*B + b: the second GEMM reads H, and operand-transform warps turn each
 *       landed H tile into G in shared memory before its MMAs (the same arithmetic as the
 *       GELU epilogue of mlp_tp_forward, so Y is bitwise mlp_tp_forward's when H is; the
 *       first GEMM is tiled as in mlp_tp_forward, so it is). Arguments, workspace and errors
 *       as mlp_tp_forward, without G.
 *   mlp_tp_backward_recompute  the backward from the kept H alone: dB = GELU(H)^T dY reads H
 *       with the same on-chip transform; every gradient is bitwise mlp_tp_backward's with the
 *       forward's G. Workspace: mlp_tp_recompute_workspace_bytes (= mlp_tp_workspace_bytes),
 *       with dH in its first T*f*2 bytes on return. Other arguments and errors as
 *       mlp_tp_backward.
 * The transform costs about 8 GELU evaluations per clock per SM next to the MMAs (one A value
 * per 512 multiply-adds of a 512-wide tile, every A tile once per output-column tile), so
 * these two GEMMs run slower than the ones that read a stored G; what they save is the G
 * activation ([T,f] bf16) and its HBM traffic. */
mlp_status mlp_tp_forward_recompute(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a,
                                    const mlp_bf16* B, const mlp_bf16* b, int T, int h, int f, int t,
                                    mlp_bf16* H, mlp_bf16* Y, void* workspace, size_t workspace_bytes,
                                    void* cuda_stream);
size_t mlp_tp_recompute_workspace_bytes(int T, int h, int f, int t);
mlp_status mlp_tp_backward_recompute(const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* B, const mlp_bf16* H,
                                     const mlp_bf16* dY, int T, int h, int f, int t, mlp_bf16* dX, mlp_bf16* dA,
                                     mlp_bf16* dB, float* da, float* db, void* workspace, size_t workspace_bytes,
                                     void* cuda_stream);

/* Synchronises `cuda_stream`, then reports and clears the device status word of the
 * current device: MLP_ETIMEOUT if a bounded device wait ran out since the last query,
 * MLP_ECUDA if the stream holds a CUDA error, else MLP_OK. */
mlp_status mlp_tp_query_device_status(void* cuda_stream);

/* The raw device status code behind the last MLP_ETIMEOUT (which wait gave up), or 0. */
int mlp_tp_last_device_code(void);

/* Where the bounded wait behind the last MLP_ETIMEOUT gave up: block index, thread index,
 * output tile and k block (-1 where not applicable). Returns the device code, or 0. */
int mlp_tp_last_device_where(int* block, int* thread, int* tile, int* kblock);

/* Human-readable name of a status. Never NULL. */
const char* mlp_tp_status_string(mlp_status s);

/* Kernel launches the library has made since it was loaded (every entry point, device and
 * stream): the difference across a region counts the region's launches, split-tail fixups
 * included. */
long long mlp_tp_launch_count(void);

/* Self-test of the bounded-wait path: launches one small kernel that waits on a barrier
 * nothing will ever complete, with a limit of `limit_ns` nanoseconds; the wait runs out,
 * the kernel returns normally, and the next mlp_tp_query_device_status() reports
 * MLP_ETIMEOUT. The GPU context stays usable. */
mlp_status mlp_tp_selftest_wait_timeout(unsigned long long limit_ns, void* cuda_stream);

/* Per-kernel timing for benchmarks. While enabled, every forward/backward call records a
 * CUDA event on its stream before its first launch and after each launch (no extra
 * synchronisation). mlp_tp_timing_collect() waits for those events, writes the summed
 * milliseconds and launch counts per kernel id into ms[MLP_NUM_KERNELS] and
 * counts[MLP_NUM_KERNELS], and forgets them. */
enum {
    MLP_K_FWD_UP = 0,        /* H = X*A + a, G = GELU(H) */
    MLP_K_FWD_DOWN = 1,      /* Y = G*B + b */
    MLP_K_BWD_DH = 2,        /* dH = (dY*B^T) (.) GELU'(H) */
    MLP_K_BWD_DX = 3,        /* dX = dH*A^T */
    MLP_K_BWD_DA = 4,        /* dA = X^T*dH */
    MLP_K_BWD_DB = 5,        /* dB = G^T*dY */
    MLP_K_COLSUM_PARTIAL = 6,/* db partial column sums (da's come from the dH GEMM) */
    MLP_K_COLSUM_FINAL = 7,  /* da, db final sums */
    MLP_K_DROPOUT_BWD = 8,   /* dY = dZ (.) keep / (1 - p) */
    MLP_K_ATTN_QKV = 9,      /* attention: QKV = X*Wqkv */
    MLP_K_ATTN_FWD = 10,     /* attention: C = softmax(mask(Q K^T / sqrt(d))) V per head, and L */
    MLP_K_ATTN_OUT = 11,     /* attention: Y = C*Wo (sum over head shards) */
    MLP_K_ATTN_DC = 12,      /* attention: dC = dY*Wo^T */
    MLP_K_ATTN_DWO = 13,     /* attention: dWo = C^T*dY */
    MLP_K_ATTN_DOT = 14,     /* attention: D = rowsum(dC (.) C) per head */
    MLP_K_ATTN_DQ = 15,      /* attention: dQ */
    MLP_K_ATTN_DKDV = 16,    /* attention: dK, dV */
    MLP_K_ATTN_DX = 17,      /* attention: dX = dQKV*Wqkv^T (sum over Q, K, V and head shards) */
    MLP_K_ATTN_DWQKV = 18,   /* attention: dWqkv = X^T*dQKV */
    MLP_NUM_KERNELS = 19
};
mlp_status mlp_tp_timing_enable(int on);
mlp_status mlp_tp_timing_collect(double* ms, int* counts);
const char* mlp_tp_kernel_name(int kernel);

/* ---- head-parallel self-attention block -----------------------------------------------
 *
 * The attention half of the Megatron layer ("Efficient Large-Scale Language Model Training
 * on GPU Clusters Using Megatron-LM", section 3, Figure 5b; "Distributed training",
 * ml-interview-book, section 2.6, and its section 3.2 head-parallel attention; "Parallelism",
 * xuewyang.github.io, "Attention"): the query, key and value weights are split by columns
 * grouped by head and the output weight by rows, so each of t shards owns a/t whole heads,
 * runs their attention with no communication, and the shards' partial outputs are summed.
 * Here all t shards live on one GPU and that sum is the K loop of the output projection's
 * tensor-core accumulator. No biases (the pages' head-parallel attention has none).
 *
 *   QKV = X*Wqkv                       Wqkv = [Wq | Wk | Wv], each [h, a*d]
 *   per head j:  S_j = Q_j K_j^T / sqrt(d)  (causal: key k > query q masked)
 *                P_j = softmax over each row of S_j,   C_j = P_j V_j
 *   C = [C_1 | ... | C_a]              Y = C*Wo,   Wo [a*d, h]
 *
 * Tokens are b sequences of s positions, batch-major: row bi*s + p of X is position p of
 * sequence bi; attention never crosses sequences. Layout (row-major, dense):
 *   X [T,h]  Wqkv [h,3*a*d]  Wo [a*d,h]  QKV [T,3*a*d]  C [T,a*d]  Y, dY, dX [T,h]
 *   L [b*a, s] fp32: L[bi*a + j, p] = log2 sum_k 2^(S_j[p,k] * log2(e)), the base-2
 *   log-sum-exp of position p's scaled scores in head j (kept for the backward pass).
 *   Head j of Q (of K, V, C) is the column block [j*d, (j+1)*d) of its part; shard i owns
 *   heads [i*a/t, (i+1)*a/t).
 * Shapes: b >= 0, s >= 1, h >= 8 and h % 8 == 0, a >= 1, d == 128 (the one head width the
 * kernels are written for; MLP_ESHAPE otherwise), t >= 1 with a % t == 0. Pointers as for
 * the MLP block (token-indexed ones may be NULL when b == 0). Results are bitwise
 * reproducible run to run (no atomics anywhere). Three launches, plus one per split GEMM
 * tail; `workspace` is optional, as for mlp_tp_forward. */
mlp_status mlp_tp_attn_forward(const mlp_bf16* X, const mlp_bf16* Wqkv, const mlp_bf16* Wo, int b, int s, int h,
                               int a, int d, int t, int causal, mlp_bf16* QKV, mlp_bf16* C, float* L, mlp_bf16* Y,
                               void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Device workspace mlp_tp_attn_backward needs (bytes; 0 for inadmissible shapes):
 * dC [T, a*d] bf16 | D [b*a, s] fp32 | dQKV [T, 3*a*d] bf16 | split-tail parts, each
 * 256-byte aligned. */
size_t mlp_tp_attn_workspace_bytes(int b, int s, int h, int a, int d, int t);

/* Backward of the attention block given dY and the forward's QKV, C and L:
 *   dC = dY*Wo^T, dWo = C^T*dY, then per head (with D = rowsum(dC_j (.) C_j))
 *   dP = dC_j V_j^T, dS = P (.) (dP - D), dQ_j = dS K_j / sqrt(d), dK_j = dS^T Q_j / sqrt(d),
 *   dV_j = P^T dC_j, and dX = dQKV*Wqkv^T (the sum over Q, K, V and over head shards),
 *   dWqkv = X^T*dQKV. dWqkv [h, 3*a*d] and dWo [a*d, h] are overwritten. The workspace
 *   (256-byte aligned, at least mlp_tp_attn_workspace_bytes) holds dQKV on return. */
mlp_status mlp_tp_attn_backward(const mlp_bf16* X, const mlp_bf16* Wqkv, const mlp_bf16* Wo, const mlp_bf16* QKV,
                                const mlp_bf16* C, const float* L, const mlp_bf16* dY, int b, int s, int h, int a,
                                int d, int t, int causal, mlp_bf16* dX, mlp_bf16* dWqkv, mlp_bf16* dWo,
                                void* workspace, size_t workspace_bytes, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* MLP_TP_H */
