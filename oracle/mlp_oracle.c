/*
 * mlp_oracle.c -- plain fp64 CPU oracle for the tensor-parallel Transformer MLP block.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the CPU-baseline leg of
 * the benchmark load this library. The CUDA path shares no code with it and never calls it.
 *
 * What it computes (row-major, rows are tokens):
 *   H = X*A + a,  G = act(H),  Y = G*B + b                               (forward)
 *   dG = dY*B^T,  dH = dG (.) act'(H),  dX = dH*A^T,
 *   dA = X^T*dH,  dB = G^T*dY,  da = colsum(dH),  db = colsum(dY)          (backward)
 * with X [T,h], A [h,f], a [f], B [f,h], b [h], dY [T,h].
 *
 * Sources:
 *  - "Efficient Large-Scale Language Model Training on GPU Clusters Using Megatron-LM"
 *    (paper summary), section 3 "Tensor Model Parallelism: The Megatron Partitioning",
 *    Figure 5a: Y = GeLU(XA), Z = Dropout(YB); A split by columns, B by rows, one sum.
 *    Section 3 "Fused element-wise kernels" names the bias+GeLU pair, which places the
 *    first bias before the activation.
 *  - "Distributed training" (ml-interview-book), section 2.6 "Tensor parallelism: why
 *    exactly two all-reduces per block": GELU(XA)B = sum_i GELU(XA_i) B_i, and the column
 *    layer's input gradient is sum_i dY_i W_i^T.
 *  - "Parallelism" (xuewyang.github.io), "The MLP, with real numbers" and "The backward
 *    pass": the per-shard backward through B, the nonlinearity and A, the sum for dX, and
 *    local weight gradients dA_i = X^T dH_i.
 *
 * Readings taken where the pages are silent: the activation is the tanh form of GELU
 * (erf GELU, ReLU with relu'(0) = 0 and the identity are selectable for tests); the output
 * bias b is added once, after the shard sum, so db = colsum(dY); shards are contiguous equal
 * column blocks of A (row blocks of B), as torch.chunk makes them.
 *
 * Nothing is rounded: inputs arrive as fp64 (or as bf16 bit patterns that convert exactly)
 * and every sum is carried in fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ACT_GELU_TANH = 0, ACT_GELU_ERF = 1, ACT_RELU = 2, ACT_IDENTITY = 3 };

/* ---- activations ------------------------------------------------------------------ */

/* GELU, tanh form (Hendrycks & Gimpel): 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))). */
static double gelu_tanh(double x)
{
    const double c = sqrt(2.0 / M_PI);
    double u = c * (x + 0.044715 * x * x * x);
    return 0.5 * x * (1.0 + tanh(u));
}

/* d/dx of the tanh form: 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) du/dx,
 * du/dx = sqrt(2/pi) (1 + 3 * 0.044715 x^2). */
static double gelu_tanh_grad(double x)
{
    const double c = sqrt(2.0 / M_PI);
    double u = c * (x + 0.044715 * x * x * x);
    double th = tanh(u);
    double du = c * (1.0 + 3.0 * 0.044715 * x * x);
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * du;
}

/* GELU, exact form: x Phi(x), Phi the standard normal CDF. */
static double gelu_erf(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }

/* d/dx x Phi(x) = Phi(x) + x phi(x). */
static double gelu_erf_grad(double x)
{
    double Phi = 0.5 * (1.0 + erf(x / sqrt(2.0)));
    double phi = exp(-0.5 * x * x) / sqrt(2.0 * M_PI);
    return Phi + x * phi;
}

static double act_fn(int act, double x)
{
    switch (act) {
    case ACT_GELU_TANH: return gelu_tanh(x);
    case ACT_GELU_ERF: return gelu_erf(x);
    case ACT_RELU: return x > 0.0 ? x : 0.0;
    default: return x;
    }
}

/* ReLU'(0) = 0: "Parallelism" (xuewyang.github.io), "The backward pass", GPU 2's ReLU
 * passes [2, 1] to [2, 0] because its input was [1, 0]. */
static double act_grad(int act, double x)
{
    switch (act) {
    case ACT_GELU_TANH: return gelu_tanh_grad(x);
    case ACT_GELU_ERF: return gelu_erf_grad(x);
    case ACT_RELU: return x > 0.0 ? 1.0 : 0.0;
    default: return 1.0;
    }
}

double oracle_act(int act, double x) { return act_fn(act, x); }
double oracle_act_grad(int act, double x) { return act_grad(act, x); }

/* ---- plain matrix products (row-major, fp64) -------------------------------------- */

/* out[M,N] = P[M,K] * Q[K,N] */
static void mm_nn(int64_t M, int64_t N, int64_t K, const double *P, const double *Q, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double *o = out + i * N;
        for (int64_t j = 0; j < N; ++j) o[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = P[i * K + k];
            const double *q = Q + k * N;
            for (int64_t j = 0; j < N; ++j) o[j] += p * q[j];
        }
    }
}

/* out[M,N] = P[M,K] * Q[N,K]^T */
static void mm_nt(int64_t M, int64_t N, int64_t K, const double *P, const double *Q, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        const double *p = P + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const double *q = Q + j * K;
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += p[k] * q[k];
            out[i * N + j] = s;
        }
    }
}

/* out[M,N] = P[K,M]^T * Q[K,N] */
static void mm_tn(int64_t M, int64_t N, int64_t K, const double *P, const double *Q, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double *o = out + i * N;
        for (int64_t j = 0; j < N; ++j) o[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = P[k * M + i];
            const double *q = Q + k * N;
            for (int64_t j = 0; j < N; ++j) o[j] += p * q[j];
        }
    }
}

/* out[N] = sum over rows of P[M,N] */
static void colsum(int64_t M, int64_t N, const double *P, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j) {
        double s = 0.0;
        for (int64_t i = 0; i < M; ++i) s += P[i * N + j];
        out[j] = s;
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---- the unsharded block ----------------------------------------------------------- */

/* Forward, Figure 5a with biases: H = X A + a; G = act(H); Y = G B + b.
 * H, G are [T,f] and are what the forward keeps for the backward ("Distributed training",
 * section 2.2: the MLP stores the GELU input and the down-projection input). */
int oracle_mlp_forward(int64_t T, int64_t h, int64_t f, int act,
                       const double *X, const double *A, const double *a,
                       const double *B, const double *b,
                       double *H, double *G, double *Y)
{
    if (T < 0 || h < 1 || f < 1) return 1;
    mm_nn(T, f, h, X, A, H);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r)
        for (int64_t j = 0; j < f; ++j) {
            double v = H[r * f + j] + a[j];
            H[r * f + j] = v;
            G[r * f + j] = act_fn(act, v);
        }
    mm_nn(T, h, f, G, B, Y);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r)
        for (int64_t n = 0; n < h; ++n) Y[r * h + n] += b[n];
    return 0;
}

/* Backward by the chain rule through Y = G B + b, G = act(H), H = X A + a:
 * dG = dY B^T; dH = dG (.) act'(H); dX = dH A^T; dA = X^T dH; dB = G^T dY;
 * da = colsum(dH); db = colsum(dY). dH (optional, [T,f]) is returned when non-NULL. */
int oracle_mlp_backward(int64_t T, int64_t h, int64_t f, int act,
                        const double *X, const double *A, const double *B,
                        const double *H, const double *G, const double *dY,
                        double *dX, double *dA, double *da, double *dB, double *db,
                        double *dH_out)
{
    if (T < 0 || h < 1 || f < 1) return 1;
    double *dH = dH_out ? dH_out : (double *)malloc(sizeof(double) * (size_t)(T * f > 0 ? T * f : 1));
    if (!dH) return 2;
    mm_nt(T, f, h, dY, B, dH); /* dG */
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r)
        for (int64_t j = 0; j < f; ++j) dH[r * f + j] *= act_grad(act, H[r * f + j]);
    mm_nt(T, h, f, dH, A, dX);
    mm_tn(h, f, T, X, dH, dA);
    mm_tn(f, h, T, G, dY, dB);
    colsum(T, f, dH, da);
    colsum(T, h, dY, db);
    if (!dH_out) free(dH);
    return 0;
}

/* ---- the sharded block, shard by shard (the pages' own form) ------------------------ */

/* Shard i owns columns [i f/t, (i+1) f/t) of A and a, and the same rows of B.
 * Forward: P_i = act(X A_i + a_i) B_i; Y = sum_i P_i + b (the g sum).
 * Backward: dG_i = dY B_i^T; dH_i = dG_i (.) act'(H_i); dX_i = dH_i A_i^T; dX = sum_i dX_i
 * (the f sum: the backward of a copy is a sum); dA_i = X^T dH_i; dB_i = G_i^T dY;
 * da_i = colsum(dH_i); db = colsum(dY).
 * Y_part and dX_part, when non-NULL, receive the t per-shard partials [t,T,h]. */
int oracle_mlp_sharded(int64_t T, int64_t h, int64_t f, int64_t t, int act,
                       const double *X, const double *A, const double *a,
                       const double *B, const double *b, const double *dY,
                       double *Y, double *dX, double *dA, double *da, double *dB, double *db,
                       double *Y_part, double *dX_part)
{
    if (T < 0 || h < 1 || f < 1 || t < 1 || f % t != 0) return 1;
    int64_t fs = f / t;
    size_t nTf = (size_t)(T * fs > 0 ? T * fs : 1), nhf = (size_t)(h * fs), nTh = (size_t)(T * h > 0 ? T * h : 1);
    double *Ai = malloc(sizeof(double) * nhf), *Bi = malloc(sizeof(double) * nhf);
    double *Hi = malloc(sizeof(double) * nTf), *Gi = malloc(sizeof(double) * nTf);
    double *dHi = malloc(sizeof(double) * nTf), *Pi = malloc(sizeof(double) * nTh);
    double *dXi = malloc(sizeof(double) * nTh), *dAi = malloc(sizeof(double) * nhf);
    double *dBi = malloc(sizeof(double) * nhf);
    if (!Ai || !Bi || !Hi || !Gi || !dHi || !Pi || !dXi || !dAi || !dBi) return 2;
    for (int64_t i = 0; i < T * h; ++i) { Y[i] = 0.0; dX[i] = 0.0; }
    for (int64_t s = 0; s < t; ++s) {
        int64_t c0 = s * fs;
        for (int64_t k = 0; k < h; ++k)
            for (int64_t j = 0; j < fs; ++j) Ai[k * fs + j] = A[k * f + c0 + j];
        for (int64_t j = 0; j < fs; ++j)
            for (int64_t n = 0; n < h; ++n) Bi[j * h + n] = B[(c0 + j) * h + n];
        /* column-parallel half: shard-local activation */
        mm_nn(T, fs, h, X, Ai, Hi);
        for (int64_t r = 0; r < T; ++r)
            for (int64_t j = 0; j < fs; ++j) {
                Hi[r * fs + j] += a[c0 + j];
                Gi[r * fs + j] = act_fn(act, Hi[r * fs + j]);
            }
        /* row-parallel half: partial output, summed over shards */
        mm_nn(T, h, fs, Gi, Bi, Pi);
        for (int64_t i = 0; i < T * h; ++i) Y[i] += Pi[i];
        if (Y_part) memcpy(Y_part + s * T * h, Pi, sizeof(double) * (size_t)(T * h));
        /* backward through the shard */
        mm_nt(T, fs, h, dY, Bi, dHi);
        for (int64_t r = 0; r < T; ++r)
            for (int64_t j = 0; j < fs; ++j) dHi[r * fs + j] *= act_grad(act, Hi[r * fs + j]);
        mm_nt(T, h, fs, dHi, Ai, dXi);
        for (int64_t i = 0; i < T * h; ++i) dX[i] += dXi[i];
        if (dX_part) memcpy(dX_part + s * T * h, dXi, sizeof(double) * (size_t)(T * h));
        mm_tn(h, fs, T, X, dHi, dAi);
        mm_tn(fs, h, T, Gi, dY, dBi);
        for (int64_t k = 0; k < h; ++k)
            for (int64_t j = 0; j < fs; ++j) dA[k * f + c0 + j] = dAi[k * fs + j];
        for (int64_t j = 0; j < fs; ++j)
            for (int64_t n = 0; n < h; ++n) dB[(c0 + j) * h + n] = dBi[j * h + n];
        colsum(T, fs, dHi, da + c0);
    }
    for (int64_t r = 0; r < T; ++r)
        for (int64_t n = 0; n < h; ++n) Y[r * h + n] += b[n];
    colsum(T, h, dY, db);
    free(Ai); free(Bi); free(Hi); free(Gi); free(dHi); free(Pi); free(dXi); free(dAi); free(dBi);
    return 0;
}

/* ---- sampled entries over bf16 inputs (large workloads) ---------------------------- */

/* bf16 bit pattern -> fp64, exact: a bf16 is the top half of an IEEE binary32. */
static double bf16d(uint16_t v)
{
    uint32_t u = (uint32_t)v << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

/* The same block as oracle_mlp_forward/backward, evaluated only where asked, with the
 * inputs given as bf16 bit patterns:
 *   for each sampled token r = rows[i]:  Y[r,:] and dX[r,:]   -> Yr[i*h+n], dXr[i*h+k]
 *   for each sampled column j = cols[c]: dA[:,j], dB[j,:], da[j] -> dAc[c*h+k], dBc[c*h+n], dac[c]
 *   and all of db.
 * Each sampled entry is the full sum of its definition; nothing is approximated. */
int oracle_mlp_sampled_bf16(int64_t T, int64_t h, int64_t f, int act,
                            const uint16_t *X, const uint16_t *A, const uint16_t *a,
                            const uint16_t *B, const uint16_t *b, const uint16_t *dY,
                            int64_t nR, const int64_t *rows, int64_t nC, const int64_t *cols,
                            double *Yr, double *dXr, double *dAc, double *dBc, double *dac,
                            double *db)
{
    if (T < 1 || h < 1 || f < 1) return 1;
    for (int64_t i = 0; i < nR; ++i) if (rows[i] < 0 || rows[i] >= T) return 1;
    for (int64_t c = 0; c < nC; ++c) if (cols[c] < 0 || cols[c] >= f) return 1;

    /* sampled tokens: one row of H, G, dG, dH each */
#pragma omp parallel
    {
        double *x = malloc(sizeof(double) * (size_t)h), *dy = malloc(sizeof(double) * (size_t)h);
        double *Hr = malloc(sizeof(double) * (size_t)f), *Gr = malloc(sizeof(double) * (size_t)f);
        double *dHr = malloc(sizeof(double) * (size_t)f);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nR; ++i) {
            int64_t r = rows[i];
            for (int64_t k = 0; k < h; ++k) { x[k] = bf16d(X[r * h + k]); dy[k] = bf16d(dY[r * h + k]); }
            for (int64_t j = 0; j < f; ++j) Hr[j] = 0.0;
            for (int64_t k = 0; k < h; ++k) {
                double xk = x[k];
                const uint16_t *Ak = A + k * f;
                for (int64_t j = 0; j < f; ++j) Hr[j] += xk * bf16d(Ak[j]);
            }
            for (int64_t j = 0; j < f; ++j) {
                Hr[j] += bf16d(a[j]);
                Gr[j] = act_fn(act, Hr[j]);
            }
            for (int64_t n = 0; n < h; ++n) Yr[i * h + n] = bf16d(b[n]);
            for (int64_t j = 0; j < f; ++j) {
                double g = Gr[j], dg = 0.0;
                const uint16_t *Bj = B + j * h;
                for (int64_t n = 0; n < h; ++n) {
                    double bjn = bf16d(Bj[n]);
                    Yr[i * h + n] += g * bjn;
                    dg += dy[n] * bjn;
                }
                dHr[j] = dg * act_grad(act, Hr[j]);
            }
            for (int64_t k = 0; k < h; ++k) {
                const uint16_t *Ak = A + k * f;
                double s = 0.0;
                for (int64_t j = 0; j < f; ++j) s += dHr[j] * bf16d(Ak[j]);
                dXr[i * h + k] = s;
            }
        }
        free(x); free(dy); free(Hr); free(Gr); free(dHr);
    }

    /* sampled columns: one column of H, G, dG, dH each, over all tokens */
#pragma omp parallel
    {
        double *Acol = malloc(sizeof(double) * (size_t)h), *Brow = malloc(sizeof(double) * (size_t)h);
        double *Hc = malloc(sizeof(double) * (size_t)T), *Gc = malloc(sizeof(double) * (size_t)T);
        double *dHc = malloc(sizeof(double) * (size_t)T);
#pragma omp for schedule(dynamic, 1)
        for (int64_t c = 0; c < nC; ++c) {
            int64_t j = cols[c];
            for (int64_t k = 0; k < h; ++k) Acol[k] = bf16d(A[k * f + j]);
            for (int64_t n = 0; n < h; ++n) Brow[n] = bf16d(B[j * h + n]);
            double aj = bf16d(a[j]);
            for (int64_t r = 0; r < T; ++r) {
                double s = 0.0, dg = 0.0;
                for (int64_t k = 0; k < h; ++k) s += bf16d(X[r * h + k]) * Acol[k];
                Hc[r] = s + aj;
                Gc[r] = act_fn(act, Hc[r]);
                for (int64_t n = 0; n < h; ++n) dg += bf16d(dY[r * h + n]) * Brow[n];
                dHc[r] = dg * act_grad(act, Hc[r]);
            }
            double sa = 0.0;
            for (int64_t r = 0; r < T; ++r) sa += dHc[r];
            dac[c] = sa;
            for (int64_t k = 0; k < h; ++k) dAc[c * h + k] = 0.0;
            for (int64_t n = 0; n < h; ++n) dBc[c * h + n] = 0.0;
            for (int64_t r = 0; r < T; ++r) {
                double dh = dHc[r], g = Gc[r];
                for (int64_t k = 0; k < h; ++k) dAc[c * h + k] += bf16d(X[r * h + k]) * dh;
                for (int64_t n = 0; n < h; ++n) dBc[c * h + n] += g * bf16d(dY[r * h + n]);
            }
        }
        free(Acol); free(Brow); free(Hc); free(Gc); free(dHc);
    }

#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < h; ++n) {
        double s = 0.0;
        for (int64_t r = 0; r < T; ++r) s += bf16d(dY[r * h + n]);
        db[n] = s;
    }
    return 0;
}

/* ---- bias + dropout + residual add on the block output ------------------------------ */

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC 2011): ten rounds of the 4x32 Philox S-box on a 128-bit counter, keyed by a 64-bit key
 * that is bumped by the Weyl constants between rounds. */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0; /* multiplier of the first pair */
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2; /* multiplier of the second pair */
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Dropout keep mask of a [T,h] tensor: element e = r*h + c draws word (e % 4) of Philox on
 * counter (lo32(e/4), hi32(e/4), lo32(offset), hi32(offset)) with key (lo32(seed),
 * hi32(seed)); its top 24 bits u24 keep the element when u24 >= floor(p * 2^24). */
int oracle_dropout_keep(int64_t T, int64_t h, double p, uint64_t seed, uint64_t offset, uint8_t *keep)
{
    if (T < 0 || h < 1 || !(p >= 0.0 && p < 1.0)) return 1;
    const uint32_t p24 = (uint32_t)floor(p * 16777216.0);
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    const int64_t n = T * h;
#pragma omp parallel for schedule(static)
    for (int64_t q = 0; q < (n + 3) / 4; ++q) {
        uint32_t ctr[4] = {(uint32_t)q, (uint32_t)((uint64_t)q >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)};
        uint32_t out[4];
        oracle_philox4x32_10(ctr, key, out);
        for (int w = 0; w < 4; ++w) {
            int64_t e = 4 * q + w;
            if (e < n) keep[e] = (uint8_t)((out[w] >> 8) >= p24);
        }
    }
    return 0;
}

/* The fused output step of "Efficient Large-Scale Language Model Training ... Megatron-LM"
 * (section 3, "Fused element-wise kernels": bias + dropout + residual add), applied to the
 * block output of Figure 5a (Z = Dropout(Y B)) with the residual stream R:
 *   Z = R + keep (.) (G B + b) / (1 - p)        with Y = G B + b from oracle_mlp_forward.
 * Backward: dL/dY = dL/dZ (.) keep / (1 - p), dL/dR = dL/dZ. */
int oracle_residual_dropout(int64_t T, int64_t h, double p, const double *Y, const double *R,
                            const uint8_t *keep, double *Z)
{
    if (T < 0 || h < 1 || !(p >= 0.0 && p < 1.0)) return 1;
    const double scale = 1.0 / (1.0 - p);
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < T * h; ++e) Z[e] = R[e] + (keep[e] ? Y[e] * scale : 0.0);
    return 0;
}

int oracle_dropout_backward(int64_t T, int64_t h, double p, const double *dZ, const uint8_t *keep, double *dY)
{
    if (T < 0 || h < 1 || !(p >= 0.0 && p < 1.0)) return 1;
    const double scale = 1.0 / (1.0 - p);
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < T * h; ++e) dY[e] = keep[e] ? dZ[e] * scale : 0.0;
    return 0;
}

/* ---- SwiGLU variant of the block ----------------------------------------------------- */

/* "Distributed training" (ml-interview-book), section 7 "Exercises", exercise 3: the SwiGLU
 * MLP Y = (SiLU(X A) (.) X Wg) B with A and Wg both split by columns and B by rows; each
 * shard's SiLU and product are shard-local, so Y = sum_i (SiLU(X A_i) (.) X Wg_i) B_i and
 * one sum remains. No biases, as on the page. SiLU(x) = x sigma(x). */
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double silu(double x) { return x * sigmoid(x); }
/* d/dx x sigma(x) = sigma(x) + x sigma(x) (1 - sigma(x)) */
static double silu_grad(double x)
{
    double s = sigmoid(x);
    return s + x * s * (1.0 - s);
}

double oracle_silu(double x) { return silu(x); }
double oracle_silu_grad(double x) { return silu_grad(x); }

/* Ha = X A, Hg = X Wg, U = SiLU(Ha) (.) Hg, Y = U B. */
int oracle_swiglu_forward(int64_t T, int64_t h, int64_t f, const double *X, const double *A, const double *Wg,
                          const double *B, double *Ha, double *Hg, double *U, double *Y)
{
    if (T < 0 || h < 1 || f < 1) return 1;
    mm_nn(T, f, h, X, A, Ha);
    mm_nn(T, f, h, X, Wg, Hg);
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < T * f; ++e) U[e] = silu(Ha[e]) * Hg[e];
    mm_nn(T, h, f, U, B, Y);
    return 0;
}

/* Chain rule: dU = dY B^T; dHa = dU (.) Hg (.) SiLU'(Ha); dHg = dU (.) SiLU(Ha);
 * dX = dHa A^T + dHg Wg^T; dA = X^T dHa; dWg = X^T dHg; dB = U^T dY. */
int oracle_swiglu_backward(int64_t T, int64_t h, int64_t f, const double *X, const double *A, const double *Wg,
                           const double *B, const double *Ha, const double *Hg, const double *U, const double *dY,
                           double *dX, double *dA, double *dWg, double *dB)
{
    if (T < 0 || h < 1 || f < 1) return 1;
    size_t n = (size_t)(T * f > 0 ? T * f : 1);
    double *dU = malloc(sizeof(double) * n), *dHa = malloc(sizeof(double) * n), *dHg = malloc(sizeof(double) * n);
    double *dX2 = malloc(sizeof(double) * (size_t)(T * h > 0 ? T * h : 1));
    if (!dU || !dHa || !dHg || !dX2) return 2;
    mm_nt(T, f, h, dY, B, dU);
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < T * f; ++e) {
        dHa[e] = dU[e] * Hg[e] * silu_grad(Ha[e]);
        dHg[e] = dU[e] * silu(Ha[e]);
    }
    mm_nt(T, h, f, dHa, A, dX);
    mm_nt(T, h, f, dHg, Wg, dX2);
    for (int64_t e = 0; e < T * h; ++e) dX[e] += dX2[e];
    mm_tn(h, f, T, X, dHa, dA);
    mm_tn(h, f, T, X, dHg, dWg);
    mm_tn(f, h, T, U, dY, dB);
    free(dU); free(dHa); free(dHg); free(dX2);
    return 0;
}

/* Shard by shard, with the explicit sums over shards of the partial outputs (forward) and
 * of the partial input gradients (backward); Y_part, dX_part (optional) get [t,T,h]. */
int oracle_swiglu_sharded(int64_t T, int64_t h, int64_t f, int64_t t, const double *X, const double *A,
                          const double *Wg, const double *B, const double *dY, double *Y, double *dX, double *dA,
                          double *dWg, double *dB, double *Y_part, double *dX_part)
{
    if (T < 0 || h < 1 || f < 1 || t < 1 || f % t != 0) return 1;
    int64_t fs = f / t;
    size_t nhf = (size_t)(h * fs), nTf = (size_t)(T * fs > 0 ? T * fs : 1), nTh = (size_t)(T * h > 0 ? T * h : 1);
    double *Ai = malloc(sizeof(double) * nhf), *Wi = malloc(sizeof(double) * nhf), *Bi = malloc(sizeof(double) * nhf);
    double *Ha = malloc(sizeof(double) * nTf), *Hg = malloc(sizeof(double) * nTf), *U = malloc(sizeof(double) * nTf);
    double *P = malloc(sizeof(double) * nTh), *dXi = malloc(sizeof(double) * nTh);
    double *dAi = malloc(sizeof(double) * nhf), *dWi = malloc(sizeof(double) * nhf), *dBi = malloc(sizeof(double) * nhf);
    if (!Ai || !Wi || !Bi || !Ha || !Hg || !U || !P || !dXi || !dAi || !dWi || !dBi) return 2;
    for (int64_t i = 0; i < T * h; ++i) { Y[i] = 0.0; dX[i] = 0.0; }
    for (int64_t s = 0; s < t; ++s) {
        int64_t c0 = s * fs;
        for (int64_t k = 0; k < h; ++k)
            for (int64_t j = 0; j < fs; ++j) {
                Ai[k * fs + j] = A[k * f + c0 + j];
                Wi[k * fs + j] = Wg[k * f + c0 + j];
            }
        for (int64_t j = 0; j < fs; ++j)
            for (int64_t n = 0; n < h; ++n) Bi[j * h + n] = B[(c0 + j) * h + n];
        oracle_swiglu_forward(T, h, fs, X, Ai, Wi, Bi, Ha, Hg, U, P);
        for (int64_t i = 0; i < T * h; ++i) Y[i] += P[i];
        if (Y_part) memcpy(Y_part + s * T * h, P, sizeof(double) * (size_t)(T * h));
        oracle_swiglu_backward(T, h, fs, X, Ai, Wi, Bi, Ha, Hg, U, dY, dXi, dAi, dWi, dBi);
        for (int64_t i = 0; i < T * h; ++i) dX[i] += dXi[i];
        if (dX_part) memcpy(dX_part + s * T * h, dXi, sizeof(double) * (size_t)(T * h));
        for (int64_t k = 0; k < h; ++k)
            for (int64_t j = 0; j < fs; ++j) {
                dA[k * f + c0 + j] = dAi[k * fs + j];
                dWg[k * f + c0 + j] = dWi[k * fs + j];
            }
        for (int64_t j = 0; j < fs; ++j)
            for (int64_t n = 0; n < h; ++n) dB[(c0 + j) * h + n] = dBi[j * h + n];
    }
    free(Ai); free(Wi); free(Bi); free(Ha); free(Hg); free(U); free(P); free(dXi); free(dAi); free(dWi); free(dBi);
    return 0;
}

/* The SwiGLU block evaluated only where asked, over bf16 inputs (as oracle_mlp_sampled_bf16):
 * sampled tokens rows[i] -> Y[r,:], dX[r,:]; sampled columns cols[c] -> dA[:,j], dWg[:,j],
 * dB[j,:]. Each entry is the full sum of its definition. */
int oracle_swiglu_sampled_bf16(int64_t T, int64_t h, int64_t f, const uint16_t *X, const uint16_t *A,
                               const uint16_t *Wg, const uint16_t *B, const uint16_t *dY, int64_t nR,
                               const int64_t *rows, int64_t nC, const int64_t *cols, double *Yr, double *dXr,
                               double *dAc, double *dWc, double *dBc)
{
    if (T < 1 || h < 1 || f < 1) return 1;
    for (int64_t i = 0; i < nR; ++i) if (rows[i] < 0 || rows[i] >= T) return 1;
    for (int64_t c = 0; c < nC; ++c) if (cols[c] < 0 || cols[c] >= f) return 1;
#pragma omp parallel
    {
        double *x = malloc(sizeof(double) * (size_t)h), *dy = malloc(sizeof(double) * (size_t)h);
        double *ha = malloc(sizeof(double) * (size_t)f), *hg = malloc(sizeof(double) * (size_t)f);
        double *dha = malloc(sizeof(double) * (size_t)f), *dhg = malloc(sizeof(double) * (size_t)f);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nR; ++i) {
            int64_t r = rows[i];
            for (int64_t k = 0; k < h; ++k) { x[k] = bf16d(X[r * h + k]); dy[k] = bf16d(dY[r * h + k]); }
            for (int64_t j = 0; j < f; ++j) { ha[j] = 0.0; hg[j] = 0.0; }
            for (int64_t k = 0; k < h; ++k)
                for (int64_t j = 0; j < f; ++j) {
                    ha[j] += x[k] * bf16d(A[k * f + j]);
                    hg[j] += x[k] * bf16d(Wg[k * f + j]);
                }
            for (int64_t n = 0; n < h; ++n) Yr[i * h + n] = 0.0;
            for (int64_t j = 0; j < f; ++j) {
                double u = silu(ha[j]) * hg[j], du = 0.0;
                for (int64_t n = 0; n < h; ++n) {
                    double bjn = bf16d(B[j * h + n]);
                    Yr[i * h + n] += u * bjn;
                    du += dy[n] * bjn;
                }
                dha[j] = du * hg[j] * silu_grad(ha[j]);
                dhg[j] = du * silu(ha[j]);
            }
            for (int64_t k = 0; k < h; ++k) {
                double s = 0.0;
                for (int64_t j = 0; j < f; ++j) s += dha[j] * bf16d(A[k * f + j]) + dhg[j] * bf16d(Wg[k * f + j]);
                dXr[i * h + k] = s;
            }
        }
        free(x); free(dy); free(ha); free(hg); free(dha); free(dhg);
    }
#pragma omp parallel
    {
        double *ac = malloc(sizeof(double) * (size_t)h), *wc = malloc(sizeof(double) * (size_t)h);
        double *br = malloc(sizeof(double) * (size_t)h);
#pragma omp for schedule(dynamic, 1)
        for (int64_t c = 0; c < nC; ++c) {
            int64_t j = cols[c];
            for (int64_t k = 0; k < h; ++k) { ac[k] = bf16d(A[k * f + j]); wc[k] = bf16d(Wg[k * f + j]); }
            for (int64_t n = 0; n < h; ++n) br[n] = bf16d(B[j * h + n]);
            for (int64_t k = 0; k < h; ++k) { dAc[c * h + k] = 0.0; dWc[c * h + k] = 0.0; }
            for (int64_t n = 0; n < h; ++n) dBc[c * h + n] = 0.0;
            for (int64_t r = 0; r < T; ++r) {
                double a = 0.0, g = 0.0, du = 0.0;
                for (int64_t k = 0; k < h; ++k) {
                    double xv = bf16d(X[r * h + k]);
                    a += xv * ac[k];
                    g += xv * wc[k];
                }
                for (int64_t n = 0; n < h; ++n) du += bf16d(dY[r * h + n]) * br[n];
                double dha = du * g * silu_grad(a), dhg = du * silu(a), u = silu(a) * g;
                for (int64_t k = 0; k < h; ++k) {
                    double xv = bf16d(X[r * h + k]);
                    dAc[c * h + k] += xv * dha;
                    dWc[c * h + k] += xv * dhg;
                }
                for (int64_t n = 0; n < h; ++n) dBc[c * h + n] += u * bf16d(dY[r * h + n]);
            }
        }
        free(ac); free(wc); free(br);
    }
    return 0;
}

/* ---- head-parallel self-attention block ---------------------------------------------- */

/* "Efficient Large-Scale Language Model Training ... Megatron-LM", section 3, Figure 5b, and
 * "Distributed training" (ml-interview-book), section 3.2 (tensor_parallel_attention): the
 * heads are split across t shards (Wq, Wk, Wv by columns grouped by head, Wo by rows), each
 * shard computes its heads' attention locally and the outputs of Wo sum over shards.
 * Tokens are [b, s] (T = b*s rows, batch-major); each head sees only its own sequence.
 *   Q = X Wq, K = X Wk, V = X Wv                               [T, hd]
 *   S = Q_h K_h^T / sqrt(d) (+ causal mask: key > query -> -inf), P = softmax_rows(S)
 *   C_h = P V_h, C = [C_1 | ... | C_a]                           [T, hd]
 *   Y = C Wo                                                     [T, h]
 * with a heads of width d (hd = a*d columns; the pages use hd = h). No biases. */
static void attn_core_forward(int64_t b, int64_t s, int64_t a, int64_t d, int causal, const double *Q,
                              const double *K, const double *V, double *P, double *C, double *L)
{
    const int64_t hd = a * d;
    const double scale = 1.0 / sqrt((double)d);
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t bi = 0; bi < b; ++bi)
        for (int64_t hh = 0; hh < a; ++hh) {
            double *Pbh = P + (bi * a + hh) * s * s;
            for (int64_t i = 0; i < s; ++i) {
                const double *q = Q + (bi * s + i) * hd + hh * d;
                double m = -INFINITY;
                for (int64_t j = 0; j < s; ++j) {
                    double v = -INFINITY;
                    if (!causal || j <= i) {
                        const double *k = K + (bi * s + j) * hd + hh * d;
                        double dot = 0.0;
                        for (int64_t e = 0; e < d; ++e) dot += q[e] * k[e];
                        v = dot * scale;
                    }
                    Pbh[i * s + j] = v;
                    if (v > m) m = v;
                }
                double sum = 0.0;
                for (int64_t j = 0; j < s; ++j) {
                    double e = (Pbh[i * s + j] == -INFINITY) ? 0.0 : exp(Pbh[i * s + j] - m);
                    Pbh[i * s + j] = e;
                    sum += e;
                }
                for (int64_t j = 0; j < s; ++j) Pbh[i * s + j] /= sum;
                /* base-2 log-sum-exp of the row's scaled scores: log2 sum_j exp(S_ij) */
                if (L) L[(bi * a + hh) * s + i] = (m + log(sum)) / log(2.0);
                double *c = C + (bi * s + i) * hd + hh * d;
                for (int64_t e = 0; e < d; ++e) c[e] = 0.0;
                for (int64_t j = 0; j < s; ++j) {
                    const double p = Pbh[i * s + j];
                    if (p == 0.0) continue;
                    const double *v = V + (bi * s + j) * hd + hh * d;
                    for (int64_t e = 0; e < d; ++e) c[e] += p * v[e];
                }
            }
        }
}

int oracle_attn_forward(int64_t b, int64_t s, int64_t h, int64_t a, int64_t d, int causal, const double *X,
                        const double *Wq, const double *Wk, const double *Wv, const double *Wo, double *Q,
                        double *K, double *V, double *P, double *C, double *Y, double *L)
{
    if (b < 1 || s < 1 || h < 1 || a < 1 || d < 1) return 1;
    const int64_t T = b * s, hd = a * d;
    mm_nn(T, hd, h, X, Wq, Q);
    mm_nn(T, hd, h, X, Wk, K);
    mm_nn(T, hd, h, X, Wv, V);
    attn_core_forward(b, s, a, d, causal, Q, K, V, P, C, L);
    mm_nn(T, h, hd, C, Wo, Y);
    return 0;
}

/* Backward given dY: dC = dY Wo^T; dWo = C^T dY; per head dV = P^T dC_h, dP = dC_h V_h^T,
 * dS = P (.) (dP - rowsum(dP (.) P)), dQ_h = dS K_h / sqrt(d), dK_h = dS^T Q_h / sqrt(d);
 * dX = dQ Wq^T + dK Wk^T + dV Wv^T; dWq = X^T dQ; dWk = X^T dK; dWv = X^T dV. */
int oracle_attn_backward(int64_t b, int64_t s, int64_t h, int64_t a, int64_t d, const double *X,
                         const double *Wq, const double *Wk, const double *Wv, const double *Wo, const double *Q,
                         const double *K, const double *V, const double *P, const double *C, const double *dY,
                         double *dX, double *dWq, double *dWk, double *dWv, double *dWo)
{
    if (b < 1 || s < 1 || h < 1 || a < 1 || d < 1) return 1;
    const int64_t T = b * s, hd = a * d;
    const double scale = 1.0 / sqrt((double)d);
    double *dC = malloc(sizeof(double) * (size_t)(T * hd)), *dQ = calloc((size_t)(T * hd), sizeof(double));
    double *dK = calloc((size_t)(T * hd), sizeof(double)), *dV = calloc((size_t)(T * hd), sizeof(double));
    double *tmp = malloc(sizeof(double) * (size_t)(T * h));
    if (!dC || !dQ || !dK || !dV || !tmp) return 2;
    mm_nt(T, hd, h, dY, Wo, dC);
    mm_tn(hd, h, T, C, dY, dWo);
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t bi = 0; bi < b; ++bi)
        for (int64_t hh = 0; hh < a; ++hh) {
            const double *Pbh = P + (bi * a + hh) * s * s;
            double *dS = malloc(sizeof(double) * (size_t)(s * s));
            for (int64_t i = 0; i < s; ++i) {
                const double *dc = dC + (bi * s + i) * hd + hh * d;
                double rs = 0.0;
                for (int64_t j = 0; j < s; ++j) {
                    const double *v = V + (bi * s + j) * hd + hh * d;
                    double dp = 0.0;
                    for (int64_t e = 0; e < d; ++e) dp += dc[e] * v[e];
                    dS[i * s + j] = dp;
                    rs += dp * Pbh[i * s + j];
                }
                for (int64_t j = 0; j < s; ++j) dS[i * s + j] = Pbh[i * s + j] * (dS[i * s + j] - rs);
            }
            for (int64_t i = 0; i < s; ++i)
                for (int64_t j = 0; j < s; ++j) {
                    const double p = Pbh[i * s + j], g = dS[i * s + j] * scale;
                    const double *dc = dC + (bi * s + i) * hd + hh * d;
                    double *dv = dV + (bi * s + j) * hd + hh * d;
                    double *dq = dQ + (bi * s + i) * hd + hh * d;
                    double *dk = dK + (bi * s + j) * hd + hh * d;
                    const double *k = K + (bi * s + j) * hd + hh * d;
                    const double *q = Q + (bi * s + i) * hd + hh * d;
                    for (int64_t e = 0; e < d; ++e) {
                        dv[e] += p * dc[e];
                        dq[e] += g * k[e];
                        dk[e] += g * q[e];
                    }
                }
            free(dS);
        }
    mm_nt(T, h, hd, dQ, Wq, dX);
    mm_nt(T, h, hd, dK, Wk, tmp);
    for (int64_t e = 0; e < T * h; ++e) dX[e] += tmp[e];
    mm_nt(T, h, hd, dV, Wv, tmp);
    for (int64_t e = 0; e < T * h; ++e) dX[e] += tmp[e];
    mm_tn(h, hd, T, X, dQ, dWq);
    mm_tn(h, hd, T, X, dK, dWk);
    mm_tn(h, hd, T, X, dV, dWv);
    free(dC); free(dQ); free(dK); free(dV); free(tmp);
    return 0;
}

/* Shard by shard: shard i owns heads [i a/t, (i+1) a/t): its columns of Wq, Wk, Wv and its
 * rows of Wo; Y = sum_i C_i Wo_i (the one sum), dX = sum_i dX_i. Y_part, dX_part (optional)
 * receive the per-shard partials [t,T,h]. */
int oracle_attn_sharded(int64_t b, int64_t s, int64_t h, int64_t a, int64_t d, int64_t t, int causal,
                        const double *X, const double *Wq, const double *Wk, const double *Wv, const double *Wo,
                        const double *dY, double *Y, double *dX, double *dWq, double *dWk, double *dWv,
                        double *dWo, double *Y_part, double *dX_part)
{
    if (b < 1 || s < 1 || h < 1 || a < 1 || d < 1 || t < 1 || a % t != 0) return 1;
    const int64_t T = b * s, hd = a * d, as = a / t, cs = as * d;
    size_t nw = (size_t)(h * cs), nt = (size_t)(T * cs), nth = (size_t)(T * h);
    double *q = malloc(sizeof(double) * nw), *k = malloc(sizeof(double) * nw), *v = malloc(sizeof(double) * nw);
    double *o = malloc(sizeof(double) * nw), *Qi = malloc(sizeof(double) * nt), *Ki = malloc(sizeof(double) * nt);
    double *Vi = malloc(sizeof(double) * nt), *Ci = malloc(sizeof(double) * nt);
    double *Pi = malloc(sizeof(double) * (size_t)(b * as * s * s)), *Yi = malloc(sizeof(double) * nth);
    double *dXi = malloc(sizeof(double) * nth), *gq = malloc(sizeof(double) * nw), *gk = malloc(sizeof(double) * nw);
    double *gv = malloc(sizeof(double) * nw), *go = malloc(sizeof(double) * nw);
    if (!q || !k || !v || !o || !Qi || !Ki || !Vi || !Ci || !Pi || !Yi || !dXi || !gq || !gk || !gv || !go) return 2;
    for (int64_t e = 0; e < T * h; ++e) { Y[e] = 0.0; dX[e] = 0.0; }
    for (int64_t sh = 0; sh < t; ++sh) {
        const int64_t c0 = sh * cs;
        for (int64_t r = 0; r < h; ++r)
            for (int64_t c = 0; c < cs; ++c) {
                q[r * cs + c] = Wq[r * hd + c0 + c];
                k[r * cs + c] = Wk[r * hd + c0 + c];
                v[r * cs + c] = Wv[r * hd + c0 + c];
            }
        for (int64_t c = 0; c < cs; ++c)
            for (int64_t n = 0; n < h; ++n) o[c * h + n] = Wo[(c0 + c) * h + n];
        oracle_attn_forward(b, s, h, as, d, causal, X, q, k, v, o, Qi, Ki, Vi, Pi, Ci, Yi, NULL);
        for (int64_t e = 0; e < T * h; ++e) Y[e] += Yi[e];
        if (Y_part) memcpy(Y_part + sh * T * h, Yi, sizeof(double) * nth);
        oracle_attn_backward(b, s, h, as, d, X, q, k, v, o, Qi, Ki, Vi, Pi, Ci, dY, dXi, gq, gk, gv, go);
        for (int64_t e = 0; e < T * h; ++e) dX[e] += dXi[e];
        if (dX_part) memcpy(dX_part + sh * T * h, dXi, sizeof(double) * nth);
        for (int64_t r = 0; r < h; ++r)
            for (int64_t c = 0; c < cs; ++c) {
                dWq[r * hd + c0 + c] = gq[r * cs + c];
                dWk[r * hd + c0 + c] = gk[r * cs + c];
                dWv[r * hd + c0 + c] = gv[r * cs + c];
            }
        for (int64_t c = 0; c < cs; ++c)
            for (int64_t n = 0; n < h; ++n) dWo[(c0 + c) * h + n] = go[c * h + n];
    }
    free(q); free(k); free(v); free(o); free(Qi); free(Ki); free(Vi); free(Ci); free(Pi); free(Yi); free(dXi);
    free(gq); free(gk); free(gv); free(go);
    return 0;
}

/* Sampled attention outputs at sizes where the whole block is too slow on a CPU: for each
 * listed head and token row, C[row, head] (d values) and L[row, head], from bf16 inputs
 * (raw bits). For every (sequence, head) touched, K and V of the head are computed over the
 * positions the sampled rows can see, then each row's scores, softmax and P V, all fp64. */
int oracle_attn_sampled_bf16(int64_t b, int64_t s, int64_t h, int64_t a, int64_t d, int causal, const uint16_t *X,
                             const uint16_t *Wq, const uint16_t *Wk, const uint16_t *Wv, const int64_t *rows,
                             int64_t nrows, const int64_t *heads, int64_t nheads, double *C_out, double *L_out)
{
    if (b < 1 || s < 1 || h < 1 || a < 1 || d < 1) return 1;
    const int64_t hd = a * d, T = b * s;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= T) return 1;
    for (int64_t k = 0; k < nheads; ++k)
        if (heads[k] < 0 || heads[k] >= a) return 1;
    double *Wcol = malloc(sizeof(double) * (size_t)(h * d * 3));
    double *Kh = malloc(sizeof(double) * (size_t)(s * d)), *Vh = malloc(sizeof(double) * (size_t)(s * d));
    double *sc = malloc(sizeof(double) * (size_t)s), *q = malloc(sizeof(double) * (size_t)d);
    if (!Wcol || !Kh || !Vh || !sc || !q) return 2;
    const double scale = 1.0 / sqrt((double)d);
    for (int64_t hk = 0; hk < nheads; ++hk) {
        const int64_t hh = heads[hk], c0 = hh * d;
        for (int64_t i = 0; i < h; ++i)
            for (int64_t e = 0; e < d; ++e) {
                Wcol[(0 * h + i) * d + e] = bf16d(Wq[i * hd + c0 + e]);
                Wcol[(1 * h + i) * d + e] = bf16d(Wk[i * hd + c0 + e]);
                Wcol[(2 * h + i) * d + e] = bf16d(Wv[i * hd + c0 + e]);
            }
        for (int64_t bi = 0; bi < b; ++bi) {
            int64_t pmax = -1;
            for (int64_t r = 0; r < nrows; ++r)
                if (rows[r] / s == bi) {
                    const int64_t p = rows[r] % s;
                    const int64_t need = causal ? p : s - 1;
                    if (need > pmax) pmax = need;
                }
            if (pmax < 0) continue;
#pragma omp parallel for schedule(static)
            for (int64_t p = 0; p <= pmax; ++p) {
                const uint16_t *x = X + (bi * s + p) * h;
                for (int64_t e = 0; e < d; ++e) { Kh[p * d + e] = 0.0; Vh[p * d + e] = 0.0; }
                for (int64_t i = 0; i < h; ++i) {
                    const double xv = bf16d(x[i]);
                    const double *wk = Wcol + (1 * h + i) * d, *wv = Wcol + (2 * h + i) * d;
                    for (int64_t e = 0; e < d; ++e) {
                        Kh[p * d + e] += xv * wk[e];
                        Vh[p * d + e] += xv * wv[e];
                    }
                }
            }
            for (int64_t r = 0; r < nrows; ++r) {
                if (rows[r] / s != bi) continue;
                const int64_t p = rows[r] % s, nk = causal ? p + 1 : s;
                const uint16_t *x = X + rows[r] * h;
                for (int64_t e = 0; e < d; ++e) q[e] = 0.0;
                for (int64_t i = 0; i < h; ++i) {
                    const double xv = bf16d(x[i]);
                    for (int64_t e = 0; e < d; ++e) q[e] += xv * Wcol[(0 * h + i) * d + e];
                }
                double m = -INFINITY;
                for (int64_t j = 0; j < nk; ++j) {
                    double dot = 0.0;
                    for (int64_t e = 0; e < d; ++e) dot += q[e] * Kh[j * d + e];
                    sc[j] = dot * scale;
                    if (sc[j] > m) m = sc[j];
                }
                double sum = 0.0;
                for (int64_t j = 0; j < nk; ++j) { sc[j] = exp(sc[j] - m); sum += sc[j]; }
                double *c = C_out + (r * nheads + hk) * d;
                for (int64_t e = 0; e < d; ++e) c[e] = 0.0;
                for (int64_t j = 0; j < nk; ++j)
                    for (int64_t e = 0; e < d; ++e) c[e] += sc[j] / sum * Vh[j * d + e];
                L_out[r * nheads + hk] = (m + log(sum)) / log(2.0);
            }
        }
    }
    free(Wcol); free(Kh); free(Vh); free(sc); free(q);
    return 0;
}
