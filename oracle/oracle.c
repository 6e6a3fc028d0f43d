/*
 * oracle.c -- plain float64 CPU oracle for the sharded GEMM forward/backward,
 * the column-then-row tensor-parallel MLP (plain and gated), the attention
 * projections with their head-aligned plan, and the vocabulary-sharded
 * cross-entropy.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA library; neither side includes or
 * links the other.
 *
 * Every function computes the plain, unsharded definition with triple loops
 * in double precision, in the order the definition states, except the two
 * functions named *_sharded*, which restate the pages' per-rank formulations
 * so that the tests can check sharded == unsharded.  OpenMP only distributes
 * independent output rows / columns over threads; it never splits a sum.
 *
 * Sources (web pages, cited by title and section):
 *   [SG]  "Sharded GEMM与Backprop：行、列、内维三种切分"
 *         (interview-support-pro.com, openai-sharded-matmul-backprop)
 *   [MC]  "多卡张量：拆开计算，再合回同一结果" (glenzli.com, distributed-execution)
 *   [TP]  "第 6 课：张量并行 TP" (learn.payai.win, train/lesson06)
 *
 * Arrays are dense row-major doubles unless stated.  Labels are int64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_SHAPE 1
#define ORC_ERR_PARTITION 2
#define ORC_ERR_LABEL 5

#define ORC_ACT_GELU_ERF 0
#define ORC_ACT_GELU_TANH 1
#define ORC_ACT_TANH 2
#define ORC_ACT_SILU 3

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * Shard plan.  [SG] "Python 参考实现" splits each axis with numpy's
 * array_split; [SG] "题意与假设" allows uneven and empty shards and
 * [SG] "手动走一遍" splits K=5 into 3/2.  array_split gives the first
 * (dim mod parts) shards one extra element.  Written as the running sum
 * of the shard sizes.
 * ---------------------------------------------------------------------- */
int orc_plan_shards(int64_t dim, int32_t parts, int64_t* off) {
    if (parts < 1) return ORC_ERR_PARTITION;
    if (dim < 0) return ORC_ERR_SHAPE;
    int64_t small = dim / parts;
    int64_t n_big = dim % parts;
    off[0] = 0;
    for (int32_t r = 0; r < parts; ++r) {
        int64_t size = (r < n_big) ? small + 1 : small;
        off[r + 1] = off[r] + size;
    }
    return ORC_OK;
}

/* Owner rank of index y: the r with off[r] <= y < off[r+1], by linear scan.
 * [MC] "04 / VOCABULARY SHARDS", indicator 1[y in V_r].  -1 if none. */
int32_t orc_owner(int64_t y, const int64_t* off, int32_t parts) {
    for (int32_t r = 0; r < parts; ++r)
        if (off[r] <= y && y < off[r + 1]) return r;
    return -1;
}

/* ------------------------------------------------------------------------
 * Unsharded GEMM forward and backward.  [SG] "题意与假设": L = <G, AB>;
 * [SG] "解题路线" step 1: dA = G B^T, dB = A^T G.
 * A is M x K, B is K x N, G is M x N.  Any output may be NULL.
 * ---------------------------------------------------------------------- */
void orc_matmul(int64_t M, int64_t K, int64_t N,
                const double* A, const double* B, const double* G,
                double* Y, double* dA, double* dB) {
    if (Y) {
        #pragma omp parallel for schedule(static)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n) {
                double s = 0.0;
                for (int64_t k = 0; k < K; ++k) s += A[m * K + k] * B[k * N + n];
                Y[m * N + n] = s;
            }
    }
    if (dA) {
        #pragma omp parallel for schedule(static)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t k = 0; k < K; ++k) {
                double s = 0.0;
                for (int64_t n = 0; n < N; ++n) s += G[m * N + n] * B[k * N + n];
                dA[m * K + k] = s;
            }
    }
    if (dB) {
        #pragma omp parallel for schedule(static)
        for (int64_t k = 0; k < K; ++k)
            for (int64_t n = 0; n < N; ++n) {
                double s = 0.0;
                for (int64_t m = 0; m < M; ++m) s += A[m * K + k] * G[m * N + n];
                dB[k * N + n] = s;
            }
    }
}

/* ------------------------------------------------------------------------
 * Element-wise activations and their derivatives.
 *   GELU_ERF : x * Phi(x), Phi the standard normal CDF written with erf --
 *              the default form of torch's gelu used by [TP] "参考答案".
 *   GELU_TANH: the tanh approximation of GELU (Hendrycks & Gimpel 2016),
 *              0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 *   TANH     : tanh, whose derivative [MC] "02 / BACKWARD" writes as 1 - H^2.
 *   SILU     : x sigma(x) with the logistic sigma(x) = 1 / (1 + e^{-x}), an
 *              element-wise activation [TP] core concept 2.A step 3 names;
 *              d/dx = sigma(x) + x sigma(x) (1 - sigma(x)).
 * ---------------------------------------------------------------------- */
static const double ORC_PI = 3.14159265358979323846;

double orc_act(int kind, double x) {
    if (kind == ORC_ACT_GELU_ERF) {
        return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
    } else if (kind == ORC_ACT_GELU_TANH) {
        double c = sqrt(2.0 / ORC_PI);
        return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
    } else if (kind == ORC_ACT_SILU) {
        return x / (1.0 + exp(-x));
    } else {
        return tanh(x);
    }
}

double orc_act_grad(int kind, double x) {
    if (kind == ORC_ACT_GELU_ERF) {
        /* d/dx [x Phi(x)] = Phi(x) + x phi(x), phi the normal density. */
        double cdf = 0.5 * (1.0 + erf(x / sqrt(2.0)));
        double pdf = exp(-0.5 * x * x) / sqrt(2.0 * ORC_PI);
        return cdf + x * pdf;
    } else if (kind == ORC_ACT_GELU_TANH) {
        /* u = tanh(c (x + a x^3)); d/dx = 0.5 (1+u) + 0.5 x (1-u^2) c (1 + 3a x^2) */
        double c = sqrt(2.0 / ORC_PI);
        double u = tanh(c * (x + 0.044715 * x * x * x));
        return 0.5 * (1.0 + u) + 0.5 * x * (1.0 - u * u) * c * (1.0 + 3.0 * 0.044715 * x * x);
    } else if (kind == ORC_ACT_SILU) {
        double sg = 1.0 / (1.0 + exp(-x));
        return sg + x * sg * (1.0 - sg);
    } else {
        double h = tanh(x);
        return 1.0 - h * h;
    }
}

/* ------------------------------------------------------------------------
 * Column-then-row MLP, unsharded definition.
 * Forward  [MC] "01 / COLUMN THEN ROW"; [TP] core concept 2.A:
 *     Hp = X W1,  Ha = phi(Hp),  Y = Ha W2.
 * Backward [MC] "02 / BACKWARD" (upstream G_Y given, no scaling):
 *     dHa = G_Y W2^T,  dZ = dHa * phi'(Hp),  dW2 = Ha^T G_Y,
 *     dW1 = X^T dZ,    dX = dZ W1^T.
 * Shapes: X T x d, W1 d x F (in,out), W2 F x d (in,out), G_Y T x d.
 *
 * orc_mlp_rows computes rows `rows[i]` of Y and dX (each row of Y and dX
 * depends on one row of X and G_Y only).  Outputs are nrows x d.
 * ---------------------------------------------------------------------- */
void orc_mlp_rows(int64_t T, int64_t d, int64_t F,
                  const double* X, const double* W1, const double* W2, const double* GY,
                  int act, int64_t nrows, const int64_t* rows,
                  double* Y, double* dX) {
    (void)T;
    #pragma omp parallel
    {
        double* hp = (double*)malloc(sizeof(double) * (size_t)(F > 0 ? F : 1));
        double* dz = (double*)malloc(sizeof(double) * (size_t)(F > 0 ? F : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t t = rows[i];
            /* Hp[t,:] = X[t,:] W1 */
            for (int64_t f = 0; f < F; ++f) hp[f] = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                double x = X[t * d + c];
                for (int64_t f = 0; f < F; ++f) hp[f] += x * W1[c * F + f];
            }
            /* Y[t,:] = phi(Hp[t,:]) W2 */
            if (Y) {
                for (int64_t c = 0; c < d; ++c) Y[i * d + c] = 0.0;
                for (int64_t f = 0; f < F; ++f) {
                    double ha = orc_act(act, hp[f]);
                    for (int64_t c = 0; c < d; ++c) Y[i * d + c] += ha * W2[f * d + c];
                }
            }
            if (dX) {
                /* dZ[t,f] = (G_Y[t,:] . W2[f,:]) * phi'(Hp[t,f]) */
                for (int64_t f = 0; f < F; ++f) {
                    double s = 0.0;
                    for (int64_t c = 0; c < d; ++c) s += GY[t * d + c] * W2[f * d + c];
                    dz[f] = s * orc_act_grad(act, hp[f]);
                }
                /* dX[t,:] = dZ[t,:] W1^T */
                for (int64_t c = 0; c < d; ++c) {
                    double s = 0.0;
                    for (int64_t f = 0; f < F; ++f) s += dz[f] * W1[c * F + f];
                    dX[i * d + c] = s;
                }
            }
        }
        free(hp);
        free(dz);
    }
}

/* orc_mlp_cols computes, for each selected hidden unit f = cols[j], column f
 * of dW1 (written to dW1[:, j], a d x ncols array) and row f of dW2 (written
 * to dW2[j, :], an ncols x d array).  Each needs column f of Hp over all T. */
void orc_mlp_cols(int64_t T, int64_t d, int64_t F,
                  const double* X, const double* W1, const double* W2, const double* GY,
                  int act, int64_t ncols, const int64_t* cols,
                  double* dW1, double* dW2) {
    #pragma omp parallel
    {
        double* ha = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double* dz = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t j = 0; j < ncols; ++j) {
            int64_t f = cols[j];
            for (int64_t t = 0; t < T; ++t) {
                double hp = 0.0;
                for (int64_t c = 0; c < d; ++c) hp += X[t * d + c] * W1[c * F + f];
                double dha = 0.0;
                for (int64_t c = 0; c < d; ++c) dha += GY[t * d + c] * W2[f * d + c];
                ha[t] = orc_act(act, hp);
                dz[t] = dha * orc_act_grad(act, hp);
            }
            if (dW1)
                for (int64_t c = 0; c < d; ++c) {
                    double s = 0.0;
                    for (int64_t t = 0; t < T; ++t) s += X[t * d + c] * dz[t];
                    dW1[c * ncols + j] = s;
                }
            if (dW2)
                for (int64_t c = 0; c < d; ++c) {
                    double s = 0.0;
                    for (int64_t t = 0; t < T; ++t) s += ha[t] * GY[t * d + c];
                    dW2[j * d + c] = s;
                }
        }
        free(ha);
        free(dz);
    }
}

/* ------------------------------------------------------------------------
 * Gated column-then-row MLP (SwiGLU when phi = SiLU), unsharded definition.
 * [TP] reference answer Q1 puts the "gate/up" projections and the
 * activation in the column-parallel layer and the "down" projection in the
 * row-parallel one; the gate and up weights are both split along F with the
 * same shard plan, so the element-wise gating stays shard-local exactly as
 * phi does in core concept 2.A step 3.  The gating product itself is the
 * usual gated linear unit (the pages give no formula; this is the plain
 * reading of "gate/up"):
 *     Hg = X Wg,  U = X Wu,  A = phi(Hg) * U,  Y = A W2.
 * Backward (upstream G_Y given, no scaling; chain rule through the product):
 *     dA = G_Y W2^T,  dU = dA * phi(Hg),  dHg = dA * U * phi'(Hg),
 *     dWg = X^T dHg,  dWu = X^T dU,  dW2 = A^T G_Y,
 *     dX = dHg Wg^T + dU Wu^T.
 * Shapes: X T x d, Wg and Wu d x F (in,out), W2 F x d (in,out), G_Y T x d.
 *
 * orc_glu_rows computes rows `rows[i]` of Y and dX (nrows x d each).
 * ---------------------------------------------------------------------- */
void orc_glu_rows(int64_t T, int64_t d, int64_t F,
                  const double* X, const double* Wg, const double* Wu, const double* W2, const double* GY,
                  int act, int64_t nrows, const int64_t* rows, double* Y, double* dX) {
    (void)T;
    #pragma omp parallel
    {
        double* hg = (double*)malloc(sizeof(double) * (size_t)(F > 0 ? F : 1));
        double* u = (double*)malloc(sizeof(double) * (size_t)(F > 0 ? F : 1));
        double* dhg = (double*)malloc(sizeof(double) * (size_t)(F > 0 ? F : 1));
        double* du = (double*)malloc(sizeof(double) * (size_t)(F > 0 ? F : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nrows; ++i) {
            int64_t t = rows[i];
            /* Hg[t,:] = X[t,:] Wg,  U[t,:] = X[t,:] Wu */
            for (int64_t f = 0; f < F; ++f) { hg[f] = 0.0; u[f] = 0.0; }
            for (int64_t c = 0; c < d; ++c) {
                double x = X[t * d + c];
                for (int64_t f = 0; f < F; ++f) {
                    hg[f] += x * Wg[c * F + f];
                    u[f] += x * Wu[c * F + f];
                }
            }
            if (Y) {
                /* Y[t,:] = (phi(Hg[t,:]) * U[t,:]) W2 */
                for (int64_t c = 0; c < d; ++c) Y[i * d + c] = 0.0;
                for (int64_t f = 0; f < F; ++f) {
                    double a = orc_act(act, hg[f]) * u[f];
                    for (int64_t c = 0; c < d; ++c) Y[i * d + c] += a * W2[f * d + c];
                }
            }
            if (dX) {
                for (int64_t f = 0; f < F; ++f) {
                    double da = 0.0; /* dA[t,f] = G_Y[t,:] . W2[f,:] */
                    for (int64_t c = 0; c < d; ++c) da += GY[t * d + c] * W2[f * d + c];
                    du[f] = da * orc_act(act, hg[f]);
                    dhg[f] = da * u[f] * orc_act_grad(act, hg[f]);
                }
                /* dX[t,:] = dHg[t,:] Wg^T + dU[t,:] Wu^T */
                for (int64_t c = 0; c < d; ++c) {
                    double s = 0.0;
                    for (int64_t f = 0; f < F; ++f) s += dhg[f] * Wg[c * F + f];
                    for (int64_t f = 0; f < F; ++f) s += du[f] * Wu[c * F + f];
                    dX[i * d + c] = s;
                }
            }
        }
        free(hg);
        free(u);
        free(dhg);
        free(du);
    }
}

/* orc_glu_cols computes, for each selected hidden unit f = cols[j], column f
 * of dWg and of dWu (written to column j of d x ncols arrays) and row f of
 * dW2 (row j of an ncols x d array).  Each needs column f of Hg and U over
 * all T.  Any output may be NULL. */
void orc_glu_cols(int64_t T, int64_t d, int64_t F,
                  const double* X, const double* Wg, const double* Wu, const double* W2, const double* GY,
                  int act, int64_t ncols, const int64_t* cols, double* dWg, double* dWu, double* dW2) {
    #pragma omp parallel
    {
        double* a = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double* dhg = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double* du = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t j = 0; j < ncols; ++j) {
            int64_t f = cols[j];
            for (int64_t t = 0; t < T; ++t) {
                double hg = 0.0, u = 0.0, da = 0.0;
                for (int64_t c = 0; c < d; ++c) hg += X[t * d + c] * Wg[c * F + f];
                for (int64_t c = 0; c < d; ++c) u += X[t * d + c] * Wu[c * F + f];
                for (int64_t c = 0; c < d; ++c) da += GY[t * d + c] * W2[f * d + c];
                a[t] = orc_act(act, hg) * u;
                du[t] = da * orc_act(act, hg);
                dhg[t] = da * u * orc_act_grad(act, hg);
            }
            for (int64_t c = 0; c < d; ++c) {
                double sg = 0.0, su = 0.0, s2 = 0.0;
                for (int64_t t = 0; t < T; ++t) {
                    sg += X[t * d + c] * dhg[t];
                    su += X[t * d + c] * du[t];
                    s2 += a[t] * GY[t * d + c];
                }
                if (dWg) dWg[c * ncols + j] = sg;
                if (dWu) dWu[c * ncols + j] = su;
                if (dW2) dW2[j * d + c] = s2;
            }
        }
        free(a);
        free(dhg);
        free(du);
    }
}

/* ------------------------------------------------------------------------
 * Head-aligned shard plan of the attention projections.
 * [TP] core concept 2.B: W_Q, W_K, W_V are split along the output head
 * dimension, each rank owning H / TP heads; W_O is split along its input
 * head dimension.  [TP] core concept 3.4: H must be divisible by TP; with
 * grouped-query attention (H_kv key/value heads, each shared by H / H_kv
 * query heads) TP = 8 for H = 32, H_kv = 8 gives every rank 4 query heads
 * and 1 KV head, while TP = 16 leaves the 8 KV heads indivisible and they
 * must be shared or replicated across ranks.  Reading taken: the KV heads
 * are split evenly when H_kv mod TP = 0, and each KV head is replicated on
 * TP / H_kv ranks when TP mod H_kv = 0; other combinations are rejected,
 * as is H mod H_kv != 0.
 * Outputs: q_off[0..tp] (query-head offsets, rank r owns heads
 * [q_off[r], q_off[r+1])), kv_first[0..tp-1] (first KV head of rank r),
 * *kv_count (KV heads per rank), *kv_replicas (ranks holding each KV head).
 * ---------------------------------------------------------------------- */
int orc_plan_heads(int32_t n_heads, int32_t n_kv_heads, int32_t tp, int64_t* q_off, int64_t* kv_first,
                   int32_t* kv_count, int32_t* kv_replicas) {
    if (tp < 1 || n_heads < 1 || n_kv_heads < 1) return ORC_ERR_PARTITION;
    if (n_heads % tp != 0) return ORC_ERR_PARTITION;          /* H mod TP = 0 */
    if (n_heads % n_kv_heads != 0) return ORC_ERR_PARTITION;  /* whole query groups */
    int32_t per_rank = n_heads / tp;
    for (int32_t r = 0; r <= tp; ++r) q_off[r] = (int64_t)r * per_rank;
    if (n_kv_heads % tp == 0) {
        *kv_count = n_kv_heads / tp;
        *kv_replicas = 1;
        for (int32_t r = 0; r < tp; ++r) kv_first[r] = (int64_t)r * (n_kv_heads / tp);
    } else if (tp % n_kv_heads == 0) {
        int32_t rep = tp / n_kv_heads;
        *kv_count = 1;
        *kv_replicas = rep;
        for (int32_t r = 0; r < tp; ++r) kv_first[r] = r / rep;
    } else {
        return ORC_ERR_PARTITION;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Attention projections, unsharded definitions ([TP] core concept 2.B; the
 * attention core between them is not part of this computation: its
 * outputs and gradients are inputs here).
 * QKV projections (column-parallel):  Q = X Wq, K = X Wk, V = X Wv;
 * given the upstream dQ, dK, dV:       dWq = X^T dQ, dWk = X^T dK,
 *                                      dWv = X^T dV,
 *                                      dX = dQ Wq^T + dK Wk^T + dV Wv^T.
 * X T x d; Wq d x nq; Wk, Wv d x nkv (in,out); nq = H dh, nkv = H_kv dh.
 * Any output may be NULL.
 * ---------------------------------------------------------------------- */
void orc_attn_qkv(int64_t T, int64_t d, int64_t nq, int64_t nkv,
                  const double* X, const double* Wq, const double* Wk, const double* Wv,
                  const double* dQ, const double* dK, const double* dV,
                  double* Q, double* K, double* V, double* dX, double* dWq, double* dWk, double* dWv) {
    const double* W[3] = {Wq, Wk, Wv};
    const double* G[3] = {dQ, dK, dV};
    double* O[3] = {Q, K, V};
    double* dW[3] = {dWq, dWk, dWv};
    const int64_t n[3] = {nq, nkv, nkv};
    for (int p = 0; p < 3; ++p) {
        if (O[p]) {
            #pragma omp parallel for schedule(static)
            for (int64_t t = 0; t < T; ++t)
                for (int64_t j = 0; j < n[p]; ++j) {
                    double s = 0.0;
                    for (int64_t c = 0; c < d; ++c) s += X[t * d + c] * W[p][c * n[p] + j];
                    O[p][t * n[p] + j] = s;
                }
        }
        if (dW[p]) {
            #pragma omp parallel for schedule(static)
            for (int64_t c = 0; c < d; ++c)
                for (int64_t j = 0; j < n[p]; ++j) {
                    double s = 0.0;
                    for (int64_t t = 0; t < T; ++t) s += X[t * d + c] * G[p][t * n[p] + j];
                    dW[p][c * n[p] + j] = s;
                }
        }
    }
    if (dX) {
        #pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t c = 0; c < d; ++c) {
                double s = 0.0;
                for (int p = 0; p < 3; ++p)
                    for (int64_t j = 0; j < n[p]; ++j) s += G[p][t * n[p] + j] * W[p][c * n[p] + j];
                dX[t * d + c] = s;
            }
    }
}

/* Output projection (row-parallel):    Y = C Wo;
 * given the upstream G_Y:              dC = G_Y Wo^T, dWo = C^T G_Y.
 * C T x nq (the attention core's context), Wo nq x d (in,out). */
void orc_attn_out(int64_t T, int64_t d, int64_t nq, const double* C, const double* Wo, const double* GY,
                  double* Y, double* dC, double* dWo) {
    if (Y) {
        #pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t c = 0; c < d; ++c) {
                double s = 0.0;
                for (int64_t j = 0; j < nq; ++j) s += C[t * nq + j] * Wo[j * d + c];
                Y[t * d + c] = s;
            }
    }
    if (dC) {
        #pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t j = 0; j < nq; ++j) {
                double s = 0.0;
                for (int64_t c = 0; c < d; ++c) s += GY[t * d + c] * Wo[j * d + c];
                dC[t * nq + j] = s;
            }
    }
    if (dWo) {
        #pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < nq; ++j)
            for (int64_t c = 0; c < d; ++c) {
                double s = 0.0;
                for (int64_t t = 0; t < T; ++t) s += C[t * nq + j] * GY[t * d + c];
                dWo[j * d + c] = s;
            }
    }
}

/* ------------------------------------------------------------------------
 * Vocabulary cross-entropy, unsharded definition, for selected tokens.
 * [MC] "04 / VOCABULARY SHARDS" (single supervised position, no label
 * smoothing): per token, z = h W,  m = max_j z_j,  s = sum_j e^{z_j - m},
 * L = log s + m - z_y,  dL/dz_j = e^{z_j - m}/s - 1[j = y];  the gradient
 * of the shared hidden is dh = dz W^T (summed over all vocabulary shards,
 * with no division by the shard count).
 * h is T x d, W is d x V (in,out), labels int64 in [0, V).
 * Outputs per selected token i: loss[i], dlogits[i, :] (V), dhidden[i, :]
 * (d), owner[i] (shard of the label under the plan for `parts`).
 * Returns ORC_ERR_LABEL if a selected label is outside [0, V).
 * ---------------------------------------------------------------------- */
int orc_ce_tokens(int64_t T, int64_t d, int64_t V,
                  const double* h, const double* W, const int64_t* labels, int32_t parts,
                  int64_t ntok, const int64_t* toks,
                  double* loss, double* dlogits, double* dhidden, int32_t* owner) {
    (void)T;
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(parts + 1));
    int rc = orc_plan_shards(V, parts, off);
    if (rc != ORC_OK) { free(off); return rc; }
    for (int64_t i = 0; i < ntok; ++i)
        if (labels[toks[i]] < 0 || labels[toks[i]] >= V) { free(off); return ORC_ERR_LABEL; }
    #pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
        double* dz = (double*)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < ntok; ++i) {
            int64_t t = toks[i];
            int64_t y = labels[t];
            for (int64_t v = 0; v < V; ++v) z[v] = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                double hv = h[t * d + c];
                for (int64_t v = 0; v < V; ++v) z[v] += hv * W[c * V + v];
            }
            double m = -INFINITY;
            for (int64_t v = 0; v < V; ++v) if (z[v] > m) m = z[v];
            double s = 0.0;
            for (int64_t v = 0; v < V; ++v) s += exp(z[v] - m);
            if (loss) loss[i] = log(s) + m - z[y];
            for (int64_t v = 0; v < V; ++v) dz[v] = exp(z[v] - m) / s - (v == y ? 1.0 : 0.0);
            if (dlogits) memcpy(dlogits + i * V, dz, sizeof(double) * (size_t)V);
            if (dhidden)
                for (int64_t c = 0; c < d; ++c) {
                    double acc = 0.0;
                    for (int64_t v = 0; v < V; ++v) acc += dz[v] * W[c * V + v];
                    dhidden[i * d + c] = acc;
                }
            if (owner) owner[i] = orc_owner(y, off, parts);
        }
        free(z);
        free(dz);
    }
    free(off);
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * The pages' sharded formulation of one position's cross-entropy, kept
 * literal so that tests can check it equals the unsharded one.
 * [MC] "04 / VOCABULARY SHARDS":
 *   m_r = max_{j in V_r} z_j,  m = max_r m_r,
 *   s_r = sum_{j in V_r} e^{z_j - m},  s = sum_r s_r,
 *   t_r = 1[y in V_r] (z_y - m),  L = log s - sum_r t_r.
 * An empty shard has m_r = -inf, s_r = 0, t_r = 0.  Outputs m_r, s_r, t_r
 * (each `parts` long) and returns L.
 * ---------------------------------------------------------------------- */
double orc_ce_sharded_one(int64_t V, const double* z, int64_t y, int32_t parts,
                          double* m_r, double* s_r, double* t_r) {
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(parts + 1));
    orc_plan_shards(V, parts, off);
    double m = -INFINITY;
    for (int32_t r = 0; r < parts; ++r) {
        double mr = -INFINITY;
        for (int64_t j = off[r]; j < off[r + 1]; ++j) if (z[j] > mr) mr = z[j];
        m_r[r] = mr;
        if (mr > m) m = mr;
    }
    double s = 0.0, tsum = 0.0;
    for (int32_t r = 0; r < parts; ++r) {
        double sr = 0.0;
        for (int64_t j = off[r]; j < off[r + 1]; ++j) sr += exp(z[j] - m);
        s_r[r] = sr;
        s += sr;
        t_r[r] = (off[r] <= y && y < off[r + 1]) ? (z[y] - m) : 0.0;
        tsum += t_r[r];
    }
    free(off);
    return log(s) - tsum;
}

/* ------------------------------------------------------------------------
 * Vocabulary cross-entropy with the extensions a real implementation needs,
 * which [MC] "04 / VOCABULARY SHARDS" lists after its example (vocabulary
 * padding, ignore_index) and [SG] "易错点与追问" raises (a loss denominator
 * that stays the same across ranks with uneven numbers of supervised
 * tokens).  Full computation over all T tokens.
 *   Columns v >= vocab_real are padding: outside the softmax, gradient 0.
 *   A label equal to ignore_index gives loss 0, gradient 0, owner -1 and
 *   does not count.
 *   reduction 0 (none) / 1 (sum): loss_reduced = sum_t L_t (not written for
 *   none); reduction 2 (mean): loss_reduced = sum_t L_t / D with D =
 *   denominator if > 0, else the number of counted labels (1 if none).
 *   dlogits, dhidden = dlogits W^T and dwhead = h^T dlogits are the
 *   gradients of sum_t L_t (none, sum) or of loss_reduced (mean).
 * Returns ORC_ERR_LABEL for a label outside [0, vocab_real) that is not
 * ignore_index, ORC_ERR_SHAPE for vocab_real outside [1, V].
 * ---------------------------------------------------------------------- */
int orc_ce_ex(int64_t T, int64_t d, int64_t V,
              const double* h, const double* W, const int64_t* labels, int32_t parts,
              int64_t ignore_index, int64_t vocab_real, int reduction, double denominator,
              double* loss, double* loss_reduced, double* dlogits, double* dhidden, double* dwhead,
              int32_t* owner) {
    if (vocab_real < 1 || vocab_real > V) return ORC_ERR_SHAPE;
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(parts + 1));
    int rc = orc_plan_shards(V, parts, off);
    if (rc != ORC_OK) { free(off); return rc; }
    int64_t count = 0;
    for (int64_t t = 0; t < T; ++t) {
        if (labels[t] == ignore_index) continue;
        if (labels[t] < 0 || labels[t] >= vocab_real) { free(off); return ORC_ERR_LABEL; }
        ++count;
    }
    const double D = (reduction == 2) ? (denominator > 0.0 ? denominator : (count > 0 ? (double)count : 1.0)) : 1.0;
    double total = 0.0;
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    for (int64_t t = 0; t < T; ++t) {
        double* dz = dlogits + t * V;
        const int64_t y = labels[t];
        if (y == ignore_index) {
            for (int64_t v = 0; v < V; ++v) dz[v] = 0.0;
            loss[t] = 0.0;
            owner[t] = -1;
            continue;
        }
        for (int64_t v = 0; v < V; ++v) z[v] = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            double hv = h[t * d + c];
            for (int64_t v = 0; v < V; ++v) z[v] += hv * W[c * V + v];
        }
        double m = -INFINITY;
        for (int64_t v = 0; v < vocab_real; ++v) if (z[v] > m) m = z[v];
        double s = 0.0;
        for (int64_t v = 0; v < vocab_real; ++v) s += exp(z[v] - m);
        loss[t] = log(s) + m - z[y];
        total += loss[t];
        for (int64_t v = 0; v < V; ++v)
            dz[v] = (v < vocab_real) ? (exp(z[v] - m) / s - (v == y ? 1.0 : 0.0)) / D : 0.0;
        owner[t] = orc_owner(y, off, parts);
    }
    if (loss_reduced && reduction != 0) *loss_reduced = total / D;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t v = 0; v < V; ++v) acc += dlogits[t * V + v] * W[c * V + v];
            dhidden[t * d + c] = acc;
        }
    if (dwhead)
        for (int64_t c = 0; c < d; ++c)
            for (int64_t v = 0; v < V; ++v) {
                double acc = 0.0;
                for (int64_t t = 0; t < T; ++t) acc += h[t * d + c] * dlogits[t * V + v];
                dwhead[c * V + v] = acc;
            }
    free(z);
    free(off);
    return ORC_OK;
}
