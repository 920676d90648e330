/*
 * Gradients of exact softmax attention, in plain fp64 -- the ORACLE for the
 * backward pass.
 *
 * TEST INFRASTRUCTURE ONLY (same rules as attn_ref.c): nothing on the product
 * path links, loads or calls this file, and it shares no code with the CUDA
 * path.
 *
 * For O = softmax(scale * Q K^T [+ causal mask]) V and an upstream gradient
 * dO = dL/dO of some scalar L, the chain rule through the definition gives,
 * with P the row-stochastic attention matrix (p_ij = 0 where j is masked):
 *
 *   dV = P^T dO
 *   dP = dO V^T
 *   D_i = sum_c dO_ic O_ic            (= sum_j p_ij dp_ij)
 *   dS = P o (dP - D)                  (softmax Jacobian, row by row)
 *   dQ = scale * dS K
 *   dK = scale * dS^T Q
 *
 * computed here directly from that definition: P from the three-pass softmax
 * of attn_ref.c (max, sum of exp, normalise), everything in fp64, the causal
 * mask being key j visible to query i iff j <= i (Nq = Nk = N).  The pages
 * name the backward pass only as the part the ~100-line kernel's author had
 * not written yet ("Show HN: Flash Attention in ~100 lines of CUDA"); the
 * formulas are the textbook derivative of the forward definition.
 *
 * Inputs: fp64 or bf16 bit patterns, contiguous [B,H,N,d]; outputs fp64
 * [B,H,N,d].  Parity status: pinned (finite differences of the oracle's own
 * forward, torch autograd through scaled_dot_product_attention in fp64, and
 * closed-form column sums; see tests/test_oracle_bwd.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

static double bf16_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * One head.  Q, K, V, dO fp64 [N,d]; writes dQ, dK, dV fp64 [N,d].
 * P and dS are kept as dense [N,N] fp64 (zero where masked).
 */
static int head_bwd(const double *Q, const double *K, const double *V,
                    const double *dO, double *dQ, double *dK, double *dV,
                    int64_t N, int64_t d, double scale, int causal) {
    double *P = (double *)calloc((size_t)N * (size_t)N, sizeof(double));
    double *dS = (double *)calloc((size_t)N * (size_t)N, sizeof(double));
    if (!P || !dS) {
        free(P);
        free(dS);
        return ORACLE_ENOMEM;
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < N; ++i) {
        const int64_t last = causal ? i : N - 1;
        double *p = P + i * N;
        /* scores, then the three-pass softmax */
        double m = -INFINITY;
        for (int64_t j = 0; j <= last; ++j) {
            double acc = 0.0;
            for (int64_t c = 0; c < d; ++c) acc += Q[i * d + c] * K[j * d + c];
            p[j] = scale * acc;
            if (p[j] > m) m = p[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j <= last; ++j) {
            p[j] = exp(p[j] - m);
            l += p[j];
        }
        for (int64_t j = 0; j <= last; ++j) p[j] /= l;
        /* D_i = sum_j p_ij dp_ij with dp_ij = dO_i . V_j */
        double Di = 0.0;
        double *ds = dS + i * N;
        for (int64_t j = 0; j <= last; ++j) {
            double dp = 0.0;
            for (int64_t c = 0; c < d; ++c) dp += dO[i * d + c] * V[j * d + c];
            ds[j] = dp; /* dp for now */
            Di += p[j] * dp;
        }
        for (int64_t j = 0; j <= last; ++j) ds[j] = p[j] * (ds[j] - Di);
    }
    /* dQ = scale * dS K */
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N; ++i)
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t j = 0; j < N; ++j) acc += dS[i * N + j] * K[j * d + c];
            dQ[i * d + c] = scale * acc;
        }
    /* dK = scale * dS^T Q, dV = P^T dO */
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t c = 0; c < d; ++c) {
            double ak = 0.0, av = 0.0;
            for (int64_t i = 0; i < N; ++i) {
                ak += dS[i * N + j] * Q[i * d + c];
                av += P[i * N + j] * dO[i * d + c];
            }
            dK[j * d + c] = scale * ak;
            dV[j * d + c] = av;
        }
    free(P);
    free(dS);
    return ORACLE_OK;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

static int check(int64_t B, int64_t H, int64_t N, int64_t d) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return ORACLE_EINVAL;
    if ((double)N * (double)N > 2.0e9) return ORACLE_EINVAL; /* dense N x N per head */
    return ORACLE_OK;
}

/* fp64 inputs. */
int attn_bwd_ref_f64(const double *q, const double *k, const double *v,
                     const double *dout, double *dq, double *dk, double *dv,
                     int64_t B, int64_t H, int64_t N, int64_t d, double scale,
                     int causal, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return ORACLE_EINVAL;
    int rc = check(B, H, N, d);
    if (rc) return rc;
    set_threads(nthreads);
    for (int64_t bh = 0; bh < B * H && rc == ORACLE_OK; ++bh) {
        const int64_t off = bh * N * d;
        rc = head_bwd(q + off, k + off, v + off, dout + off, dq + off, dk + off,
                      dv + off, N, d, scale, causal);
    }
    return rc;
}

/* bf16 inputs (bit patterns), decoded head by head. */
int attn_bwd_ref_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const uint16_t *dout, double *dq, double *dk, double *dv,
                      int64_t B, int64_t H, int64_t N, int64_t d, double scale,
                      int causal, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return ORACLE_EINVAL;
    int rc = check(B, H, N, d);
    if (rc) return rc;
    set_threads(nthreads);
    const size_t n = (size_t)N * (size_t)d;
    double *buf = (double *)malloc(4 * n * sizeof(double));
    if (!buf) return ORACLE_ENOMEM;
    double *Q = buf, *K = buf + n, *V = buf + 2 * n, *dO = buf + 3 * n;
    for (int64_t bh = 0; bh < B * H && rc == ORACLE_OK; ++bh) {
        const int64_t off = bh * (int64_t)n;
        for (size_t t = 0; t < n; ++t) {
            Q[t] = bf16_to_f64(q[off + t]);
            K[t] = bf16_to_f64(k[off + t]);
            V[t] = bf16_to_f64(v[off + t]);
            dO[t] = bf16_to_f64(dout[off + t]);
        }
        rc = head_bwd(Q, K, V, dO, dq + off, dk + off, dv + off, N, d, scale, causal);
    }
    free(buf);
    return rc;
}
