/*
 * Exact softmax attention, forward, in plain fp64 -- the ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * path under exact_attention_51_gb300/csrc.
 *
 * What it computes (the plain definition, not the tiled algorithm):
 *
 *   s_ij  = scale * sum_c q_ic k_jc                     for visible j
 *   m_i   = max_j s_ij                                  (pass 1)
 *   l_i   = sum_j exp(s_ij - m_i)                       (pass 2)
 *   o_ic  = sum_j exp(s_ij - m_i) v_jc / l_i            (pass 3)
 *   lse_i = m_i + ln l_i
 *
 * "visible j" is every key 0..Nk-1, or 0..i+Nk-Nq when causal (the lower
 * "triangular matrix" of the scores, aligned to the bottom-right corner when
 * there are more keys than queries, Nk >= Nq; with Nq = Nk = N key j is
 * visible to query i iff j <= i).  The diagonal is always visible, so no row
 * is empty.
 *
 * Sources: "Tri Dao: prediction" (highsignal podcast transcript) -- exact
 * attention whose softmax needs a sum across the row of the attention matrix,
 * which the fused method must still reproduce exactly ("still get the right
 * answer"); "FlashAttention-3" HN thread -- the softmax of the triangular
 * matrix (causal mask).  The online-softmax rescaling the fast path uses is
 * NOT reproduced here: the oracle is the three-pass definition the rescaling
 * has to agree with.
 *
 * Inputs are bf16 bit patterns (what the GPU reads) decoded here by a 16-bit
 * shift into the high half of an IEEE binary32, e4m3 codes with one
 * dequantisation scale per tensor (decoded by the OCP 8-bit format's
 * definition), or plain fp64 arrays (used by the pin tests).  Layout: contiguous [B,H,N,d] row-major for q, k, v, o and
 * [B,H,N] for lse.  All arithmetic is fp64 with libm exp/log.
 *
 * Parity status: pinned (tiled-vs-two-pass brute force, closed forms,
 * invariants and a library cross-check; see tests/test_oracle.py).
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

/* bf16 -> fp64: the 16 stored bits are the top half of a binary32. */
static double bf16_bits_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * One query row i against one head's keys and values (fp64, row-major
 * [Nk,d]); `off` = Nk - Nq shifts the causal diagonal.  `s` is caller-provided
 * scratch of Nk doubles.
 */
static void attend_row(const double *q_i, const double *K, const double *V,
                       int64_t Nk, int64_t d, int64_t i, int64_t off, double scale,
                       int causal, double *s, double *o_i, double *lse_i) {
    int64_t last = causal ? i + off : Nk - 1; /* visible keys are 0..last */

    /* scores */
    for (int64_t j = 0; j <= last; ++j) {
        const double *k_j = K + j * d;
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c) acc += q_i[c] * k_j[c];
        s[j] = scale * acc;
    }
    /* pass 1: row maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j <= last; ++j)
        if (s[j] > m) m = s[j];
    /* pass 2: normaliser; s is overwritten with exp(s - m) */
    double l = 0.0;
    for (int64_t j = 0; j <= last; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    /* pass 3: probability-weighted sum of value rows */
    for (int64_t c = 0; c < d; ++c) o_i[c] = 0.0;
    for (int64_t j = 0; j <= last; ++j) {
        const double p = s[j] / l;
        const double *v_j = V + j * d;
        for (int64_t c = 0; c < d; ++c) o_i[c] += p * v_j[c];
    }
    *lse_i = m + log(l);
}

static int check_sizes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int causal) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return ORACLE_EINVAL;
    if (causal && Nk < Nq) return ORACLE_EINVAL; /* first rows would see no key */
    /* keep B*H*N*d well inside int64 */
    const double n = (double)(Nq > Nk ? Nq : Nk);
    if ((double)B * (double)H * n * (double)d > 4.0e18) return ORACLE_EINVAL;
    return ORACLE_OK;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/*
 * Rows of one head: `rows` lists query indices i (0..Nq-1) of head (b,h);
 * outputs go to o_out[r*d..] and lse_out[r] for the r-th listed row.
 * Q rows are fp64 [Nq,d], K and V fp64 [Nk,d] of that head.
 */
static int head_rows(const double *Qh, const double *Kh, const double *Vh,
                     int64_t Nq, int64_t Nk, int64_t d, double scale, int causal,
                     const int64_t *rows, int64_t nrows, double *o_out,
                     double *lse_out) {
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)Nk * sizeof(double));
        if (!s) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!s) continue;
            const int64_t i = rows ? rows[r] : r;
            attend_row(Qh + i * d, Kh, Vh, Nk, d, i, Nk - Nq, scale, causal, s,
                       o_out + r * d, lse_out + r);
        }
        free(s);
    }
    return err ? ORACLE_ENOMEM : ORACLE_OK;
}

/* ---------------------------------------------------------------- fp64 in */

/* Whole tensors, fp64 inputs: q, o [B,H,Nq,d], k, v [B,H,Nk,d], lse [B,H,Nq]. */
int attn_ref_f64_qk(const double *q, const double *k, const double *v, double *o,
                    double *lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                    int64_t d, double scale, int causal, int nthreads) {
    if (!q || !k || !v || !o || !lse) return ORACLE_EINVAL;
    int rc = check_sizes(B, H, Nq, Nk, d, causal);
    if (rc) return rc;
    set_threads(nthreads);
    for (int64_t bh = 0; bh < B * H; ++bh) {
        rc = head_rows(q + bh * Nq * d, k + bh * Nk * d, v + bh * Nk * d, Nq, Nk, d,
                       scale, causal, NULL, Nq, o + bh * Nq * d, lse + bh * Nq);
        if (rc) return rc;
    }
    return ORACLE_OK;
}

/* Whole tensors, fp64 inputs, Nq = Nk = N. */
int attn_ref_f64(const double *q, const double *k, const double *v, double *o,
                 double *lse, int64_t B, int64_t H, int64_t N, int64_t d,
                 double scale, int causal, int nthreads) {
    return attn_ref_f64_qk(q, k, v, o, lse, B, H, N, N, d, scale, causal, nthreads);
}

/* ---------------------------------------------------------------- bf16 in */

static void decode_head(const uint16_t *src, double *dst, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) dst[t] = bf16_bits_to_f64(src[t]);
}

/*
 * Selected rows, bf16 inputs: q [B,H,Nq,d], k, v [B,H,Nk,d].  rows[r] is a
 * flat query-row id (b*H + h)*Nq + i and may come in any order; the r-th
 * result goes to o_rows[r*d..] and lse_rows[r].  Each head that owns at least
 * one listed row is decoded to fp64 once per call.
 */
int attn_ref_bf16_qk_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d,
                          double scale, int causal, const int64_t *rows, int64_t nrows,
                          double *o_rows, double *lse_rows, int nthreads) {
    if (!q || !k || !v || !rows || !o_rows || !lse_rows || nrows < 0)
        return ORACLE_EINVAL;
    int rc = check_sizes(B, H, Nq, Nk, d, causal);
    if (rc) return rc;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * Nq) return ORACLE_EINVAL;
    set_threads(nthreads);

    const size_t q_elems = (size_t)Nq * (size_t)d, kv_elems = (size_t)Nk * (size_t)d;
    double *Qh = (double *)malloc(q_elems * sizeof(double));
    double *Kh = (double *)malloc(kv_elems * sizeof(double));
    double *Vh = (double *)malloc(kv_elems * sizeof(double));
    int64_t *sel = (int64_t *)malloc((size_t)(nrows ? nrows : 1) * sizeof(int64_t));
    int64_t *pos = (int64_t *)malloc((size_t)(nrows ? nrows : 1) * sizeof(int64_t));
    double *o_tmp = (double *)malloc((size_t)(nrows ? nrows : 1) * (size_t)d * sizeof(double));
    double *l_tmp = (double *)malloc((size_t)(nrows ? nrows : 1) * sizeof(double));
    if (!Qh || !Kh || !Vh || !sel || !pos || !o_tmp || !l_tmp) {
        rc = ORACLE_ENOMEM;
        goto done;
    }
    for (int64_t bh = 0; bh < B * H && rc == ORACLE_OK; ++bh) {
        int64_t cnt = 0;
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] / Nq == bh) {
                sel[cnt] = rows[r] % Nq;
                pos[cnt] = r;
                ++cnt;
            }
        if (cnt == 0) continue;
        decode_head(q + bh * (int64_t)q_elems, Qh, (int64_t)q_elems);
        decode_head(k + bh * (int64_t)kv_elems, Kh, (int64_t)kv_elems);
        decode_head(v + bh * (int64_t)kv_elems, Vh, (int64_t)kv_elems);
        rc = head_rows(Qh, Kh, Vh, Nq, Nk, d, scale, causal, sel, cnt, o_tmp, l_tmp);
        for (int64_t t = 0; t < cnt && rc == ORACLE_OK; ++t) {
            memcpy(o_rows + pos[t] * d, o_tmp + t * d, (size_t)d * sizeof(double));
            lse_rows[pos[t]] = l_tmp[t];
        }
    }
done:
    free(Qh); free(Kh); free(Vh); free(sel); free(pos); free(o_tmp); free(l_tmp);
    return rc;
}

/* Selected rows, bf16 inputs, Nq = Nk = N. */
int attn_ref_bf16_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       int64_t B, int64_t H, int64_t N, int64_t d, double scale,
                       int causal, const int64_t *rows, int64_t nrows,
                       double *o_rows, double *lse_rows, int nthreads) {
    return attn_ref_bf16_qk_rows(q, k, v, B, H, N, N, d, scale, causal, rows, nrows,
                                 o_rows, lse_rows, nthreads);
}

/* Whole tensors, bf16 inputs: q, o [B,H,Nq,d], k, v [B,H,Nk,d], lse [B,H,Nq]. */
int attn_ref_bf16_qk(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     double *o, double *lse, int64_t B, int64_t H, int64_t Nq,
                     int64_t Nk, int64_t d, double scale, int causal, int nthreads) {
    if (!q || !k || !v || !o || !lse) return ORACLE_EINVAL;
    int rc = check_sizes(B, H, Nq, Nk, d, causal);
    if (rc) return rc;
    set_threads(nthreads);
    const size_t q_elems = (size_t)Nq * (size_t)d, kv_elems = (size_t)Nk * (size_t)d;
    double *Qh = (double *)malloc(q_elems * sizeof(double));
    double *Kh = (double *)malloc(kv_elems * sizeof(double));
    double *Vh = (double *)malloc(kv_elems * sizeof(double));
    if (!Qh || !Kh || !Vh) {
        free(Qh); free(Kh); free(Vh);
        return ORACLE_ENOMEM;
    }
    for (int64_t bh = 0; bh < B * H && rc == ORACLE_OK; ++bh) {
        decode_head(q + bh * (int64_t)q_elems, Qh, (int64_t)q_elems);
        decode_head(k + bh * (int64_t)kv_elems, Kh, (int64_t)kv_elems);
        decode_head(v + bh * (int64_t)kv_elems, Vh, (int64_t)kv_elems);
        rc = head_rows(Qh, Kh, Vh, Nq, Nk, d, scale, causal, NULL, Nq,
                       o + bh * (int64_t)q_elems, lse + bh * Nq);
    }
    free(Qh); free(Kh); free(Vh);
    return rc;
}

/* Whole tensors, bf16 inputs, Nq = Nk = N. */
int attn_ref_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  double *o, double *lse, int64_t B, int64_t H, int64_t N,
                  int64_t d, double scale, int causal, int nthreads) {
    return attn_ref_bf16_qk(q, k, v, o, lse, B, H, N, N, d, scale, causal, nthreads);
}

/* ---------------------------------------------------------------- e4m3 in */

/*
 * OCP 8-bit floating point (OFP8), E4M3 variant -> fp64: bit 7 sign, bits 6..3
 * exponent (bias 7), bits 2..0 mantissa; exponent field 0 holds subnormals
 * (m / 8) * 2^-6; exponent 15 with mantissa 7 is NaN; there are no infinities,
 * so S.1111.110 = +-448 is the largest finite value.
 */
static double e4m3_to_f64(uint8_t c) {
    const int e = (c >> 3) & 15, m = c & 7;
    double x;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        x = ldexp((double)m / 8.0, -6);
    else
        x = ldexp(1.0 + (double)m / 8.0, e - 7);
    return (c & 0x80) ? -x : x;
}

static void decode_head_e4m3(const uint8_t *src, double descale, double *dst, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) dst[t] = descale * e4m3_to_f64(src[t]);
}

/* Decodes one code (for the pin tests). */
double attn_ref_e4m3_decode(int code) { return e4m3_to_f64((uint8_t)(code & 0xff)); }

/*
 * e4m3 inputs with per-tensor dequantisation scales: attention of
 * (sq * Q8, sk * K8, sv * V8) by the same definition, q [B,H,Nq,d] and k, v
 * [B,H,Nk,d] (causal needs Nk >= Nq, diagonal at the bottom-right as for bf16
 * inputs).  rows == NULL: every row, o [B,H,Nq,d] and lse [B,H,Nq]; else the
 * nrows flat row ids (b*H + h)*Nq + i in rows[], results packed in o[r*d..] /
 * lse[r] in that order.
 */
int attn_ref_e4m3_qk(const uint8_t *q, const uint8_t *k, const uint8_t *v, double sq,
                     double sk, double sv, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                     int64_t d, double scale, int causal, const int64_t *rows, int64_t nrows,
                     double *o, double *lse, int nthreads) {
    if (!q || !k || !v || !o || !lse || (rows && nrows < 0)) return ORACLE_EINVAL;
    int rc = check_sizes(B, H, Nq, Nk, d, causal);
    if (rc) return rc;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= B * H * Nq) return ORACLE_EINVAL;
    set_threads(nthreads);
    const size_t q_elems = (size_t)Nq * (size_t)d, kv_elems = (size_t)Nk * (size_t)d;
    const int64_t cap = rows ? (nrows ? nrows : 1) : 1;
    double *Qh = (double *)malloc(q_elems * sizeof(double));
    double *Kh = (double *)malloc(kv_elems * sizeof(double));
    double *Vh = (double *)malloc(kv_elems * sizeof(double));
    int64_t *sel = (int64_t *)malloc((size_t)cap * sizeof(int64_t));
    int64_t *pos = (int64_t *)malloc((size_t)cap * sizeof(int64_t));
    double *o_tmp = (double *)malloc((size_t)cap * (size_t)d * sizeof(double));
    double *l_tmp = (double *)malloc((size_t)cap * sizeof(double));
    if (!Qh || !Kh || !Vh || !sel || !pos || !o_tmp || !l_tmp) {
        rc = ORACLE_ENOMEM;
        goto done;
    }
    for (int64_t bh = 0; bh < B * H && rc == ORACLE_OK; ++bh) {
        int64_t cnt = 0;
        if (rows) {
            for (int64_t r = 0; r < nrows; ++r)
                if (rows[r] / Nq == bh) {
                    sel[cnt] = rows[r] % Nq;
                    pos[cnt] = r;
                    ++cnt;
                }
            if (cnt == 0) continue;
        }
        decode_head_e4m3(q + bh * (int64_t)q_elems, sq, Qh, (int64_t)q_elems);
        decode_head_e4m3(k + bh * (int64_t)kv_elems, sk, Kh, (int64_t)kv_elems);
        decode_head_e4m3(v + bh * (int64_t)kv_elems, sv, Vh, (int64_t)kv_elems);
        if (!rows) {
            rc = head_rows(Qh, Kh, Vh, Nq, Nk, d, scale, causal, NULL, Nq,
                           o + bh * (int64_t)q_elems, lse + bh * Nq);
            continue;
        }
        rc = head_rows(Qh, Kh, Vh, Nq, Nk, d, scale, causal, sel, cnt, o_tmp, l_tmp);
        for (int64_t t = 0; t < cnt && rc == ORACLE_OK; ++t) {
            memcpy(o + pos[t] * d, o_tmp + t * d, (size_t)d * sizeof(double));
            lse[pos[t]] = l_tmp[t];
        }
    }
done:
    free(Qh); free(Kh); free(Vh); free(sel); free(pos); free(o_tmp); free(l_tmp);
    return rc;
}

/* e4m3 inputs, Nq = Nk = N. */
int attn_ref_e4m3(const uint8_t *q, const uint8_t *k, const uint8_t *v, double sq,
                  double sk, double sv, int64_t B, int64_t H, int64_t N, int64_t d,
                  double scale, int causal, const int64_t *rows, int64_t nrows,
                  double *o, double *lse, int nthreads) {
    return attn_ref_e4m3_qk(q, k, v, sq, sk, sv, B, H, N, N, d, scale, causal, rows, nrows, o,
                            lse, nthreads);
}

/* Threads OpenMP will use for a parallel region (1 without OpenMP). */
int attn_ref_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
