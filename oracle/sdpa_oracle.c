/*
 * Plain fp64 CPU oracle for scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do. It shares no code, header or constant with the CUDA library.
 *
 * What it computes (written straight from the definitions, no tiling, no
 * online softmax, no reordering beyond the per-row loops below):
 *
 *   "Inside NVIDIA's cuDNN Graph API" (tradepoint.io), section 5
 *   "SDPA (Flash Attention) with causal masking": the op is
 *   O = softmax(attn_scale * Q K^T + causal mask) V, with the causal mask
 *   aligned top-left (diagonal_alignment TOP_LEFT, right_bound 0), i.e.
 *   query row i may attend to key j iff j <= i.  The same alignment is the
 *   TransformerEngine PR #2964 note that the causal mask becomes
 *   set_diagonal_band_right_bound(0).
 *
 *   cudnn-frontend PR #554, commit "dense backward" notes: the per-row
 *   statistic is aten's logsumexp of the scaled scores, fp32, shape
 *   (B, H, S); packed THD statistics are token-major (T, H).
 *
 *   The analytic backward of softmax attention (standard calculus, no page
 *   prints it): D_i = sum_k dO[i,k] O[i,k]; dP_ij = dO_i . V_j;
 *   dS_ij = P_ij (dP_ij - D_i); dQ_i = scale sum_j dS_ij K_j;
 *   dK_j = scale sum_i dS_ij Q_i; dV_j = sum_i P_ij dO_i.
 *
 * Allowed key set of query row i.  The masks of the cudnn-frontend PR #554
 * `sdpa` op (its `is_causal`, `causal_bottom_right` and `window_left`
 * arguments) all leave a contiguous range:
 *   A_i = { j : lo_i <= j < hi_i },  delta = n_kv - n_q for the bottom-right
 *   alignment and 0 otherwise,
 *   hi_i = n_kv, or min(n_kv, i + delta + 1) under a causal mask,
 *   lo_i = 0, or max(0, i + delta - window_left) when window_left >= 0
 * (window_left keys to the left of the diagonal stay visible, the
 * window_size = (left, right) convention of the same PR's varlen path with
 * -1 meaning unbounded).  Top-left causal without a window is the prefix
 * j <= i of section 5 above.  A row whose set is empty is "dead": O_i = 0,
 * LSE_i = -inf, and it contributes nothing to any gradient (cudnn-frontend
 * PR #554, FP8 d512 notes on fully-masked rows and the zero-length-KV THD
 * test).
 *
 * Grouped key/value heads (the same PR's GQA cases, h_kv < h_q): query head
 * hq reads key/value head hq / (h_q / h_kv); the gradient of a key/value
 * head is the sum of its group's per-query-head gradients ("GQA reduces" in
 * the PR's backward chain, dK/dV summed over h_q / h_kv query heads).
 *
 * All arrays are fp64.  Each attention problem is one (batch, head) or one
 * (sequence, head) slice, addressed by a base pointer and a row stride in
 * elements, so dense BHSD and packed THD both reduce to it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { MASK_NONE = 0, MASK_TOP_LEFT = 1, MASK_BOTTOM_RIGHT = 2 };

/* Visible keys [*lo, *hi) of query row i (see the header). */
static void key_range(int i, int n_q, int n_kv, int mask, int window_left, int *lo, int *hi)
{
    int delta = (mask == MASK_BOTTOM_RIGHT) ? n_kv - n_q : 0;
    int h = n_kv;
    if (mask != MASK_NONE && i + delta + 1 < h) h = i + delta + 1;
    if (h < 0) h = 0;
    int l = 0;
    if (window_left >= 0 && i + delta - window_left > l) l = i + delta - window_left;
    if (l > h) l = h;
    *lo = l;
    *hi = h;
}

static double dot(const double *a, const double *b, int d)
{
    double s = 0.0;
    for (int t = 0; t < d; ++t) s += a[t] * b[t];
    return s;
}

/* One query row: fills p[0..na) with the softmax probabilities, returns LSE.
 * s_ij = scale * q.k_j;  m = max_j s_ij;  LSE = m + ln sum_j exp(s_ij - m);
 * P_ij = exp(s_ij - LSE). */
static double row_probs(const double *q, const double *k, int64_t k_rs, int na,
                        int d, double scale, double *p)
{
    if (na == 0) return -INFINITY;
    double m = -INFINITY;
    for (int j = 0; j < na; ++j) {
        p[j] = scale * dot(q, k + (int64_t)j * k_rs, d);
        if (p[j] > m) m = p[j];
    }
    double sum = 0.0;
    for (int j = 0; j < na; ++j) sum += exp(p[j] - m);
    double lse = m + log(sum);
    for (int j = 0; j < na; ++j) p[j] = exp(p[j] - lse);
    return lse;
}

/* O_i = sum_j P_ij V_j */
static void row_output(const double *p, const double *v, int64_t v_rs, int na,
                       int d, double *o)
{
    for (int t = 0; t < d; ++t) o[t] = 0.0;
    for (int j = 0; j < na; ++j) {
        const double *vj = v + (int64_t)j * v_rs;
        for (int t = 0; t < d; ++t) o[t] += p[j] * vj[t];
    }
}

/* Forward of one problem, rows listed in `rows` (or all rows if rows==NULL).
 * Outputs go to o + r*o_rs and lse + r*lse_rs where r is the position in the
 * row list (or the row index itself when rows==NULL). */
static void fwd_problem(const double *q, int64_t q_rs, const double *k, int64_t k_rs,
                        const double *v, int64_t v_rs, double *o, int64_t o_rs,
                        double *lse, int64_t lse_rs, int n_q, int n_kv, int d,
                        double scale, int mask, int window_left, const int32_t *rows,
                        int n_rows)
{
    int count = rows ? n_rows : n_q;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(n_kv > 0 ? n_kv : 1));
#pragma omp for schedule(dynamic, 4)
        for (int r = 0; r < count; ++r) {
            int i = rows ? rows[r] : r;
            int lo, hi;
            key_range(i, n_q, n_kv, mask, window_left, &lo, &hi);
            double l = row_probs(q + (int64_t)i * q_rs, k + (int64_t)lo * k_rs, k_rs, hi - lo,
                                 d, scale, p);
            row_output(p, v + (int64_t)lo * v_rs, v_rs, hi - lo, d, o + (int64_t)r * o_rs);
            if (lse) lse[(int64_t)r * lse_rs] = l;
        }
        free(p);
    }
}

/* Backward of one problem.  Pass 1 (independent rows i): LSE_i, D_i and dQ_i.
 * Pass 2 (independent key rows j): dK_j and dV_j, re-deriving P_ij and dS_ij
 * from the pass-1 LSE_i and D_i.  Either pass can be restricted to a list of
 * rows; the statistics of pass 1 are always computed for every row because
 * pass 2 needs all of them. */
static void bwd_problem(const double *q, int64_t q_rs, const double *k, int64_t k_rs,
                        const double *v, int64_t v_rs, const double *dout, int64_t do_rs,
                        double *dq, int64_t dq_rs, double *dk, int64_t dk_rs,
                        double *dv, int64_t dv_rs, int n_q, int n_kv, int d,
                        double scale, int mask, int window_left,
                        const int32_t *q_rows, int n_q_rows,
                        const int32_t *kv_rows, int n_kv_rows)
{
    double *lse = (double *)malloc(sizeof(double) * (size_t)(n_q > 0 ? n_q : 1));
    double *D = (double *)malloc(sizeof(double) * (size_t)(n_q > 0 ? n_q : 1));
    /* dq output slot of row i, or -1 when dQ_i is not requested */
    int32_t *dq_slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_q > 0 ? n_q : 1));
    for (int i = 0; i < n_q; ++i) dq_slot[i] = q_rows ? -1 : i;
    if (q_rows)
        for (int r = 0; r < n_q_rows; ++r) dq_slot[q_rows[r]] = r;

#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(n_kv > 0 ? n_kv : 1));
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
        for (int i = 0; i < n_q; ++i) {
            int lo, hi;
            key_range(i, n_q, n_kv, mask, window_left, &lo, &hi);
            const double *qi = q + (int64_t)i * q_rs;
            const double *doi = dout + (int64_t)i * do_rs;
            lse[i] = row_probs(qi, k + (int64_t)lo * k_rs, k_rs, hi - lo, d, scale, p);
            row_output(p, v + (int64_t)lo * v_rs, v_rs, hi - lo, d, o);
            D[i] = dot(doi, o, d);
            int slot = dq_slot[i];
            if (slot < 0) continue;
            double *dqi = dq + (int64_t)slot * dq_rs;
            for (int t = 0; t < d; ++t) dqi[t] = 0.0;
            for (int j = lo; j < hi; ++j) {
                const double *kj = k + (int64_t)j * k_rs;
                double dp = dot(doi, v + (int64_t)j * v_rs, d);
                double ds = p[j - lo] * (dp - D[i]);
                for (int t = 0; t < d; ++t) dqi[t] += scale * ds * kj[t];
            }
        }
        free(p);
        free(o);
    }

    int count = kv_rows ? n_kv_rows : n_kv;
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < count; ++r) {
        int j = kv_rows ? kv_rows[r] : r;
        const double *kj = k + (int64_t)j * k_rs;
        const double *vj = v + (int64_t)j * v_rs;
        double *dkj = dk + (int64_t)r * dk_rs;
        double *dvj = dv + (int64_t)r * dv_rs;
        for (int t = 0; t < d; ++t) { dkj[t] = 0.0; dvj[t] = 0.0; }
        for (int i = 0; i < n_q; ++i) {
            int lo, hi;
            key_range(i, n_q, n_kv, mask, window_left, &lo, &hi);
            if (j < lo || j >= hi) continue;
            const double *qi = q + (int64_t)i * q_rs;
            const double *doi = dout + (int64_t)i * do_rs;
            double pij = exp(scale * dot(qi, kj, d) - lse[i]);
            double dp = dot(doi, vj, d);
            double ds = pij * (dp - D[i]);
            for (int t = 0; t < d; ++t) {
                dvj[t] += pij * doi[t];
                dkj[t] += scale * ds * qi[t];
            }
        }
    }
    free(lse);
    free(D);
    free(dq_slot);
}

/* ------------------------------------------------------------------ */
/* Exported entry points                                                */
/* ------------------------------------------------------------------ */

/* Mask of the entry points that take a `causal` flag: top-left or none. */
static int causal_mask(int causal) { return causal ? MASK_TOP_LEFT : MASK_NONE; }

/* Selected rows of one problem; outputs packed [n_rows, d] and [n_rows].
 * mask: 0 none, 1 causal top-left, 2 causal bottom-right; window_left < 0
 * means no left bound. */
void oracle_attn_fwd_rows_ex(const double *q, int64_t q_rs, const double *k, int64_t k_rs,
                             const double *v, int64_t v_rs, double *o, double *lse,
                             int n_q, int n_kv, int d, double scale, int mask,
                             int window_left, const int32_t *rows, int n_rows)
{
    fwd_problem(q, q_rs, k, k_rs, v, v_rs, o, d, lse, 1, n_q, n_kv, d, scale, mask,
                window_left, rows, n_rows);
}

void oracle_attn_fwd_rows(const double *q, int64_t q_rs, const double *k, int64_t k_rs,
                          const double *v, int64_t v_rs, double *o, double *lse,
                          int n_q, int n_kv, int d, double scale, int causal,
                          const int32_t *rows, int n_rows)
{
    oracle_attn_fwd_rows_ex(q, q_rs, k, k_rs, v, v_rs, o, lse, n_q, n_kv, d, scale,
                            causal_mask(causal), -1, rows, n_rows);
}

/* Selected dQ rows and dK/dV rows of one problem; outputs packed. */
void oracle_attn_bwd_rows_ex(const double *q, int64_t q_rs, const double *k, int64_t k_rs,
                             const double *v, int64_t v_rs, const double *dout,
                             int64_t do_rs, double *dq, double *dk, double *dv, int n_q,
                             int n_kv, int d, double scale, int mask, int window_left,
                             const int32_t *q_rows, int n_q_rows, const int32_t *kv_rows,
                             int n_kv_rows)
{
    bwd_problem(q, q_rs, k, k_rs, v, v_rs, dout, do_rs, dq, d, dk, d, dv, d, n_q,
                n_kv, d, scale, mask, window_left, q_rows, n_q_rows, kv_rows, n_kv_rows);
}

void oracle_attn_bwd_rows(const double *q, int64_t q_rs, const double *k, int64_t k_rs,
                          const double *v, int64_t v_rs, const double *dout, int64_t do_rs,
                          double *dq, double *dk, double *dv, int n_q, int n_kv, int d,
                          double scale, int causal, const int32_t *q_rows, int n_q_rows,
                          const int32_t *kv_rows, int n_kv_rows)
{
    oracle_attn_bwd_rows_ex(q, q_rs, k, k_rs, v, v_rs, dout, do_rs, dq, dk, dv, n_q, n_kv,
                            d, scale, causal_mask(causal), -1, q_rows, n_q_rows, kv_rows,
                            n_kv_rows);
}

/* Dense BHSD with grouped key/value heads: q,o [b,h,s_q,d]; k,v
 * [b,h_kv,s_kv,d]; lse [b,h,s_q]; h a multiple of h_kv. */
void oracle_sdpa_fwd_ex(const double *q, const double *k, const double *v, double *o,
                        double *lse, int b, int h, int h_kv, int s_q, int s_kv, int d,
                        double scale, int mask, int window_left)
{
    int g = h / h_kv;
    for (int bb = 0; bb < b; ++bb)
        for (int hq = 0; hq < h; ++hq) {
            int64_t qs = (int64_t)bb * h + hq, ks = (int64_t)bb * h_kv + hq / g;
            fwd_problem(q + qs * s_q * d, d, k + ks * s_kv * d, d, v + ks * s_kv * d, d,
                        o + qs * s_q * d, d, lse + qs * s_q, 1, s_q, s_kv, d, scale, mask,
                        window_left, NULL, 0);
        }
}

void oracle_sdpa_fwd(const double *q, const double *k, const double *v, double *o,
                     double *lse, int b, int h, int s_q, int s_kv, int d,
                     double scale, int causal)
{
    oracle_sdpa_fwd_ex(q, k, v, o, lse, b, h, h, s_q, s_kv, d, scale, causal_mask(causal), -1);
}

/* Dense backward with grouped key/value heads: dk, dv [b,h_kv,s_kv,d] are the
 * sums over each group's query heads. */
void oracle_sdpa_bwd_ex(const double *q, const double *k, const double *v,
                        const double *dout, double *dq, double *dk, double *dv, int b,
                        int h, int h_kv, int s_q, int s_kv, int d, double scale, int mask,
                        int window_left)
{
    int g = h / h_kv;
    size_t kv_elems = (size_t)s_kv * d;
    double *tk = (double *)malloc(sizeof(double) * (kv_elems ? kv_elems : 1));
    double *tv = (double *)malloc(sizeof(double) * (kv_elems ? kv_elems : 1));
    memset(dk, 0, sizeof(double) * (size_t)b * h_kv * kv_elems);
    memset(dv, 0, sizeof(double) * (size_t)b * h_kv * kv_elems);
    for (int bb = 0; bb < b; ++bb)
        for (int hq = 0; hq < h; ++hq) {
            int64_t qs = (int64_t)bb * h + hq, ks = (int64_t)bb * h_kv + hq / g;
            bwd_problem(q + qs * s_q * d, d, k + ks * s_kv * d, d, v + ks * s_kv * d, d,
                        dout + qs * s_q * d, d, dq + qs * s_q * d, d, tk, d, tv, d, s_q,
                        s_kv, d, scale, mask, window_left, NULL, 0, NULL, 0);
            for (size_t e = 0; e < kv_elems; ++e) {
                dk[ks * (int64_t)kv_elems + (int64_t)e] += tk[e];
                dv[ks * (int64_t)kv_elems + (int64_t)e] += tv[e];
            }
        }
    free(tk);
    free(tv);
}

void oracle_sdpa_bwd(const double *q, const double *k, const double *v,
                     const double *dout, double *dq, double *dk, double *dv, int b,
                     int h, int s_q, int s_kv, int d, double scale, int causal)
{
    oracle_sdpa_bwd_ex(q, k, v, dout, dq, dk, dv, b, h, h, s_q, s_kv, d, scale,
                       causal_mask(causal), -1);
}

/* Packed THD: q,o [total_q,h,d]; k,v [total_kv,h_kv,d]; lse [total_q,h];
 * sequence n owns query tokens [cu_q[n], cu_q[n+1]) and key tokens
 * [cu_kv[n], cu_kv[n+1]); the mask is applied per sequence (its own n_q and
 * n_kv give the bottom-right offset). */
void oracle_sdpa_varlen_fwd_ex(const double *q, const double *k, const double *v,
                               double *o, double *lse, const int32_t *cu_q,
                               const int32_t *cu_kv, int num_seqs, int h, int h_kv, int d,
                               double scale, int mask, int window_left)
{
    int g = h / h_kv;
    int64_t qrs = (int64_t)h * d, krs = (int64_t)h_kv * d;
    for (int n = 0; n < num_seqs; ++n) {
        int nq = cu_q[n + 1] - cu_q[n], nkv = cu_kv[n + 1] - cu_kv[n];
        for (int hh = 0; hh < h; ++hh) {
            int64_t qo = (int64_t)cu_q[n] * qrs + (int64_t)hh * d;
            int64_t ko = (int64_t)cu_kv[n] * krs + (int64_t)(hh / g) * d;
            fwd_problem(q + qo, qrs, k + ko, krs, v + ko, krs, o + qo, qrs,
                        lse + (int64_t)cu_q[n] * h + hh, h, nq, nkv, d, scale, mask,
                        window_left, NULL, 0);
        }
    }
}

void oracle_sdpa_varlen_fwd(const double *q, const double *k, const double *v,
                            double *o, double *lse, const int32_t *cu_q,
                            const int32_t *cu_kv, int num_seqs, int h, int d,
                            double scale, int causal)
{
    oracle_sdpa_varlen_fwd_ex(q, k, v, o, lse, cu_q, cu_kv, num_seqs, h, h, d, scale,
                              causal_mask(causal), -1);
}

void oracle_sdpa_varlen_bwd_ex(const double *q, const double *k, const double *v,
                               const double *dout, double *dq, double *dk, double *dv,
                               const int32_t *cu_q, const int32_t *cu_kv, int num_seqs,
                               int h, int h_kv, int d, double scale, int mask,
                               int window_left)
{
    int g = h / h_kv;
    int64_t qrs = (int64_t)h * d, krs = (int64_t)h_kv * d;
    int max_kv = 0;
    for (int n = 0; n < num_seqs; ++n)
        if (cu_kv[n + 1] - cu_kv[n] > max_kv) max_kv = cu_kv[n + 1] - cu_kv[n];
    size_t tmp_elems = (size_t)max_kv * d;
    double *tk = (double *)malloc(sizeof(double) * (tmp_elems ? tmp_elems : 1));
    double *tv = (double *)malloc(sizeof(double) * (tmp_elems ? tmp_elems : 1));
    memset(dk, 0, sizeof(double) * (size_t)cu_kv[num_seqs] * h_kv * d);
    memset(dv, 0, sizeof(double) * (size_t)cu_kv[num_seqs] * h_kv * d);
    for (int n = 0; n < num_seqs; ++n) {
        int nq = cu_q[n + 1] - cu_q[n], nkv = cu_kv[n + 1] - cu_kv[n];
        for (int hh = 0; hh < h; ++hh) {
            int64_t qo = (int64_t)cu_q[n] * qrs + (int64_t)hh * d;
            int64_t ko = (int64_t)cu_kv[n] * krs + (int64_t)(hh / g) * d;
            bwd_problem(q + qo, qrs, k + ko, krs, v + ko, krs, dout + qo, qrs, dq + qo,
                        qrs, tk, d, tv, d, nq, nkv, d, scale, mask, window_left, NULL, 0,
                        NULL, 0);
            for (int j = 0; j < nkv; ++j)
                for (int t = 0; t < d; ++t) {
                    dk[ko + (int64_t)j * krs + t] += tk[(int64_t)j * d + t];
                    dv[ko + (int64_t)j * krs + t] += tv[(int64_t)j * d + t];
                }
        }
    }
    free(tk);
    free(tv);
}

void oracle_sdpa_varlen_bwd(const double *q, const double *k, const double *v,
                            const double *dout, double *dq, double *dk, double *dv,
                            const int32_t *cu_q, const int32_t *cu_kv, int num_seqs,
                            int h, int d, double scale, int causal)
{
    oracle_sdpa_varlen_bwd_ex(q, k, v, dout, dq, dk, dv, cu_q, cu_kv, num_seqs, h, h, d,
                              scale, causal_mask(causal), -1);
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 inputs                                                      */
/* ------------------------------------------------------------------ */

/* One 8-bit E4M3 code (the OCP "FN" encoding the cudnn-frontend PR #554 FP8
 * kernels take as input): sign bit 7, exponent bits 6..3 with bias 7,
 * mantissa bits 2..0.  Exponent field 0 is subnormal, (m / 8) * 2^-6; the
 * code S.1111.111 is NaN; there are no infinities, so the largest finite
 * magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_decode(uint8_t x)
{
    int sign = x >> 7, e = (x >> 3) & 15, m = x & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* dst[i] = decode(src[i]) * descale: the real value an FP8 tensor with a
 * per-tensor descale stands for. */
void oracle_e4m3_to_f64(const uint8_t *src, double *dst, int64_t n, double descale)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = oracle_e4m3_decode(src[i]) * descale;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
