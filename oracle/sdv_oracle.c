/*
 * sdv_oracle.c -- plain fp64 CPU oracle of the batched lossless
 * draft-verification step with test-time self-selection.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product path.  It shares no code
 * with the CUDA library.  Every step is written in the order the method states
 * it, with no blocking, fusion or reordering; the only parallelism is over
 * independent sequences, or over the independent rows of one sequence.  See
 * sdv_oracle.h for the passages followed.
 */
#include "sdv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11).  Pinned by the published            */
/* known-answer vectors and by cuRAND's Philox4_32_10 generator.            */
/* ------------------------------------------------------------------------ */

/* Multipliers and Weyl key increments of Philox4x32 as published. */
#define PHILOX_MUL0 0xD2511F53u
#define PHILOX_MUL1 0xCD9E8D57u
#define PHILOX_WEYL0 0x9E3779B9u
#define PHILOX_WEYL1 0xBB67AE85u

void sdvo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_WEYL0;
            k1 += PHILOX_WEYL1;
        }
        /* One round: two 32x32->64 products; the high halves are mixed with
         * the other two words and the key, the low halves pass through. */
        uint64_t prod0 = (uint64_t)PHILOX_MUL0 * (uint64_t)x0;
        uint64_t prod1 = (uint64_t)PHILOX_MUL1 * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

double sdvo_uniform24(uint32_t word)
{
    return (double)(word >> 8) * (1.0 / 16777216.0);
}

void sdvo_uniforms(uint64_t seed, uint32_t b, uint32_t j, double* u, double* w)
{
    uint32_t ctr[4] = {j, b, 0u, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    sdvo_philox4x32_10(ctr, key, out);
    if (u) *u = sdvo_uniform24(out[0]);
    if (w) *w = sdvo_uniform24(out[1]);
}

/* ------------------------------------------------------------------------ */
/* Temperature softmax of one row.  Pinned by closed forms (uniform rows,    */
/* two-element rows, shifts) and by scipy's logsumexp.                      */
/* ------------------------------------------------------------------------ */

double sdvo_logit(const void* row, int dtype, int64_t index)
{
    if (dtype == SDVO_BF16) {
        /* bf16 is the top half of an IEEE binary32: widen exactly. */
        uint16_t h = ((const uint16_t*)row)[index];
        uint32_t bits = (uint32_t)h << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)row)[index];
}

double sdvo_row_lse(const void* row, int dtype, int64_t V, double T)
{
    /* Pass 1: the maximum of z_v = l_v / T (and a scan for NaN / +inf). */
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double z = sdvo_logit(row, dtype, v) / T;
        if (isnan(z) || z == INFINITY) return NAN;
        if (z > m) m = z;
    }
    if (m == -INFINITY) return -INFINITY;
    /* Pass 2: LSE = m + log sum_v exp(z_v - m). */
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double z = sdvo_logit(row, dtype, v) / T;
        s += exp(z - m);
    }
    return m + log(s);
}

double sdvo_logprob(const void* row, int dtype, int64_t x, double T, double lse)
{
    return sdvo_logit(row, dtype, x) / T - lse;
}

/* ------------------------------------------------------------------------ */
/* Acceptance rule, streak score, self-selection.  Pinned by the closed form */
/* E_{x~q}[min(1,p/q)] = sum_v min(p_v,q_v), by exact enumeration of the    */
/* committed-token law (K = 1 equals p; the K = 2 counter-example law), by  */
/* Monte Carlo of E[L] = S, and by the q == p invariant.                    */
/* ------------------------------------------------------------------------ */

double sdvo_accept_ratio(double lp, double lq)
{
    if (lq == -INFINITY) return 1.0;       /* q(x) = 0 <= p(x): accept        */
    if (lp == -INFINITY) return 0.0;       /* p(x) = 0 < q(x): never accept   */
    if (lq <= lp) return 1.0;              /* q(x) <= p(x): accept at once     */
    return exp(lp - lq);                   /* else accept with prob p/q        */
}

double sdvo_accept_ratio_greedy(double lp)
{
    if (lp == -INFINITY) return 0.0;       /* p(x) = 0: never accept          */
    if (lp >= 0.0) return 1.0;
    return exp(lp);                        /* accept with probability p(x)     */
}

double sdvo_streak_score(const double* a, int gamma)
{
    double score = 0.0, prefix = 1.0;
    for (int j = 0; j < gamma; ++j) {
        prefix *= a[j];
        score += prefix;
    }
    return score;
}

int sdvo_argmax_first(const double* s, int K)
{
    int best = 0;
    for (int k = 1; k < K; ++k)
        if (s[k] > s[best]) best = k;
    return best;
}

int sdvo_accept_length(const double* a, const double* u, int gamma)
{
    for (int j = 0; j < gamma; ++j) {
        int accepted = (a[j] >= 1.0) || (u[j] < a[j]);
        if (!accepted) return j;
    }
    return gamma;
}

/* ------------------------------------------------------------------------ */
/* Inverse-CDF draw.  Pinned by exact interval integration over w on tiny    */
/* rows and by the rule that zero-weight ids are never drawn.               */
/* ------------------------------------------------------------------------ */

int64_t sdvo_inverse_cdf(const double* r, int64_t V, double w, double* R_out,
                         double* t_out, double* c_prev_out, double* c_v_out)
{
    double R = 0.0;
    for (int64_t v = 0; v < V; ++v) R += r[v];
    if (R_out) *R_out = R;
    if (!(R > 0.0)) return -1;
    double t = w * R;
    if (t_out) *t_out = t;
    double c = 0.0, c_prev = 0.0;
    int64_t last_pos = -1;
    for (int64_t v = 0; v < V; ++v) {
        c_prev = c;
        c += r[v];
        if (r[v] > 0.0) last_pos = v;
        if (c > t) {
            if (c_prev_out) *c_prev_out = c_prev;
            if (c_v_out) *c_v_out = c;
            return v;
        }
    }
    /* Rounding left t at or above the total: the last id with mass. */
    if (c_prev_out) *c_prev_out = c;
    if (c_v_out) *c_v_out = c;
    return last_pos;
}

/* ------------------------------------------------------------------------ */
/* The full step for one sequence.                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    int K, gamma, dtype;
    int64_t V;
} shape_t;

static const void* p_row(const void* base, const shape_t* sh, int b, int k, int j)
{
    size_t elt = sh->dtype == SDVO_BF16 ? 2 : 4;
    int64_t idx = (((int64_t)b * sh->K + k) * (sh->gamma + 1) + j) * sh->V;
    return (const char*)base + (size_t)idx * elt;
}

static const void* q_row(const void* base, const shape_t* sh, int b, int k, int j)
{
    size_t elt = sh->dtype == SDVO_BF16 ? 2 : 4;
    int64_t idx = (((int64_t)b * sh->K + k) * sh->gamma + j) * sh->V;
    return (const char*)base + (size_t)idx * elt;
}

/* One sequence.  Its drafts are Lb tokens long (0 <= Lb <= gamma; the
 * arrays keep their gamma stride and positions >= Lb are not read): the
 * scores, the scan and the draw use positions j < Lb, and with every token
 * accepted the bonus token comes from the verifier row at position Lb. */
static int verify_one(const shape_t* sh, int b, const void* p_logits,
                      const void* q_logits, const int32_t* drafts, double T, int Lb,
                      const double* u, const double* w, int32_t* sel_out,
                      int32_t* len_out, int32_t* tok_out, double* lse_out,
                      double* scores_out, double* ratio_out, int32_t* band_out,
                      double* resid_out, int row_threads, int greedy)
{
    const int K = sh->K, G = sh->gamma, dtype = sh->dtype;
    const int64_t V = sh->V;
    const int nrow = 2 * G + 1;
    int err = 0;
    *sel_out = -1; *len_out = -1; *tok_out = -1;
    if (band_out) *band_out = 0;
    if (resid_out) *resid_out = NAN;

    if (!(T > 0.0) || isinf(T)) err |= SDVO_BAD_TEMP;
    if (Lb < 0 || Lb > G) err |= SDVO_BAD_DRAFT;
    for (int k = 0; k < K && !err; ++k)
        for (int j = 0; j < Lb; ++j) {
            int32_t x = drafts[((int64_t)b * K + k) * G + j];
            if (x < 0 || (int64_t)x >= V) err |= SDVO_BAD_DRAFT;
        }
    if (err) return err;

    const size_t nkg = (size_t)K * (G > 0 ? G : 1);
    double* lse = (double*)malloc(sizeof(double) * (size_t)K * nrow);
    double* a = (double*)malloc(sizeof(double) * nkg * 3);
    double* S = (double*)malloc(sizeof(double) * (size_t)K * 3);
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    if (!lse || !a || !S || !r) { free(lse); free(a); free(S); free(r); return -1; }
    double* a_lo = a + nkg;
    double* a_hi = a + 2 * nkg;
    double* S_lo = S + K;
    double* S_hi = S + 2 * K;

    /* Temperature softmax of every p row (j = 0..G) and q row (j < G); the
     * rows are independent, so they may be spread over threads. */
#ifdef _OPENMP
#pragma omp parallel for num_threads(row_threads > 1 ? row_threads : 1) schedule(dynamic, 4) if (row_threads > 1)
#endif
    for (int i = 0; i < K * nrow; ++i) {
        const int k = i / nrow, r = i % nrow;
        if (r <= Lb)
            lse[i] = sdvo_row_lse(p_row(p_logits, sh, b, k, r), dtype, V, T);
        else if (r > G && r - G - 1 < Lb && !greedy)
            lse[i] = sdvo_row_lse(q_row(q_logits, sh, b, k, r - G - 1), dtype, V, T);
        else
            lse[i] = NAN;     /* a row past the drafts, or a q row under greedy acceptance */
    }
    (void)row_threads;
    for (int i = 0; i < K * nrow; ++i) {
        const int r = i % nrow;
        const int used = r <= Lb || (r > G && r - G - 1 < Lb && !greedy);
        if (used && !isfinite(lse[i])) err |= SDVO_BAD_ROW;
    }
    if (lse_out) memcpy(lse_out, lse, sizeof(double) * (size_t)K * nrow);
    if (err) goto done;

    /* Ratios a = min(1, p(x)/q(x)) at every drafted token, then the expected
     * accepted streak of every draft.  lo/hi: the same ratios with p/q moved
     * by a relative 1e-5 (exact cases -- q(x) = 0, p(x) = 0, equal
     * log-probabilities -- stay put); they only feed the boundary band. */
    for (size_t i = 0; i < nkg * 3; ++i) a[i] = NAN;
    for (int k = 0; k < K; ++k) {
        for (int j = 0; j < Lb; ++j) {
            int32_t x = drafts[((int64_t)b * K + k) * G + j];
            double lp = sdvo_logprob(p_row(p_logits, sh, b, k, j), dtype, x, T, lse[k * nrow + j]);
            if (greedy) {
                /* greedy acceptance: the ratio is p(x) itself */
                a[k * G + j] = sdvo_accept_ratio_greedy(lp);
                if (lp == -INFINITY || lp >= 0.0) {
                    a_lo[k * G + j] = a_hi[k * G + j] = a[k * G + j];
                } else {
                    double r = exp(lp);
                    a_lo[k * G + j] = fmin(1.0, r * (1.0 - 1e-5));
                    a_hi[k * G + j] = fmin(1.0, r * (1.0 + 1e-5));
                }
                continue;
            }
            double lq = sdvo_logprob(q_row(q_logits, sh, b, k, j), dtype, x, T, lse[k * nrow + G + 1 + j]);
            a[k * G + j] = sdvo_accept_ratio(lp, lq);
            if (lq == -INFINITY || lp == -INFINITY || lp == lq) {
                a_lo[k * G + j] = a_hi[k * G + j] = a[k * G + j];
            } else {
                double r = exp(lp - lq);
                a_lo[k * G + j] = fmin(1.0, r * (1.0 - 1e-5));
                a_hi[k * G + j] = fmin(1.0, r * (1.0 + 1e-5));
            }
        }
        S[k] = sdvo_streak_score(a + (size_t)k * G, Lb);
        S_lo[k] = sdvo_streak_score(a_lo + (size_t)k * G, Lb);
        S_hi[k] = sdvo_streak_score(a_hi + (size_t)k * G, Lb);
    }
    if (scores_out) memcpy(scores_out, S, sizeof(double) * (size_t)K);
    if (ratio_out && G > 0) memcpy(ratio_out, a, sizeof(double) * (size_t)K * G);

    /* Self-selection: the draft with the largest expected streak.  Boundary
     * when the perturbed scores could reorder the first maximum. */
    int sel = sdvo_argmax_first(S, K);
    int band = 0;
    for (int k = 0; k < K; ++k) {
        if (k == sel) continue;
        if ((k < sel && S_hi[k] >= S_lo[sel]) || (k > sel && S_hi[k] > S_lo[sel]))
            band |= SDVO_BAND_SELECT;
    }

    /* Left-to-right acceptance of the selected draft. */
    const double* as = a + (size_t)sel * G;
    int L = sdvo_accept_length(as, u, Lb);
    for (int j = 0; j < Lb && j <= L; ++j)
        if (fabs(u[j] - as[j]) <= 1e-5 * as[j]) band |= SDVO_BAND_ACCEPT;

    /* Replacement at the first rejection (residual max(0, p - q)), or the
     * bonus token from p at position Lb when every draft token was accepted. */
    int64_t tok;
    double R = 0.0, t = 0.0, c_prev = 0.0, c_v = 0.0;
    const void* prow = p_row(p_logits, sh, b, sel, L);
    double lse_p = lse[sel * nrow + L];
    if (L < Lb && greedy) {
        /* greedy: draw from p with the rejected token zeroed out */
        const int32_t xr = drafts[((int64_t)b * K + sel) * G + L];
        for (int64_t v = 0; v < V; ++v)
            r[v] = v == xr ? 0.0 : exp(sdvo_logit(prow, dtype, v) / T - lse_p);
        tok = sdvo_inverse_cdf(r, V, w[L], &R, &t, &c_prev, &c_v);
        if (resid_out) *resid_out = R;
        if (R < 1e-3) band |= SDVO_BAND_RESID;
        if (tok < 0) {
            for (int64_t v = 0; v < V; ++v)
                r[v] = exp(sdvo_logit(prow, dtype, v) / T - lse_p);
            tok = sdvo_inverse_cdf(r, V, w[L], &R, &t, &c_prev, &c_v);
        }
    } else if (L < Lb) {
        const void* qrow = q_row(q_logits, sh, b, sel, L);
        double lse_q = lse[sel * nrow + G + 1 + L];
        for (int64_t v = 0; v < V; ++v) {
            double pv = exp(sdvo_logit(prow, dtype, v) / T - lse_p);
            double qv = exp(sdvo_logit(qrow, dtype, v) / T - lse_q);
            double d = pv - qv;
            r[v] = d > 0.0 ? d : 0.0;
        }
        tok = sdvo_inverse_cdf(r, V, w[L], &R, &t, &c_prev, &c_v);
        if (resid_out) *resid_out = R;
        if (R < 1e-3) band |= SDVO_BAND_RESID;
        if (tok < 0) {
            /* Zero residual mass (p == q on this row up to rounding): draw
             * from p instead. */
            for (int64_t v = 0; v < V; ++v)
                r[v] = exp(sdvo_logit(prow, dtype, v) / T - lse_p);
            tok = sdvo_inverse_cdf(r, V, w[L], &R, &t, &c_prev, &c_v);
        }
    } else {
        for (int64_t v = 0; v < V; ++v)
            r[v] = exp(sdvo_logit(prow, dtype, v) / T - lse_p);
        tok = sdvo_inverse_cdf(r, V, w[Lb], &R, &t, &c_prev, &c_v);
    }
    if (fabs(t - c_v) <= 1e-5 * R || fabs(t - c_prev) <= 1e-5 * R) band |= SDVO_BAND_CDF;

    *sel_out = sel;
    *len_out = L;
    *tok_out = (int32_t)tok;
    if (band_out) *band_out = band;

done:
    free(lse); free(a); free(S); free(r);
    return err;
}

static int run_batch(int B, int K, int gamma, int64_t V, int dtype, int greedy,
                     const void* p_logits, const void* q_logits,
                     const int32_t* drafts, const double* temps, const int32_t* lens,
                     const double* u_in, const double* w_in, int use_philox,
                     uint64_t seed, int32_t b0,
                     int32_t* sel, int32_t* accept_len, int32_t* next_token,
                     double* lse, double* scores, double* ratio,
                     int32_t* band, int32_t* err, double* resid_mass, int nthreads)
{
    shape_t sh = {K, gamma, dtype, V};
    int any = 0;
    if (B < 0 || K < 1 || gamma < 0 || V < 1 || (dtype != SDVO_BF16 && dtype != SDVO_F32))
        return -1;
    const int nrow = 2 * gamma + 1;
    /* Threads go to independent sequences when there are enough of them,
     * else to the independent rows of each sequence. */
    int nt = nthreads > 1 ? nthreads : 1;
    const int seq_threads = B >= nt ? nt : 1;
    const int row_threads = B >= nt ? 1 : nt;
#ifdef _OPENMP
#pragma omp parallel for num_threads(seq_threads) schedule(dynamic, 1) reduction(| : any) if (seq_threads > 1)
#endif
    for (int b = 0; b < B; ++b) {
        double* u = (double*)malloc(sizeof(double) * (size_t)(gamma + 1));
        double* w = (double*)malloc(sizeof(double) * (size_t)(gamma + 1));
        if (!u || !w) { free(u); free(w); any |= -1; continue; }
        for (int j = 0; j <= gamma; ++j) {
            if (use_philox) {
                sdvo_uniforms(seed, (uint32_t)(b0 + b), (uint32_t)j, &u[j], &w[j]);
            } else {
                u[j] = j < gamma ? u_in[(int64_t)b * gamma + j] : 0.0;
                w[j] = w_in[(int64_t)b * (gamma + 1) + j];
            }
        }
        int e = verify_one(&sh, b, p_logits, q_logits, drafts, temps[b],
                           lens ? lens[b] : gamma, u, w,
                           &sel[b], &accept_len[b], &next_token[b],
                           lse ? lse + (int64_t)b * K * nrow : NULL,
                           scores ? scores + (int64_t)b * K : NULL,
                           ratio ? ratio + (int64_t)b * K * gamma : NULL,
                           band ? band + b : NULL,
                           resid_mass ? resid_mass + b : NULL, row_threads, greedy);
        if (err) err[b] = e;
        any |= e;
        free(u); free(w);
    }
    (void)seq_threads;
    return any;
}

int sdvo_verify_uniforms(int B, int K, int gamma, int64_t V, int dtype,
                         const void* p_logits, const void* q_logits,
                         const int32_t* drafts, const double* temps,
                         const double* u, const double* w,
                         int32_t* sel, int32_t* accept_len, int32_t* next_token,
                         double* lse, double* scores, double* ratio,
                         int32_t* band, int32_t* err, double* resid_mass,
                         int nthreads)
{
    return run_batch(B, K, gamma, V, dtype, 0, p_logits, q_logits, drafts, temps, NULL, u, w, 0, 0, 0,
                     sel, accept_len, next_token, lse, scores, ratio, band, err, resid_mass,
                     nthreads);
}

int sdvo_verify_greedy_uniforms(int B, int K, int gamma, int64_t V, int dtype,
                                const void* p_logits, const int32_t* drafts,
                                const double* temps, const double* u, const double* w,
                                int32_t* sel, int32_t* accept_len, int32_t* next_token,
                                double* lse, double* scores, double* ratio,
                                int32_t* band, int32_t* err, double* resid_mass,
                                int nthreads)
{
    return run_batch(B, K, gamma, V, dtype, 1, p_logits, NULL, drafts, temps, NULL, u, w, 0, 0, 0,
                     sel, accept_len, next_token, lse, scores, ratio, band, err, resid_mass,
                     nthreads);
}

int sdvo_verify(int B, int K, int gamma, int64_t V, int dtype,
                const void* p_logits, const void* q_logits,
                const int32_t* drafts, const double* temps, uint64_t seed,
                int32_t b0,
                int32_t* sel, int32_t* accept_len, int32_t* next_token,
                double* lse, double* scores, double* ratio,
                int32_t* band, int32_t* err, double* resid_mass,
                int nthreads)
{
    return run_batch(B, K, gamma, V, dtype, 0, p_logits, q_logits, drafts, temps, NULL, NULL, NULL, 1,
                     seed, b0, sel, accept_len, next_token, lse, scores, ratio, band, err,
                     resid_mass, nthreads);
}

int sdvo_verify_greedy(int B, int K, int gamma, int64_t V, int dtype,
                       const void* p_logits, const int32_t* drafts,
                       const double* temps, uint64_t seed, int32_t b0,
                       int32_t* sel, int32_t* accept_len, int32_t* next_token,
                       double* lse, double* scores, double* ratio,
                       int32_t* band, int32_t* err, double* resid_mass,
                       int nthreads)
{
    return run_batch(B, K, gamma, V, dtype, 1, p_logits, NULL, drafts, temps, NULL, NULL, NULL, 1,
                     seed, b0, sel, accept_len, next_token, lse, scores, ratio, band, err,
                     resid_mass, nthreads);
}

int sdvo_verify_lens(int B, int K, int gamma, int64_t V, int dtype, int greedy,
                     const void* p_logits, const void* q_logits,
                     const int32_t* drafts, const double* temps, const int32_t* lens,
                     uint64_t seed, int32_t b0,
                     int32_t* sel, int32_t* accept_len, int32_t* next_token,
                     double* lse, double* scores, double* ratio,
                     int32_t* band, int32_t* err, double* resid_mass,
                     int nthreads)
{
    return run_batch(B, K, gamma, V, dtype, greedy ? 1 : 0, p_logits, greedy ? NULL : q_logits,
                     drafts, temps, lens, NULL, NULL, 1, seed, b0, sel, accept_len, next_token,
                     lse, scores, ratio, band, err, resid_mass, nthreads);
}

int sdvo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}


/* ------------------------------------------------------------------------ */
/* Causal-consistency path search: candidate pruning and the beam.  Pinned  */
/* by brute force: the kept set is the smallest most-likely set reaching    */
/* tau, and the beam equals the exact top paths of the whole lattice.       */
/* ------------------------------------------------------------------------ */

typedef struct {
    double z;     /* l / T (orders like the probability) */
    int64_t v;
} cps_entry_t;

static int cps_cmp(const void* a, const void* b)
{
    const cps_entry_t* x = (const cps_entry_t*)a;
    const cps_entry_t* y = (const cps_entry_t*)b;
    if (x->z > y->z) return -1;
    if (x->z < y->z) return 1;
    return x->v < y->v ? -1 : (x->v > y->v ? 1 : 0);
}

int sdvo_cps_prune_row(const void* row, int dtype, int64_t V, double T, double tau, int mmax,
                       int32_t* ids, double* logp, double* mass_before, double* mass_after)
{
    double lse = sdvo_row_lse(row, dtype, V, T);
    if (!isfinite(lse)) {
        /* NaN / +inf logits, or no token of positive probability: the row
         * offers no candidates */
        if (mass_before) *mass_before = 0.0;
        if (mass_after) *mass_after = 0.0;
        return 0;
    }
    cps_entry_t* e = (cps_entry_t*)malloc(sizeof(cps_entry_t) * (size_t)V);
    if (!e) return -1;
    for (int64_t v = 0; v < V; ++v) {
        e[v].z = sdvo_logit(row, dtype, v) / T;
        e[v].v = v;
    }
    qsort(e, (size_t)V, sizeof(cps_entry_t), cps_cmp);
    double mass = 0.0, before = 0.0;
    int n = 0;
    while (n < mmax && n < V) {
        if (e[n].z == -INFINITY) break;       /* probability zero: never a candidate */
        double lp = e[n].z - lse;
        ids[n] = (int32_t)e[n].v;
        logp[n] = lp;
        before = mass;
        mass += exp(lp);
        ++n;
        if (mass >= tau) break;
    }
    if (mass_before) *mass_before = before;
    if (mass_after) *mass_after = mass;
    free(e);
    return n;
}

/* One beam entry: the order key (sum of the chosen tokens' raw logits), the
 * score (sum of their log-probabilities) and the candidate rank chosen at
 * every position. */
typedef struct {
    double key;
    double score;
    int32_t* ranks;
} cps_beam_t;

/* order: key desc, then candidate ranks lexicographically asc */
static int cps_beam_before(const double ka, const int32_t* ra, const double kb, const int32_t* rb,
                           int len)
{
    if (ka > kb) return 1;
    if (ka < kb) return 0;
    for (int i = 0; i < len; ++i) {
        if (ra[i] < rb[i]) return 1;
        if (ra[i] > rb[i]) return 0;
    }
    return 0;
}

static int cps_one(int b, int gamma, int64_t V, int dtype, const void* q, double T, double tau,
                   int mmax, int beam, int32_t eos_id, int32_t* cand_ids, double* cand_logp,
                   int32_t* ncand, int32_t* lat_len, int32_t* paths, double* path_logp,
                   int32_t* npaths, int32_t* band_out)
{
    size_t elt = dtype == SDVO_BF16 ? 2 : 4;
    int band = 0;
    int32_t* ci = cand_ids + (int64_t)b * gamma * mmax;
    double* cl = cand_logp + (int64_t)b * gamma * mmax;
    int32_t* nc = ncand + (int64_t)b * gamma;
    for (int i = 0; i < gamma * mmax; ++i) { ci[i] = -1; cl[i] = -INFINITY; }
    /* Prune every position; the lattice ends at the first position whose
     * most likely token is EOS, which is kept alone as the last token. */
    int Lc = gamma;
    for (int j = 0; j < gamma; ++j) {
        const void* row = (const char*)q + (size_t)(((int64_t)b * gamma + j) * V) * elt;
        double mb = 0.0, ma = 0.0;
        int n = sdvo_cps_prune_row(row, dtype, V, T, tau, mmax, ci + j * mmax, cl + j * mmax, &mb, &ma);
        if (n < 0) return -1;
        nc[j] = n;
        /* band: the decision to stop (mass with the last kept token reaches
         * tau) or to go on (mass before it was below tau) was within 1e-5 */
        if (j < Lc && ((n < mmax && fabs(ma - tau) <= 1e-5) || (n > 1 && fabs(mb - tau) <= 1e-5)))
            band |= SDVO_CPS_BAND_MASS;
        if (j < Lc && eos_id >= 0 && ci[j * mmax] == eos_id) {
            Lc = j + 1;
            nc[j] = 1;
            for (int i = 1; i < mmax; ++i) { ci[j * mmax + i] = -1; cl[j * mmax + i] = -INFINITY; }
        }
    }
    for (int j = Lc; j < gamma; ++j) {
        nc[j] = 0;
        for (int i = 0; i < mmax; ++i) { ci[j * mmax + i] = -1; cl[j * mmax + i] = -INFINITY; }
    }
    lat_len[b] = Lc;

    /* Beam search, left to right, keeping the `beam` best prefixes.  A path's
     * score is the sum of its log-probabilities, l_j(x_j) / T - lse_j; the
     * temperature and every position's normaliser are shared by all paths of
     * the sequence, so paths rank as the sums of their raw logits, taken
     * left to right in fp64 (exact for bf16 logits).  The candidates of a
     * step are taken one by one into a sorted list of at most `beam`. */
    const int W = beam;
    cps_beam_t* cur = (cps_beam_t*)calloc((size_t)W + 1, sizeof(cps_beam_t));
    cps_beam_t* nxt = (cps_beam_t*)calloc((size_t)W + 1, sizeof(cps_beam_t));
    int32_t* store = (int32_t*)calloc((size_t)(2 * (W + 1)) * (gamma > 0 ? gamma : 1), sizeof(int32_t));
    int32_t* tmp = (int32_t*)calloc((size_t)(gamma > 0 ? gamma : 1), sizeof(int32_t));
    double* rl = (double*)calloc((size_t)gamma * mmax, sizeof(double));
    if (!cur || !nxt || !store || !tmp || !rl) {
        free(cur); free(nxt); free(store); free(tmp); free(rl);
        return -1;
    }
    for (int j = 0; j < Lc; ++j) {
        const void* row = (const char*)q + (size_t)(((int64_t)b * gamma + j) * V) * elt;
        for (int r = 0; r < nc[j]; ++r) rl[j * mmax + r] = sdvo_logit(row, dtype, ci[j * mmax + r]);
    }
    for (int i = 0; i <= W; ++i) {
        cur[i].ranks = store + (size_t)i * gamma;
        nxt[i].ranks = store + (size_t)(W + 1 + i) * gamma;
    }
    int ncur = 1;
    cur[0].key = 0.0;
    cur[0].score = 0.0;
    for (int j = 0; j < Lc; ++j) {
        int nn = 0;
        for (int w = 0; w < ncur; ++w) {
            for (int r = 0; r < nc[j]; ++r) {
                double key = cur[w].key + rl[j * mmax + r];
                for (int i = 0; i < j; ++i) tmp[i] = cur[w].ranks[i];
                tmp[j] = r;
                /* insert into nxt (sorted, at most W entries) */
                int pos = nn;
                while (pos > 0 && cps_beam_before(key, tmp, nxt[pos - 1].key, nxt[pos - 1].ranks, j + 1))
                    --pos;
                if (pos >= W) continue;
                int last = nn < W ? nn : W - 1;
                int32_t* spare = nxt[last].ranks;
                for (int i = last; i > pos; --i) nxt[i] = nxt[i - 1];
                nxt[pos].ranks = spare;
                nxt[pos].key = key;
                nxt[pos].score = cur[w].score + cl[j * mmax + r];
                for (int i = 0; i <= j; ++i) nxt[pos].ranks[i] = tmp[i];
                if (nn < W) ++nn;
            }
        }
        ncur = nn;
        cps_beam_t* t = cur; cur = nxt; nxt = t;
    }
    int32_t* pb = paths + (int64_t)b * W * gamma;
    double* sb = path_logp + (int64_t)b * W;
    for (int w = 0; w < W; ++w) {
        sb[w] = -INFINITY;
        for (int j = 0; j < gamma; ++j) pb[w * gamma + j] = -1;
    }
    for (int w = 0; w < ncur; ++w) {
        sb[w] = cur[w].score;
        for (int j = 0; j < Lc; ++j) pb[w * gamma + j] = ci[j * mmax + cur[w].ranks[j]];
    }
    npaths[b] = ncur;
    if (band_out) band_out[b] = band;
    free(cur); free(nxt); free(store); free(tmp); free(rl);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Adaptive draft length.  Pinned by hand-worked traces of the rule (growth */
/* to the cap, holding under EOS saturation, shrinking to the floor, the    */
/* window's averaging) and by its invariants.                               */
/* ------------------------------------------------------------------------ */

/* state layout: [0] steps seen, then W entries of (k, g, a) in a ring */
int sdvo_adl_state_words(int W)
{
    return 1 + 3 * W;
}

int sdvo_adl_step(int B, int W, int kmin, int kmax, int up, int down, const int32_t* gen_len,
                  const int32_t* acc_len, int32_t* k, int32_t* state)
{
    if (B < 0 || W < 1 || kmin < 1 || kmax < kmin || up < 0 || down < 0) return -1;
    for (int b = 0; b < B; ++b)
        if (k[b] < kmin || k[b] > kmax) return -1;
    const int words = sdvo_adl_state_words(W);
    for (int b = 0; b < B; ++b) {
        int32_t* st = state + (int64_t)b * words;
        int64_t kb = k[b];
        /* this step's lengths, clamped to what a step can produce */
        int64_t g = gen_len[b];
        if (g < 0) g = 0;
        if (g > kb) g = kb;
        int64_t a = acc_len[b];
        if (a < 0) a = 0;
        if (a > g) a = g;
        /* record the step in the window */
        int64_t seen = st[0];
        int slot = (int)(seen % W);
        st[1 + 3 * slot + 0] = (int32_t)kb;
        st[1 + 3 * slot + 1] = (int32_t)g;
        st[1 + 3 * slot + 2] = (int32_t)a;
        seen += 1;
        /* once the window is full the counter stays in [W, 2W): W + the ring
         * position of the next slot, so it never overflows */
        st[0] = (int32_t)(seen < W ? seen : W + (seen % W));
        /* averages over the window, compared as sums */
        int n = seen < W ? (int)seen : W;
        int64_t sk = 0, sg = 0, sa = 0;
        for (int i = 0; i < n; ++i) {
            sk += st[1 + 3 * i + 0];
            sg += st[1 + 3 * i + 1];
            sa += st[1 + 3 * i + 2];
        }
        int keeps_pace = sa >= sg;
        int fills = sg >= sk;
        int64_t next;
        if (keeps_pace && fills)
            next = kb + up;           /* expand */
        else if (keeps_pace)
            next = kb;                /* generation saturated: hold */
        else
            next = kb - down;         /* acceptance falls behind: shrink */
        if (next > kmax) next = kmax;
        if (next < kmin) next = kmin;
        k[b] = (int32_t)next;
    }
    return 0;
}

int sdvo_cps(int B, int gamma, int64_t V, int dtype, const void* q, const double* temps,
             double tau, int mmax, int beam, int32_t eos_id,
             int32_t* cand_ids, double* cand_logp, int32_t* ncand, int32_t* lat_len,
             int32_t* paths, double* path_logp, int32_t* npaths, int32_t* band, int nthreads)
{
    if (B < 1 || gamma < 1 || V < 1 || mmax < 1 || beam < 1) return -1;
    int any = 0;
#ifdef _OPENMP
    int nt = nthreads > 1 ? nthreads : 1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1) reduction(| : any) if (nt > 1)
#endif
    for (int b = 0; b < B; ++b)
        any |= cps_one(b, gamma, V, dtype, q, temps[b], tau, mmax, beam, eos_id, cand_ids,
                       cand_logp, ncand, lat_len, paths, path_logp, npaths, band);
    (void)nthreads;
    return any;
}
