/*
 * sdv_oracle.h -- plain, slow, fp64 CPU oracle of the batched lossless
 * draft-verification step with test-time self-selection.
 *
 * TEST INFRASTRUCTURE ONLY.  This library exists to check the CUDA path.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code, header, table or constant with the CUDA
 * library, and it includes nothing from it.
 *
 * Passages followed (page title, section):
 *   - "SpecDiff-2: Scaling Diffusion Drafter Alignment For Faster Speculative
 *     Decoding" (paperlayer summary), section 2 "Prelim: speculative
 *     decoding": left-to-right commit with the standard lossless acceptance
 *     rule, immediate acceptance when q(x|s) <= p(x|s), a replacement token
 *     from the normalised residual at the first rejection.
 *   - same page, Figure 2 and section 3: position-wise acceptance alpha_j and
 *     the accepted streak.
 *   - same page, section 5.2 "Test-time alignment: self-selection
 *     acceptance": K joint drafts ranked by a streak-oriented verifier score,
 *     the best is verified losslessly, verifier probabilities are reused.
 *   - "DiffuSpec: Unlocking Diffusion Language Models for Speculative
 *     Decoding" (paperlayer summary), section 3: residual replacement,
 *     unbiasedness.
 * The score formula sum_j prod_{i<=j} min(1, p/q), the Philox keying, the
 * bonus token and the argument layout are a reading of the method: the pages
 * state these quantities only in prose.
 *
 * Parity status of each function is stated next to it; every function here
 * is pinned by a test that does not re-derive the function itself.
 */
#ifndef SDV_ORACLE_H
#define SDV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SDVO_BF16 0
#define SDVO_F32 1

/* Boundary-band flags (one word per sequence).  A trial whose flag is set may
 * be decided differently by a correct fp32 implementation. */
#define SDVO_BAND_ACCEPT 1   /* |u_j - a_j| <= 1e-5 a_j at a decided position  */
#define SDVO_BAND_CDF 2      /* |t - C_v| <= 1e-5 R at the chosen v or v-1      */
#define SDVO_BAND_SELECT 4   /* moving any p/q by 1e-5 (relative) could change  */
                             /* the first maximum of the streak scores          */
#define SDVO_BAND_RESID 8    /* residual mass R < 1e-3 (ill-conditioned draw)   */

/* Status codes of sdvo_verify / sdvo_verify_uniforms (per sequence in err[]). */
#define SDVO_OK 0
#define SDVO_BAD_DRAFT 1     /* draft id outside [0, V)                          */
#define SDVO_BAD_ROW 2       /* a row holds NaN/+inf or is all -inf              */
#define SDVO_BAD_TEMP 4      /* temperature not finite or <= 0                   */

/* Philox4x32-10 block function (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC'11): 10 rounds of the 4x32 Philox
 * S-box, key bumped by the Weyl constants between rounds. */
void sdvo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* 24-bit uniform in [0, 1 - 2^-24]: (word >> 8) * 2^-24. */
double sdvo_uniform24(uint32_t word);

/* Uniforms for sequence b, position j: counter (j, b, 0, 0), key (seed low
 * word, seed high word).  Word 0 -> acceptance uniform u, word 1 -> sampling
 * uniform w. */
void sdvo_uniforms(uint64_t seed, uint32_t b, uint32_t j, double* u, double* w);

/* Decode logit `index` of a row stored as bf16 (raw 16-bit words) or fp32. */
double sdvo_logit(const void* row, int dtype, int64_t index);

/* Log-sum-exp of z_v = l_v / T over one row, two passes (max, then sum of
 * exp(z - max)).  Returns NaN if the row holds NaN or +inf, -inf if every
 * entry is -inf. */
double sdvo_row_lse(const void* row, int dtype, int64_t V, double T);

/* log-probability log p(x) = l_x / T - LSE. */
double sdvo_logprob(const void* row, int dtype, int64_t x, double T, double lse);

/* Acceptance ratio a = min(1, p(x)/q(x)) from log-probabilities.  q(x) = 0
 * (lq = -inf) counts as q <= p, so a = 1; p(x) = 0 < q(x) gives a = 0. */
double sdvo_accept_ratio(double lp, double lq);

/* Greedy acceptance ratio from the verifier alone: a = p(x) (the drafted
 * token's verifier probability; "SpecDiff-2: Scaling Diffusion Drafter
 * Alignment For Faster Speculative Decoding", section 5.2 and appendix B.4). */
double sdvo_accept_ratio_greedy(double lp);

/* Expected accepted streak S = sum_{j<gamma} prod_{i<=j} a_i. */
double sdvo_streak_score(const double* a, int gamma);

/* Index of the first maximum of s[0..K). */
int sdvo_argmax_first(const double* s, int K);

/* Accepted length: the first j with not(a_j >= 1 or u_j < a_j), else gamma. */
int sdvo_accept_length(const double* a, const double* u, int gamma);

/* Inverse CDF over non-negative weights r[0..V): R = sum r (increasing id
 * order), t = w R, returns the first v with C_v = sum_{i<=v} r_i > t.  If no v
 * qualifies (rounding), the last v with r_v > 0.  Returns -1 if R == 0.
 * Optional outputs: *R_out, *t_out, *c_prev_out (C_{v-1}), *c_v_out (C_v). */
int64_t sdvo_inverse_cdf(const double* r, int64_t V, double w, double* R_out,
                         double* t_out, double* c_prev_out, double* c_v_out);

/* Full step for a batch with explicit uniforms u[B][gamma] and
 * w[B][gamma+1] (random numbers passed in as inputs).
 *   p_logits [B][K][gamma+1][V], q_logits [B][K][gamma][V] (dtype), drafts
 *   [B][K][gamma] int32, temps [B] (> 0).
 *   Outputs (each may be NULL except sel/accept_len/next_token):
 *   sel[B], accept_len[B], next_token[B]   (-1 for a sequence with err != 0)
 *   lse[B][K][2 gamma + 1]: p rows j=0..gamma, then q rows j=0..gamma-1
 *   scores[B][K], ratio[B][K][gamma], band[B], err[B], resid_mass[B].
 * Returns the OR of all err[] words.  nthreads > 1 runs sequences in
 * parallel (independent problems); 0 or 1 runs serially. */
int sdvo_verify_uniforms(int B, int K, int gamma, int64_t V, int dtype,
                         const void* p_logits, const void* q_logits,
                         const int32_t* drafts, const double* temps,
                         const double* u, const double* w,
                         int32_t* sel, int32_t* accept_len, int32_t* next_token,
                         double* lse, double* scores, double* ratio,
                         int32_t* band, int32_t* err, double* resid_mass,
                         int nthreads);

/* Same, with the Philox uniforms of sdvo_uniforms(seed, b0 + b, j); b0 is the
 * index of the first sequence of this batch within the full call, so a
 * sample of sequences can be checked on its own. */
int sdvo_verify(int B, int K, int gamma, int64_t V, int dtype,
                const void* p_logits, const void* q_logits,
                const int32_t* drafts, const double* temps, uint64_t seed,
                int32_t b0,
                int32_t* sel, int32_t* accept_len, int32_t* next_token,
                double* lse, double* scores, double* ratio,
                int32_t* band, int32_t* err, double* resid_mass,
                int nthreads);

/* Greedy acceptance (same page, section 5.2 and appendix B.4): no drafter
 * rows.  a_j = p_j(x_j); S_k and the selection as above; accept iff
 * u_j < p_j(x_j); at the first rejection L draw from p_L with x_L zeroed out
 * (renormalised); if all are accepted, the bonus token from p_gamma.  The
 * q entries of lse[] are NaN. */
int sdvo_verify_greedy_uniforms(int B, int K, int gamma, int64_t V, int dtype,
                                const void* p_logits, const int32_t* drafts,
                                const double* temps, const double* u, const double* w,
                                int32_t* sel, int32_t* accept_len, int32_t* next_token,
                                double* lse, double* scores, double* ratio,
                                int32_t* band, int32_t* err, double* resid_mass,
                                int nthreads);
int sdvo_verify_greedy(int B, int K, int gamma, int64_t V, int dtype,
                       const void* p_logits, const int32_t* drafts,
                       const double* temps, uint64_t seed, int32_t b0,
                       int32_t* sel, int32_t* accept_len, int32_t* next_token,
                       double* lse, double* scores, double* ratio,
                       int32_t* band, int32_t* err, double* resid_mass,
                       int nthreads);

/* Either rule (greedy = 0: the standard rule, 1: greedy acceptance, q_logits
 * unused) with a draft length per sequence: lens[b] in [0, gamma] (the arrays
 * keep their gamma stride; positions at or past lens[b] are not read).  The
 * scores and the scan run over j < lens[b]; with every token accepted the
 * bonus token comes from p at position lens[b], drawn with the uniform
 * w_{lens[b]}.  lse[] entries of rows not read are NaN; a length outside
 * [0, gamma] is a draft error. */
int sdvo_verify_lens(int B, int K, int gamma, int64_t V, int dtype, int greedy,
                     const void* p_logits, const void* q_logits,
                     const int32_t* drafts, const double* temps, const int32_t* lens,
                     uint64_t seed, int32_t b0,
                     int32_t* sel, int32_t* accept_len, int32_t* next_token,
                     double* lse, double* scores, double* ratio,
                     int32_t* band, int32_t* err, double* resid_mass,
                     int nthreads);

/* ------------------------------------------------------------------------ */
/* Causal-consistency path search ("DiffuSpec: Unlocking Diffusion Language   */
/* Models for Speculative Decoding", section 4.2; settings of section 5.3).   */
/* ------------------------------------------------------------------------ */

/* Band flags of a CPS result (one word per sequence). */
#define SDVO_CPS_BAND_MASS 1   /* a cumulative mass within 1e-5 of tau at a cut  */

/* Candidates of one drafter row: softmax(l / T), tokens in order of
 * (probability desc, id asc); keep the shortest prefix whose mass reaches tau,
 * at most mmax tokens; a token of probability zero is never kept.  Writes ids
 * and natural-log probabilities, returns the count (0 for a row with a NaN or
 * +inf logit or none finite); *mass_before / *mass_after get the mass without
 * / with the last kept token (for the band check). */
int sdvo_cps_prune_row(const void* row, int dtype, int64_t V, double T, double tau, int mmax,
                       int32_t* ids, double* logp, double* mass_before, double* mass_after);

/* Pruning of every row of q [B][gamma][V], the lattice cut at the first
 * position whose most likely token is eos_id (kept as the last token; eos_id <
 * 0: no cut), and a left-to-right beam of width `beam` over the lattice,
 * scoring a path by the sum of its log-probabilities (drafter confidence).
 * Paths rank as the sums of their raw logits (the temperature and the
 * positions' normalisers are common to all paths), summed left to right in
 * fp64; ties go to the path whose candidate ranks come first
 * lexicographically.  With this separable score the beam returns the exact
 * `beam` best paths.
 * Outputs: cand_ids / cand_logp [B][gamma][mmax] (-1 / -inf past the count),
 * ncand [B][gamma] (0 past the lattice), lat_len [B], paths [B][beam][gamma]
 * (-1 past the lattice), path_logp [B][beam] (-inf for missing paths),
 * npaths [B], band [B] (may be NULL). */
int sdvo_cps(int B, int gamma, int64_t V, int dtype, const void* q, const double* temps,
             double tau, int mmax, int beam, int32_t eos_id,
             int32_t* cand_ids, double* cand_logp, int32_t* ncand, int32_t* lat_len,
             int32_t* paths, double* path_logp, int32_t* npaths, int32_t* band, int nthreads);

/* ------------------------------------------------------------------------ */
/* Adaptive draft length ("DiffuSpec", section 4.3; appendix C).  The page  */
/* gives the controller's inputs and direction, not a formula.  Reading:    */
/* over the last W steps of a sequence (k_i drafted, g_i generated up to    */
/* and including the first EOS, a_i accepted), acceptance keeps pace when   */
/* sum a >= sum g, and generation fills the drafts when sum g >= sum k.     */
/* Then k grows by `up` (at most kmax); if acceptance keeps pace but        */
/* generation saturates (EOS before the draft end), k holds; if acceptance  */
/* falls behind, k shrinks by `down` (at least kmin).  Inputs are clamped   */
/* to 0 <= g <= k and 0 <= a <= g before they enter the window.             */
/* ------------------------------------------------------------------------ */

/* Number of int32 words of one sequence's controller state for window W. */
int sdvo_adl_state_words(int W);

/* One step for B sequences: k [B] holds the draft length each sequence just
 * used and receives the next one; gen_len / acc_len [B] are that step's
 * generated and accepted lengths; state [B][sdvo_adl_state_words(W)] starts
 * zeroed.  Returns 0, or -1 for invalid parameters (W < 1, kmin < 1,
 * kmax < kmin, up < 0, down < 0, a k outside [kmin, kmax]). */
int sdvo_adl_step(int B, int W, int kmin, int kmax, int up, int down, const int32_t* gen_len,
                  const int32_t* acc_len, int32_t* k, int32_t* state);

/* Number of threads the build can run (1 without OpenMP). */
int sdvo_max_threads(void);

#ifdef __cplusplus
}
#endif

#endif
