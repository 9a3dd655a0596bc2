/*
 * sdv.h -- C ABI of libsdv: batched lossless draft verification with
 * test-time self-selection, for speculative decoding with diffusion drafters,
 * on one NVIDIA GB300 (sm_103a).
 *
 * What one call computes, for every sequence b of a batch of B, given K
 * candidate drafts of gamma tokens each:
 *
 *   1. Temperature softmax of every verifier row p(.|s, x_<j) (j = 0..gamma)
 *      and drafter row q_j (j = 0..gamma-1) over the full vocabulary V.
 *      ("SpecDiff-2: Scaling Diffusion Drafter Alignment For Faster
 *      Speculative Decoding", section 2: the verifier scores all positions in
 *      parallel and exposes q(.|s) and p(.|s).)
 *   2. Per drafted token the acceptance ratio a = min(1, p(x)/q(x)), and per
 *      draft the expected accepted streak S_k = sum_j prod_{i<=j} a_i
 *      (same page, Figure 2 and section 3: position-wise acceptance and
 *      accepted streaks).
 *   3. Self-selection: sel = argmax_k S_k, ties to the lowest k (same page,
 *      section 5.2: K drafts from one denoising pass are ranked by a
 *      streak-oriented verifier score and the best is verified; the verifier
 *      probabilities of the ranking are reused for acceptance).
 *   4. The standard left-to-right acceptance rule on draft sel: token j is
 *      accepted when q <= p, else when u_j < p/q; the first rejection ends the
 *      scan (same page, section 2; "DiffuSpec: Unlocking Diffusion Language
 *      Models for Speculative Decoding", section 3).
 *   5. At the first rejection L < gamma, a replacement token drawn from the
 *      normalised residual max(0, p_L - q_L) (same passages); when all gamma
 *      tokens are accepted, a bonus token drawn from p_gamma.
 *
 * Random numbers: Philox4x32-10 (Salmon et al., SC'11) with key
 * (seed & 0xffffffff, seed >> 32) and counter (j, b, 0, 0); word 0 gives the
 * acceptance uniform u_j, word 1 the sampling uniform w_j, each as
 * (word >> 8) * 2^-24.  The uniforms do not depend on k.  Inverse-CDF draws
 * return the first id v whose cumulative mass exceeds w * (total mass).
 *
 * Layout: every tensor is contiguous, row-major, on the device of the
 * context unless stated otherwise.
 *   p_logits  [B][K][gamma+1][V]  bf16 or fp32
 *   q_logits  [B][K][gamma][V]    same dtype as p_logits ([B][gamma][V] with
 *                                 SDV_FLAG_SHARED_Q, see sdv_create_ex)
 *   drafts    [B][K][gamma]       int32 token ids
 *   out_sel, out_accept_len, out_next_token  [B] int32
 * V * sizeof(element) must be a multiple of 16 bytes and both logit buffers
 * 16-byte aligned (every row then starts on a 16-byte boundary).
 *
 * Ownership: the caller owns every tensor.  A context owns its workspace
 * (allocated by sdv_create, freed by sdv_destroy) and borrows the stream.
 *
 * Errors: argument errors are returned synchronously and nothing is
 * enqueued.  Data errors found on the device (a draft id outside [0, V), a row
 * holding NaN or +inf or only -inf, a per-sequence temperature that is not a
 * finite positive number) set the outputs of that sequence to -1 and are
 * reported by the next sdv_sync.  A context is not thread-safe; use one
 * context per stream.  Outputs are a pure function of (inputs, temperature,
 * seed).
 *
 * CUDA graphs: sdv_verify, sdv_verify_ex, sdv_verify_len, sdv_verify_qstat,
 * sdv_cps, sdv_cps_ex, sdv_cps_prune, sdv_cps_beam and sdv_adl_step check
 * their arguments on the host and enqueue kernels; they allocate nothing,
 * copy nothing and never wait.  Each may therefore be captured into a CUDA graph, in any capture
 * mode, when the stream it launches on (the context's, for the verify calls:
 * see sdv_set_stream) is the capturing stream, with kernel timing off.  Make
 * one uncaptured call of each shape first (the path search may set a kernel
 * attribute on its first call with a large lattice).  A replay recomputes the
 * step from the current contents of the captured buffers, with the scalars of
 * the capture (temperature, seed, tau, ...).  sdv_verify_host and sdv_sync
 * wait for the stream and cannot be captured.
 */
#ifndef SDV_H
#define SDV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sdv_ctx sdv_ctx;

typedef enum {
    SDV_OK = 0,
    SDV_ERR_ARG = 1,          /* bad argument; nothing was enqueued              */
    SDV_ERR_CUDA = 2,         /* a CUDA runtime call failed, or a device wait    */
                              /* gave up after its iteration limit               */
    SDV_ERR_OOM = 3,          /* workspace allocation failed                     */
    SDV_ERR_DEVICE_DATA = 4,  /* bad draft id / non-finite row / bad per-seq T   */
    SDV_ERR_SCRATCH = 5       /* sdv_verify_static: the shape needs more scratch */
                              /* than SDV_STATIC_SCRATCH_BYTES                   */
} sdv_status;

typedef enum { SDV_BF16 = 0, SDV_F32 = 1 } sdv_dtype;

/*
 * Create a context for batches of shape (B, K, gamma, V) on the current CUDA
 * device, enqueuing on `stream` (a cudaStream_t; NULL = the legacy default
 * stream).  Requires B >= 1, K >= 1, gamma >= 1, V >= 1, V * elt % 16 == 0.
 * Allocates the workspace (partial row statistics, per-sequence tasks, a
 * status word: a few MB at most).  The select pass holds about
 * K * (20 * gamma + 12) bytes per sequence in shared memory; a shape beyond
 * the device's per-block limit (227 KB on GB300, where K = 64 at gamma = 128
 * fits) is refused with SDV_ERR_ARG.  On error *out is NULL.
 */
sdv_status sdv_create(sdv_ctx** out, int B, int K, int gamma, int V,
                      sdv_dtype dtype, void* stream);

/*
 * Layout flags for sdv_create_ex.
 *
 * SDV_FLAG_SHARED_Q: the K drafts of a sequence are sampled from the
 * position-wise marginals of one denoising pass ("SpecDiff-2: Scaling
 * Diffusion Drafter Alignment For Faster Speculative Decoding", section 5.2),
 * so the drafter rows do not depend on k: q_logits is [B][gamma][V] and row
 * (b, j) serves every draft k.  Each marginal row is read once, which cuts the
 * drafter bytes K-fold.  Results equal those of the full layout with q
 * broadcast over k.
 */
#define SDV_FLAG_SHARED_Q 1u

/*
 * SDV_FLAG_GREEDY: greedy acceptance, which verifies the selected draft
 * without drafting probabilities (same page, section 5.2 and appendix B.4;
 * usable with drafters of another tokenizer).  No drafter rows are read:
 * q_logits may be NULL.  a_j = p_j(x_j), the streak score is
 * S_k = sum_j prod_{i<=j} p_i(x_i), token j is accepted when u_j < p_j(x_j),
 * and at the first rejection L the replacement is drawn from p_L with x_L
 * zeroed out (renormalised); with every token accepted, the bonus token comes
 * from p_gamma.  out_lse is then [B][K][gamma+1].  Cannot be combined with
 * SDV_FLAG_SHARED_Q.
 */
#define SDV_FLAG_GREEDY 2u

/*
 * SDV_FLAG_SHARED_PREFIX_ROW: the verifier row at position 0 of every draft
 * conditions only on the shared prefix s (same page, section 5.2: the K
 * drafts extend one prefix), so it is one row per sequence: row (b, 0, 0) of
 * p_logits serves every draft k and rows (b, k > 0, 0) are not read (their
 * contents do not matter).  p_logits keeps its [B][K][gamma+1][V] shape.
 * Results equal those of the full layout with row (b, 0, 0) copied to every
 * k.  Combines with either flag above.
 */
#define SDV_FLAG_SHARED_PREFIX_ROW 4u

/* sdv_create with layout flags (0 = the full [B][K][gamma][V] q layout). */
sdv_status sdv_create_ex(sdv_ctx** out, int B, int K, int gamma, int V,
                         sdv_dtype dtype, void* stream, unsigned flags);

/*
 * Enqueue one verification step with one temperature for all sequences
 * (temperature > 0, finite; it scales both p and q).  Returns after
 * enqueuing; the outputs are valid once the stream has reached this point.
 */
sdv_status sdv_verify(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                      const int32_t* drafts, float temperature, uint64_t seed,
                      int32_t* out_sel, int32_t* out_accept_len,
                      int32_t* out_next_token);

/*
 * As sdv_verify, plus:
 *   temperature_per_seq  device float [B] or NULL (NULL: use `temperature`)
 *   out_scores           device float [B][K] expected streaks, or NULL
 *   out_lse              device float [B][K][2 gamma + 1] row log-sum-exp of
 *                        l / T (p rows j = 0..gamma, then q rows j = 0..gamma-1),
 *                        or NULL
 */
sdv_status sdv_verify_ex(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                         const int32_t* drafts, float temperature,
                         const float* temperature_per_seq, uint64_t seed,
                         int32_t* out_sel, int32_t* out_accept_len,
                         int32_t* out_next_token, float* out_scores,
                         float* out_lse);

/*
 * As sdv_verify_ex, with a draft length per sequence ("DiffuSpec: Unlocking
 * Diffusion Language Models for Speculative Decoding", sections 4.2-4.3: the
 * draft length adapts per step, and a path ends at its first EOS).
 *   draft_len  device int32 [B], 0 <= draft_len[b] <= gamma (required)
 * The arrays keep their gamma stride; for sequence b only the drafts at
 * positions j < draft_len[b] count, so the caller may leave the rest as
 * they are.  The streak scores and the acceptance scan run over those
 * positions, and with all of them accepted the bonus token comes from the
 * verifier row at position draft_len[b], drawn with that position's uniform.
 * Rows past a sequence's length are not read: the p rows j > draft_len[b] and
 * the q rows j >= draft_len[b].  Their out_lse entries are NaN.  The result
 * for b equals that of sdv_verify_ex on the drafts cut to draft_len[b].  A
 * length outside [0, gamma] is a data error for that sequence: its outputs
 * are -1, and sdv_sync reports SDV_ERR_DEVICE_DATA.
 */
sdv_status sdv_verify_len(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                          const int32_t* drafts, const int32_t* draft_len, float temperature,
                          const float* temperature_per_seq, uint64_t seed, int32_t* out_sel,
                          int32_t* out_accept_len, int32_t* out_next_token, float* out_scores,
                          float* out_lse);

/*
 * As sdv_verify_len (draft_len may be NULL: every draft has gamma tokens),
 * with the drafter rows' softmax statistics supplied by the caller instead of
 * computed here.  In a decode step the path search has just streamed the same
 * marginals (sdv_cps_ex writes these statistics), so the verification reads
 * the q rows only at the drafted tokens and, for a rejection, in the residual
 * draw: one full pass over the marginals per step instead of two.
 *   q_row_stat  device float [rows_q][4], 16-byte aligned, one entry per q
 *               row in q_logits' row order ([B][gamma] with
 *               SDV_FLAG_SHARED_Q, else [B][K][gamma]):
 *               {m, s, c, 0} with c = 1.4426950408889634f / T, an fp32
 *               division (T the row's sequence's temperature), m the row's
 *               largest logit and s = sum over the row of 2^((logit - m) * c)
 * The result is that of sdv_verify_len up to the rounding of s (the sum is
 * taken in another order).  An entry whose c differs from the c this call
 * computes for its sequence is a data error for that sequence (outputs -1,
 * SDV_ERR_DEVICE_DATA from sdv_sync).  A row whose m or s is not finite, or
 * s <= 0, is a bad row as for sdv_verify_ex.  Not with SDV_FLAG_GREEDY
 * (which reads no q rows): SDV_ERR_ARG.
 */
sdv_status sdv_verify_qstat(sdv_ctx* ctx, const void* p_logits, const void* q_logits,
                            const int32_t* drafts, const int32_t* draft_len,
                            const float* q_row_stat, float temperature,
                            const float* temperature_per_seq, uint64_t seed, int32_t* out_sel,
                            int32_t* out_accept_len, int32_t* out_next_token, float* out_scores,
                            float* out_lse);

/*
 * End-to-end variant for callers whose data lives in HOST memory: copies the
 * inputs to device buffers owned by the context (allocated on the first call,
 * the size of one batch's inputs), runs sdv_verify_ex, copies the three
 * outputs back and waits for the stream.  All pointers are host pointers
 * (pinned memory gives full copy bandwidth); temperature_per_seq may be NULL.
 * Returns the status of the step, as sdv_sync would.
 */
sdv_status sdv_verify_host(sdv_ctx* ctx, const void* p_logits_host,
                           const void* q_logits_host, const int32_t* drafts_host,
                           float temperature, const float* temperature_per_seq_host,
                           uint64_t seed, int32_t* out_sel_host,
                           int32_t* out_accept_len_host,
                           int32_t* out_next_token_host);

/*
 * Wait for the context's stream and return the device-side status of every
 * step enqueued since the previous sdv_sync (then cleared): SDV_OK,
 * SDV_ERR_DEVICE_DATA or SDV_ERR_CUDA.  SDV_ERR_CUDA with the text "a bounded
 * device wait gave up" means that the sampling pass waited for its row copy
 * longer than its poll limit; it then wrote -1 to all three outputs of the
 * sequences concerned, and the context stays usable.
 */
sdv_status sdv_sync(sdv_ctx* ctx);

/* Text of the last error seen by this context ("" if none).  The pointer is
 * valid until the next call on the context. */
const char* sdv_last_error(const sdv_ctx* ctx);

/* Free the workspace and the context (NULL is a no-op).  Waits for the
 * context's stream first. */
void sdv_destroy(sdv_ctx* ctx);

/* Launch plan of a context, for tests and benchmarks: CTAs of the row pass,
 * 16-byte vectors per row chunk, chunks per row, CTAs per sequence (cluster
 * size) of the sampling pass.  Any pointer may be NULL. */
sdv_status sdv_plan(const sdv_ctx* ctx, int* rowpass_ctas, int64_t* chunk_vectors,
                    int* chunks_per_row, int* sample_cluster);

/*
 * Fault-path test hook (not part of the method; the pages have no
 * counterpart).  With SDV_HOOK_SAMPLE_NO_COPY set, the sampling pass of later
 * steps arms its barrier for the row copy but issues no copy and polls only a
 * few times, so that its bounded wait runs out with nothing in flight: the
 * step writes -1 to every sequence's three outputs and sdv_sync returns
 * SDV_ERR_CUDA ("a bounded device wait gave up").  This is how the timeout
 * path is tested without faulting or hanging a GPU.  hooks = 0 restores
 * normal steps; unknown bits give SDV_ERR_ARG.
 */
#define SDV_HOOK_SAMPLE_NO_COPY 1u
sdv_status sdv_set_test_hooks(sdv_ctx* ctx, unsigned hooks);

/* Replace the stream of a context (a cudaStream_t): later calls enqueue on
 * it.  The caller orders it after work already enqueued on the old stream.
 * To capture a step into a CUDA graph, set the capturing stream first. */
sdv_status sdv_set_stream(sdv_ctx* ctx, void* stream);

/*
 * Kernel timing.  While enabled, every step records CUDA events on the
 * context's stream before the row pass and after each of its three kernels
 * (row pass, select/scan, sample), for up to 65536 steps.  sdv_profile_read
 * waits for the recorded steps, writes the mean device time in milliseconds
 * of each kernel to ms_avg[0..2] and the number of steps to *steps, and
 * clears the record.  Enabling with enable = 0 stops recording.
 */
sdv_status sdv_profile_enable(sdv_ctx* ctx, int enable);
sdv_status sdv_profile_read(sdv_ctx* ctx, float* ms_avg, int* steps);

/*
 * Causal-consistency path search over drafter marginals ("DiffuSpec:
 * Unlocking Diffusion Language Models for Speculative Decoding", section 4.2;
 * the page's settings, section 5.3: beam 3, mmax 15, tau 0.8).  Produces
 * left-to-right drafts from one denoising pass's position-wise marginals:
 *   1. each row q[b][j] is pruned to the shortest list of its most likely
 *      tokens (probability of softmax(q / T) descending, ties to the lower id)
 *      whose mass reaches tau, at most mmax tokens; a token of probability
 *      zero (logit -inf) is never a candidate;
 *   2. the lattice ends at the first position whose most likely token is
 *      eos_id, which is kept alone as the last token (eos_id < 0: no cut);
 *   3. the paths a beam of width `beam` keeps over the lattice, scoring a
 *      path by the sum of its log-probabilities (drafter confidence; the
 *      page's causal fluency proxy is not specified there and is not used).
 *      The temperature and each position's normaliser are common to all of a
 *      sequence's paths, so paths rank by the sum of their raw logits (in
 *      fp64, exact for bf16 logits); equal sums go to the path whose
 *      candidate ranks come first lexicographically.  With a score that sums
 *      over positions the beam keeps the `beam` best paths of the lattice,
 *      and these are found best first rather than position by position.  The
 *      result is those paths, best first, each with its log-probability
 *      summed in fp32 in a fixed order.
 * The paths serve as the K = beam drafts of a verification step
 * (SDV_FLAG_SHARED_Q, with the same q).
 * Arguments: q_marginals device [B][gamma][V] bf16 or fp32 (16-byte aligned,
 * V * elt % 16 == 0); temperature, or device temperature_per_seq [B];
 * 0 <= tau <= 1; 1 <= mmax <= 16; 1 <= beam <= 16; gamma <= 1024;
 * eos_id < V.  Outputs (device, caller-owned): out_cand_ids / out_cand_logp /
 * out_cand_logit [B][gamma][mmax] (candidate ids, natural-log probabilities
 * and raw logits; -1 / -inf / -inf past the count), out_ncand [B][gamma] (0
 * past the lattice), out_paths [B][beam][gamma] (-1 past the lattice or past
 * npaths), out_path_logp [B][beam] (-inf past npaths), out_npaths [B],
 * out_lat_len [B] or NULL.  A row holding NaN, +inf or only -inf gets no
 * candidates and its sequence no path.  Stateless: allocates nothing, only
 * enqueues on `stream`.
 */
sdv_status sdv_cps(int B, int gamma, int V, sdv_dtype dtype, void* stream,
                   const void* q_marginals, float temperature,
                   const float* temperature_per_seq, float tau, int mmax, int beam,
                   int eos_id, int32_t* out_cand_ids, float* out_cand_logp,
                   float* out_cand_logit, int32_t* out_ncand, int32_t* out_paths,
                   float* out_path_logp, int32_t* out_npaths, int32_t* out_lat_len);

/*
 * sdv_cps that also writes every marginal row's softmax statistics, as the
 * pruning pass computes them, to out_row_stat (device float [B][gamma][4],
 * 16-byte aligned, or NULL): {m, s, c, 0} with c = 1.4426950408889634f / T
 * (fp32), m the row's largest logit and s = sum of 2^((logit - m) * c).  sdv_verify_qstat takes
 * them so that the verification of the paths does not stream the marginals a
 * second time.
 */
sdv_status sdv_cps_ex(int B, int gamma, int V, sdv_dtype dtype, void* stream,
                      const void* q_marginals, float temperature,
                      const float* temperature_per_seq, float tau, int mmax, int beam,
                      int eos_id, int32_t* out_cand_ids, float* out_cand_logp,
                      float* out_cand_logit, int32_t* out_ncand, int32_t* out_paths,
                      float* out_path_logp, int32_t* out_npaths, int32_t* out_lat_len,
                      float* out_row_stat);

/*
 * The two halves of sdv_cps, for callers that inspect or reuse the pruned
 * lattice.  sdv_cps_prune is step 1 for every row (no EOS cut): it reads
 * q_marginals / temperature(_per_seq) and writes out_cand_ids, out_cand_logp,
 * out_cand_logit and out_ncand exactly as sdv_cps documents them, before the
 * cut.  sdv_cps_beam is steps 2-3: it reads the lattice (as sdv_cps_prune
 * wrote it: each position's candidates in decreasing order of logit, at most
 * mmax of them; a count of 0 or less leaves the sequence without a path),
 * trims it in place at an EOS end (one candidate at the EOS
 * position, none past it) and writes the paths.  V is only used to check
 * eos_id.  Argument rules, ownership and errors as for sdv_cps; sdv_cps is
 * sdv_cps_prune followed by sdv_cps_beam on `stream`.
 */
sdv_status sdv_cps_prune(int B, int gamma, int V, sdv_dtype dtype, void* stream,
                         const void* q_marginals, float temperature,
                         const float* temperature_per_seq, float tau, int mmax,
                         int32_t* out_cand_ids, float* out_cand_logp, float* out_cand_logit,
                         int32_t* out_ncand);
sdv_status sdv_cps_beam(int B, int gamma, int V, int mmax, int beam, int eos_id, void* stream,
                        int32_t* cand_ids, float* cand_logp, float* cand_logit, int32_t* ncand,
                        int32_t* out_paths, float* out_path_logp, int32_t* out_npaths,
                        int32_t* out_lat_len);

/*
 * Adaptive draft length ("DiffuSpec: Unlocking Diffusion Language Models for
 * Speculative Decoding", section 4.3 and appendix C).  The page states the
 * controller's inputs and direction only; this is the plainest rule that
 * fits it.  Per sequence, a window of the last `window` steps records the
 * draft length k used, the EOS-aware generated length g (tokens up to and
 * including the first EOS of the chosen draft, e.g. sdv_cps's lattice length)
 * and the accepted length a (e.g. sdv_verify's out_len); g is clamped to
 * [0, k] and a to [0, g].  Acceptance keeps pace when the window's a sum to
 * its g; generation fills the drafts when its g sum to its k.  The next
 * length is k + up if both hold, k if only the first holds (generation
 * saturated: EOS before the end of the draft), k - down otherwise, clamped to
 * [kmin, kmax].
 * Limits: 1 <= window <= 64; 1 <= kmin <= kmax <= 2^20; 0 <= up, down <= 2^20.
 * sdv_adl_state_words(window): int32 words of one sequence's state (-1 for a
 * bad window).  The state [B][words] is caller-owned and starts zeroed; its
 * layout is private to the library.
 * sdv_adl_step_host: host pointers; k [B] holds the lengths just used and
 * receives the next ones.  SDV_ERR_ARG for bad limits or any k outside
 * [kmin, kmax] (then nothing is updated).
 * sdv_adl_step: the same on device pointers, enqueued on `stream` (one thread
 * per sequence); a sequence whose k lies outside [kmin, kmax] is left as it
 * is and sets bit 16 in *status (device int32, may be NULL), which the caller
 * clears.  Host-checked argument errors return SDV_ERR_ARG.
 */
#define SDV_ADL_MAX_WINDOW 64
#define SDV_STATUS_BAD_LENGTH 16
int sdv_adl_state_words(int window);
sdv_status sdv_adl_step_host(int B, int window, int kmin, int kmax, int up, int down,
                             const int32_t* gen_len, const int32_t* acc_len, int32_t* k,
                             int32_t* state);
sdv_status sdv_adl_step(int B, int window, int kmin, int kmax, int up, int down, void* stream,
                        const int32_t* gen_len, const int32_t* acc_len, int32_t* k,
                        int32_t* state, int32_t* status);

/*
 * sdv_verify_static -- the step of sdv_verify_ex for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry point:
 * it exists for deployment, not for the method.
 *
 * Who needs it: code that must not call cudaMalloc -- a process whose device
 * memory belongs entirely to another allocator (a serving engine's pool, which
 * would otherwise see memory vanish behind its back), a plug-in loaded into
 * such a process, code that runs where allocation is forbidden.  sdv_create
 * allocates a workspace; this call does not.  It takes no context and
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 *
 * Scratch: the row-pass partials, per-sequence tasks and status word live in
 * one static device array of SDV_STATIC_SCRATCH_BYTES (8 MiB), which every GPU
 * that loads libsdv holds until the process exits.  A shape whose scratch does
 * not fit is rejected with SDV_ERR_SCRATCH before anything is enqueued (as a
 * guide: partials take 8 bytes per row chunk, at least one chunk per row, so
 * B*K*(2*gamma+1) must stay below about one million rows).
 *
 * Set-up: the first call on a device, with that device current, looks up the
 * device address of the array (cudaGetSymbolAddress), the device's limits,
 * and raises the kernels' shared-memory limits; later calls on that device
 * do none of this.
 *
 * Arguments: as sdv_verify_ex, with the shape (B, K, gamma, V, dtype) and the
 * stream (a cudaStream_t, NULL = legacy default stream) passed on every call;
 * all tensors are caller-owned device memory (logits 16-byte aligned, the
 * int32 / float arrays 4-byte aligned).  Outputs are the same values
 * sdv_verify_ex writes.  Argument errors -- including a host pointer or a
 * misaligned one -- return SDV_ERR_ARG and nothing is enqueued.  The call only
 * enqueues; there is no sdv_sync for it: a sequence with bad data (draft id
 * out of range, non-finite row, bad per-sequence temperature), or whose
 * sampling pass gave up waiting for its row copy, gets -1 in all three
 * outputs.
 *
 * Sharing: every call uses the same array and leaves its contents behind (the
 * status word is cleared at the start of each call; the rest is written before
 * it is read).  Calls that overlap on the GPU -- on two streams or from two
 * host threads -- race on the array; the caller must serialise them.
 */
#define SDV_STATIC_SCRATCH_BYTES (8u << 20)
sdv_status sdv_verify_static(int B, int K, int gamma, int V, sdv_dtype dtype, void* stream,
                             const void* p_logits, const void* q_logits,
                             const int32_t* drafts, float temperature,
                             const float* temperature_per_seq, uint64_t seed,
                             int32_t* out_sel, int32_t* out_accept_len,
                             int32_t* out_next_token);

#ifdef __cplusplus
}
#endif

#endif /* SDV_H */
