/*
 * smp.h -- C ABI of libsmp: batched exact top-k / top-p truncation and
 * sampling over a [B, V] logits matrix, hand-written for sm_103a (GB300).
 *
 * The contract (AI Infra KB note M012, section 02 "which candidates do top-k
 * and top-p keep"; CMU 11-868 lecture 9 notes, section 3.3), per row:
 *   1. temperature T: T == 0 takes a separate greedy argmax path and never
 *      divides; T > 0 scales z = fl32(x / T)  (KB note section 02; "Sampling
 *      system design" post, section on temperature);
 *   2. legal-token mask: illegal tokens and -inf logits are excluded
 *      (KB note section 05);
 *   3. top-k: keep the K = min(top_k, |legal|) highest logits and
 *      renormalise; ties at the boundary keep the earliest token ids
 *      (Qrita paper notes, key design 3);
 *   4. top-p: keep the shortest prefix, in descending probability, whose
 *      renormalised mass reaches top_p (">=", the lecture's exercise 7
 *      answer), again keeping the earliest ids among equal values;
 *   5. renormalise and draw by inverse CDF in token-id order with
 *      u = Philox4x32-10(seed, offset) (KB note section 02 figure note and
 *      section 06 on explicit random state).
 * An empty candidate set is an error; no substitute token is ever produced
 * (KB note section 03, section 07).
 *
 * Entry points: smp_topk_topp_mask (kept sets), smp_sample (draws),
 * smp_sample_logprob and smp_top_logprobs (draws with their log-
 * probabilities), smp_argmax (greedy), smp_sample_noalloc (no handle, no
 * allocation), smp_repetition_penalty (an in-place logits processor to run
 * before sampling), smp_gumbel_sample (a sort-free Gumbel-max draw over a
 * kept set, for comparison) and smp_spec_verify (speculative-decoding
 * verification against the kept sets' probabilities); smp_set_kernel
 * chooses between the two sampler kernels and smp_set_wait_limit bounds the
 * device-side waits.
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees, copies to the host or synchronises inside a
 *     call.  Work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) on the handle's device.
 *   - logits: row-major [B][ld] of `dtype`, ld >= V (elements).  Rows whose
 *     start is 16-byte aligned are staged with bulk TMA copies; others with
 *     plain loads (slower, same results).
 *   - bitmask: nullable, uint32 [B][W], W = ceil(V/32), row stride W words.
 *     Bit (j % 32) of word (j / 32) allows token j (1 = allowed).  Bits at or
 *     past V are ignored.  NULL = every token allowed.
 *   - kept_mask: same packed layout as bitmask, [B][W], 1 = token kept.
 *   - The return value is the call status: SMP_OK, SMP_ERR_INVALID_PARAM for
 *     bad arguments (NULL required pointers, B < 0, V < 1, ld < V, unknown
 *     dtype), SMP_ERR_CAPACITY when B or V exceed the smp_create limits or V
 *     exceeds what one thread-block cluster can hold, SMP_ERR_CUDA when the
 *     launch fails.  Per-row outcomes go to row_status.
 *   - A row whose status is not SMP_OK gets token -1, kept_count 0, an
 *     all-zero kept_mask row and all-zero probabilities.
 *   - RNG: every row reads exactly one Philox4x32-10 block, key =
 *     (lo32 seed[r], hi32 seed[r]), counter = (lo32 offset[r], hi32
 *     offset[r], 0, 0); u = (word0 >> 8) * 2^-24.  The library keeps no RNG
 *     state: the caller advances offsets by the amount consumed (one block
 *     per row per call), e.g. offset[r] = base + r and base += B per step.
 *     Replaying a captured graph with frozen offsets repeats the draws.
 */
#ifndef SMP_H
#define SMP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct smp_ctx* smp_handle;
typedef void* smp_stream; /* a cudaStream_t */

typedef enum { SMP_F32 = 0, SMP_BF16 = 1, SMP_F16 = 2 } smp_dtype;

enum {
  SMP_OK = 0,
  SMP_ERR_EMPTY = 1,         /* row: no legal finite candidate            */
  SMP_ERR_NONFINITE = 2,     /* row: NaN or +inf in a legal slot          */
  SMP_ERR_INVALID_PARAM = 3, /* row: bad temperature/top_k/top_p; call: bad argument */
  SMP_ERR_TIMEOUT = 4,       /* row: a bounded device wait expired        */
  SMP_ERR_CUDA = 5,          /* call: CUDA error at launch or setup       */
  SMP_ERR_CAPACITY = 6       /* call: B or V beyond the handle's limits   */
};

/* Per-row sampling parameters, all DEVICE arrays of length B ("Sampling
 * system design" post: every sequence carries its own SamplingParams).
 *   temperature: >= 0 (0 = greedy); NaN or < 0 -> row SMP_ERR_INVALID_PARAM
 *   top_k      : >= 1; values above V mean V; < 1 -> SMP_ERR_INVALID_PARAM
 *   top_p      : in (0, 1]; 1 disables top-p; else SMP_ERR_INVALID_PARAM
 *   seed, offset: Philox key and counter (see above). */
typedef struct {
  const float* temperature;
  const int32_t* top_k;
  const float* top_p;
  const uint64_t* seed;
  const uint64_t* offset;
} smp_row_params;

/* Create a handle bound to CUDA device `device` for calls with B <=
 * max_batch and V <= max_vocab.  Queries the device, configures the kernels
 * (shared memory, CTAs per SM) and builds the host-side sigma-truncation
 * table (Qrita paper notes, key design 1 and "training strategy": delta =
 * Phi^-1(1 - k/V) from a precomputed table).  Allocates the handle's one
 * device workspace (1,968,896 bytes: the job board on which rows with large
 * top-p sets share their passes over the row across CTAs); calls allocate
 * nothing.
 * Calls on one handle must not run concurrently (issue them on one stream).
 * Returns SMP_OK, SMP_ERR_INVALID_PARAM or SMP_ERR_CUDA. */
int smp_create(smp_handle* h, int device, int max_batch, int max_vocab);

/* Release a handle and its workspace (NULL is accepted). */
int smp_destroy(smp_handle h);

/* Kept set of every row: after temperature, mask, top-k and top-p (steps
 * 1-4 above), write kept_mask [B][W] and kept_count [B].  Greedy rows keep
 * {argmax} with probability 1.  probs_out (nullable) receives [B][V] fp32
 * final probabilities (0 outside the kept set) -- a test aid that costs 4*V
 * bytes of writes per row.  No random number is drawn. */
int smp_topk_topp_mask(smp_handle h, const void* logits, smp_dtype dtype, int B, int V,
                       int64_t ld, const uint32_t* bitmask, const smp_row_params* params,
                       uint32_t* kept_mask, int32_t* kept_count, int32_t* row_status,
                       float* probs_out, smp_stream stream);

/* Full contract (steps 1-5): tokens [B] and row_status [B]; kept_mask and
 * kept_count (both nullable) as in smp_topk_topp_mask. */
int smp_sample(smp_handle h, const void* logits, smp_dtype dtype, int B, int V, int64_t ld,
               const uint32_t* bitmask, const smp_row_params* params, int32_t* tokens,
               int32_t* row_status, uint32_t* kept_mask, int32_t* kept_count,
               smp_stream stream);

/* smp_sample plus the log-probability of each drawn token ("Sampling system
 * design" post, section on logprobs: a sampler that returns logprobs returns
 * the selected token's log-probability and states the distribution it is
 * taken under).  The distribution here is the PROCESSED one the token was
 * drawn from: after temperature, mask, top-k and top-p, renormalised over
 * the kept set -- the final probability smp_topk_topp_mask writes to
 * probs_out for that token.  logprobs: DEVICE float [B], required.
 * Greedy rows (kept set {argmax}) get 0; rows whose status is not SMP_OK
 * get NaN.  Other arguments, outputs and statuses are those of smp_sample;
 * the tokens drawn are the same as smp_sample's for the same inputs. */
int smp_sample_logprob(smp_handle h, const void* logits, smp_dtype dtype, int B, int V,
                       int64_t ld, const uint32_t* bitmask, const smp_row_params* params,
                       int32_t* tokens, float* logprobs, int32_t* row_status,
                       uint32_t* kept_mask, int32_t* kept_count, smp_stream stream);

/* Top logprobs: the n most likely tokens of each row's kept set with their
 * log-probabilities ("Sampling system design" post, section on logprobs),
 * under the same processed distribution as smp_sample_logprob.  Inputs are
 * that call's outputs for the same logits and parameters: kept_mask
 * [B][ceil(V/32)], tokens [B] and logprobs [B] (all DEVICE).  Per row the
 * kept tokens are ranked by logit (descending, smallest id first among equal
 * logits); top_ids [B][n] receives the first n ids, top_logprobs [B][n]
 * their log-probabilities, computed as
 *     logprobs[r] + (fl32(x_j / T) - fl32(x_tok / T))
 * (two kept tokens' log-probabilities differ by their scaled logits' difference;
 * greedy rows: 0 for the argmax).  Slots past the kept set's size get id -1
 * and -inf; rows whose token is -1 (an error row) get -1 and NaN.
 * 1 <= n <= 32 (larger n: SMP_ERR_CAPACITY).  Call status as for
 * smp_gumbel_sample.  Work: one pass over each row's kept mask and its kept
 * logits (a cluster of up to 8 CTAs per row). */
int smp_top_logprobs(smp_handle h, const void* logits, smp_dtype dtype, int B, int V, int64_t ld,
                     const uint32_t* kept_mask, const float* temperature, const int32_t* tokens,
                     const float* logprobs, int n, int32_t* top_ids, float* top_logprobs,
                     smp_stream stream);

/* Greedy path alone (KB note section 02; lecture 9 answer 1): the legal
 * finite token with the largest logit, the smallest id on ties.  Rows with
 * no legal finite logit get SMP_ERR_EMPTY, rows with NaN / +inf in a legal
 * slot SMP_ERR_NONFINITE. */
int smp_argmax(smp_handle h, const void* logits, smp_dtype dtype, int B, int V, int64_t ld,
               const uint32_t* bitmask, int32_t* tokens, int32_t* row_status,
               smp_stream stream);

/* smp_sample without a handle and without any device allocation.  The pages
 * this library follows have no counterpart: it exists for callers that may
 * not call cudaMalloc.  One example is a plugin inside a serving runtime that
 * reserves nearly all device memory for its KV cache at start-up and hands
 * out memory only through its own pool.  Another is a stateless hook with
 * nowhere to keep a handle between calls.
 * Arguments, outputs and statuses are those of smp_sample.  The call runs on
 * the CURRENT CUDA device.  The caller passes every input and output.
 * Scratch: the job board that smp_create would allocate is instead a static
 * device array of 1,968,896 bytes.  Every device that loads the library
 * holds it until the process exits.
 * Set-up: the first call on each device does the set-up, with that device
 * current.  It configures the kernels, looks up the array's device address
 * and clears the array on `stream`.  Make that first call before any stream
 * capture.  Every call looks the address up again (a host-side query); when
 * it has changed, as after cudaDeviceReset, the set-up runs again.
 * Limit: V may be at most 128 staging chunks, that is 786,432 tokens for fp32
 * and 1,572,864 for bf16/fp16.  Larger V returns SMP_ERR_CAPACITY and
 * launches nothing.  B has no limit of its own.
 * Sharing: all calls on a device share the one array.  Each launch leaves
 * the board cleared when it ends.  Calls that overlap on the GPU race on it,
 * so issue them in order, e.g. on one stream.  Calls through a handle use
 * that handle's own workspace and do not race with these. */
int smp_sample_noalloc(const void* logits, smp_dtype dtype, int B, int V, int64_t ld,
                       const uint32_t* bitmask, const smp_row_params* params, int32_t* tokens,
                       int32_t* row_status, uint32_t* kept_mask, int32_t* kept_count,
                       smp_stream stream);

/* Speculative-decoding verification with the exact accept / reject rule
 * (lecture notes "Decoding: Sampling, Beam Search and Speculative Decoding",
 * section 5.2, after Leviathan et al. 2023 and Chen et al. 2023), for B
 * sequences that each carry G draft tokens.  The output tokens are then
 * distributed exactly as the target's distributions, whatever the draft.
 * Per sequence s, for i = 0, 1, ...: with d = draft_tokens[s][i], accept d
 * iff u_acc(i) * q_i(d) < p_i(d) (probability min(1, p/q)); at the first
 * rejection draw one token from norm(max(0, p_i - q_i)) and stop; if all G
 * drafts are accepted, draw one more token from p_G.  A draw is the inverse
 * CDF in token-id order: the first id whose cumulative weight exceeds u
 * times the total, with weights held as exact integers floor(w * 2^42) so
 * that the result does not depend on summation order.
 *   target_probs: fp32 [B][G+1][ld]: p_i, the target's probabilities at
 *                 draft positions 0..G-1 and at the bonus position G (for
 *                 example probs_out of smp_topk_topp_mask on the target's
 *                 logits).  Base address 16-byte aligned.
 *   draft_probs : fp32 [B][G][ld]: q_i, the distributions the drafts were
 *                 drawn from; 16-byte aligned; NULL allowed when G == 0.
 *   draft_tokens: int32 [B][G]; NULL allowed when G == 0.
 *   B >= 0; 0 <= G <= 31; 1 <= V <= 1,048,576; ld >= V, a multiple of 4.
 *   seed, offset: uint64 [B].  Position i (0..G) uses the Philox4x32-10
 *                 block at counter offset[s] + i (key as for smp_sample):
 *                 u_acc(i) = (word0 >> 8) * 2^-24, and the draw at position
 *                 i uses u_res(i) = (word1 >> 8) * 2^-24.  A call consumes
 *                 G + 1 blocks per sequence: advance offsets by G + 1.
 * Outputs (DEVICE, caller-owned): out_tokens int32 [B][G+1] (the accepted
 * drafts, then the drawn token, then -1), n_accepted int32 [B] (0..G),
 * row_status int32 [B]:
 *   SMP_ERR_INVALID_PARAM -- a draft token outside [0, V), or a probability
 *     the rule reads (p_i(d_i) and q_i(d_i) for every i < G, and every entry
 *     of the drawn row or rows) that is NaN or outside [0, 1];
 *   SMP_ERR_EMPTY -- the drawn weights sum to zero (for example p_i <= q_i
 *     everywhere after a rejection).
 * Such a sequence gets out_tokens all -1 and n_accepted 0.
 * Call status: SMP_ERR_INVALID_PARAM for NULL required pointers, unaligned
 * probabilities, ld not a multiple of 4 or ld < V; SMP_ERR_CAPACITY for G >
 * 31, V beyond 1,048,576 or B / V beyond the handle's limits; SMP_ERR_CUDA
 * when the launch fails.  Work: one launch, a cluster of up to 8 CTAs per
 * sequence; it reads two probabilities per draft token and the one drawn row
 * (p_j and q_j after a rejection) once.  No workspace is used. */
int smp_spec_verify(smp_handle h, const float* target_probs, const float* draft_probs,
                    const int32_t* draft_tokens, int B, int G, int V, int64_t ld,
                    const uint64_t* seed, const uint64_t* offset, int32_t* out_tokens,
                    int32_t* n_accepted, int32_t* row_status, smp_stream stream);

/* Repetition penalty, applied IN PLACE to the logits before sampling
 * ("Sampling system design" post, section on the repetition penalty: a
 * logits processor that reads each sequence's history tokens and lowers the
 * logits of tokens already seen).  The post leaves the formula open; this is
 * the CTRL rule (Keskar et al. 2019): for row r, theta = penalty[r], and
 * every DISTINCT token t among history[r][0..H-1],
 *     x_t <- x_t / theta  if x_t > 0,   x_t <- x_t * theta  otherwise,
 * computed in binary32 with correct rounding and stored back in the logits'
 * format with round-to-nearest-even (-inf stays -inf; theta = 1 changes
 * nothing).  Tokens that appear several times are penalised once.
 *   logits    : DEVICE [B][ld] of dtype, modified in place.
 *   history   : DEVICE int32 [B][history_ld], H entries per row; entries
 *               outside [0, V) are padding.  NULL allowed when H == 0.
 *   penalty   : DEVICE float [B]; a value that is not finite and > 0 leaves
 *               the row unchanged with row_status SMP_ERR_INVALID_PARAM.
 *   row_status: DEVICE int32 [B], required (SMP_OK or the above).
 * Call status: SMP_ERR_INVALID_PARAM for NULL required pointers, B < 0,
 * V < 1, ld < V, H < 0, history_ld < H or an unknown dtype;
 * SMP_ERR_CAPACITY for B or V beyond the handle's limits or V above
 * 1,572,864; SMP_ERR_CUDA when the launch fails.  Work: one launch, one CTA
 * per row; it reads the history and reads and writes only the logits of the
 * history's tokens (never the whole row).  Issue it on the sampler's stream
 * before smp_sample. */
int smp_repetition_penalty(smp_handle h, void* logits, smp_dtype dtype, int B, int V, int64_t ld,
                           const int32_t* history, int H, int64_t history_ld,
                           const float* penalty, int32_t* row_status, smp_stream stream);

/* Gumbel-max sampling over a kept set: a sort-free second sampler family
 * for distribution and timing comparisons (lecture notes "Decoding:
 * Sampling, Beam Search and Speculative Decoding", section 3.2: the argmax of
 * z_i + g_i, with g_i = -log(-log(u_i)) independent Gumbel noise, is a draw
 * from softmax(z)).  Per row: candidates are the tokens whose kept_mask bit
 * is set (kept_mask NULL: every token) and whose logit is not -inf; z_i =
 * fl32(x_i / T); u_i = ((w >> 8) + 1/2) * 2^-24 with w word (i mod 4) of the
 * Philox4x32-10 block at key (lo32 seed[r], hi32 seed[r]) and counter
 * (lo32 offset[r], hi32 offset[r], i / 4, 0x47554D42); the token is the
 * argmax of z_i + g_i (fp32; smallest id on ties); T == 0 takes the argmax
 * of x.  With the kept_mask that smp_topk_topp_mask writes, the draw follows
 * the same top-k / top-p distribution as smp_sample's (different draws: it
 * uses its own random numbers and no prefix sum).
 *   kept_mask : DEVICE uint32 [B][ceil(V/32)], nullable (layout of bitmask).
 *   temperature, seed, offset: DEVICE [B]; tokens, row_status: DEVICE [B].
 * Row status: SMP_ERR_INVALID_PARAM (T NaN or < 0), SMP_ERR_NONFINITE (NaN
 * or +inf among the candidates), SMP_ERR_EMPTY (no candidate); token -1.
 * Call status: SMP_ERR_INVALID_PARAM for NULL required pointers, B < 0,
 * V < 1, ld < V or an unknown dtype; SMP_ERR_CAPACITY beyond the handle's
 * limits; SMP_ERR_CUDA when the launch fails.  Work: one pass over each row
 * (a cluster of up to 8 CTAs per row); no workspace. */
int smp_gumbel_sample(smp_handle h, const void* logits, smp_dtype dtype, int B, int V, int64_t ld,
                      const uint32_t* kept_mask, const float* temperature, const uint64_t* seed,
                      const uint64_t* offset, int32_t* tokens, int32_t* row_status,
                      smp_stream stream);

/* Optional per-row diagnostics for subsequent calls on this handle: when
 * row_info is not NULL, each call writes int32 [B][4] to it (DEVICE memory
 * owned by the caller, at least max_batch*4 entries): {path, band size,
 * selection rounds, refinement rounds}.  path: 0 error, 1 greedy, 2 all
 * legal kept, 3 sigma-truncation hit, 4 full-row refinement.  NULL turns it
 * off.  Not thread-safe against concurrent calls on the same handle. */
int smp_set_row_info(smp_handle h, int32_t* row_info);

/* Which sampler kernel later calls on this handle launch (the results are the
 * same; only the time differs).  SMP_KERNEL_BOARD (the default): one CTA per
 * row, two resident per SM, with a device job board through which CTAs that
 * are done take chunks of the slow rows.  SMP_KERNEL_SPLIT (bf16 / fp16
 * logits only; other dtypes keep the board kernel): each row split over a
 * thread-block cluster of up to 8 CTAs that stream their slices once through
 * a shared-memory ring and combine over distributed shared memory; fastest
 * when top-k bounds every row, slower on rows whose top-p set runs to tens of
 * thousands of tokens.  Returns SMP_ERR_INVALID_PARAM for another value.  Not
 * thread-safe against concurrent calls on the same handle. */
enum { SMP_KERNEL_BOARD = 0, SMP_KERNEL_SPLIT = 1 };
int smp_set_kernel(smp_handle h, int kernel);

/* Bound on each device-side wait of later calls on this handle, in SM clock
 * cycles (cycles <= 0 restores the default, 4e9: about two seconds).  The
 * waits are those for a staged copy to land and for other CTAs' chunks of a
 * shared row.  A row whose wait runs out returns SMP_ERR_TIMEOUT with token
 * -1 and count 0 (its kept mask and probabilities are unspecified); no token
 * is ever substituted.  A CTA whose wait ran out stages nothing more in that
 * launch (its later rows also return SMP_ERR_TIMEOUT) and, before it exits,
 * waits for its copies still in flight with the default bound.  The next call
 * starts clean.  Meant for tests and diagnostics: a very small bound makes
 * rows time out on purpose.  Not thread-safe against concurrent calls on the
 * same handle. */
int smp_set_wait_limit(smp_handle h, long long cycles);

/* Launch plan of a call with B rows of V tokens of `dtype` on this handle's
 * device, for the kernel smp_set_kernel chose: CTAs per row (the
 * thread-block cluster; 1 for the board kernel), slice length (tokens per
 * CTA; the board kernel's staging chunk), dynamic shared memory per CTA
 * (bytes) and candidate-list capacity per CTA.  Any output pointer may be
 * NULL.  Returns SMP_ERR_CAPACITY when V cannot be held. */
int smp_plan(smp_handle h, smp_dtype dtype, int B, int V, int* cluster, int* slice,
             int* smem_bytes, int* capacity);

/* Static description of a status code. */
const char* smp_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* SMP_H */
