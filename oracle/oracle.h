/*
 * oracle.h -- plain CPU oracle for batched top-k / top-p truncation and sampling.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only tests/, the package's smoke check and the CPU-baseline
 * leg of bench.py use it.  It shares no code, header or constant with the CUDA
 * library; it carries its own status codes, its own fp16/bf16 decoders and its
 * own Philox4x32-10.
 *
 * What it computes (the contract of "AI Infra KB M012", sections 02-03, and of
 * the CMU 11-868 lecture 9 notes, section 3.3), per row:
 *   temperature (0 = separate greedy argmax path) -> legal-token mask ->
 *   top-k with renormalisation -> top-p as the shortest prefix of descending
 *   probability whose mass reaches p -> renormalise -> inverse-CDF draw in
 *   token-id order.
 * Ranking is by (logit descending, token id ascending): ties keep the earliest
 * ids (Qrita paper notes, key design 3).  Everything after the fp32 scaling
 * z = fl32(x / temperature) is done in double.
 */
#ifndef TSS_ORACLE_H
#define TSS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_EMPTY = 1, ORC_NONFINITE = 2, ORC_INVALID = 3 };
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2 };

/* flags[] bits */
enum { ORC_FLAG_TOPP_BOUNDARY = 1, ORC_FLAG_CDF_BOUNDARY = 2 };

float orc_bf16_to_f32(uint16_t h);
float orc_f16_to_f32(uint16_t h);

/* Philox4x32-10 block function (Salmon, Moraes, Dror, Shaw, SC'11). */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
/* u in [0,1) for a row: key = (lo32 seed, hi32 seed), counter = (lo32 off,
 * hi32 off, 0, 0); u = (word0 >> 8) * 2^-24. */
double orc_uniform(uint64_t seed, uint64_t offset);

/*
 * Core selection on one row given in double precision.
 *   n       : vocabulary size
 *   x       : value used for ranking (the fp32 logit, as a double)
 *   z       : value used for the softmax (fl32(x / T), as a double)
 *   legal   : 1 = candidate (mask allows it and x != -inf), 0 = excluded
 *   top_k   : already validated, >= 1 (clamped to n inside)
 *   top_p   : already validated, in (0, 1]
 *   u       : uniform draw in [0, 1)
 * Outputs (all nullable): kept[n] (1 = in the final kept set), prob[n]
 * (final renormalised probability, 0 outside the kept set), token, counts,
 * boundary flags.  Returns ORC_OK or ORC_EMPTY.
 */
int orc_select_core(int n, const double* x, const double* z, const unsigned char* legal,
                    int32_t top_k, double top_p, double u,
                    unsigned char* kept, double* prob, int32_t* token,
                    int32_t* n_topk, int32_t* n_kept, int32_t* flags);

/*
 * Whole batch.  logits is [B][ld] of dtype; bitmask is [B][ceil(V/32)] or
 * NULL (bit j%32 of word j/32, 1 = allowed).  Per-row parameter arrays have
 * length B.  mode: 0 = sample, 1 = argmax only (every row greedy).
 * Outputs: status, token (-1 on error rows), kept_count, kept_mask
 * [B][ceil(V/32)] (nullable), probs [B][V] (nullable), flags, u (nullable).
 * Rows are independent; n_threads > 1 runs them in parallel.
 */
int orc_batch(const void* logits, int dtype, int B, int V, int64_t ld,
              const uint32_t* bitmask,
              const float* temperature, const int32_t* top_k, const float* top_p,
              const uint64_t* seed, const uint64_t* offset, int mode,
              int32_t* status, int32_t* token, int32_t* kept_count,
              uint32_t* kept_mask, double* probs, int32_t* flags, double* u_out,
              int n_threads);

/*
 * Speculative-decoding verification with the exact accept / reject rule
 * (lecture notes "Decoding: Sampling, Beam Search and Speculative Decoding",
 * section 5.2, after Leviathan et al. 2023 and Chen et al. 2023).  One
 * sequence with G draft tokens d[0..G-1]; q_i is the draft distribution at
 * draft position i, p_i the target distribution at position i (i = 0..G).
 * For i = 0, 1, ...: accept d_i iff u_acc[i] * q_i(d_i) < p_i(d_i) (that is,
 * with probability min(1, p/q)); at the first rejection draw the token from
 * norm(max(0, p_i - q_i)) with u_res[i] and stop; if all G are accepted,
 * draw one more token from p_G with u_res[G].  A draw is the inverse CDF in
 * token-id order: the first id whose cumulative weight exceeds u * S, over
 * the reals: the residual is p - q of the given binary32 values, taken in
 * double, S and the prefixes are compensated sums, and u = k * 2^-24.
 *   p       : [G+1] rows of V floats, row stride ld
 *   q       : [G] rows of V floats, row stride ld (NULL when G == 0)
 *   u_acc   : [G] uniforms in [0,1); u_res: [G+1] uniforms in [0,1)
 * Outputs: out_tokens[G+1] (accepted drafts, then the drawn token, then -1),
 * n_acc, and margin = distance of u_res to the nearest switch point of the
 * draw, in units of u (infinity when the draw has a single candidate).
 * Status: ORC_INVALID when a draft token is outside [0, V) or a probability
 * the rule reads (p_i(d_i), q_i(d_i) for every i < G; the whole drawn row or
 * rows) is NaN or outside [0, 1]; ORC_EMPTY when the drawn weights sum to 0.
 * Every output of a sequence with a status other than ORC_OK is -1 / 0.
 */
int orc_spec_verify_u(int G, int V, const float* p, const float* q, int64_t ld,
                      const int32_t* d, const double* u_acc, const double* u_res,
                      int32_t* out_tokens, int32_t* n_acc, double* margin);

/*
 * A second, labelled variant (not the definition): the same rule with the
 * draw taken in the precision the CUDA library states for its integer
 * decision -- the residual as the binary32 difference p - q, each weight the
 * integer floor(w * 2^42), the target floor(k * S / 2^24).  It differs from
 * orc_spec_verify_u only where u * S lies within the weights' rounding of a
 * switch point.  No margin output.
 */
int orc_spec_verify_fx_u(int G, int V, const float* p, const float* q, int64_t ld,
                         const int32_t* d, const double* u_acc, const double* u_res,
                         int32_t* out_tokens, int32_t* n_acc);

/*
 * Batch of B sequences with Philox4x32-10 uniforms: for draft position i
 * (i = 0..G) the block at key (lo32 seed[s], hi32 seed[s]) and counter
 * offset[s] + i gives u_acc[i] = (word0 >> 8) * 2^-24 and
 * u_res[i] = (word1 >> 8) * 2^-24.  p: [B][G+1][ld], q: [B][G][ld],
 * d: [B][G], out_tokens: [B][G+1].  fixed = 0: orc_spec_verify_u (the
 * definition); fixed = 1: orc_spec_verify_fx_u (margin set to infinity).
 */
int orc_spec_verify(int B, int G, int V, const float* p, const float* q, int64_t ld,
                    const int32_t* d, const uint64_t* seed, const uint64_t* offset,
                    int32_t* out_tokens, int32_t* n_acc, int32_t* status, double* margin,
                    int fixed, int n_threads);

/* float -> bfloat16 / binary16 with round-to-nearest-even (NaN stays NaN,
 * overflow gives infinity). */
uint16_t orc_f32_to_bf16(float f);
uint16_t orc_f32_to_f16(float f);

/*
 * Repetition penalty, in place ("Sampling system design" post, section on the
 * repetition penalty; the formula, which the post leaves open, is the CTRL
 * rule of Keskar et al. 2019).  For row r and every DISTINCT token t of
 * history[r][0..H-1] (row stride hld; entries outside [0, V) are padding):
 * x = x / penalty[r] if x > 0, else x * penalty[r], in binary32, stored back
 * in the logits' format with round-to-nearest-even.  A penalty that is not
 * finite and > 0 leaves the row unchanged and sets status[r] = ORC_INVALID.
 */
int orc_repetition_penalty(void* logits, int dtype, int B, int V, int64_t ld,
                           const int32_t* history, int H, int64_t hld, const float* penalty,
                           int32_t* status);

/*
 * Gumbel-max sampling (lecture notes, section 3.2: the argmax of
 * z_i + g_i with g_i = -log(-log(u_i)) is a draw from softmax(z)), a
 * sort-free second sampler for comparison.  Per row: candidates are the
 * tokens whose kept_mask bit is set (kept_mask [B][ceil(V/32)], NULL = all)
 * and whose logit is not -inf; z_i = fl32(x_i / T); u_i from
 * orc_gumbel_uniform; T == 0 takes the argmax of x (first maximum).  The
 * perturbed values are evaluated in double; margin[r] = best - second best.
 * Status: ORC_INVALID (T NaN or < 0), ORC_NONFINITE (NaN / +inf among the
 * candidates), ORC_EMPTY (no candidate); token -1 on those rows.
 */
double orc_gumbel_uniform(uint64_t seed, uint64_t offset, int i);
int orc_gumbel_sample(const void* logits, int dtype, int B, int V, int64_t ld,
                      const uint32_t* kept_mask, const float* temperature,
                      const uint64_t* seed, const uint64_t* offset, int32_t* token,
                      int32_t* status, double* margin, int n_threads);

#ifdef __cplusplus
}
#endif
#endif
