/*
 * oracle.c -- plain, slow CPU oracle for batched top-k / top-p truncation and
 * sampling.  TEST INFRASTRUCTURE ONLY: the product path never links it.
 *
 * It writes out the definitions directly: a full sort of every row by
 * (logit descending, id ascending), a double-precision softmax, prefix cuts
 * for top-k and top-p, and a linear inverse-CDF scan in token-id order.  No
 * blocking, truncation heuristic, pivot search or fusion: those belong to the
 * fast path this oracle is used to check.
 *
 * Citations are to the pages' titles and sections:
 *   [KB]   AI Infra KB note M012 (token selection after the LM head)
 *   [BLOG] "Sampling system design: from logits to controllable generation"
 *          (mini vLLM series)
 *   [QR]   "Qrita: High-performance Top-k and Top-p using Pivot-based
 *          Truncation and Selection" (paper notes)
 *   [LEC]  CMU 11-868 lecture 9 notes, "Decoding: Sampling, Beam Search and
 *          Speculative Decoding"
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------- */
/* Input decoding.  Both conversions are exact; written from the IEEE 754  */
/* binary16 layout and the bfloat16 definition (upper half of a binary32). */
/* ---------------------------------------------------------------------- */

float orc_bf16_to_f32(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

float orc_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int mant = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)mant, -24); /* zero or subnormal: mant * 2^-24 */
  } else if (expo == 31) {
    v = mant ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + mant), expo - 25); /* (1 + mant/1024) * 2^(e-15) */
  }
  return (float)(sign ? -v : v);
}

static float load_logit(const void* row, int dtype, int i) {
  switch (dtype) {
    case ORC_F32: return ((const float*)row)[i];
    case ORC_BF16: return orc_bf16_to_f32(((const uint16_t*)row)[i]);
    default: return orc_f16_to_f32(((const uint16_t*)row)[i]);
  }
}

static int mask_allows(const uint32_t* mask_row, int i) {
  if (!mask_row) return 1;
  return (int)((mask_row[i >> 5] >> (i & 31)) & 1u);
}

/* ---------------------------------------------------------------------- */
/* Philox4x32-10, from the round function and key schedule published by    */
/* Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as     */
/* 1, 2, 3" (SC'11).  [KB] section 06 asks for explicit (seed, offset)     */
/* random state; the counter/key layout below is this build's choice.      */
/* ---------------------------------------------------------------------- */

#define ORC_PHILOX_M0 0xD2511F53u
#define ORC_PHILOX_M1 0xCD9E8D57u
#define ORC_PHILOX_W0 0x9E3779B9u
#define ORC_PHILOX_W1 0xBB67AE85u

void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
  uint32_t k[2] = {key_in[0], key_in[1]};
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k[0] += ORC_PHILOX_W0;
      k[1] += ORC_PHILOX_W1;
    }
    uint64_t p0 = (uint64_t)ORC_PHILOX_M0 * (uint64_t)c[0];
    uint64_t p1 = (uint64_t)ORC_PHILOX_M1 * (uint64_t)c[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c[1] ^ k[0];
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c[3] ^ k[1];
    uint32_t n3 = lo0;
    c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
  }
  out[0] = c[0]; out[1] = c[1]; out[2] = c[2]; out[3] = c[3];
}

double orc_uniform(uint64_t seed, uint64_t offset) {
  uint32_t ctr[4] = {(uint32_t)offset, (uint32_t)(offset >> 32), 0u, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

/* ---------------------------------------------------------------------- */
/* Core selection                                                          */
/* ---------------------------------------------------------------------- */

typedef struct {
  double x;
  int id;
} orc_item;

/* (x descending, id ascending): a total order, so any sort of the ids by
 * this key equals a stable sort by x alone.  Ties keep the earliest ids
 * ([QR] key design 3). */
static int rank_cmp(const void* a, const void* b) {
  const orc_item* p = (const orc_item*)a;
  const orc_item* q = (const orc_item*)b;
  if (p->x > q->x) return -1;
  if (p->x < q->x) return 1;
  return (p->id < q->id) ? -1 : (p->id > q->id);
}

static int id_cmp(const void* a, const void* b) {
  int p = *(const int*)a, q = *(const int*)b;
  return (p > q) - (p < q);
}

int orc_select_core(int n, const double* x, const double* z, const unsigned char* legal,
                    int32_t top_k, double top_p, double u,
                    unsigned char* kept, double* prob, int32_t* token,
                    int32_t* n_topk, int32_t* n_kept, int32_t* flags) {
  if (kept) memset(kept, 0, (size_t)n);
  if (prob) for (int i = 0; i < n; ++i) prob[i] = 0.0;
  if (token) *token = -1;
  if (n_topk) *n_topk = 0;
  if (n_kept) *n_kept = 0;
  if (flags) *flags = 0;

  /* Legal set L: [KB] section 05 sets illegal logits to -inf before the
   * draw; the front end folds that into legal[]. */
  int nl = 0;
  for (int i = 0; i < n; ++i) nl += legal[i] ? 1 : 0;
  if (nl == 0) return ORC_EMPTY; /* [KB] section 03: an empty set is an error */

  orc_item* order = (orc_item*)malloc(sizeof(orc_item) * (size_t)nl);
  double* w = (double*)malloc(sizeof(double) * (size_t)n);
  int* sp = (int*)malloc(sizeof(int) * (size_t)nl);
  int j = 0;
  for (int i = 0; i < n; ++i)
    if (legal[i]) { order[j].x = x[i]; order[j].id = i; ++j; }

  /* Rank L by (x desc, id asc). */
  qsort(order, (size_t)nl, sizeof(orc_item), rank_cmp);

  /* Softmax over L in double ([LEC] 3.3: temperature divides the logits,
   * then normalise). */
  double m = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (legal[i] && z[i] > m) m = z[i];
  double total = 0.0;
  for (int i = 0; i < n; ++i) {
    w[i] = legal[i] ? exp(z[i] - m) : 0.0;
    total += w[i];
  }

  /* Top-k: keep the first K of the rank order and renormalise ([KB] 02,
   * [LEC] 3.3).  K = min(top_k, |L|). */
  int K = top_k < nl ? top_k : nl;
  double mass_k = 0.0;
  for (int r = 0; r < K; ++r) mass_k += w[order[r].id] / total;

  /* Top-p: the shortest prefix of the top-k order whose renormalised mass
   * reaches p (">=": the worked answer to exercise 7 of [LEC] keeps the prefix
   * whose mass equals p).  If rounding leaves every prefix short, keep all K. */
  int nstar = K;
  double cum_at = 0.0, cum_before = 0.0;
  if (top_p < 1.0) {
    double cum = 0.0;
    for (int r = 0; r < K; ++r) {
      double q = (w[order[r].id] / total) / mass_k;
      double prev = cum;
      cum += q;
      if (cum >= top_p) { nstar = r + 1; cum_at = cum; cum_before = prev; break; }
    }
    if (flags) {
      if (fabs(cum_at - top_p) <= 1e-5 || (nstar > 1 && fabs(top_p - cum_before) <= 1e-5))
        *flags |= ORC_FLAG_TOPP_BOUNDARY;
    }
  }

  /* Final renormalisation over S_p. */
  double mass_p = 0.0;
  for (int r = 0; r < nstar; ++r) mass_p += (w[order[r].id] / total) / mass_k;

  for (int r = 0; r < nstar; ++r) {
    int id = order[r].id;
    if (kept) kept[id] = 1;
    if (prob) prob[id] = ((w[id] / total) / mass_k) / mass_p;
    sp[r] = id;
  }

  /* Inverse-CDF draw in token-id order ([KB] section 02 figure note): the
   * token is the first id whose cumulative probability exceeds u; if
   * rounding leaves none, the last kept id. */
  qsort(sp, (size_t)nstar, sizeof(int), id_cmp);
  double cum = 0.0, dmin = INFINITY;
  int tok = sp[nstar - 1];
  int found = 0;
  for (int r = 0; r < nstar; ++r) {
    int id = sp[r];
    cum += ((w[id] / total) / mass_k) / mass_p;
    double d = fabs(cum - u);
    if (d < dmin) dmin = d;
    if (!found && cum > u) { tok = id; found = 1; }
  }
  if (flags && dmin <= 1e-6) *flags |= ORC_FLAG_CDF_BOUNDARY;

  if (token) *token = tok;
  if (n_topk) *n_topk = K;
  if (n_kept) *n_kept = nstar;
  free(order);
  free(w);
  free(sp);
  return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Row front end: decode, validate, legal set, greedy path, fp32 scaling.  */
/* ---------------------------------------------------------------------- */

static int row_params_valid(float t, int32_t k, float p) {
  /* [BLOG] parameter validation: reject negative temperature, top_p > 1 and
   * non-positive top_k (the build's reading: top_k < 1 is invalid). */
  if (isnan(t) || t < 0.0f) return 0;
  if (k < 1) return 0;
  if (isnan(p) || !(p > 0.0f) || p > 1.0f) return 0;
  return 1;
}

static int oracle_row(const void* row, int dtype, int V, const uint32_t* mask_row,
                      float t, int32_t k, float p, uint64_t seed, uint64_t offset, int mode,
                      int32_t* token, int32_t* kept_count, uint32_t* kept_mask_row,
                      double* probs_row, int32_t* flags, double* u_out) {
  int W = (V + 31) / 32;
  *token = -1;
  *kept_count = 0;
  *flags = 0;
  if (kept_mask_row) memset(kept_mask_row, 0, sizeof(uint32_t) * (size_t)W);
  if (probs_row) for (int i = 0; i < V; ++i) probs_row[i] = 0.0;
  double u = orc_uniform(seed, offset);
  if (u_out) *u_out = u;

  if (mode == 1) {
    t = 0.0f; k = 1; p = 1.0f; /* argmax entry point: every row greedy */
  }
  if (!row_params_valid(t, k, p)) return ORC_INVALID;
  if (k > V) k = V;

  float* xs = (float*)malloc(sizeof(float) * (size_t)V);
  unsigned char* legal = (unsigned char*)malloc((size_t)V);
  int nonfinite = 0, nl = 0;
  for (int i = 0; i < V; ++i) {
    xs[i] = load_logit(row, dtype, i);
    legal[i] = (unsigned char)(mask_allows(mask_row, i) && !(isinf(xs[i]) && xs[i] < 0));
    if (legal[i]) {
      ++nl;
      if (isnan(xs[i]) || isinf(xs[i])) nonfinite = 1; /* [KB] 07: explicit error */
    }
  }
  int status = ORC_OK;
  if (nonfinite) status = ORC_NONFINITE;
  else if (nl == 0) status = ORC_EMPTY;
  else if (t == 0.0f) {
    /* Greedy is a separate argmax path ([KB] 02, [BLOG]); ties go to the
     * earlier vocabulary id ([LEC] answer 1). */
    int best = -1;
    for (int i = 0; i < V; ++i)
      if (legal[i] && (best < 0 || xs[i] > xs[best])) best = i;
    *token = best;
    *kept_count = 1;
    if (kept_mask_row) kept_mask_row[best >> 5] |= 1u << (best & 31);
    if (probs_row) probs_row[best] = 1.0;
  } else {
    double* xd = (double*)malloc(sizeof(double) * (size_t)V);
    double* zd = (double*)malloc(sizeof(double) * (size_t)V);
    unsigned char* kept = (unsigned char*)malloc((size_t)V);
    for (int i = 0; i < V; ++i) {
      xd[i] = legal[i] ? (double)xs[i] : 0.0;
      /* z = fl32(x / T): correctly rounded binary32 division. */
      float zf = legal[i] ? xs[i] / t : 0.0f;
      zd[i] = (double)zf;
    }
    int32_t tok, ntk, nkp, fl;
    status = orc_select_core(V, xd, zd, legal, k, (double)p, u, kept, probs_row, &tok, &ntk,
                             &nkp, &fl);
    if (status == ORC_OK) {
      *token = tok;
      *kept_count = nkp;
      *flags = fl;
      if (kept_mask_row)
        for (int i = 0; i < V; ++i)
          if (kept[i]) kept_mask_row[i >> 5] |= 1u << (i & 31);
    }
    free(xd);
    free(zd);
    free(kept);
  }
  if (status != ORC_OK) {
    *token = -1;
    *kept_count = 0;
    if (kept_mask_row) memset(kept_mask_row, 0, sizeof(uint32_t) * (size_t)W);
    if (probs_row) for (int i = 0; i < V; ++i) probs_row[i] = 0.0;
  }
  free(xs);
  free(legal);
  return status;
}

int orc_batch(const void* logits, int dtype, int B, int V, int64_t ld,
              const uint32_t* bitmask,
              const float* temperature, const int32_t* top_k, const float* top_p,
              const uint64_t* seed, const uint64_t* offset, int mode,
              int32_t* status, int32_t* token, int32_t* kept_count,
              uint32_t* kept_mask, double* probs, int32_t* flags, double* u_out,
              int n_threads) {
  int W = (V + 31) / 32;
  size_t es = (dtype == ORC_F32) ? 4 : 2;
  if (n_threads < 1) n_threads = 1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
  for (int r = 0; r < B; ++r) {
    const char* row = (const char*)logits + (size_t)r * (size_t)ld * es;
    const uint32_t* mrow = bitmask ? bitmask + (size_t)r * (size_t)W : NULL;
    status[r] = oracle_row(row, dtype, V, mrow, mode == 1 ? 0.0f : temperature[r],
                           mode == 1 ? 1 : top_k[r], mode == 1 ? 1.0f : top_p[r],
                           seed ? seed[r] : 0, offset ? offset[r] : 0, mode,
                           &token[r], &kept_count[r],
                           kept_mask ? kept_mask + (size_t)r * (size_t)W : NULL,
                           probs ? probs + (size_t)r * (size_t)V : NULL,
                           &flags[r], u_out ? &u_out[r] : NULL);
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Speculative-decoding verification, exact rule (lecture notes "Decoding: */
/* Sampling, Beam Search and Speculative Decoding", section 5.2, after     */
/* Leviathan et al. 2023 and Chen et al. 2023): accept the draft token x   */
/* with probability min(1, p(x)/q(x)); at the first rejection draw from    */
/* norm(max(0, p - q)) and stop; after G acceptances draw a bonus token    */
/* from the target's distribution at position G.                           */
/* ---------------------------------------------------------------------- */

static int prob_ok(float v) { return !isnan(v) && v >= 0.0f && v <= 1.0f; }

/* Compensated (Neumaier) running sum: the result is the exact sum rounded
   once, up to a relative error of about 2^-106 for the sums taken here. */
typedef struct {
  double s, c;
} nsum;
static void nsum_add(nsum* a, double x) {
  double t = a->s + x;
  if (fabs(a->s) >= fabs(x)) a->c += (a->s - t) + x;
  else a->c += (x - t) + a->s;
  a->s = t;
}
static double nsum_val(const nsum* a) { return a->s + a->c; }

/* The checks and acceptance tests both variants share: returns the position
   j of the draw (G when every draft is accepted) or -1 for ORC_INVALID. */
static int spec_accept(int G, int V, const float* p, const float* q, int64_t ld, const int32_t* d,
                       const double* u_acc) {
  for (int i = 0; i < G; ++i) {
    if (d[i] < 0 || d[i] >= V) return -1;
    if (!prob_ok(p[(size_t)i * ld + d[i]]) || !prob_ok(q[(size_t)i * ld + d[i]])) return -1;
  }
  /* acceptance tests in order; u * q < p is exact in double (24 x 24 bits) */
  int j = G;
  for (int i = 0; i < G; ++i) {
    const double a = (double)p[(size_t)i * ld + d[i]];
    const double b = (double)q[(size_t)i * ld + d[i]];
    if (u_acc[i] * b < a) continue;
    j = i;
    break;
  }
  return j;
}
/* The rows the draw at position j reads: p_j, and q_j after a rejection
   (NULL after G acceptances); 0 when one of their values is not a
   probability. */
static int spec_rows(int j, int G, int V, const float* p, const float* q, int64_t ld,
                     const float** pr, const float** qr) {
  *pr = p + (size_t)j * ld;
  *qr = (j < G) ? q + (size_t)j * ld : NULL;
  for (int x = 0; x < V; ++x)
    if (!prob_ok((*pr)[x]) || (*qr && !prob_ok((*qr)[x]))) return 0;
  return 1;
}
/* Residual weight of id x over the reals: max(0, p(x) - q(x)), or p(x). */
static double spec_res(const float* pr, const float* qr, int x) {
  const double r = qr ? (double)pr[x] - (double)qr[x] : (double)pr[x];
  return r > 0.0 ? r : 0.0;
}

int orc_spec_verify_u(int G, int V, const float* p, const float* q, int64_t ld,
                      const int32_t* d, const double* u_acc, const double* u_res,
                      int32_t* out_tokens, int32_t* n_acc, double* margin) {
  for (int i = 0; i <= G; ++i) out_tokens[i] = -1;
  *n_acc = 0;
  *margin = INFINITY;
  const int j = spec_accept(G, V, p, q, ld, d, u_acc);
  if (j < 0) return ORC_INVALID;
  /* the drawn position: residual max(0, p_j - q_j) after a rejection, the
     target row p_G after G acceptances; the weights are real numbers (the
     difference of the two binary32 values, in double), their total and the
     prefixes compensated sums */
  const float *pr, *qr;
  if (!spec_rows(j, G, V, p, q, ld, &pr, &qr)) return ORC_INVALID;
  nsum S = {0.0, 0.0};
  for (int x = 0; x < V; ++x) nsum_add(&S, spec_res(pr, qr, x));
  const double St = nsum_val(&S);
  if (!(St > 0.0)) return ORC_EMPTY;
  /* inverse CDF in id order: the first id whose cumulative weight exceeds
     u * S; the margin is the distance of u * S to the nearest prefix that
     separates two candidates, over S */
  const double t = u_res[j] * St;
  int tok = -1, last = -1;
  double best = INFINITY;
  nsum cum = {0.0, 0.0};
  for (int x = 0; x < V; ++x) {
    const double r = spec_res(pr, qr, x);
    if (!(r > 0.0)) continue;
    last = x;
    nsum_add(&cum, r);
    const double c = nsum_val(&cum);
    if (tok < 0 && c > t) tok = x;
    if (c < St) {
      const double dist = fabs(c - t) / St;
      if (dist < best) best = dist;
    }
  }
  if (tok < 0) tok = last; /* u * S rounds up to S: the last candidate */
  for (int i = 0; i < j; ++i) out_tokens[i] = d[i];
  out_tokens[j] = tok;
  *n_acc = j;
  *margin = best;
  return ORC_OK;
}

int orc_spec_verify_fx_u(int G, int V, const float* p, const float* q, int64_t ld,
                         const int32_t* d, const double* u_acc, const double* u_res,
                         int32_t* out_tokens, int32_t* n_acc) {
  for (int i = 0; i <= G; ++i) out_tokens[i] = -1;
  *n_acc = 0;
  const int j = spec_accept(G, V, p, q, ld, d, u_acc);
  if (j < 0) return ORC_INVALID;
  /* the residual as the binary32 difference, each weight the integer
     floor(w * 2^42); sums and prefixes of these are exact */
  const float *pr, *qr;
  if (!spec_rows(j, G, V, p, q, ld, &pr, &qr)) return ORC_INVALID;
  uint64_t S = 0;
  for (int x = 0; x < V; ++x) {
    float r = qr ? pr[x] - qr[x] : pr[x];
    if (!(r > 0.0f)) r = 0.0f;
    S += (uint64_t)floor(ldexp((double)r, 42));
  }
  if (S == 0) return ORC_EMPTY;
  /* with integer prefixes P, P > u * S iff P > floor(k * S / 2^24), u = k 2^-24 */
  const uint64_t k = (uint64_t)ldexp(u_res[j], 24);
  const uint64_t T = (uint64_t)(((unsigned __int128)S * k) >> 24);
  int tok = -1;
  uint64_t cum = 0;
  for (int x = 0; x < V && tok < 0; ++x) {
    float r = qr ? pr[x] - qr[x] : pr[x];
    if (!(r > 0.0f)) continue;
    cum += (uint64_t)floor(ldexp((double)r, 42));
    if (cum > T) tok = x;
  }
  for (int i = 0; i < j; ++i) out_tokens[i] = d[i];
  out_tokens[j] = tok;
  *n_acc = j;
  return ORC_OK;
}

static void spec_uniforms(int G, uint64_t seed, uint64_t offset, double* ua, double* ur) {
  for (int i = 0; i <= G; ++i) {
    uint64_t c = offset + (uint64_t)i;
    uint32_t ctr[4] = {(uint32_t)c, (uint32_t)(c >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    if (i < G) ua[i] = (double)(out[0] >> 8) * (1.0 / 16777216.0);
    ur[i] = (double)(out[1] >> 8) * (1.0 / 16777216.0);
  }
}

int orc_spec_verify(int B, int G, int V, const float* p, const float* q, int64_t ld,
                    const int32_t* d, const uint64_t* seed, const uint64_t* offset,
                    int32_t* out_tokens, int32_t* n_acc, int32_t* status, double* margin,
                    int fixed, int n_threads) {
  if (n_threads < 1) n_threads = 1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
  for (int s = 0; s < B; ++s) {
    double ua[64], ur[65];
    spec_uniforms(G, seed[s], offset[s], ua, ur);
    int32_t* ot = out_tokens + (size_t)s * (size_t)(G + 1);
    const float* ps = p + (size_t)s * (size_t)(G + 1) * (size_t)ld;
    const float* qs = G ? q + (size_t)s * (size_t)G * (size_t)ld : NULL;
    const int32_t* ds = d + (size_t)s * (size_t)G;
    if (fixed) {
      status[s] = orc_spec_verify_fx_u(G, V, ps, qs, ld, ds, ua, ur, ot, &n_acc[s]);
      margin[s] = INFINITY;
    } else {
      status[s] = orc_spec_verify_u(G, V, ps, qs, ld, ds, ua, ur, ot, &n_acc[s], &margin[s]);
    }
    if (status[s] != ORC_OK) {
      for (int i = 0; i <= G; ++i) ot[i] = -1;
      n_acc[s] = 0;
      margin[s] = INFINITY;
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Repetition penalty ("Sampling system design" post, section on the      */
/* repetition penalty: a logits processor that reads the sequence's       */
/* history and lowers the logits of tokens already seen).  The pages leave */
/* the formula open; this build takes the CTRL rule (Keskar et al. 2019):  */
/* x / theta for a positive logit, x * theta otherwise, once per distinct  */
/* token of the history, in binary32, stored back in the logits' format   */
/* with round-to-nearest-even.                                             */
/* ---------------------------------------------------------------------- */

uint16_t orc_f32_to_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, sizeof b);
  if (isnan(f)) return (uint16_t)(((b >> 16) & 0x8000u) | 0x7fc0u);
  /* round to nearest, ties to even, on the 16 bits kept */
  uint32_t r = b + 0x7fffu + ((b >> 16) & 1u);
  return (uint16_t)(r >> 16);
}

uint16_t orc_f32_to_f16(float f) {
  uint16_t sign = signbit(f) ? 0x8000u : 0u;
  double a = fabs((double)f);
  if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u); /* rounds past 65504 */
  if (a < ldexp(1.0, -14)) {
    /* subnormal (or zero): units of 2^-24, ties to even; 1024 units is the
       smallest normal, which the same code word encodes */
    double q = rint(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)q);
  }
  int e;
  frexp(a, &e); /* a = m * 2^e, m in [0.5, 1): the leading bit weighs 2^(e-1) */
  e -= 1;
  double q = rint(ldexp(a, 10 - e)); /* significand with 10 fraction bits */
  if (q >= 2048.0) {
    q = 1024.0;
    e += 1;
  }
  if (e + 15 >= 31) return (uint16_t)(sign | 0x7c00u);
  return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(q - 1024.0));
}

int orc_repetition_penalty(void* logits, int dtype, int B, int V, int64_t ld,
                           const int32_t* history, int H, int64_t hld, const float* penalty,
                           int32_t* status) {
  size_t es = (dtype == ORC_F32) ? 4 : 2;
  unsigned char* seen = (unsigned char*)malloc((size_t)(V > 0 ? V : 1));
  if (!seen) return -1;
  for (int r = 0; r < B; ++r) {
    float th = penalty[r];
    if (!(th > 0.0f) || isinf(th)) {
      status[r] = ORC_INVALID;
      continue;
    }
    status[r] = ORC_OK;
    memset(seen, 0, (size_t)V);
    char* row = (char*)logits + (size_t)r * (size_t)ld * es;
    for (int i = 0; i < H; ++i) {
      int t = history[(size_t)r * (size_t)hld + i];
      if (t < 0 || t >= V || seen[t]) continue; /* padding, or already penalised */
      seen[t] = 1;
      float x = load_logit(row, dtype, t);
      float y = (x > 0.0f) ? x / th : x * th;
      if (dtype == ORC_F32) ((float*)row)[t] = y;
      else if (dtype == ORC_BF16) ((uint16_t*)row)[t] = orc_f32_to_bf16(y);
      else ((uint16_t*)row)[t] = orc_f32_to_f16(y);
    }
  }
  free(seen);
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Gumbel-max sampling over a kept set (lecture notes "Decoding: Sampling, */
/* Beam Search and Speculative Decoding", section 3.2: argmax of the       */
/* logits plus Gumbel noise is a draw from their softmax): a sort-free     */
/* second sampler family, used for comparison with the inverse-CDF draw.   */
/* ---------------------------------------------------------------------- */

/* The uniform of element i of a row: word (i mod 4) of the Philox4x32-10
   block at key (lo32 seed, hi32 seed), counter (lo32 offset, hi32 offset,
   i / 4, 0x47554D42), mapped to the open interval (0, 1) as
   ((w >> 8) + 1/2) * 2^-24. */
double orc_gumbel_uniform(uint64_t seed, uint64_t offset, int i) {
  uint32_t ctr[4] = {(uint32_t)offset, (uint32_t)(offset >> 32), (uint32_t)(i >> 2),
                     0x47554D42u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return ((double)(out[i & 3] >> 8) + 0.5) * (1.0 / 16777216.0);
}

int orc_gumbel_sample(const void* logits, int dtype, int B, int V, int64_t ld,
                      const uint32_t* kept_mask, const float* temperature,
                      const uint64_t* seed, const uint64_t* offset, int32_t* token,
                      int32_t* status, double* margin, int n_threads) {
  int W = (V + 31) / 32;
  size_t es = (dtype == ORC_F32) ? 4 : 2;
  if (n_threads < 1) n_threads = 1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
  for (int r = 0; r < B; ++r) {
    const char* row = (const char*)logits + (size_t)r * (size_t)ld * es;
    const uint32_t* mrow = kept_mask ? kept_mask + (size_t)r * (size_t)W : NULL;
    float t = temperature[r];
    token[r] = -1;
    margin[r] = INFINITY;
    if (!(t >= 0.0f)) {
      status[r] = ORC_INVALID;
      continue;
    }
    int best = -1, nonfinite = 0;
    double bv = -INFINITY, second = -INFINITY;
    for (int i = 0; i < V; ++i) {
      if (!mask_allows(mrow, i)) continue;
      float x = load_logit(row, dtype, i);
      if (isinf(x) && x < 0) continue;
      if (isnan(x) || isinf(x)) {
        nonfinite = 1;
        break;
      }
      double v;
      if (t == 0.0f) {
        v = (double)x; /* greedy: no noise, the first maximum wins */
      } else {
        double u = orc_gumbel_uniform(seed[r], offset[r], i);
        v = (double)(x / t) - log(-log(u));
      }
      if (v > bv) {
        second = bv;
        bv = v;
        best = i;
      } else if (v > second) {
        second = v;
      }
    }
    if (nonfinite) {
      status[r] = ORC_NONFINITE;
      continue;
    }
    if (best < 0) {
      status[r] = ORC_EMPTY;
      continue;
    }
    status[r] = ORC_OK;
    token[r] = best;
    margin[r] = bv - second;
  }
  return 0;
}
