// smp_kernel.cuh -- per-row driver and the kernel entry of the sampler.
//
// Per row (contract of the AI Infra KB note M012, sections 02-03):
//   temperature (0 = greedy argmax) -> legal mask -> top-k (earliest ids win
//   ties) -> top-p (shortest prefix, value descending then id ascending,
//   whose mass reaches p) -> renormalise -> inverse-CDF draw in token-id
//   order with a Philox4x32-10 uniform.
//
// Rows are routed by their parameters:
//   argmax    temperature 0, top_k = 1, or the argmax entry point;
//   keep-all  top_k >= V and top_p = 1: every legal token is kept;
//   list      top_k <= KLIST: sigma-truncated candidate list, resolved on chip;
//   general   everything else, and lists that fail validation: the mass
//             stream with a list attempt, then the weight-histogram bracket,
//             then exact radix descent.
#pragma once

#include "smp_general.cuh"

namespace smp {

// ---------------------------------------------------------------------------
// Outputs
// ---------------------------------------------------------------------------
template <int DT>
__device__ void zero_outputs(Ctx<DT>& X) {
  const KArgs& a = *X.a;
  if (a.kept_mask) {
    uint32_t* m = a.kept_mask + (size_t)X.row * X.W;
    for (int w = threadIdx.x; w < X.W; w += NT) m[w] = 0u;
  }
  if (a.probs && a.mode == MODE_MASK) {
    float* p = a.probs + (size_t)X.row * X.V;
    for (int i = threadIdx.x; i < X.V; i += NT) p[i] = 0.f;
  }
}

// Status, token, count and diagnostics of the row (one thread writes).
template <int DT>
__device__ void put_row(Ctx<DT>& X, int status, int token, int count, int path, int nlist) {
  const KArgs& a = *X.a;
  a.status[X.row] = status;
  if (a.tokens) a.tokens[X.row] = (status == ST_OK) ? token : -1;
  if (a.logprob && status != ST_OK) a.logprob[X.row] = __int_as_float(0x7fffffff);
  if (a.kept_count) a.kept_count[X.row] = (status == ST_OK) ? count : 0;
  if (a.row_info) {
    int* ri = a.row_info + (size_t)X.row * 4;
    ri[0] = (status == ST_OK) ? path : PATH_ERROR;
    ri[1] = nlist;
  }
}
template <int DT>
__device__ void write_row(Ctx<DT>& X, int status, int token, int count, int path) {
  if (threadIdx.x == 0) put_row(X, status, token, count, path, X.sh->n);
}

// Error row; `where` (a source line) goes to the row diagnostics.
template <int DT>
__device__ __noinline__ void error_row(Ctx<DT>& Xr, int status, int where = 0) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  __syncthreads();
  if (X.sh->primed) {
    // the row ends before its first pass: take the issued chunks off the ring
    ring_wait(X, 0);
    if (X.nch > 1) ring_wait(X, 1);
    __syncthreads();
    if (threadIdx.x == 0) X.sh->primed = 0;
  }
  zero_outputs(X);
  write_row(X, status, -1, 0, PATH_ERROR);
  if (threadIdx.x == 0 && X.a->row_info) X.a->row_info[(size_t)X.row * 4 + 2] = where;
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Kept set resolved inside the list (the list holds every element of S_p):
// top-k (K > 0: the K-th entry; K = 0: every entry is in S_k), top-p (target
// Pq > 0 in fixed point, else p times the S_k mass), count, draw and outputs.
// Outputs were zeroed beforehand.  Runs on a group of G threads; returns false
// (nothing written) when the list does not hold the top-p boundary.
// ---------------------------------------------------------------------------
template <int G, int DT>
__device__ bool list_solve(Ctx<DT>& X, int n, int K, float p, uint64_t Pq, float m_z, double u,
                           int path) {
  const KArgs& a = *X.a;
  const uint32_t* lk = X.lk;
  const int* li = X.li;
  uint32_t vK = 0u;
  int idK = -1;
  if (K > 0 && !list_resolve_k<G>(X, n, K, vK, idK)) return false;
  list_weights<G, DT, false>(X, n, m_z, 0.f, vK, idK);
  Res R;
  R.vK = R.vP = vK;
  R.idK = R.idP = idK;
  uint64_t mp = 0;
  int nk = 0;
  if (p < 1.f) {
    if (!list_resolve_p<G, DT, false>(X, n, Pq, p, m_z, 0.f, R, mp, &nk)) return false;
  } else {
    const float* wq = list_w(X);
    uint64_t s = 0;
    for (int i = gtid<G>(); i < n; i += G) s += to_fx(wq[i]);
    mp = gsum_q<G>(s, X.sh->rq[1]);
    nk = (K > 0) ? K : n;
  }
  int tok = -1;
  if (a.mode == MODE_SAMPLE)
    tok = (G == NT && nk <= NT) ? list_draw_small(X, n, R.vP, R.idP, mp, u)
                                : list_draw<G>(X, n, R.vP, R.idP, mp, u);
  const float* wq = list_w(X);
  const double inv = 1099511627776.0 / (double)mp;
  for (int i = gtid<G>(); i < n; i += G) {
    const int id = li[i];
    if (!in_set(lk[i], id, R.vP, R.idP)) continue;
    if (a.kept_mask) red_or_global(a.kept_mask + (size_t)X.row * X.W + (id >> 5), 1u << (id & 31));
    if (a.probs && a.mode == MODE_MASK)
      a.probs[(size_t)X.row * X.V + id] = (float)((double)wq[i] * inv);
    if (a.logprob && id == tok) a.logprob[X.row] = (float)fmin(log((double)wq[i] * inv), 0.0);
  }
  if (gtid<G>() == 0) put_row(X, ST_OK, tok, nk, path, n);
  return true;
}

// list_solve on one warp (short lists) or the whole CTA; every thread returns
// the same verdict.
template <int DT>
__device__ __noinline__ bool list_finish(Ctx<DT>& X, int n, int K, float p, uint64_t Pq, float m_z,
                                         double u, int path, uint32_t kbase, uint32_t kmax) {
  // every list entry has kbase <= key <= kmax (the stream's threshold and its
  // largest append)
  if (threadIdx.x == 0) {
    X.sh->bu[4] = kbase;
    X.sh->bu[5] = max(kmax, kbase);
  }
  zero_outputs(X);
  __syncthreads();
  const bool ok = list_solve<NT>(X, n, K, p, Pq, m_z, u, path);
  __syncthreads();
  return ok;
}

// Log of the drawn token's final probability for a kept set decided over the
// whole row: the contract's weight expf(fl32(x / T) - zr) over the kept mass
// mtot relative to the same reference, as probs_pass writes probabilities.
template <int DT>
__device__ void put_logprob(Ctx<DT>& X, int tok, float zr, double mtot) {
  if (threadIdx.x != 0 || !X.a->logprob || tok < 0) return;
  uint32_t b;
  if constexpr (DT == DT_F32) b = reinterpret_cast<const uint32_t*>(X.src)[tok];
  else b = reinterpret_cast<const uint16_t*>(X.src)[tok];
  const float x = bits_value<DT>(b);
  // (a probability a rounding above 1 is taken as 1)
  X.a->logprob[X.row] = (float)fmin(log((double)expf(__fdiv_rn(x, X.temp) - zr) / mtot), 0.0);
}

// ---------------------------------------------------------------------------
// Kept set decided by a boundary over the whole row: kept pass (mask, count,
// masses), draw and probabilities.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ void finish_by_pass(Ctx<DT>& X, uint32_t vF, int idF, float ref, double u,
                                            int path) {
  const KArgs& a = *X.a;
  const float nm = -ref * X.c2;
  const int nk = kept_pass(X, vF, idF, nm);
  double mtot = 0.0;
  int tok = -1;
  if (a.mode == MODE_SAMPLE || (a.probs && a.mode == MODE_MASK))
    tok = sample_tail(X, u, vF, idF, nm, nullptr, mtot);
  if (a.probs && a.mode == MODE_MASK) probs_pass(X, vF, idF, __fdiv_rn(ref, X.temp), mtot);
  if (X.sh->timeout) return error_row(X, ST_TIMEOUT, __LINE__);
  put_logprob(X, tok, __fdiv_rn(ref, X.temp), mtot);
  write_row(X, ST_OK, tok, nk, path);
  __syncthreads();
}

// Kept set = {above the bracket} (written by band_kept_pass) + the band list
// entries in {key > vF} + {key == vF, id <= idF}: their mask bits and
// per-cell masses are merged, then the draw and probabilities follow.
template <int DT>
__device__ __noinline__ void finish_band(Ctx<DT>& X, int n, const BandOut& bo, uint32_t vF,
                                         int idF, float m, double u, int path) {
  const KArgs& a = *X.a;
  const float nm = -m * X.c2;
  uint64_t* extra = cell_extra(X);
  const float* wq = list_w(X);
  const uint32_t* lk = X.lk;
  const int* li = X.li;
  // per-cell fixed-point masses of the kept band entries, summed as two
  // 21-bit pieces in 32-bit counters (no carries, no returned values: every
  // weight is at most 1, so a piece is below 2^21 and a cell's sum below 2^32)
  uint32_t* p0 = reinterpret_cast<uint32_t*>(list_scratch(X) + 2048);
  uint32_t* p1 = p0 + MAXCH * NWARP;
  __syncthreads();
  for (int f = threadIdx.x; f < X.nch * NWARP; f += NT) {
    p0[f] = 0u;
    p1[f] = 0u;
  }
  __syncthreads();
  // each thread takes a contiguous run of entries (list order follows the
  // row's chunks, so a run mostly stays in one cell) and adds a cell's sum
  // when the run leaves it: few shared atomics, and no lanes of a warp
  // queueing on one address
  int nk = 0;
  const int per = (n + NT - 1) / NT;
  const int i0 = threadIdx.x * per, i1 = min(n, i0 + per);
  int fc = -1;
  uint32_t a0 = 0u, a1 = 0u;
  for (int i = i0; i < i1; ++i) {
    const int id = li[i];
    if (!in_set(lk[i], id, vF, idF)) continue;
    ++nk;
    if (a.kept_mask) red_or_global(a.kept_mask + (size_t)X.row * X.W + (id >> 5), 1u << (id & 31));
    const uint64_t q = to_fx(wq[i]);
    const int f = cell_of<DT>(id);
    if (f != fc) {
      if (fc >= 0) {
        atomicAdd(&p0[fc], a0);
        atomicAdd(&p1[fc], a1);
      }
      fc = f;
      a0 = a1 = 0u;
    }
    a0 += (uint32_t)(q & 0x1fffffull);
    a1 += (uint32_t)(q >> 21);
  }
  if (fc >= 0) {
    atomicAdd(&p0[fc], a0);
    atomicAdd(&p1[fc], a1);
  }
  __syncthreads();
  for (int f = threadIdx.x; f < X.nch * NWARP; f += NT)
    extra[f] = (uint64_t)p0[f] + ((uint64_t)p1[f] << 21);
  nk = bsum_i(nk, X.sh->ri[1]) + bo.above_n;
  double mtot = 0.0;
  int tok = -1;
  if (a.mode == MODE_SAMPLE || (a.probs && a.mode == MODE_MASK))
    tok = sample_tail(X, u, vF, idF, nm, extra, mtot);
  if (a.probs && a.mode == MODE_MASK) probs_pass(X, vF, idF, __fdiv_rn(m, X.temp), mtot);
  if (X.sh->timeout) return error_row(X, ST_TIMEOUT, __LINE__);
  put_logprob(X, tok, __fdiv_rn(m, X.temp), mtot);
  write_row(X, ST_OK, tok, nk, path);
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Band jobs.  The owner of a bracketed row publishes its band pass, runs its
// chunks from the front, waits (bounded) for the chunks helpers claimed from
// the back, and gathers the list, the cell masses and the count above the
// bracket.
// ---------------------------------------------------------------------------
// The owner's side of band job j: its band pass from the front, a bounded wait
// for the helpers' chunks, then their list entries (after the owner's), cells
// and count.  Returns the list length (-1 if a bounded wait expired).
template <int DT>
__device__ __noinline__ int run_job(Ctx<DT>& X, int j, int b_lo, int b_hi, float nref, float nm,
                                    BandOut& bo) {
  Board* bd = X.a->board;
  int own_above = 0;
  const int first = band_owner_pass(X, j, b_lo, b_hi, nref, nm, own_above);
  if (!wait_job(X, j, X.nch - first)) return -1;
  volatile JobHdr* H = &bd->hdr[j];
  const int n_own = X.sh->n;
  const int n_h = H->list_n;
  bo.above_n = own_above + H->above_n;
  bo.above_q = 0;
  const int ln = n_own + n_h;
  if (ln <= CAP) {
    // helpers' entries: loads batched ahead of the stores
    constexpr int PB = 8;
#pragma unroll 1
    for (int i0 = 0; i0 < n_h; i0 += NT * PB) {
      uint32_t k[PB];
      int id[PB];
#pragma unroll
      for (int q = 0; q < PB; ++q) {
        const int i = i0 + q * NT + threadIdx.x;
        if (i < n_h) {
          k[q] = __ldcg(&bd->lk[j][i]);
          id[q] = __ldcg(&bd->li[j][i]);
        }
      }
#pragma unroll
      for (int q = 0; q < PB; ++q) {
        const int i = i0 + q * NT + threadIdx.x;
        if (i < n_h) {
          X.lk[n_own + i] = k[q];
          X.li[n_own + i] = id[q];
        }
      }
    }
  }
  for (int f = first * NWARP + threadIdx.x; f < X.nch * NWARP; f += NT)
    X.sh->cmass[f / NWARP][f % NWARP] = __ldcg(&bd->cmass[j][f]);
  __syncthreads();
  if (threadIdx.x == 0) X.sh->n = ln;
  __syncthreads();
  return ln;
}

// Band pass over a weight-histogram bracket, shared on the job board when a
// slot is free, else run by this CTA alone.  Returns the list length.
template <int DT>
__device__ int band_any(Ctx<DT>& X, int b_lo, int b_hi, float nref, float nm, BandOut& bo) {
  float xa, xb;
  band_thresholds<DT>(X.c2, nref, b_lo, b_hi, xa, xb);
  const int j = publish_job(X, JOB_BAND, X.nch, b_lo, b_hi, nref, nm, xa, xb);
  int ln;
  if (j >= 0) {
    ln = run_job(X, j, b_lo, b_hi, nref, nm, bo);
  } else {
    bo = band_kept_pass(X, b_lo, b_hi, nref, nm);
    ln = X.sh->n;
  }
  if (ln >= 0) bo.above_q = cells_fixed_mass(X);
  bo.xa = xa;
  bo.xb = xb;
  return ln;
}

// After its own rows, a CTA runs published tasks until every CTA has finished
// its rows (so no job can still appear); the last CTA out resets the board.
template <int DT>
__device__ __noinline__ void help_and_exit(Ctx<DT>& X) {
  Board* bd = X.a->board;
  if (!bd) return;
  if (threadIdx.x == 0) atomicAdd(&bd->ctas_done, 1);
  const long long t0 = clock64();
  const long long lim = X.a->wait_limit;
#pragma unroll 1
  while (true) {
    if (threadIdx.x < 32) {
      // warp 0 looks at every job slot at once (lane q: slot q), then tries
      // the open ones from a slot that depends on the CTA, so that helpers
      // spread over the jobs
      static_assert(MAXJOBS <= 32, "one lane per job slot");
      volatile Board* vb = bd;
      const int lane = threadIdx.x;
      const unsigned long long e = vb->hdr[lane].ends;  // unpublished slots read as closed
      const bool open = ends_front(e) < ends_back(e);
      const uint32_t m = __ballot_sync(0xffffffffu, open);
      int jj = -1, tt = -1, stop = 0, kind = 0;
      // after an expired wait this CTA takes no more tasks
      if (lane == 0 && X.sh->timeout) {
        stop = 1;
      } else if (lane == 0) {
        const int rot = (int)(blockIdx.x % 32u);
        const uint32_t rm = (m >> rot) | (rot ? (m << (32 - rot)) : 0u);
        uint32_t left = rm;
        while (left && jj < 0) {
          const int q = (__ffs(left) - 1 + rot) & 31;
          left &= left - 1u;
          // a chunk from the back of the row (see JobHdr)
          const unsigned long long old = atomicAdd(&bd->hdr[q].ends, ~0ull);
          const int d = ends_back(old) - 1;
          if (d >= ends_front(old)) {
            jj = q;
            tt = d;
            kind = ends_kind(old);
          }
        }
        __threadfence();  // the job's header is read after the claim
        if (jj < 0 && !m) {
          if (vb->ctas_done >= (int)gridDim.x || clock64() - t0 > lim) stop = 1;
          else __nanosleep(200);
        }
        X.sh->bi[0] = jj;
        X.sh->bi[1] = tt;
        X.sh->bi[2] = stop;
        X.sh->bi[3] = kind;
      }
    }
    __syncthreads();
    const int jj = X.sh->bi[0], tt = X.sh->bi[1], stop = X.sh->bi[2], kind = X.sh->bi[3];
    __syncthreads();
    if (stop) break;
    if (jj >= 0) {
      if (kind == JOB_STREAM) stream_task(X, jj, tt);
      else band_task(X, jj, tt);
    }
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&bd->exits, 1) == (int)gridDim.x - 1) {
      const int nj = min(bd->njobs, MAXJOBS);
      for (int q = 0; q < nj; ++q) {
        JobHdr* H = &bd->hdr[q];
        H->ends = 0ull;  // reads as closed until the next publish
        H->done = H->list_n = H->above_n = 0;
        H->mxk = 0u;
        H->nleg = H->nf = H->bad = 0;
      }
      bd->njobs = 0;
      bd->ctas_done = 0;
      bd->next_row = 0;
      bd->exits = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Radix descent to a boundary.  COUNT (MASS = false): the target-th largest
// legal element (ties: earliest ids).  MASS: the top-p boundary of S_k (vK,
// idK) for mass p * M_k, M_k taken from the first histogram.  Returns false if
// no boundary was found (only possible when a bounded wait gave up mid-pass).
// ---------------------------------------------------------------------------
template <int DT, bool MASS>
__device__ __noinline__ bool descend(Ctx<DT>& X, uint64_t target, float p, uint32_t vK, int idK,
                                     float m, uint32_t& v_out, int& id_out) {
  constexpr int SIG = ElemT<DT>::SIG;
  constexpr int NLV = (SIG == 16) ? 2 : 3;  // digit widths: 11 + 5, or 11 + 11 + 10
  const float nm = -m * X.c2;
  uint32_t prefix = 0u;
  int plen = 0;
  Cross cr;
  cr.cnt = 0;
#pragma unroll 1
  for (int lv = 0; lv < NLV; ++lv) {
    const int nbits = (lv == 0) ? HB : ((SIG == 16) ? 5 : (lv == 1 ? HB : 10));
    const int shift = SIG - plen - nbits;
    uint32_t ac;
    uint64_t am;
    hist_pass<DT, MASS>(X, prefix, plen, shift, nbits, vK, idK, nm, ac, am);
    if (MASS && lv == 0) {
      const uint64_t mk = hist_total(X, nbits);
      target = (uint64_t)ceil((double)p * (double)mk);
      if (target == 0) target = 1;
    }
    cr = hist_cross<DT, MASS>(X, nbits, MASS ? am : (uint64_t)ac, target);
    if (!cr.ok) return false;
    prefix = (prefix << nbits) | (uint32_t)cr.bin;
    plen += nbits;
    if (cr.cnt <= (uint32_t)CAP) break;
  }
  const uint32_t lo = prefix << (SIG - plen);
  const uint64_t hi = ((uint64_t)prefix + 1u) << (SIG - plen);
  if (cr.cnt <= (uint32_t)CAP) {
    uint32_t ac;
    uint64_t am;
    band_pass<DT, MASS>(X, lo, hi, vK, idK, nm, ac, am);
    const int n = min(X.sh->n, CAP);
    list_range(X, n);
    if (!MASS) return list_resolve_k<NT>(X, n, (int)(target - ac), v_out, id_out);
    list_weights<NT, DT, true>(X, n, 0.f, nm, vK, idK);
    Res R;
    R.vK = vK;
    R.idK = idK;
    uint64_t km;
    if (!list_resolve_p<NT, DT, true>(X, n, target - am, 1.f, 0.f, nm, R, km)) return false;
    v_out = R.vP;
    id_out = R.idP;
    return true;
  }
  // one value with more than CAP copies
  v_out = prefix;
  if (!MASS) {
    const int keep = (int)(target - cr.before);
    id_out = (keep < (int)cr.cnt) ? tie_pass(X, prefix, keep, 0u, NOID) : NOID;
  } else {
    const uint64_t qv = fx_weight(key_value<DT>(prefix), X.c2, nm);
    if (qv == 0) return false;
    const uint64_t j = (target - cr.before + qv - 1) / qv;
    id_out = (j < (uint64_t)cr.cnt) ? tie_pass(X, prefix, (int)j, vK, idK)
                                   : ((prefix == vK) ? idK : NOID);
  }
  return true;
}

// ---------------------------------------------------------------------------
// Row classes
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ void row_argmax(Ctx<DT>& X) {
  const KArgs& a = *X.a;
  uint32_t bk;
  int bid, nf = 0;
  argmax_stream(X, bk, bid, nf);
  if (X.sh->timeout) return error_row(X, ST_TIMEOUT, __LINE__);
  if (nf) return error_row(X, ST_NONFINITE);
  if (bk == 0u) return error_row(X, ST_EMPTY);
  zero_outputs(X);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (a.kept_mask) a.kept_mask[(size_t)X.row * X.W + (bid >> 5)] = 1u << (bid & 31);
    if (a.probs && a.mode == MODE_MASK) a.probs[(size_t)X.row * X.V + bid] = 1.f;
    if (a.logprob) a.logprob[X.row] = 0.f;  // the kept set is {argmax}
    put_row(X, ST_OK, bid, 1, PATH_GREEDY, 0);
  }
  __syncthreads();
}

// Mass stream; a second stream with the row maximum as reference when the
// first chunk's maximum was far below it (weights would overflow).
template <int DT, bool ALLM>
__device__ __forceinline__ ExpOut mass_stream(Ctx<DT>& X, float Kt, float vest, float p_hist) {
  ExpOut E;
  float ref = __int_as_float(0x7fffffff);
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    E = exp_stream<DT, ALLM, !ALLM>(X, Kt, vest, ref, p_hist);
    if (X.sh->timeout || E.nf || E.nleg == 0 || !((E.mx - E.ref) * X.c2 > 100.f)) break;
    ref = E.mx;
  }
  return E;
}

template <int DT>
__device__ __noinline__ void row_keepall(Ctx<DT>& X, double u, float vest) {
  const KArgs& a = *X.a;
  const ExpOut E = mass_stream<DT, true>(X, 0.f, vest, 0.f);
  if (X.sh->timeout) return error_row(X, ST_TIMEOUT, __LINE__);
  if (E.nf) return error_row(X, ST_NONFINITE);
  if (E.nleg == 0) return error_row(X, ST_EMPTY);
  const float nm = -E.ref * X.c2;
  double mtot = 0.0;
  int tok = -1;
  if (a.mode == MODE_SAMPLE || (a.probs && a.mode == MODE_MASK))
    tok = sample_tail(X, u, 0u, -1, nm, nullptr, mtot);
  if (a.probs && a.mode == MODE_MASK) probs_pass(X, 0u, -1, __fdiv_rn(E.ref, X.temp), mtot);
  if (X.sh->timeout) return error_row(X, ST_TIMEOUT, __LINE__);
  put_logprob(X, tok, __fdiv_rn(E.ref, X.temp), mtot);
  write_row(X, ST_OK, tok, E.nleg, PATH_ALL);
  __syncthreads();
}

// Returns false when the list does not validate (the row then takes the
// general path).
template <int DT>
__device__ __noinline__ bool row_list(Ctx<DT>& X, int K, float p, double u, float vest) {
  const bool take_all = vest <= (float)(CAP - CAP / 8);
  const float Kt = (float)(K + K / 4 + 64);
  int nf = 0;
  uint32_t tkey;
  const uint32_t kmax = list_stream(X, Kt, vest, take_all, nf, tkey);
  if (X.sh->timeout) {
    error_row(X, ST_TIMEOUT, __LINE__);
    return true;
  }
  const int nl = X.sh->n;
  if (nl > CAP || (nl < K && !(take_all && nl > 0))) {
    if (take_all && nl == 0) {
      error_row(X, nf ? ST_NONFINITE : ST_EMPTY);
      return true;
    }
    return false;
  }
  if (nf || kmax >= ElemT<DT>::KPINF) {
    error_row(X, ST_NONFINITE);
    return true;
  }
  const float m_z = __fdiv_rn(key_value<DT>(kmax), X.temp);
  if (!list_finish(X, nl, min(K, nl), p, 0, m_z, u, PATH_SIGMA, tkey, kmax))
    error_row(X, ST_TIMEOUT, __LINE__);
  return true;
}

// Band pass over a top-p bracket [b_lo, b_hi] (bins relative to nref), then
// the exact boundary inside the band list; true when the row is finished.
// Every kept-mask word is rewritten by the band pass, so a failed attempt
// leaves nothing behind for the next one.
template <int DT>
__device__ __noinline__ bool band_try_p(Ctx<DT>& X, int b_lo, int b_hi, float nref, float nm,
                                        uint64_t Pq, float m, double u) {
  BandOut bo;
  const int ln = band_any(X, b_lo, b_hi, nref, nm, bo);
  if (X.sh->timeout) return false;
  const int nb = min(max(ln, 0), CAP);
  // the band's key range is the thresholds' (every entry has xb <= x < xa)
  if (threadIdx.x == 0) {
    const uint32_t k_lo = bits_key<DT>(DT == DT_F32 ? pack_down<DT>(bo.xb) : (pack_down<DT>(bo.xb) & 0xffffu));
    const uint32_t k_hi = (bo.xa < INFINITY)
        ? bits_key<DT>(DT == DT_F32 ? pack_down<DT>(bo.xa) : (pack_down<DT>(bo.xa) & 0xffffu)) - 1u
        : ElemT<DT>::KPINF - 1u;
    X.sh->bu[4] = k_lo;
    X.sh->bu[5] = max(k_hi, k_lo);
  }
  __syncthreads();
  if (ln >= 0 && ln <= CAP && Pq > bo.above_q) {
    list_weights<NT, DT, true>(X, nb, 0.f, nm, 0u, -1);
    Res R;
    R.vK = 0u;
    R.idK = -1;
    uint64_t km;
    if (list_resolve_p<NT, DT, true>(X, nb, Pq - bo.above_q, 1.f, 0.f, nm, R, km)) {
      finish_band(X, nb, bo, R.vP, R.idP, m, u, PATH_FULL);
      return true;
    }
  }
  return false;
}

template <int DT>
__device__ __noinline__ void row_general(Ctx<DT>& X, int K, float p, double u, float vest) {
  // list target: the top-k set plus margin, or (no top-k boundary expected)
  // 512 -- top-p sets are short unless the row is flat, and flat rows take
  // the histogram bracket anyway
  const int Kt = (K < X.V && (float)K < vest && K <= (CAP * 3) / 4) ? K + K / 4 + 64 : 512;
  // a top-p row without top-k boundary may build its weight histogram in the
  // stream (when the first chunk predicts a kept set beyond the list)
  const bool g1 = !((float)K < vest) && p < 1.f;
  const ExpOut E = mass_stream<DT, false>(X, (float)Kt, vest, g1 ? p : 0.f);
  if (X.sh->timeout) return error_row(X, ST_TIMEOUT, __LINE__);
  if (E.nf) return error_row(X, ST_NONFINITE);
  if (E.nleg == 0) return error_row(X, ST_EMPTY);
  const float m = E.mx;
  const float m_z = __fdiv_rn(m, X.temp);
  const float nm = -m * X.c2;
  const int keff = min(K, E.nleg);
  const bool needK = keff < E.nleg;
  const int n = min(X.sh->n, CAP);
  const bool list_ok = !E.ovf;
  // row mass relative to the maximum, fixed point
  const double zq = E.z * exp2((double)((E.ref - m) * X.c2)) * 1099511627776.0;

  // 1. the whole kept set inside the sigma-truncated list
  if (list_ok) {
    if (needK && n >= keff) {
      if (list_finish(X, n, keff, p, 0, m_z, u, PATH_SIGMA, E.tkey, E.lkmax)) return;
    } else if (!needK && p < 1.f && E.lmass >= (double)p * E.z * (1.0 - 1e-4)) {
      // the list (a rank prefix of the legal set) carries p of the row's mass
      const uint64_t Pq = max((uint64_t)1, (uint64_t)ceil((double)p * zq));
      if (list_finish(X, n, 0, p, Pq, m_z, u, PATH_SIGMA, E.tkey, E.lkmax)) return;
    }
  }
  // 2. a weight histogram (relative to the maximum), then one band pass over
  //    the bracket it gives
  int b_lo, b_hi;
  if (!needK && p < 1.f) {
    const uint64_t Pq = max((uint64_t)1, (uint64_t)ceil((double)p * zq));
    // the stream's sampled histogram first (bins relative to its reference),
    // then a full histogram pass relative to the maximum
    if (E.hist && wh_bracket_sampled(X, (1.0 - (double)p) * E.z, (float)ElemT<DT>::EPV, b_lo, b_hi)) {
      if (band_try_p(X, b_lo, b_hi, -E.ref * X.c2, nm, Pq, m, u)) return;
      if (X.sh->timeout) return error_row(X, ST_TIMEOUT, __LINE__);
    }
    whist_pass(X, nm, true);
    if (wh_bracket(X, true, 0, (double)p * zq / 1099511627776.0, 0.f, b_lo, b_hi)) {
      if (band_try_p(X, b_lo, b_hi, nm, nm, Pq, m, u)) return;
      if (X.sh->timeout) return error_row(X, ST_TIMEOUT, __LINE__);
    }
  } else if (needK) {
    whist_pass(X, nm, false);
    if (wh_bracket(X, false, keff, 0.0, 0.f, b_lo, b_hi)) {
      BandOut bo;
      const int ln = band_any(X, b_lo, b_hi, nm, nm, bo);
      if (X.sh->timeout) return error_row(X, ST_TIMEOUT, __LINE__);
      const int nb = min(max(ln, 0), CAP);
      list_range(X, nb);
      uint32_t vK;
      int idK;
      if (ln >= 0 && ln <= CAP && keff > bo.above_n &&
          list_resolve_k<NT>(X, nb, keff - bo.above_n, vK, idK)) {
        list_weights<NT, DT, true>(X, nb, 0.f, nm, vK, idK);
        if (p >= 1.f) return finish_band(X, nb, bo, vK, idK, m, u, PATH_FULL);
        uint64_t s = 0;
        const float* wq = list_w(X);
        for (int i = threadIdx.x; i < nb; i += NT) s += to_fx(wq[i]);
        const uint64_t mk = bo.above_q + bsum_q(s, X.sh->rq[1]);
        const uint64_t Pq = max((uint64_t)1, (uint64_t)ceil((double)p * (double)mk));
        if (Pq > bo.above_q) {
          Res R;
          R.vK = vK;
          R.idK = idK;
          uint64_t km;
          if (list_resolve_p<NT, DT, true>(X, nb, Pq - bo.above_q, 1.f, 0.f, nm, R, km))
            return finish_band(X, nb, bo, R.vP, R.idP, m, u, PATH_FULL);
        } else {
          uint32_t vP;
          int idP;
          if (!descend<DT, true>(X, 0, p, vK, idK, m, vP, idP)) return error_row(X, ST_TIMEOUT, __LINE__);
          return finish_by_pass(X, vP, idP, m, u, PATH_FULL);
        }
      }
    }
  }
  // 3. exact radix descent
  uint32_t vK = 0u;
  int idK = -1;
  if (needK && !descend<DT, false>(X, (uint64_t)keff, 1.f, 0u, -1, m, vK, idK))
    return error_row(X, ST_TIMEOUT, __LINE__);
  if (p < 1.f) {
    uint32_t vP;
    int idP;
    if (!descend<DT, true>(X, 0, p, vK, idK, m, vP, idP)) return error_row(X, ST_TIMEOUT, __LINE__);
    return finish_by_pass(X, vP, idP, m, u, PATH_FULL);
  }
  return finish_by_pass(X, vK, idK, m, u, PATH_FULL);
}

// ---------------------------------------------------------------------------
// One row.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ void process_row(Ctx<DT>& X, int row) {
  const KArgs& a = *X.a;
  X.row = row;
  X.src = reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)a.ld * ElemT<DT>::ES;
  X.bm = a.bitmask ? a.bitmask + (size_t)row * X.W : nullptr;
  __syncthreads();
  ring_prime(X);
  // an expired wait leaves the ring's phases unknown: this CTA streams no more
  if (X.sh->timeout) return error_row(X, ST_TIMEOUT, __LINE__);

  float T = 0.f, p = 1.f;
  int topk = 1;
  if (a.mode != MODE_ARGMAX) {
    T = a.temperature[row];
    topk = a.top_k[row];
    p = a.top_p[row];
    if (!(T >= 0.f) || topk < 1 || !(p > 0.f) || !(p <= 1.f)) return error_row(X, ST_INVALID);
  }
  const int K = min(topk, X.V);
  X.temp = T;
  // (an infinite temperature keeps a tiny positive slope so that -inf still
  //  maps to a zero weight)
  X.c2 = (T > 0.f) ? fmaxf(1.4426950408889634f / T, 1e-30f) : 0.f;
  if (a.mode == MODE_ARGMAX || T == 0.f || K == 1) return row_argmax(X);
  const double u = (a.mode == MODE_SAMPLE) ? philox_uniform(a.seed[row], a.offset[row]) : 0.0;

  // legal-count estimate: the bitmask's population, else V
  float vest = (float)X.V;
  if (X.bm) {
    int pc = 0;
    for (int w = threadIdx.x; w < X.W; w += NT) {
      uint32_t b = __ldg(X.bm + w);
      if (w == X.W - 1 && (X.V & 31)) b &= (1u << (X.V & 31)) - 1u;
      pc += __popc(b);
    }
    vest = fmaxf((float)bsum_i(pc, X.sh->ri[1]), 1.f);
  }
  if (K >= X.V && p >= 1.f) return row_keepall(X, u, vest);
  if (K <= KLIST && row_list(X, K, p, u, vest)) return;
  row_general(X, K, p, u, vest);
}

template <int DT>
__global__ void __launch_bounds__(NT, 2) smp_kernel(const __grid_constant__ KArgs a) {
  extern __shared__ unsigned char smem_raw[];
  char* base = reinterpret_cast<char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  // One context per warp in shared memory: every lane of a warp holds the
  // same values, and functions that copy it into registers (LocalCtx) or read
  // it in place then load from shared memory instead of the local-memory
  // stack, which the L1 share left beside two CTAs' shared memory cannot hold.
  __shared__ Ctx<DT> ctxw[NWARP];
  Ctx<DT>& X = ctxw[threadIdx.x >> 5];
  X.a = &a;
  X.ring = base;
  X.lk = reinterpret_cast<uint32_t*>(base + SMEM_RING);
  X.li = reinterpret_cast<int*>(base + SMEM_RING + CAP * 4);
  X.wh = reinterpret_cast<uint32_t*>(base + SMEM_RING + SMEM_LIST);
  X.sh = reinterpret_cast<Sh*>(base + SMEM_RING + SMEM_LIST + SMEM_HIST);
  X.V = a.V;
  X.W = a.W;
  X.nch = (a.V + ElemT<DT>::CE - 1) / ElemT<DT>::CE;
  X.use_tma = a.use_tma;
  X.parity = 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&X.sh->full[s], 1);
    fence_mbar_init();
    X.sh->timeout = 0;
    X.sh->n = 0;
    X.sh->primed = 0;
    for (int s = 0; s < NSTAGE; ++s) X.sh->niss[s] = 0;
  }
  __syncthreads();
  if (a.board) {
    // rows are handed out in order as CTAs free up, so that rows of unequal
    // cost (and B beyond the resident grid) balance over the CTAs
#pragma unroll 1
    while (true) {
      if (threadIdx.x == 0) X.sh->row_next = atomicAdd(&a.board->next_row, 1);
      __syncthreads();
      const int row = X.sh->row_next;
      __syncthreads();
      if (row >= a.B) break;
      process_row(X, row);
    }
  } else {
    for (int row = blockIdx.x; row < a.B; row += gridDim.x) process_row(X, row);
  }
  help_and_exit(X);
  // After an expired wait: wait again, bounded by a fixed two seconds, for
  // the last copy issued into each stage before the CTA exits (at most one
  // per stage is outstanding, as nothing is issued after the expiry).
  __syncthreads();
  if (threadIdx.x == 0 && X.sh->timeout) {
    for (int s = 0; s < NSTAGE; ++s) {
      const int n = X.sh->niss[s];
      if (n > 0) mbar_wait_bounded(&X.sh->full[s], (uint32_t)(n - 1) & 1u, 4000000000ll);
    }
  }
}

}  // namespace smp
