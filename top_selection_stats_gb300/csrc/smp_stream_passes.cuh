// smp_stream_passes.cuh -- the single-pass row streams of the sampling kernel.
//
//   argmax_stream : greedy rows and top-k = 1: packed max test per vector, the
//                   exact argmax (earliest id) only on vectors that beat the
//                   warp's running maximum.
//   list_stream   : top-k rows (k <= KLIST): sigma truncation (Qrita paper
//                   notes, key design 1) -- a threshold t = mu + delta * sigma
//                   from the first chunk, one packed compare per vector, and
//                   the elements >= t appended to the candidate list.
//   exp_stream    : rows whose kept set can be large: the softmax mass of every
//                   legal element (base-2 hardware exponential relative to the
//                   first chunk's maximum), the legal count and the maximum;
//                   keep-all rows also write the kept mask and per-chunk
//                   masses; other rows fill a sigma-truncated list and a
//                   histogram of the weights (WHS bins per factor of two).
#pragma once

#include "smp_list.cuh"

namespace smp {

// Mean and deviation of the legal finite elements of a staged chunk, and
// their maximum (-inf if none), in one pass and one block reduction.
template <int DT>
__device__ __forceinline__ void chunk_stats(Ctx<DT>& X, const char* stage, float& mu, float& sd,
                                         int& cnt, float* mx_out = nullptr) {
  constexpr int EPV = ElemT<DT>::EPV;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float s1 = 0.f, s2 = 0.f, n = 0.f, mn = INFINITY, mx = -INFINITY;
#pragma unroll 1
  for (int it = 0; it < ITW; ++it) {
    const uint4 r = load_vec(X, stage, 0, warp_vec<DT>(it));
    float x[EPV];
    unpack<DT>(r, x);
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      if (x[j] > -INFINITY && x[j] < INFINITY) {
        n += 1.f;
        s1 += x[j];
        s2 += x[j] * x[j];
        mn = fminf(mn, x[j]);
        mx = fmaxf(mx, x[j]);
      }
    }
  }
  n = warp_sum(n);
  s1 = warp_sum(s1);
  s2 = warp_sum(s2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __syncthreads();
  if (lane == 0) {
    X.sh->r5[0][warp] = n;
    X.sh->r5[1][warp] = s1;
    X.sh->r5[2][warp] = s2;
    X.sh->r5[3][warp] = mn;
    X.sh->r5[4][warp] = mx;
  }
  __syncthreads();
  n = s1 = s2 = 0.f;
  mn = INFINITY;
  mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {  // in warp order: every thread the same sums
    n += X.sh->r5[0][w];
    s1 += X.sh->r5[1][w];
    s2 += X.sh->r5[2][w];
    mn = fminf(mn, X.sh->r5[3][w]);
    mx = fmaxf(mx, X.sh->r5[4][w]);
  }
  if (mx_out) *mx_out = mx;
  cnt = (int)n;
  mu = n > 0.f ? s1 / n : 0.f;
  sd = sqrtf(n > 0.f ? fmaxf(s2 / n - mu * mu, 0.f) : 0.f);
  // A few far-negative legal values (a penalised or suppressed token) would
  // inflate the deviation and lift the threshold: when the smallest value
  // lies more than 4 deviations below the mean, up to two more passes over
  // the staged chunk leave those values out (the upper tail, where the
  // candidates are, is always kept).
  if (!(mn < mu - 4.f * sd)) return;
#pragma unroll 1
  for (int rep = 0; rep < 2; ++rep) {
    const float lo = mu - 4.f * sd;
    float r1 = 0.f, r2 = 0.f, rn = 0.f;
#pragma unroll 1
    for (int it = 0; it < ITW; ++it) {
      const uint4 r = load_vec(X, stage, 0, warp_vec<DT>(it));
      float x[EPV];
      unpack<DT>(r, x);
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        if (x[j] >= lo && x[j] < INFINITY) {
          rn += 1.f;
          r1 += x[j];
          r2 += x[j] * x[j];
        }
      }
    }
    rn = bsum_f(rn, X.sh->rf[0]);
    if (!(rn < n) || rn < 1.f) break;  // nothing left out: the estimate stands
    r1 = bsum_f(r1, X.sh->rf[1]);
    r2 = bsum_f(r2, X.sh->rf[2]);
    n = rn;
    mu = r1 / n;
    sd = sqrtf(fmaxf(r2 / n - mu * mu, 0.f));
  }
}

// t = mu + delta(q) * sd, delta(q) = Phi^-1(1 - q) interpolated from the host
// table over log2 q in [-24, 0] (step 1/4).  q >= 1 gives -inf.
__device__ __forceinline__ float sigma_threshold(const KArgs& a, float mu, float sd, float q) {
  if (!(q < 1.f)) return -INFINITY;
  float pos = (log2f(fmaxf(q, 1e-30f)) + 24.f) * 4.f;
  pos = fminf(fmaxf(pos, 0.f), (float)(DTAB - 1));
  const int i = min((int)pos, DTAB - 2);
  const float f = pos - (float)i;
  const float d = a.delta[i] * (1.f - f) + a.delta[i + 1] * f;
  return mu + d * sd;
}

// Threshold packed in the element type (rounded toward -inf) and its exact
// float value; anything at or below the lowest finite value takes every
// legal element.
template <int DT>
__device__ __forceinline__ void make_threshold(float t, uint32_t& t2, float& tf) {
  const float low = key_value<DT>(ElemT<DT>::KLOW);
  if (!(t > low)) t = low;
  t2 = pack_down<DT>(t);
  tf = (DT == DT_F32) ? __uint_as_float(t2) : bits_value<DT>(t2 & 0xffffu);
}

// Threshold of a sigma-truncated list from the staged first chunk.
template <int DT>
__device__ __forceinline__ void list_threshold(Ctx<DT>& X, const char* stage, float Kt, float vest,
                                               uint32_t& t2, float& tf, float* mx_out = nullptr) {
  float mu, sd;
  int n1;
  chunk_stats(X, stage, mu, sd, n1, mx_out);
  const float t = (n1 >= 64) ? sigma_threshold(*X.a, mu, sd, Kt / vest) : -INFINITY;
  make_threshold<DT>(t, t2, tf);
}


// ---------------------------------------------------------------------------
// Argmax over the legal finite elements: (largest key, earliest id).
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ void argmax_stream(Ctx<DT>& Xr, uint32_t& best_key, int& best_id, int& nf) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  const int v0 = warp_vec<DT>(0);
  uint32_t wkey = 0u;
  int wid = NOID;
  float runf = -INFINITY;
  uint32_t run2 = ninf2<DT>();
  int bad = 0;
  ring_begin(X);
  RingIt<DT> R(X);
#pragma unroll 1
  while (R.c < X.nch) {
    const char* stage = R.wait(X);
    uint4 r[ITW];
#pragma unroll
    for (int it = 0; it < ITW; ++it) r[it] = load_vec(X, stage, R.c, v0 + 32 * it);
    uint32_t hits = 0u;
    if (R.c == 0) {
      // seed the warp's running maximum with its first chunk: only vectors
      // holding that maximum (or NaN) take the exact path
      float m = -INFINITY;
#pragma unroll
      for (int it = 0; it < ITW; ++it) m = fmaxf(m, vmax_nan_f<DT>(r[it]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (m > -INFINITY) {
        runf = nextafterf(m, -INFINITY);  // elements >= m pass the strict test
        run2 = pack_down<DT>(runf);
      }
    }
#pragma unroll
    for (int it = 0; it < ITW; ++it) hits |= any_gt<DT>(r[it], run2, runf) ? (1u << it) : 0u;
    if (__any_sync(0xffffffffu, hits != 0u)) {
      uint32_t lk = 0u;
      int lid = NOID;
#pragma unroll 1
      for (int it = 0; it < ITW; ++it) {
        if (!((hits >> it) & 1u)) continue;
        const int vi = v0 + 32 * it;
        const uint4 rv = load_vec(X, stage, R.c, vi);
        const int id0 = R.c * CE + vi * EPV;
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
          const uint32_t b = elem_bits<DT>(rv, j);
          const float x = bits_value<DT>(b);
          if (x != x || x == INFINITY) {
            bad = 1;
          } else if (x > runf) {
            const uint32_t k = bits_key<DT>(b);
            if (k > lk) {
              lk = k;
              lid = id0 + j;
            }
          }
        }
      }
      const uint32_t mk = __reduce_max_sync(0xffffffffu, lk);
      if (mk > wkey) {
        wid = (int)__reduce_min_sync(0xffffffffu, (uint32_t)((lk == mk) ? lid : NOID));
        wkey = mk;
        runf = key_value<DT>(mk);
        run2 = pack_down<DT>(runf);
      }
    }
    R.release(X);
  }
  best_key = bmax_u(wkey, X.sh->ru[0]);
  best_id = (int)bmin_u((uint32_t)((wkey == best_key) ? wid : NOID), X.sh->ru[1]);
  nf = bsum_i(bad, X.sh->ri[0]);
}

// ---------------------------------------------------------------------------
// Sigma-truncated list.  Kt is the number of candidates aimed at; take_all
// puts every legal element in the list.  Once the list overflows the rest of
// the row is only drained.  Returns the largest key appended (0: none); nf
// counts NaN / +inf seen in legal slots; tkey is the threshold's key.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ uint32_t list_stream(Ctx<DT>& Xr, float Kt, float vest, bool take_all,
                                             int& nf, uint32_t& tkey) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  if (threadIdx.x == 0) X.sh->n = 0;
  const int v0 = warp_vec<DT>(0);
  uint32_t t2;
  float tf;
  make_threshold<DT>(-INFINITY, t2, tf);
  uint32_t kmax = 0u;
  int bad = 0;
  ring_begin(X);
  RingIt<DT> R(X);
#pragma unroll 1
  while (R.c < X.nch) {
    const char* stage = R.wait(X);
    if (R.c == 0 && !take_all) list_threshold(X, stage, Kt, vest, t2, tf);
    uint4 r[ITW];
#pragma unroll
    for (int it = 0; it < ITW; ++it) r[it] = load_vec(X, stage, R.c, v0 + 32 * it);
    uint32_t hits = 0u;
#pragma unroll
    for (int it = 0; it < ITW; ++it) hits |= any_ge<DT>(r[it], t2, tf) ? (1u << it) : 0u;
    // once the list overflowed the row falls back: the pass only drains
    // (one reservation per warp and chunk; the vectors are still in registers)
    if (__any_sync(0xffffffffu, hits != 0u) && X.sh->n <= CAP) {
      uint32_t cms[ITW];
      int cnt = 0;
#pragma unroll
      for (int it = 0; it < ITW; ++it) {
        cms[it] = ((hits >> it) & 1u) ? ge_mask<DT>(r[it], t2, tf, bad) : 0u;
        cnt += __popc(cms[it]);
      }
      const int inc = warp_incl_scan(cnt);
      const int tot = __shfl_sync(0xffffffffu, inc, 31);
      int base = 0;
      if ((threadIdx.x & 31) == 31 && tot) base = atomicAdd(&X.sh->n, tot);
      base = __shfl_sync(0xffffffffu, base, 31);
      int pos = base + inc - cnt;
#pragma unroll
      for (int it = 0; it < ITW; ++it) {
        uint32_t cm = cms[it];
        const int id0 = R.c * CE + (v0 + 32 * it) * EPV;
        while (cm) {
          const int j = __ffs(cm) - 1;
          cm &= cm - 1u;
          const uint32_t k = bits_key<DT>(elem_bits_dyn<DT>(r[it], j));
          kmax = max(kmax, k);
          if (pos < CAP) {
            X.lk[pos] = k;
            X.li[pos] = id0 + j;
          }
          ++pos;
        }
      }
    }
    R.release(X);
  }
  nf = bsum_i(bad, X.sh->ri[0]);
  tkey = bits_key<DT>((DT == DT_F32) ? t2 : (t2 & 0xffffu));  // every entry's key is >= tkey
  return bmax_u(kmax, X.sh->ru[0]);
}

// ---------------------------------------------------------------------------
// Softmax-mass stream.  Weights 2^((x - ref) * log2(e) / T) with ref the first
// chunk's maximum (or ref_in when given).  ALLM (keep-all rows): kept mask
// words written on the fly, per-chunk per-warp masses in sh->cmass.  EMIT: a
// sigma-truncated list with Kt candidates aimed at.  The maximum, the NaN /
// +inf flag and the -inf test ride on packed extrema accumulated per thread.
// ---------------------------------------------------------------------------
struct ExpOut {
  double z;    // sum of weights (relative to ref)
  float ref;   // reference value
  float mx;    // maximum legal value
  int nleg;    // legal finite count
  int nf;      // NaN / +inf seen
  int ovf;     // list overflow (EMIT)
  double lmass;  // mass of the list's elements (EMIT, relative to ref)
  uint32_t tkey, lkmax;  // the list threshold's key and the largest key listed (EMIT)
  int hist;              // a weight histogram (relative to ref) of one element in EPV was built
};

// Sum of the EPV weights of a vector: a tree (short dependency chains).
template <int EPV>
__device__ __forceinline__ float tree_sum(const float (&w)[EPV]) {
  if constexpr (EPV == 8) {
    return ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
  } else {
    return (w[0] + w[1]) + (w[2] + w[3]);
  }
}

// Excess-weighted weight-histogram entry for y = WHOFF - WHS * a, a = (x - ref)
// * log2(e) / T: bin floor(y) clamped to [0, WBINS); the element adds 2^11 *
// 2^f, f = (1 - frac(y)) / WHS its weight's excess over the bin's lower edge
// (2^f by its quadratic expansion, error < 2e-5).  Clamped elements add 2^11.
// Floors are taken by round-down adds of a power-of-two constant, not by
// float -> int conversions (a slower pipe).
__device__ __forceinline__ void whist_entry(float y, int& b, uint32_t& add) {
  // t = 1.5 * 2^23 + floor(y) for -1 <= y < 2^22 (y below -1 clamps to bin 0)
  const float t = __fadd_rd(fmaxf(y, -1.f), 12582912.0f);
  const int fyi = __float_as_int(t) - 0x4B400000;
  b = min(max(fyi, 0), WBINS - 1);
  const float fy = __fsub_rn(t, 12582912.0f);
  const float f = (b == fyi) ? (1.f - (y - fy)) * (1.f / WHS) : 0.f;
  const float v = fmaf(f, fmaf(f, 491.96f, 1419.57f), 2048.5f);  // in [2048.5, 2143)
  add = (uint32_t)(__float_as_int(__fadd_rd(v, 8388608.0f)) - 0x4B000000);
}
__device__ __forceinline__ void whist_add(uint32_t* wh, float x, float c2, float nref) {
  int b;
  uint32_t add;
  whist_entry(fmaf(fmaf(x, c2, nref), -(float)WHS, (float)WHOFF), b, add);
  atomicAdd(&wh[b], add);
}

// ---------------------------------------------------------------------------
// Job board primitives.  publish_job writes a job's header for this CTA's row,
// then (after a fence) the claim word that opens it (the owner keeps chunk 0,
// and chunk 1 of a stream job), and returns its slot, or -1 without a board
// or a free slot.  OwnerClaims walks the owner's claims from the front, one
// chunk ahead of the ring.  wait_job waits, bounded, until the helpers report
// n chunks of job j done.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ends_front(unsigned long long e) { return (int)(e >> 32); }
__device__ __forceinline__ int ends_back(unsigned long long e) {
  return (int)((uint32_t)e & (ENDS_KIND - 1u)) - (int)ENDS_OFF;
}
__device__ __forceinline__ int ends_kind(unsigned long long e) {
  return ((uint32_t)e & ENDS_KIND) ? JOB_STREAM : JOB_BAND;
}

template <int DT>
__device__ int publish_job(Ctx<DT>& X, int kind, int nch, int b_lo, int b_hi, float nref,
                           float nm, float xa = INFINITY, float xb = INFINITY) {
  Board* bd = X.a->board;
  if (!bd) return -1;
  if (threadIdx.x == 0) {
    const int j = atomicAdd(&bd->njobs, 1);
    X.sh->bi[0] = (j < MAXJOBS) ? j : -1;
  }
  __syncthreads();
  const int j = X.sh->bi[0];
  __syncthreads();
  if (j < 0) return -1;
  if (kind == JOB_STREAM)
    for (int b = threadIdx.x; b < WBINS; b += NT) bd->wh[j][b] = 0u;
  if (threadIdx.x == 0) {
    JobHdr* H = &bd->hdr[j];
    H->row = X.row;
    H->kind = kind;
    H->nch = nch;
    H->b_lo = b_lo;
    H->b_hi = b_hi;
    H->nref = nref;
    H->nm = nm;
    H->c2 = X.c2;
    H->xa = xa;
    H->xb = xb;
  }
  __threadfence();
  __syncthreads();
  // opened last: the owner holds chunk 0 of a band job and chunks 0 and 1 of
  // a stream job (its ring already has them)
  if (threadIdx.x == 0)
    atomicExch(&bd->hdr[j].ends,
               ((kind == JOB_BAND ? 1ull : 2ull) << 32) |
                   (unsigned long long)((uint32_t)nch + ENDS_OFF + (kind == JOB_STREAM ? ENDS_KIND : 0u)));
  return j;
}

// The owner's claims, made by thread 0.  decide(d) claims chunk d, issues it
// into stage d % NSTAGE when the claim succeeds and leaves the answer in
// sh->bi[6 + d % 2]; the other threads may read it (owns) only after a block
// barrier that follows the call.  After the first failed claim, `first` is
// the first helper chunk.
template <int DT>
struct OwnerClaims {
  JobHdr* H;
  int live, first;
  __device__ __forceinline__ void start(Ctx<DT>& X, JobHdr* h, int nch) {
    H = h;
    live = 1;
    first = nch;
  }
  // The claim of chunk d is taken when the owner is ready to stage it (after
  // chunk d - 2), not earlier, so that helpers arriving meanwhile take it.
  __device__ __forceinline__ void decide(Ctx<DT>& X, int d) {
    if (threadIdx.x != 0) return;
    int own = 0;
    if (live) {
      const unsigned long long old = atomicAdd(&H->ends, 1ull << 32);
      const int f = ends_front(old);
      if (f < ends_back(old)) {
        own = 1;
        issue_chunk(X, d, d % NSTAGE);
      } else {
        live = 0;
        first = f;
      }
    }
    X.sh->bi[6 + (d & 1)] = own;
  }
  __device__ __forceinline__ bool owns(const Ctx<DT>& X, int d) const {
    return X.sh->bi[6 + (d & 1)] != 0;
  }
};

template <int DT>
__device__ bool wait_job(Ctx<DT>& X, int j, int n) {
  if (threadIdx.x == 0) {
    volatile JobHdr* H = &X.a->board->hdr[j];
    const long long t0 = clock64();
    int ok = 1;
    while (H->done < n) {
      if (clock64() - t0 > X.a->wait_limit) {
        ok = 0;
        break;
      }
      __nanosleep(100);
    }
    __threadfence();
    if (ok && H->bad) ok = 0;  // a helper's chunk never landed
    X.sh->bi[0] = ok;
    if (!ok) X.sh->timeout = 1;
  }
  __syncthreads();
  const bool ok = X.sh->bi[0] != 0;
  __syncthreads();
  return ok;
}

// Mass (returned: this thread's float sum), legal count, packed maximum and
// sampled weight-histogram entries (one element per vector) of one staged
// chunk: the body of a shared mass stream, the same arithmetic whichever CTA
// runs the chunk.
template <int DT>
__device__ __forceinline__ float mass_hist_chunk(const Ctx<DT>& X, const char* stage, int c,
                                                 float c2, float nref, uint32_t* wh,
                                                 uint32_t& amax, int& nleg) {
  constexpr int EPV = ElemT<DT>::EPV;
  const int v0 = warp_vec<DT>(0);
  float cs = 0.f;
#pragma unroll
  for (int it = 0; it < ITW; ++it) {
    const uint4 r = load_vec(X, stage, c, v0 + 32 * it);
    amax = pmax<DT>(amax, vmax2<DT>(r));
    float x[EPV], w[EPV];
    unpack<DT>(r, x);
#pragma unroll
    for (int q = 0; q < EPV; ++q) w[q] = fast_exp2(fmaf(x[q], c2, nref));  // -inf -> 0
    cs += tree_sum<EPV>(w);
#pragma unroll
    for (int q = 0; q < EPV; ++q) nleg += (x[q] > -INFINITY) ? 1 : 0;
    // the sampled element of this vector (as in the owner's stream)
    const int qs = (v0 + 32 * it) & (EPV - 1);
    float xs = x[0];
#pragma unroll
    for (int q = 1; q < EPV; ++q) xs = (qs == q) ? x[q] : xs;
    if (xs > -INFINITY) whist_add(wh, xs, c2, nref);
  }
  return cs;
}

// ---------------------------------------------------------------------------
// Chunks of a published mass stream (job j), run by a helper from chunk c on:
// while a chunk is processed the next one is claimed and its copy issued into
// the other stage, so the helper stays on the job until its chunks run out.
// Per chunk: the per-warp masses.  Once, at the end: the legal count, largest
// value, NaN / +inf flag and weight histogram (built in this CTA's histogram
// area, then added to the job's) and the number of chunks done.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ void stream_task(Ctx<DT>& Xr, int j, int c) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  const KArgs& a = *X.a;
  Board* bd = a.board;
  volatile JobHdr* H = &bd->hdr[j];
  const int row = H->row;
  const float nref = H->nref, c2 = H->c2;
  X.row = row;
  X.src = reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)a.ld * ElemT<DT>::ES;
  X.bm = a.bitmask ? a.bitmask + (size_t)row * X.W : nullptr;
  X.c2 = c2;
  // the chunk's copy first, the histogram clear while it is in flight (the
  // previous task's last barrier freed both stages)
  int s = 0;
  if (threadIdx.x == 0) issue_chunk(X, c, s);
  uint32_t* wh = X.wh;
  for (int b = threadIdx.x; b < WBINS; b += NT) wh[b] = 0u;
  __syncthreads();
  uint32_t amax = p_ninf<DT>();
  int nleg = 0, ndone = 0;
#pragma unroll 1
  for (int it = 0;; ++it) {
    if (threadIdx.x == 0) {
      const int d = helper_claim(bd, j, X.sh->timeout);
      if (d >= 0) issue_chunk(X, d, s ^ 1);
      X.sh->bi[6 + (it & 1)] = d;
    }
    const char* stage = ring_wait_at(X, c, s);
    const float cs = mass_hist_chunk<DT>(X, stage, c, c2, nref, wh, amax, nleg);
    const float ws = warp_sum(cs);
    if ((threadIdx.x & 31) == 0) bd->cmass[j][c * NWARP + (threadIdx.x >> 5)] = ws;
    ++ndone;
    __syncthreads();  // the stage is free, the next claim visible
    c = X.sh->bi[6 + (it & 1)];
    if (c < 0) break;
    s ^= 1;
  }
  const float tmax = p2f_max<DT>(amax);
  const int nf = bsum_i((tmax < INFINITY) ? 0 : 1, X.sh->ri[1]);  // (its barrier ends the histogram)
  for (int b = threadIdx.x; b < WBINS; b += NT) {
    const uint32_t v = wh[b];
    if (v) atomicAdd(&bd->wh[j][b], v);
  }
  const float mx = bmax_f(nf ? -INFINITY : tmax, X.sh->rf[0]);
  nleg = bsum_i(nleg, X.sh->ri[0]);
  if (threadIdx.x == 0) {
    if (X.sh->timeout) atomicOr((int*)&H->bad, 1);
    if (nf) atomicOr((int*)&H->nf, 1);
    else if (mx > -INFINITY) atomicMax((unsigned int*)&H->mxk, fkey(mx));
    if (nleg) atomicAdd((int*)&H->nleg, nleg);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd((int*)&H->done, ndone);
}

template <int DT, bool ALLM, bool EMIT>
__device__ __noinline__ ExpOut exp_stream(Ctx<DT>& Xr, float Kt, float vest, float ref_in,
                                          float p_hist) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  constexpr uint32_t FULLB = (1u << EPV) - 1u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int v0 = warp_vec<DT>(0);
  uint32_t* mrow = (ALLM && X.a->kept_mask) ? X.a->kept_mask + (size_t)X.row * X.W : nullptr;
  if (threadIdx.x == 0) X.sh->n = 0;
  uint32_t t2 = p_pinf<DT>();
  float tf = INFINITY;
  float ref = ref_in, nref = 0.f;
  const float c2 = X.c2;
  float lm = 0.f;
  uint32_t lkm = 0u;
  bool hist = false;
  uint32_t* wh = X.wh;
  uint32_t amax = p_ninf<DT>();
  int nleg = 0;
  int js = -1;  // board slot of the shared rest of the stream
  ring_begin(X);
  RingIt<DT> R(X);
#pragma unroll 1
  while (R.c < X.nch) {
    const int c = R.c;
    const char* stage = R.wait(X);
    if (c == 0) {
      if (EMIT) {
        // the list threshold and the reference (the first chunk's maximum)
        // from one pass over the chunk
        float m = -INFINITY;
        list_threshold(X, stage, Kt, vest, t2, tf, &m);
        if (ref_in != ref_in) ref = (m > -INFINITY) ? m : 0.f;
      } else if (ref_in != ref_in) {  // reference = the first chunk's maximum
        float m = -INFINITY;
#pragma unroll 1
        for (int it = 0; it < ITW; ++it) {
          float x[EPV];
          unpack<DT>(load_vec(X, stage, 0, v0 + 32 * it), x);
#pragma unroll
          for (int j = 0; j < EPV; ++j)
            if (x[j] < INFINITY) m = fmaxf(m, x[j]);
        }
        ref = bmax_f(m, X.sh->rf[0]);
        if (!(ref > -INFINITY)) ref = 0.f;
      }
      nref = -ref * c2;
      if (EMIT) {
        if (p_hist > 0.f) {
          // top-p row: if the first chunk's mass at or above the list
          // threshold is below p of its mass, the kept set will not fit the
          // list -- build the weight histogram on the way (bins relative to
          // ref, excess-weighted counts)
          float z0 = 0.f, m0 = 0.f;
#pragma unroll 1
          for (int it = 0; it < ITW; ++it) {
            float x[EPV];
            unpack<DT>(load_vec(X, stage, 0, v0 + 32 * it), x);
#pragma unroll
            for (int j = 0; j < EPV; ++j) {
              const float w = fast_exp2(fmaf(x[j], c2, nref));
              z0 += w;
              if (x[j] >= tf) m0 += w;
            }
          }
          z0 = bsum_f(z0, X.sh->rf[1]);
          m0 = bsum_f(m0, X.sh->rf[2]);
          hist = m0 < p_hist * z0;
          if (hist) {
            // a sampled weight histogram: element (vector index mod EPV) of
            // every vector, one in EPV of the row; no list (it could not hold
            // the kept set).  The rest of the stream goes on the job board:
            // this CTA streams from the front, helpers take chunks from the
            // back (this loop ends after chunk 0).
            for (int b = threadIdx.x; b < WBINS; b += NT) wh[b] = 0u;
            __syncthreads();
            t2 = p_pinf<DT>();
            tf = INFINITY;
            if (X.nch > 2) {
              js = publish_job(X, JOB_STREAM, X.nch, 0, 0, nref, 0.f);
              if (js >= 0) X.nch = 1;
            }
          }
        }
      }
    }
    float cs = 0.f;
    uint32_t hits = 0u, cmin = p_pinf<DT>();
#pragma unroll
    for (int it = 0; it < ITW; ++it) {
      const uint4 r = load_vec(X, stage, c, v0 + 32 * it);
      const uint32_t m2 = vmax2<DT>(r);
      amax = pmax<DT>(amax, m2);
      cmin = pmin<DT>(cmin, vmin2<DT>(r));
      if (EMIT && p_any_ge<DT>(m2, t2, tf)) hits |= 1u << it;
      float x[EPV], w[EPV];
      unpack<DT>(r, x);
#pragma unroll
      for (int j = 0; j < EPV; ++j) w[j] = fast_exp2(fmaf(x[j], c2, nref));  // -inf -> 0
      cs += tree_sum<EPV>(w);
      if (EMIT && hist) {
        // the sampled element of this vector (index v0 + 32 it + lane)
        const int q = (v0 + 32 * it) & (EPV - 1);
        float xs = x[0];
#pragma unroll
        for (int j = 1; j < EPV; ++j) xs = (q == j) ? x[j] : xs;
        if (xs > -INFINITY) whist_add(wh, xs, c2, nref);
      }
    }
    // legal count and kept-mask words: every slot legal unless the chunk
    // holds -inf somewhere in this warp
    const bool neg = !(p2f_min<DT>(cmin) > -INFINITY);
    if (!__any_sync(0xffffffffu, neg)) {
      nleg += EPV * ITW;
      if (ALLM && mrow) {
#pragma unroll
        for (int it = 0; it < ITW; ++it) {
          const int wi = (c * CE + (v0 + 32 * it) * EPV) >> 5;
          if ((lane & (32 / EPV - 1)) == 0 && wi < X.W) mrow[wi] = 0xffffffffu;
        }
      }
    } else {
#pragma unroll 1
      for (int it = 0; it < ITW; ++it) {
        const int vi = v0 + 32 * it;
        uint32_t kb = FULLB;
        if (neg) {
          float x[EPV];
          unpack<DT>(load_vec(X, stage, c, vi), x);
          kb = 0u;
#pragma unroll
          for (int j = 0; j < EPV; ++j)
            if (x[j] > -INFINITY) kb |= 1u << j;
        }
        nleg += __popc(kb);
        if (ALLM && mrow) {
          uint32_t wv;
          int wi;
          if constexpr (EPV == 8) {
            wv = kb << (8 * (lane & 3));
            wv |= __shfl_xor_sync(0xffffffffu, wv, 1);
            wv |= __shfl_xor_sync(0xffffffffu, wv, 2);
            wi = ((lane & 3) == 0) ? ((c * CE + vi * EPV) >> 5) : -1;
          } else {
            wv = kb << (4 * (lane & 7));
            wv |= __shfl_xor_sync(0xffffffffu, wv, 1);
            wv |= __shfl_xor_sync(0xffffffffu, wv, 2);
            wv |= __shfl_xor_sync(0xffffffffu, wv, 4);
            wi = ((lane & 7) == 0) ? ((c * CE + vi * EPV) >> 5) : -1;
          }
          if (wi >= 0 && wi < X.W) mrow[wi] = wv;
        }
      }
    }
    if (EMIT && __any_sync(0xffffffffu, hits != 0u) && X.sh->n <= CAP) {
      int dummy = 0;
      lkm = max(lkm, warp_append_hits<DT, true>(X, stage, c, hits, t2, tf, dummy, c2, nref, lm));
    }
    const float ws = warp_sum(cs);
    if (lane == 0) X.sh->cmass[c][warp] = ws;
    R.release(X);
  }
  const int nch = Xr.nch;
  int helpers = 0;  // chunks of the shared stream that helpers ran
  if (EMIT && js >= 0) {
    // the owner's side of the shared stream: chunk 1 is in flight, chunks
    // from 2 on are the owner's while its claims succeed
    Board* bd = X.a->board;
    OwnerClaims<DT> oc;
    oc.start(X, &bd->hdr[js], nch);
    __syncthreads();  // every warp is done with chunk 0: its stage takes chunk 2
    oc.decide(X, 2);
#pragma unroll 1
    for (int c = 1; c < nch; ++c) {
      if (c >= 2 && !oc.owns(X, c)) break;
      const char* stage = ring_wait(X, c);
      const float cs = mass_hist_chunk<DT>(X, stage, c, c2, nref, wh, amax, nleg);
      const float ws = warp_sum(cs);
      if (lane == 0) X.sh->cmass[c][warp] = ws;
      __syncthreads();
      oc.decide(X, c + 2);
    }
    if (threadIdx.x == 0) X.sh->bi[0] = oc.first;
    __syncthreads();
    const int first = X.sh->bi[0];
    helpers = nch - first;
    if (wait_job(X, js, helpers)) {
      for (int b = threadIdx.x; b < WBINS; b += NT) wh[b] += __ldcg(&bd->wh[js][b]);
      for (int f = first * NWARP + threadIdx.x; f < nch * NWARP; f += NT)
        X.sh->cmass[f / NWARP][f % NWARP] = __ldcg(&bd->cmass[js][f]);
    }
    __syncthreads();
  }
  const float tmax = p2f_max<DT>(amax);
  ExpOut o;
  // row mass: the per-(chunk, warp) cells summed in chunk order, the same
  // whether or not the stream was shared (the barrier: every warp's cells of
  // its last chunk are written)
  __syncthreads();
  double zc = 0.0;
  if (threadIdx.x < nch) {
#pragma unroll
    for (int w = 0; w < NWARP; ++w) zc += (double)X.sh->cmass[threadIdx.x][w];
  }
  o.z = bsum_d(zc, X.sh->rd[0]);
  o.ref = ref;
  o.nf = bsum_i((tmax < INFINITY) ? 0 : 1, X.sh->ri[1]);  // NaN or +inf in a legal slot
  o.mx = bmax_f(o.nf ? -INFINITY : tmax, X.sh->rf[0]);
  o.nleg = bsum_i(nleg, X.sh->ri[0]);
  o.ovf = X.sh->n > CAP;
  if (EMIT && js >= 0) {
    // the helpers' counts, flags and maximum (their cells and histogram
    // were merged above)
    volatile JobHdr* H = &X.a->board->hdr[js];
    if (helpers > 0) {
      o.nleg += H->nleg;
      o.nf |= H->nf;
      const uint32_t mk = H->mxk;
      o.mx = o.nf ? -INFINITY : fmaxf(o.mx, mk ? key_to_float(mk) : -INFINITY);
    }
    o.ovf = 1;  // the list saw chunk 0 only
  }
  o.lmass = EMIT ? bsum_d((double)lm, X.sh->rd[1]) : 0.0;
  o.tkey = bits_key<DT>((DT == DT_F32) ? t2 : (t2 & 0xffffu));
  o.lkmax = EMIT ? bmax_u(lkm, X.sh->ru[0]) : 0u;
  o.hist = hist ? 1 : 0;
  if (hist) o.ovf = 1;  // no list was kept
  return o;
}

// ---------------------------------------------------------------------------
// Weight-histogram pass: legal elements binned by a = (x - m) * log2(e) / T
// (nm = -m * log2(e) / T), WHS bins per factor of two.  hmass: each element
// adds 2^11 * 2^f, f = (1 - frac(y)) / WHS its weight's excess over the bin's
// lower edge (2^f by its quadratic expansion, error < 2e-5); else 1.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ void whist_pass(Ctx<DT>& Xr, float nm, bool hmass) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  constexpr int EPV = ElemT<DT>::EPV;
  uint32_t* wh = X.wh;
  for (int b = threadIdx.x; b < WBINS; b += NT) wh[b] = 0u;
  const int v0 = warp_vec<DT>(0);
  const float c2 = X.c2;
  ring_begin(X);
  RingIt<DT> R(X);
#pragma unroll 1
  while (R.c < X.nch) {
    const char* stage = R.wait(X);
#pragma unroll 1
    for (int it = 0; it < ITW; ++it) {
      float x[EPV];
      unpack<DT>(load_vec(X, stage, R.c, v0 + 32 * it), x);
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        if (!(x[j] > -INFINITY)) continue;
        const float y = fmaf(fmaf(x[j], c2, nm), -(float)WHS, (float)WHOFF);
        int b;
        uint32_t add;
        whist_entry(y, b, add);
        atomicAdd(&wh[b], hmass ? add : 1u);
      }
    }
    R.release(X);
  }
  __syncthreads();
}

}  // namespace smp
