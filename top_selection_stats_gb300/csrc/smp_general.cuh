// smp_general.cuh -- exact selection for rows whose kept set does not fit the
// candidate list (flat rows under top-p, top_k beyond the list, failed sigma
// bands), and the passes shared by every row whose kept set is decided by a
// (value, id) boundary.
//
// Weight-histogram bracket.  The mass stream histograms the legal elements by
// a = (x - ref) * log2(e) / T (WHS bins per factor of two).  Counts per bin
// are exact, so the bin holding the k-th element is known; masses per bin are
// bounded by count * 2^a at the bin's edges, so the bins that can hold the
// top-p boundary form a short bracket.  One band pass then collects the
// bracket into the list (where the boundary and its tie quota are resolved
// exactly), and at the same time writes the kept mask, count and per-chunk
// masses of everything above the bracket, which is kept whatever the exact
// boundary.
//
// Radix descent (fallback).  Each pass re-reads the row and builds a 2^11-bin
// histogram -- counts for a top-k boundary, fixed-point masses for a top-p
// boundary -- of the next key digit inside the current prefix, until the
// bin holding the boundary has at most CAP elements; a band pass collects it.
// A single value with more than CAP copies is resolved by a tie pass that
// ranks its copies in id order.  Masses are integers (2^-40 units of the row
// maximum's weight), so every decision is independent of summation order.
#pragma once

#include "smp_stream_passes.cuh"

namespace smp {

template <int DT>
__device__ __forceinline__ float vmax_f(const uint4 r) {
  float x[ElemT<DT>::EPV];
  unpack<DT>(r, x);
  float m = x[0];
#pragma unroll
  for (int j = 1; j < ElemT<DT>::EPV; ++j) m = fmaxf(m, x[j]);
  return m;
}

// Weight 2^((x - m) * log2(e) / T) in fixed point (nm = -m * log2(e) / T).
__device__ __forceinline__ uint64_t fx_weight(float x, float c2, float nm) {
  return to_fx(fast_exp2(fmaf(x, c2, nm)));
}

// Weight-histogram bin of x (nref = -ref * log2(e) / T, as in the mass stream).
__device__ __forceinline__ int wbin(float x, float c2, float nref) {
  const float a = fmaf(x, c2, nref);
  return min(max(floor_small(fmaf(a, -(float)WHS, (float)WHOFF)), 0), WBINS - 1);
}

// Writes the kept-mask word of 32 consecutive elements held by 4 (16-bit) or
// 8 (fp32) consecutive lanes; all lanes of the warp call it.
template <int DT>
__device__ __forceinline__ void put_mask_word(const Ctx<DT>& X, uint32_t* mrow, uint32_t kb,
                                              int id0) {
  constexpr int EPV = ElemT<DT>::EPV;
  const int lane = threadIdx.x & 31;
  uint32_t wv;
  int wi;
  if constexpr (EPV == 8) {
    wv = kb << (8 * (lane & 3));
    wv |= __shfl_xor_sync(0xffffffffu, wv, 1);
    wv |= __shfl_xor_sync(0xffffffffu, wv, 2);
    wi = ((lane & 3) == 0) ? (id0 >> 5) : -1;
  } else {
    wv = kb << (4 * (lane & 7));
    wv |= __shfl_xor_sync(0xffffffffu, wv, 1);
    wv |= __shfl_xor_sync(0xffffffffu, wv, 2);
    wv |= __shfl_xor_sync(0xffffffffu, wv, 4);
    wi = ((lane & 7) == 0) ? (id0 >> 5) : -1;
  }
  if (mrow && wi >= 0 && wi < X.W) mrow[wi] = wv;
}

// Per-(chunk, warp) cell of row element id (the order of the kept masses).
template <int DT>
__device__ __forceinline__ int cell_of(int id) {
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE, VW = ElemT<DT>::VW;
  return (id / CE) * NWARP + ((id % CE) / EPV) / VW;
}
// Fixed-point kept masses of list entries, per cell (in the ring scratch),
// and two 32-bit partial counters per cell after them.
template <int DT>
__device__ __forceinline__ uint64_t* cell_extra(const Ctx<DT>& X) {
  return list_scratch(X) + 1024;
}
static_assert(CAP * 4 + (2048 + MAXCH * NWARP) * 8 <= SMEM_RING, "cell masses live in the ring");

// ---------------------------------------------------------------------------
// Bracket from the weight histogram.  Bins (descending weight) 0..WBINS-1.
//   K mode : counts; the bin holding the k-th element (counts are exact).
//   P mode : masses (units of the reference weight) from excess-weighted
//            counts; the bins where the running mass crosses PZ * (1 -/+
//            1e-3), the margin covering the 2^-11 quantisation of the excess
//            and the rounding of the mass stream's sums.
// Returns false when the bracket holds (or may hold) more than CAP elements.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ bool wh_bracket(Ctx<DT>& Xr, bool pmode, int K, double PZ, float amax,
                                        int& b_lo, int& b_hi) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  const uint32_t* wh = X.wh;
  constexpr int BPT = WBINS / NT;
  const int t = threadIdx.x;
  float v[BPT];
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < BPT; ++q) {
    const int b = t * BPT + q;
    // P mode: wh[b] / 2^11 counts the bin's elements in units of its lower
    // edge weight 2^((WHOFF - b - 1) / WHS); the clamped end bins are bounded
    // by amax above and 0 below
    v[q] = (float)wh[b];
    if (pmode) {
      const float lo_w = (b == WBINS - 1) ? 0.f : exp2f((float)(WHOFF - b - 1) * (1.f / WHS));
      v[q] = (b == 0) ? v[q] * (1.f / 2048.f) * exp2f(fmaxf(amax, (float)WHOFF / WHS))
                      : v[q] * (1.f / 2048.f) * lo_w;
    }
    s += v[q];
  }
  float tot;
  float cum = bscan_excl<float>(s, X.sh->rf[0], tot);
  if (t == 0) {
    X.sh->bi[0] = WBINS;
    X.sh->bi[1] = -1;
  }
  __syncthreads();
  const float lo_t = pmode ? (float)(PZ * (1.0 - 1e-3)) : (float)K;
  const float hi_t = pmode ? (float)(PZ * (1.0 + 1e-3)) : (float)K;
#pragma unroll
  for (int q = 0; q < BPT; ++q) {
    const int b = t * BPT + q;
    if (v[q] > 0.f && cum + v[q] >= lo_t) atomicMin(&X.sh->bi[0], b);
    if (v[q] > 0.f && cum < hi_t) atomicMax(&X.sh->bi[1], b);
    cum += v[q];
  }
  __syncthreads();
  b_lo = X.sh->bi[0];
  b_hi = X.sh->bi[1];
  if (b_lo >= WBINS || b_hi < b_lo) {
    __syncthreads();
    return false;
  }
  int n = 0;
#pragma unroll
  for (int q = 0; q < BPT; ++q) {
    const int b = t * BPT + q;
    if (b >= b_lo && b <= b_hi) n += pmode ? (int)(wh[b] >> 11) + 1 : (int)wh[b];
  }
  n = bsum_i(n, X.sh->ri[1]);
  return n <= CAP;
}

// ---------------------------------------------------------------------------
// Bracket from a sampled weight histogram (one element in `scale`, excess-
// weighted counts relative to the stream's reference).  The kept set is the
// heaviest prefix reaching p of the row mass M, so its boundary bin b* is the
// first whose lighter part L(b* + 1) (the mass of bins b* + 1 ... WBINS - 1)
// is at most T1 = (1 - p) M.  L is estimated as scale times the sampled mass;
// the bracket runs from the point estimate of b* outward over the bins where
// that estimate is within a margin of T1 (four standard deviations of the
// sampling error).  Returns false when the bracket would hold more than CAP
// elements by the sample's count.  The exact band pass decides the result.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ bool wh_bracket_sampled(Ctx<DT>& Xr, double T1, float scale, int& b_lo,
                                                int& b_hi) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  const uint32_t* wh = X.wh;
  constexpr int BPT = WBINS / NT;
  const int t = threadIdx.x;
  // per bin: sampled mass (units of the reference weight) and sum of squares
  // bound (mass times the bin's upper weight)
  float v[BPT], q2[BPT];
  float s = 0.f, s2 = 0.f;
#pragma unroll
  for (int q = 0; q < BPT; ++q) {
    const int b = t * BPT + q;
    const float lo_w = (b == WBINS - 1) ? 0.f : exp2f((float)(WHOFF - b - 1) * (1.f / WHS));
    const float hi_w = exp2f((float)(WHOFF - b) * (1.f / WHS));
    v[q] = (float)wh[b] * (1.f / 2048.f) * lo_w;
    q2[q] = v[q] * hi_w;
    s += v[q];
    s2 += q2[q];
  }
  float tot, tot2;
  float c = bscan_excl<float>(s, X.sh->rf[0], tot);
  float c2 = bscan_excl<float>(s2, X.sh->rf[1], tot2);
  if (t == 0) {
    X.sh->bi[0] = WBINS;
    X.sh->bi[1] = WBINS;
    X.sh->bi[2] = -1;
  }
  __syncthreads();
  const float T1f = (float)T1;
  // L(b + 1) estimates and margins; the point estimate of b* and the
  // lightest bin where L(b + 1) is surely below T1
  float Lq[BPT], dq[BPT];
#pragma unroll
  for (int q = 0; q < BPT; ++q) {
    const int b = t * BPT + q;
    c += v[q];  // mass of bins 0 .. b
    c2 += q2[q];
    Lq[q] = scale * fmaxf(tot - c, 0.f);
    dq[q] = 4.f * scale * sqrtf(fmaxf(tot2 - c2, 0.f)) + 1e-3f * T1f;
    if (Lq[q] <= T1f) atomicMin(&X.sh->bi[0], b);
    if (Lq[q] + dq[q] <= T1f) atomicMin(&X.sh->bi[1], b);
  }
  __syncthreads();
  // the heaviest end: just below the last bin above the estimate where the
  // boundary is surely not (heavier bins carry the sampled heads, whose
  // sampling error says nothing about the bins near the boundary)
  const int bhat = X.sh->bi[0];
#pragma unroll
  for (int q = 0; q < BPT; ++q) {
    const int b = t * BPT + q;
    if (b < bhat && Lq[q] - dq[q] > T1f) atomicMax(&X.sh->bi[2], b);
  }
  __syncthreads();
  b_lo = X.sh->bi[2] + 1;
  b_hi = min(X.sh->bi[1], WBINS - 1);
  if (bhat >= WBINS || b_hi >= WBINS - 1 || b_hi < b_lo) {
    __syncthreads();
    return false;
  }
  int n = 0;
#pragma unroll
  for (int q = 0; q < BPT; ++q) {
    const int b = t * BPT + q;
    if (b >= b_lo && b <= b_hi) n += (int)(wh[b] >> 11) + 1;
  }
  n = bsum_i(n, X.sh->ri[1]);
  return (float)n * scale <= (float)CAP;
}

// ---------------------------------------------------------------------------
// Band-and-kept pass over a weight-histogram bracket [b_lo, b_hi]: legal
// elements of bins inside go to the list; those of bins above (larger
// weights) are kept: kept-mask bits, count, per-(chunk, warp) masses relative
// to the row maximum (nm) and their fixed-point total.  Every mask word is
// written (bracket elements still 0).
// ---------------------------------------------------------------------------
struct BandOut {
  int above_n;
  uint64_t above_q;  // fixed-point mass above the bracket (from the per-cell sums)
  float xa, xb;      // the bracket's value thresholds (band: xb <= x < xa)
};

// Fixed-point mass of the per-(chunk, warp) cells in sh->cmass: every cell
// converted on its own (integer operations) and the integers summed, so the
// total does not depend on which CTA computed which chunk or on the order.
template <int DT>
__device__ uint64_t cells_fixed_mass(Ctx<DT>& X) {
  uint64_t s = 0;
  for (int f = threadIdx.x; f < X.nch * NWARP; f += NT) s += to_fx(X.sh->cmass[f / NWARP][f % NWARP]);
  return bsum_q(s, X.sh->rq[1]);
}
// Smallest legal value x whose weight-histogram bin (relative to nref) is at
// most bmax, or +inf: the bin is monotone in x, so a bisection over the
// element type's order-preserving keys finds it.
template <int DT>
__device__ float first_value_in_bins(float c2, float nref, int bmax) {
  uint32_t lo = ElemT<DT>::KLOW - 1u, hi = ElemT<DT>::KPINF;  // sentinels: lo fails, hi passes
  while (hi - lo > 1u) {
    const uint32_t mid = lo + ((hi - lo) >> 1);
    if (wbin(key_value<DT>(mid), c2, nref) <= bmax) hi = mid;
    else lo = mid;
  }
  return (hi == ElemT<DT>::KPINF) ? INFINITY : key_value<DT>(hi);
}
// Value thresholds of a bracket [b_lo, b_hi]: above it <=> x >= xa; inside
// it <=> xb <= x < xa.
template <int DT>
__device__ void band_thresholds(float c2, float nref, int b_lo, int b_hi, float& xa, float& xb) {
  xa = first_value_in_bins<DT>(c2, nref, b_lo - 1);
  xb = first_value_in_bins<DT>(c2, nref, b_hi);
}

// Band classification of one staged chunk (the body of every band pass, the
// same arithmetic whichever CTA runs the chunk): bracket elements go to this
// CTA's list (sh->n), elements above the bracket get their kept-mask bits and
// count (nk) and add their weights relative to the row maximum (nm) to the
// returned per-thread mass.  The bracket is tested as two value thresholds
// (packed compares), and the chunk's bracket elements are appended behind
// one list reservation per warp.
template <int DT>
__device__ __forceinline__ float band_chunk(Ctx<DT>& X, const char* stage, int c, float xa,
                                            float xb, float c2, float nm, uint32_t* mrow, int& nk) {
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  const uint32_t xa2 = pack_down<DT>(xa), xb2 = pack_down<DT>(xb);
  int dummy = 0;
  float cs = 0.f;
  uint32_t cms[ITW];
  uint32_t anyb = 0u;
#pragma unroll
  for (int it = 0; it < ITW; ++it) {
    const int vi = warp_vec<DT>(it);
    const uint4 r = load_vec(X, stage, c, vi);
    const int id0 = c * CE + vi * EPV;
    const uint32_t kb = ge_mask<DT>(r, xa2, xa, dummy);
    cms[it] = ge_mask<DT>(r, xb2, xb, dummy) & ~kb;
    anyb |= cms[it];
    if (__any_sync(0xffffffffu, kb != 0u)) {
      float x[EPV];
      unpack<DT>(r, x);
#pragma unroll
      for (int q = 0; q < EPV; ++q)
        if ((kb >> q) & 1u) cs += fast_exp2(fmaf(x[q], c2, nm));
    }
    nk += __popc(kb);
    put_mask_word<DT>(X, mrow, kb, id0);
  }
  if (__any_sync(0xffffffffu, anyb != 0u)) {
    int cnt = 0;
#pragma unroll
    for (int it = 0; it < ITW; ++it) cnt += __popc(cms[it]);
    const int inc = warp_incl_scan(cnt);
    const int tot = __shfl_sync(0xffffffffu, inc, 31);
    int base = 0;
    if ((threadIdx.x & 31) == 31 && tot) base = atomicAdd(&X.sh->n, tot);
    base = __shfl_sync(0xffffffffu, base, 31);
    int pos = base + inc - cnt;
#pragma unroll
    for (int it = 0; it < ITW; ++it) {
      uint32_t cm = cms[it];
      if (!cm) continue;
      const int vi = warp_vec<DT>(it);
      const uint4 r = load_vec(X, stage, c, vi);
      const int id0 = c * CE + vi * EPV;
      while (cm) {
        const int q = __ffs(cm) - 1;
        cm &= cm - 1u;
        if (pos < CAP) {
          X.lk[pos] = bits_key<DT>(elem_bits_dyn<DT>(r, q));
          X.li[pos] = id0 + q;
        }
        ++pos;
      }
    }
  }
  return cs;
}

// The band pass of a row alone (no board slot): every chunk through the ring.
template <int DT>
__device__ __noinline__ BandOut band_kept_pass(Ctx<DT>& Xr, int b_lo, int b_hi, float nref, float nm) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* mrow = X.a->kept_mask ? X.a->kept_mask + (size_t)X.row * X.W : nullptr;
  if (threadIdx.x == 0) X.sh->n = 0;
  int nk = 0;
  float xa, xb;
  band_thresholds<DT>(X.c2, nref, b_lo, b_hi, xa, xb);
  ring_begin(X);
#pragma unroll 1
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = warp_wait(X, c);
    const float ws = warp_sum(band_chunk<DT>(X, stage, c, xa, xb, X.c2, nm, mrow, nk));
    if (lane == 0) X.sh->cmass[c][warp] = ws;
    warp_release(X, c);
  }
  BandOut o;
  o.above_n = bsum_i(nk, X.sh->ri[0]);
  o.above_q = 0;
  return o;
}

// The owner's side of a band job (slot j): the band pass over the chunks this
// CTA claims from the front (one block barrier per chunk).
// Returns the first helper chunk; the list (sh->n entries), the cells and
// above_n cover the owner's chunks.
template <int DT>
__device__ __noinline__ int band_owner_pass(Ctx<DT>& Xr, int j, int b_lo, int b_hi, float nref,
                                            float nm, int& above_n) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* mrow = X.a->kept_mask ? X.a->kept_mask + (size_t)X.row * X.W : nullptr;
  if (threadIdx.x == 0) X.sh->n = 0;
  int nk = 0;
  const float xa = X.a->board->hdr[j].xa, xb = X.a->board->hdr[j].xb;
  OwnerClaims<DT> oc;
  oc.start(X, &X.a->board->hdr[j], X.nch);
  // chunk 0 is the owner's; each further chunk is claimed only when the owner
  // is done with the previous one, so helpers (by then usually plentiful)
  // take most of the pass
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) X.sh->done[s] = 0;
    issue_chunk(X, 0, 0);
  }
  __syncthreads();
#pragma unroll 1
  for (int c = 0; c < X.nch; ++c) {
    if (c >= 1 && !oc.owns(X, c)) break;
    const char* stage = ring_wait(X, c);
    const float ws = warp_sum(band_chunk<DT>(X, stage, c, xa, xb, X.c2, nm, mrow, nk));
    if (lane == 0) X.sh->cmass[c][warp] = ws;
    __syncthreads();
    oc.decide(X, c + 1);
    __syncthreads();  // every thread reads the claim of chunk c + 1 after thread 0 made it
  }
  if (threadIdx.x == 0) X.sh->bi[1] = oc.first;
  above_n = bsum_i(nk, X.sh->ri[0]);
  const int first = X.sh->bi[1];
  __syncthreads();
  return first;
}

// ---------------------------------------------------------------------------
// Chunks of a published band pass (job j), run by a helper from chunk c on
// (the next chunk claimed and its copy issued while one is processed):
// band_chunk into this CTA's list area, the cells to the job; at the end the
// entries are copied behind one reservation in the job's list and the counts
// go to its header.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ void band_task(Ctx<DT>& Xr, int j, int c) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const KArgs& a = *X.a;
  Board* bd = a.board;
  volatile JobHdr* H = &bd->hdr[j];
  const int row = H->row;
  const float nm = H->nm, c2 = H->c2, xa = H->xa, xb = H->xb;
  X.row = row;
  X.src = reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)a.ld * ElemT<DT>::ES;
  X.bm = a.bitmask ? a.bitmask + (size_t)row * X.W : nullptr;
  X.c2 = c2;
  uint32_t* mrow = a.kept_mask ? a.kept_mask + (size_t)row * X.W : nullptr;
  int s = 0;
  if (threadIdx.x == 0) {
    issue_chunk(X, c, s);  // (the previous task's last barrier freed both stages)
    X.sh->n = 0;
  }
  __syncthreads();
  int nk = 0, ndone = 0;
#pragma unroll 1
  for (int it = 0;; ++it) {
    if (threadIdx.x == 0) {
      const int d = helper_claim(bd, j, X.sh->timeout);
      if (d >= 0) issue_chunk(X, d, s ^ 1);
      X.sh->bi[6 + (it & 1)] = d;
    }
    const char* stage = ring_wait_at(X, c, s);
    const float ws = warp_sum(band_chunk<DT>(X, stage, c, xa, xb, c2, nm, mrow, nk));
    if (lane == 0) bd->cmass[j][c * NWARP + warp] = ws;
    ++ndone;
    __syncthreads();  // the stage is free, the next claim visible
    c = X.sh->bi[6 + (it & 1)];
    if (c < 0) break;
    s ^= 1;
  }
  nk = __reduce_add_sync(0xffffffffu, nk);
  if (lane == 0 && nk) atomicAdd((int*)&H->above_n, nk);
  __syncthreads();
  const int n = X.sh->n;
  if (threadIdx.x == 0) X.sh->bi[4] = n ? atomicAdd((int*)&H->list_n, n) : 0;
  __syncthreads();
  const int base = X.sh->bi[4];
  const int ncopy = min(min(n, CAP), CAP - base);
  for (int i = threadIdx.x; i < ncopy; i += NT) {
    bd->lk[j][base + i] = X.lk[i];
    bd->li[j][base + i] = X.li[i];
  }
  if (threadIdx.x == 0 && X.sh->timeout) atomicOr((int*)&H->bad, 1);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd((int*)&H->done, ndone);
}

// ---------------------------------------------------------------------------
// Descent histogram pass over the legal elements whose key has the plen-bit
// prefix `prefix`: bins of key bits [shift, shift + nbits).  MASS histograms
// count only S_k members (vK, idK) and also add their fixed-point masses.
// Elements above the prefix region are summed into above_c / above_m.
// ---------------------------------------------------------------------------
template <int DT, bool MASS>
__device__ __noinline__ void hist_pass(Ctx<DT>& Xr, uint32_t prefix, int plen, int shift, int nbits,
                                       uint32_t vK, int idK, float nm, uint32_t& above_c,
                                       uint64_t& above_m) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE, SIG = ElemT<DT>::SIG;
  const int nb = 1 << nbits;
  uint32_t* hc = X.lk;
  uint64_t* hm = reinterpret_cast<uint64_t*>(X.lk + HBINS);
  __syncthreads();
  for (int b = threadIdx.x; b < nb; b += NT) {
    hc[b] = 0u;
    hm[b] = 0;
  }
  const uint32_t lo_key = plen ? (prefix << (SIG - plen)) : 0u;
  const float lo_val = (plen && lo_key > ElemT<DT>::KLOW) ? key_value<DT>(lo_key) : -INFINITY;
  uint32_t ac = 0u;
  uint64_t am = 0;
  ring_begin(X);
#pragma unroll 1
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = warp_wait(X, c);
#pragma unroll 1
    for (int it = 0; it < ITW; ++it) {
      const int vi = warp_vec<DT>(it);
      const uint4 r = load_vec(X, stage, c, vi);
      if (!(vmax_f<DT>(r) >= lo_val)) continue;  // the whole vector is below the region
      const int id0 = c * CE + vi * EPV;
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        const uint32_t b = elem_bits<DT>(r, j);
        const float x = bits_value<DT>(b);
        if (!(x > -INFINITY)) continue;
        const uint32_t k = bits_key<DT>(b);
        if (MASS && !in_set(k, id0 + j, vK, idK)) continue;
        const uint32_t top = plen ? (k >> (SIG - plen)) : 0u;
        if (top < prefix) continue;
        const uint64_t w = MASS ? fx_weight(x, X.c2, nm) : 1ull;
        if (top == prefix) {
          const int d = (int)((k >> shift) & (uint32_t)(nb - 1));
          atomicAdd(&hc[d], 1u);
          if (MASS) smem_add_u64(&hm[d], w);
        } else {
          ++ac;
          am += w;
        }
      }
    }
    warp_release(X, c);
  }
  above_c = (uint32_t)bsum_i((int)ac, X.sh->ri[0]);
  above_m = bsum_q(am, X.sh->rq[1]);
}

// The bin (scanning from the largest digit down) where the running weight,
// starting at `above`, reaches target.
struct Cross {
  int bin, ok;
  uint64_t before, val;
  uint32_t cnt;
};
template <int DT, bool MASS>
__device__ __noinline__ Cross hist_cross(Ctx<DT>& Xr, int nbits, uint64_t above, uint64_t target) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  const int nb = 1 << nbits;
  const uint32_t* hc = X.lk;
  const uint64_t* hm = reinterpret_cast<const uint64_t*>(X.lk + HBINS);
  const int bpt = nb >= NT ? nb / NT : 1;
  const int t = threadIdx.x;
  const int hi = nb - 1 - t * bpt;  // this thread's bins: hi, hi - 1, ..., hi - bpt + 1
  uint64_t loc = 0;
  if (hi >= 0)
    for (int q = 0; q < bpt; ++q) loc += MASS ? hm[hi - q] : (uint64_t)hc[hi - q];
  uint64_t tot;
  const uint64_t ex = bscan_excl<uint64_t>(loc, X.sh->rq[0], tot);
  if (t == 0) X.sh->bi[0] = -1;
  __syncthreads();
  if (hi >= 0) {
    uint64_t cum = above + ex;
    for (int q = 0; q < bpt; ++q) {
      const int b = hi - q;
      const uint64_t v = MASS ? hm[b] : (uint64_t)hc[b];
      if (v > 0 && cum < target && cum + v >= target) {
        X.sh->bi[0] = b;
        X.sh->bq[0] = cum;
        X.sh->bq[1] = v;
        X.sh->bu[0] = hc[b];
      }
      cum += v;
    }
  }
  __syncthreads();
  Cross o;
  o.bin = X.sh->bi[0];
  o.ok = o.bin >= 0;
  o.before = X.sh->bq[0];
  o.val = X.sh->bq[1];
  o.cnt = X.sh->bu[0];
  return o;
}

// Sum of a MASS histogram (the mass of S_k at the first descent level).
template <int DT>
__device__ uint64_t hist_total(Ctx<DT>& X, int nbits) {
  const uint64_t* hm = reinterpret_cast<const uint64_t*>(X.lk + HBINS);
  uint64_t s = 0;
  for (int b = threadIdx.x; b < (1 << nbits); b += NT) s += hm[b];
  return bsum_q(s, X.sh->rq[1]);
}

// Band pass: every legal element with lo <= key < hi (MASS: every S_k member)
// goes to the list; legal elements with key >= hi are counted (and, MASS, the
// S_k members' masses summed).
template <int DT, bool MASS>
__device__ __noinline__ void band_pass(Ctx<DT>& Xr, uint32_t lo, uint64_t hi, uint32_t vK, int idK,
                                       float nm, uint32_t& above_c, uint64_t& above_m) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  const float lo_val = (lo > ElemT<DT>::KLOW) ? key_value<DT>(lo) : -INFINITY;
  if (threadIdx.x == 0) X.sh->n = 0;
  uint32_t ac = 0u;
  uint64_t am = 0;
  ring_begin(X);
#pragma unroll 1
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = warp_wait(X, c);
#pragma unroll 1
    for (int it = 0; it < ITW; ++it) {
      const int vi = warp_vec<DT>(it);
      const uint4 r = load_vec(X, stage, c, vi);
      const int id0 = c * CE + vi * EPV;
      uint32_t cm = 0u;
      if (vmax_f<DT>(r) >= lo_val) {
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
          const uint32_t b = elem_bits<DT>(r, j);
          const float x = bits_value<DT>(b);
          if (!(x > -INFINITY)) continue;
          const uint32_t k = bits_key<DT>(b);
          if ((uint64_t)k >= hi) {
            ++ac;
            if (MASS && in_set(k, id0 + j, vK, idK)) am += fx_weight(x, X.c2, nm);
          } else if (k >= lo && (!MASS || in_set(k, id0 + j, vK, idK))) {
            cm |= 1u << j;  // a MASS band holds S_k members only, as its histogram
          }
        }
      }
      if (__any_sync(0xffffffffu, cm != 0u)) list_append(X, r, id0, cm);
    }
    warp_release(X, c);
  }
  above_c = (uint32_t)bsum_i((int)ac, X.sh->ri[0]);
  above_m = bsum_q(am, X.sh->rq[1]);
}

// ---------------------------------------------------------------------------
// Tie pass: id of the rank-th (1-based) legal element, in id order, among
// those with key v that belong to S_k (vK, idK).
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ int tie_pass(Ctx<DT>& Xr, uint32_t v, int rank, uint32_t vK, int idK) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int c = threadIdx.x; c < X.nch; c += NT) X.sh->ctie[c] = 0;
  ring_begin(X);
#pragma unroll 1
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = warp_wait(X, c);
    int cnt = 0;
#pragma unroll 1
    for (int it = 0; it < ITW; ++it) {
      const int vi = warp_vec<DT>(it);
      const uint4 r = load_vec(X, stage, c, vi);
      const int id0 = c * CE + vi * EPV;
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        const uint32_t b = elem_bits<DT>(r, j);
        if (!(bits_value<DT>(b) > -INFINITY)) continue;
        const uint32_t k = bits_key<DT>(b);
        cnt += (k == v && in_set(k, id0 + j, vK, idK)) ? 1 : 0;
      }
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (lane == 0 && cnt) atomicAdd(&X.sh->ctie[c], cnt);
    warp_release(X, c);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int cum = 0, cs = -1;
    for (int c = 0; c < X.nch; ++c) {
      if (cum + X.sh->ctie[c] >= rank) {
        cs = c;
        break;
      }
      cum += X.sh->ctie[c];
    }
    X.sh->bi[2] = cs;
    X.sh->bi[3] = rank - cum;
    X.sh->bi[4] = NOID;
  }
  __syncthreads();
  const int cs = X.sh->bi[2];
  const int want = X.sh->bi[3];
  if (cs < 0) return NOID;
  // rank the ties of chunk cs in element order (warp, it, lane, element)
  __syncthreads();
  if (threadIdx.x == 0) issue_chunk(X, cs, cs % NSTAGE);
  const char* stage = ring_wait(X, cs);
  int cnt[ITW];
  uint32_t bits[ITW];
#pragma unroll
  for (int it = 0; it < ITW; ++it) {
    const int vi = warp_vec<DT>(it);
    const uint4 r = load_vec(X, stage, cs, vi);
    const int id0 = cs * CE + vi * EPV;
    uint32_t bb = 0u;
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      const uint32_t b = elem_bits<DT>(r, j);
      if (!(bits_value<DT>(b) > -INFINITY)) continue;
      const uint32_t k = bits_key<DT>(b);
      if (k == v && in_set(k, id0 + j, vK, idK)) bb |= 1u << j;
    }
    bits[it] = bb;
    cnt[it] = __popc(bb);
  }
  int incl[ITW], wt = 0, tw[ITW];
#pragma unroll
  for (int it = 0; it < ITW; ++it) {
    incl[it] = warp_incl_scan(cnt[it]);
    tw[it] = __shfl_sync(0xffffffffu, incl[it], 31);
    wt += tw[it];
  }
  __syncthreads();
  if (lane == 0) X.sh->ri[1][warp] = wt;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += X.sh->ri[1][w];
#pragma unroll
  for (int it = 0; it < ITW; ++it) {
    const int b0 = base + incl[it] - cnt[it];
    if (want > b0 && want <= b0 + cnt[it]) {
      uint32_t bb = bits[it];
      for (int q = 1; q < want - b0; ++q) bb &= bb - 1u;
      X.sh->bi[4] = cs * CE + warp_vec<DT>(it) * EPV + (__ffs(bb) - 1);
    }
    base += tw[it];
  }
  __syncthreads();
  return X.sh->bi[4];
}

// ---------------------------------------------------------------------------
// Kept pass: the kept set is {legal, key > vF} + {legal, key == vF, id <= idF}.
// Writes the kept mask, counts the kept elements and records per-(chunk,
// warp) masses (weights relative to ref: nm = -ref * log2(e) / T).
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ int kept_pass(Ctx<DT>& Xr, uint32_t vF, int idF, float nm) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* mrow = X.a->kept_mask ? X.a->kept_mask + (size_t)X.row * X.W : nullptr;
  const float v_val = (vF >= ElemT<DT>::KLOW) ? key_value<DT>(vF) : -INFINITY;
  int nk = 0;
  ring_begin(X);
#pragma unroll 1
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = warp_wait(X, c);
    float cs = 0.f;
#pragma unroll 1
    for (int it = 0; it < ITW; ++it) {
      const int vi = warp_vec<DT>(it);
      const uint4 r = load_vec(X, stage, c, vi);
      const int id0 = c * CE + vi * EPV;
      uint32_t kb = 0u;
      if (vmax_f<DT>(r) >= v_val) {
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
          const uint32_t b = elem_bits<DT>(r, j);
          const float x = bits_value<DT>(b);
          if (!(x > -INFINITY)) continue;
          if (in_set(bits_key<DT>(b), id0 + j, vF, idF)) {
            kb |= 1u << j;
            cs += fast_exp2(fmaf(x, X.c2, nm));
          }
        }
      }
      nk += __popc(kb);
      put_mask_word<DT>(X, mrow, kb, id0);
    }
    const float ws = warp_sum(cs);
    if (lane == 0) X.sh->cmass[c][warp] = ws;
    warp_release(X, c);
  }
  return bsum_i(nk, X.sh->ri[0]);
}

// ---------------------------------------------------------------------------
// Inverse-CDF draw over a kept set recorded per (chunk, warp) cell by
// kept_pass, band_kept_pass or the keep-all stream (plus, when extra is given,
// fixed-point masses of kept list entries per cell): T = u * (sum of the cell
// masses, in order); the cell holding T is re-read and scanned in id order.
// Returns the token (the last kept element of that cell if rounding leaves T
// past its end) and the total mass in mtot.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __noinline__ int sample_tail(Ctx<DT>& Xr, double u, uint32_t vF, int idF, float nm,
                                        const uint64_t* extra, double& mtot) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nf = X.nch * NWARP;
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) X.sh->bi[5] = -1;
    __syncwarp();
    const int per = (nf + 31) / 32;
    const int f0 = lane * per, f1 = min(nf, f0 + per);
    // cell masses as fixed-point integers in units of 2^-sc, the scale taken
    // from the largest cell so that the total of all cells stays below 2^61:
    // exact sums and compares, and no fp64 arithmetic (slow on this GPU)
    float mx = 0.f;
    for (int f = f0; f < f1; ++f) {
      float v = X.sh->cmass[f / NWARP][f % NWARP];
      if (extra) v += __ull2float_rz(extra[f] >> 20) * (1.f / 1048576.f);
      mx = fmaxf(mx, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // every cell < 2^(ex + 1); at most 2^11 cells
    const int ex = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;
    const int sc = max(0, min(61 - 11 - (ex + 1), 100));
    auto cell_fx = [&](int f) -> uint64_t {
      uint64_t v = fx_scaled(X.sh->cmass[f / NWARP][f % NWARP], sc);
      if (extra) v += (sc >= FX) ? (extra[f] << (sc - FX)) : (extra[f] >> (FX - sc));
      return v;
    };
    uint64_t s = 0;
    for (int f = f0; f < f1; ++f) s += cell_fx(f);
    const uint64_t inc = warp_incl_scan(s);
    const uint64_t tot = __shfl_sync(0xffffffffu, inc, 31);
    // T = u * tot with u = k * 2^-24
    const uint64_t k24 = (uint64_t)(u * 16777216.0);
    const uint64_t T = __umul64hi(tot, k24 << 40);
    uint64_t cum = inc - s;
    int hit = -1, last = -1;
    uint64_t before = 0;
    for (int f = f0; f < f1; ++f) {
      const uint64_t v = cell_fx(f);
      if (hit < 0 && v > 0 && cum <= T && cum + v > T) {
        hit = f;
        before = cum;
      }
      if (v > 0) last = f;
      cum += v;
    }
    // the first cell in order holding T; if rounding leaves none, the last
    // one with mass
    const uint32_t bal = __ballot_sync(0xffffffffu, hit >= 0);
    const int lst = (int)__reduce_max_sync(0xffffffffu, (uint32_t)(last + 1)) - 1;
    if (bal) {
      const int src = __ffs(bal) - 1;
      if (lane == src) {
        X.sh->bi[5] = hit;
        X.sh->bd[0] = ldexp((double)(T - before), -sc);
      }
    } else if (lane == 0) {
      X.sh->bi[5] = lst;
      X.sh->bd[0] = 1e300;  // past the end: take the last kept element
    }
    if (lane == 0) X.sh->bd[1] = ldexp((double)tot, -sc);
  }
  __syncthreads();
  mtot = X.sh->bd[1];
  const int f = X.sh->bi[5];
  if (f < 0) return -1;
  const int cs = f / NWARP, ws = f % NWARP;
  const double Tl = X.sh->bd[0];
  if (threadIdx.x == 0) issue_chunk(X, cs, cs % NSTAGE);
  const char* stage = ring_wait(X, cs);
  // the cell's scan, one vector per thread (its VW vectors are consecutive
  // in id order), in fp32 relative to the cell start (its error is a few fp32
  // ulps of the cell's mass; fp64 arithmetic is slow here)
  constexpr int VW = ElemT<DT>::VW;
  const float Tf = (float)Tl;
  const int t = threadIdx.x;
  float w[EPV];
  int id0 = 0, lastk = -1;
#pragma unroll
  for (int j = 0; j < EPV; ++j) w[j] = 0.f;
  if (t < VW) {
    const int vi = ws * VW + t;
    const uint4 r = load_vec(X, stage, cs, vi);
    id0 = cs * CE + vi * EPV;
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      const uint32_t b = elem_bits<DT>(r, j);
      const float x = bits_value<DT>(b);
      if (x > -INFINITY && in_set(bits_key<DT>(b), id0 + j, vF, idF)) {
        w[j] = fast_exp2(fmaf(x, X.c2, nm));
        lastk = id0 + j;
      }
    }
  }
  const float vs = tree_sum<EPV>(w);
  float tot;
  const float pre = bscan_excl<float>(vs, X.sh->rf[0], tot);
  if (t == 0) {
    X.sh->bi[6] = NOID;
    X.sh->bi[2] = -1;
  }
  __syncthreads();
  // the first vector in id order whose end passes T (the smallest id wins)
  if (vs > 0.f && pre + vs > Tf) {
    float cum = pre;
    int tok = -1, lastj = -1;
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      if (w[j] > 0.f) lastj = id0 + j;
      cum += w[j];
      if (tok < 0 && w[j] > 0.f && cum > Tf) tok = id0 + j;
    }
    atomicMin(&X.sh->bi[6], tok >= 0 ? tok : lastj);
  }
  if (lastk >= 0) atomicMax(&X.sh->bi[2], lastk);
  __syncthreads();
  const int found = X.sh->bi[6];
  const int res = (found != NOID) ? found : X.sh->bi[2];
  __syncthreads();
  return res;
}

// Probabilities of a boundary-decided kept set: the contract's weight
// expf(fl32(x / T) - fl32(ref / T)) over mtot (the kept mass relative to ref)
// for kept elements, 0 elsewhere.
template <int DT>
__device__ __noinline__ void probs_pass(Ctx<DT>& Xr, uint32_t vF, int idF, float zr, double mtot) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  float* prow = X.a->probs + (size_t)X.row * X.V;
  ring_begin(X);
#pragma unroll 1
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = warp_wait(X, c);
#pragma unroll 1
    for (int it = 0; it < ITW; ++it) {
      const int vi = warp_vec<DT>(it);
      const uint4 r = load_vec(X, stage, c, vi);
      const int id0 = c * CE + vi * EPV;
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        if (id0 + j >= X.V) break;
        const uint32_t b = elem_bits<DT>(r, j);
        const float x = bits_value<DT>(b);
        float pr = 0.f;
        if (x > -INFINITY && in_set(bits_key<DT>(b), id0 + j, vF, idF))
          pr = (float)((double)expf(__fdiv_rn(x, X.temp) - zr) / mtot);
        prow[id0 + j] = pr;
      }
    }
    warp_release(X, c);
  }
}

}  // namespace smp
