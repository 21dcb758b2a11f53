// smp_stream_main.cuh -- per-row driver of the streaming kernel (see
// smp_stream.cuh for the pipeline and the helpers).  Every pass is an
// explicit loop over the ring so that accumulators stay in registers.
#pragma once

namespace smp {

// Legal-masked vector of chunk c at stage-local vector index v.
template <int DT>
__device__ __forceinline__ uint4 load_masked(const Ctx<DT>& X, const char* stage, int c, int v) {
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  uint4 r = *reinterpret_cast<const uint4*>(stage + (size_t)v * 16);
  if (X.bm) {
    const uint32_t lb = mask_bits(X, c * CE + v * EPV);
    if (lb != (1u << EPV) - 1u) r = apply_mask<DT>(r, lb);
  }
  return r;
}

// Mask word assembly: lane l holds EPV consecutive bits; LPW lanes form one
// 32-bit word (ordered warp mapping), written by the first lane of the group.
template <int DT>
__device__ __forceinline__ void store_mask_word(uint32_t* mrow, int W, int gid0, uint32_t bits) {
  constexpr int EPV = ElemT<DT>::EPV;
  constexpr int LPW = 32 / EPV;
  const int lane = threadIdx.x & 31;
  uint32_t word = bits << (EPV * (lane % LPW));
#pragma unroll
  for (int o = 1; o < LPW; o <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, o);
  const int gw = gid0 >> 5;
  if ((lane % LPW) == 0 && gw < W) mrow[gw] = word;
}

// Copies of key kB in chunk c: each warp's starting rank in the row (id
// order) given tie_base copies in earlier chunks; returns the chunk's total.
template <int DT>
__device__ __forceinline__ int tie_prefix(const Ctx<DT>& X, const char* stage, int c, uint32_t kB,
                                          int tie_base, int& warp_start) {
  constexpr int EPV = ElemT<DT>::EPV, ITW = ElemT<DT>::ITW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float vB = key_to_float(kB);
  int t = 0;
  for (int it = 0; it < ITW; ++it) {
    const uint4 r = load_masked(X, stage, c, warp_vec<DT>(it));
    if (!__any_sync(0xffffffffu, vmax<DT>(r) >= vB)) continue;
    float x[EPV];
    unpack<DT>(r, x);
#pragma unroll
    for (int j = 0; j < EPV; ++j) t += (!is_neg_inf(x[j]) && fkey(x[j]) == kB) ? 1 : 0;
  }
  t = __reduce_add_sync(0xffffffffu, t);
  if (lane == 0) X.sh->wst[warp] = t;
  __syncthreads();
  int start = tie_base, tot = 0;
  for (int w = 0; w < NWARP; ++w) {
    if (w < warp) start += X.sh->wst[w];
    tot += X.sh->wst[w];
  }
  __syncthreads();
  warp_start = start;
  return tot;
}

// Membership bits of one vector: key > kB, or a copy of kB whose rank in the
// row is below nB (all = every legal element).  Warp-collective.
template <int DT>
__device__ __forceinline__ uint32_t classify(const float (&x)[ElemT<DT>::EPV], uint32_t kB, int nB,
                                             bool all, int& tie_run) {
  constexpr int EPV = ElemT<DT>::EPV;
  uint32_t bits = 0u, tbits = 0u;
#pragma unroll
  for (int j = 0; j < EPV; ++j) {
    if (is_neg_inf(x[j])) continue;
    if (all) {
      bits |= 1u << j;
      continue;
    }
    const uint32_t k = fkey(x[j]);
    if (k > kB) bits |= 1u << j;
    else if (k == kB) tbits |= 1u << j;
  }
  if (!all) {
    const int nt = __popc(tbits);
    const int incl = warp_incl_scan(nt);
    int rr = tie_run + incl - nt;
#pragma unroll
    for (int j = 0; j < EPV; ++j)
      if ((tbits >> j) & 1u) {
        if (rr < nB) bits |= 1u << j;
        ++rr;
      }
    tie_run += __shfl_sync(0xffffffffu, incl, 31);
  }
  return bits;
}

// Fast weight relative to the row max: 2^((x - max) * log2(e) / T).
template <int DT>
__device__ __forceinline__ float fastw(const Ctx<DT>& X, float x) {
  return fast_exp2((x - X.gmax) * X.c2);
}

// ---------------------------------------------------------------------------
// Kept set not gathered (all legal tokens, or the refinement path): a
// streamed pass writes the mask words and the per-chunk member mass, and
// records the copies of kB before each chunk (for the tie quota of the draw).
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ int member_pass(Ctx<DT>& X, uint32_t kB, int nB, bool all) {
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE, ITW = ElemT<DT>::ITW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* mrow = X.a->kept_mask ? X.a->kept_mask + (size_t)X.row * X.W : nullptr;
  const float vB = all ? -INFINITY : key_to_float(kB);
  int tie_base = 0, count = 0;
  ring_begin(X);
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = ring_wait(X, c);
    if (threadIdx.x == 0) X.sh->chunk_ties[c] = tie_base;
    int tie_run = 0, ties = 0;
    if (!all) ties = tie_prefix(X, stage, c, kB, tie_base, tie_run);
    float msum = 0.f;
    int cnt = 0;
    for (int it = 0; it < ITW; ++it) {
      const int v = warp_vec<DT>(it);
      const uint4 r = load_masked(X, stage, c, v);
      uint32_t bits = 0u;
      if (all || __any_sync(0xffffffffu, vmax<DT>(r) >= vB)) {
        float x[EPV];
        unpack<DT>(r, x);
        bits = classify<DT>(x, kB, nB, all, tie_run);
#pragma unroll
        for (int j = 0; j < EPV; ++j)
          if ((bits >> j) & 1u) msum += fastw(X, x[j]);
        cnt += __popc(bits);
      }
      if (mrow) store_mask_word<DT>(mrow, X.W, c * CE + v * EPV, bits);
    }
    tie_base += ties;
    const double wm = warp_sum((double)msum);
    const int wc = __reduce_add_sync(0xffffffffu, cnt);
    if (lane == 0) {
      X.sh->bd[11][warp] = wm;
      X.sh->bi[11][warp] = wc;
    }
    __syncthreads();
    double m = 0.0;
    int cc = 0;
    for (int w = 0; w < NWARP; ++w) {
      m += X.sh->bd[11][w];
      cc += X.sh->bi[11][w];
    }
    if (threadIdx.x == 0) X.sh->chunk_mass[c] = m;
    count += cc;
    ring_release(X, c);
  }
  __syncthreads();
  return count;
}

// Load chunk c into stage 0 with plain loads (the ring is idle).
template <int DT>
__device__ __forceinline__ void load_chunk_plain(const Ctx<DT>& X, int c) {
  constexpr int CE = ElemT<DT>::CE, ES = ElemT<DT>::ES;
  char* stage = X.ring;
  const int ne = min(CE, X.V - c * CE);
  const char* g = X.src + (size_t)c * CE * ES;
  for (int e = threadIdx.x; e < CE; e += NT) {
    if constexpr (ES == 4) {
      reinterpret_cast<uint32_t*>(stage)[e] =
          (e < ne) ? reinterpret_cast<const uint32_t*>(g)[e] : 0xff800000u;
    } else {
      constexpr unsigned short NEG = (DT == DT_BF16) ? 0xff80u : 0xfc00u;
      reinterpret_cast<unsigned short*>(stage)[e] =
          (e < ne) ? reinterpret_cast<const unsigned short*>(g)[e] : NEG;
    }
  }
  __syncthreads();
}

// The draw for a kept set known chunk by chunk (chunk_mass relative to the
// row max, chunk_ties = copies of kB before each chunk): the chunk holding
// u * M_p is reloaded; its warps' masses locate the warp, then the lane and
// the element, in id order.
template <int DT>
__device__ __forceinline__ int draw_streamed(Ctx<DT>& X, uint32_t kB, int nB, bool all, double Mp,
                                             double u) {
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE, ITW = ElemT<DT>::ITW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const double T = u * Mp;
  int cs = -1, lastc = -1;
  double pre = 0.0, P = 0.0, Plast = 0.0;
  for (int c = 0; c < X.nch; ++c) {
    const double m = X.sh->chunk_mass[c];
    if (m > 0.0) {
      lastc = c;
      Plast = pre;
    }
    if (cs < 0 && m > 0.0 && pre + m > T) {
      cs = c;
      P = pre;
    }
    pre += m;
  }
  if (cs < 0) {
    cs = lastc;
    P = Plast;
  }
  if (cs < 0) return -1;
  __syncthreads();
  load_chunk_plain(X, cs);
  const char* stage = X.ring;
  const float vB = all ? -INFINITY : key_to_float(kB);
  int warp_start = 0;
  if (!all) tie_prefix(X, stage, cs, kB, X.sh->chunk_ties[cs], warp_start);
  // per-warp member mass of the chunk
  {
    int tie_run = warp_start;
    float msum = 0.f;
    int cnt = 0;
    for (int it = 0; it < ITW; ++it) {
      const uint4 r = load_masked(X, stage, cs, warp_vec<DT>(it));
      if (!all && !__any_sync(0xffffffffu, vmax<DT>(r) >= vB)) continue;
      float x[EPV];
      unpack<DT>(r, x);
      const uint32_t bits = classify<DT>(x, kB, nB, all, tie_run);
#pragma unroll
      for (int j = 0; j < EPV; ++j)
        if ((bits >> j) & 1u) msum += fastw(X, x[j]);
      cnt += __popc(bits);
    }
    const double wm = warp_sum((double)msum);
    const int wc = __reduce_add_sync(0xffffffffu, cnt);
    if (lane == 0) {
      X.sh->bd[12][warp] = wm;
      X.sh->bi[12][warp] = wc;
    }
    __syncthreads();
  }
  int tw = -1, lw = -1;
  double wpre = P, tbase = 0.0, lbase = P;
  for (int w = 0; w < NWARP; ++w) {
    if (X.sh->bi[12][w] > 0) {
      lw = w;
      lbase = wpre;
    }
    if (tw < 0 && X.sh->bd[12][w] > 0.0 && wpre + X.sh->bd[12][w] > T) {
      tw = w;
      tbase = wpre;
    }
    wpre += X.sh->bd[12][w];
  }
  if (tw < 0) {
    tw = lw;
    tbase = lbase;
  }
  if (warp == tw) {
    int tie_run = warp_start;
    double base = tbase;
    int found = -1, lastm = -1;
    for (int it = 0; it < ITW && found < 0; ++it) {
      const int v = warp_vec<DT>(it);
      const uint4 r = load_masked(X, stage, cs, v);
      if (!all && !__any_sync(0xffffffffu, vmax<DT>(r) >= vB)) continue;
      float x[EPV];
      unpack<DT>(r, x);
      const uint32_t bits = classify<DT>(x, kB, nB, all, tie_run);
      float wl[EPV];
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        wl[j] = ((bits >> j) & 1u) ? fastw(X, x[j]) : 0.f;
        ls += wl[j];
      }
      const float li = warp_incl_scan(ls);
      const float tot = __shfl_sync(0xffffffffu, li, 31);
      const bool cross = (base + (double)li > T) && ls > 0.f;
      const unsigned cm = __ballot_sync(0xffffffffu, cross);
      const int gid0 = cs * CE + v * EPV;
      if (bits) lastm = gid0 + (31 - __clz(bits));
      lastm = (int)__reduce_max_sync(0xffffffffu, (unsigned)(lastm + 1)) - 1;
      if (cm) {
        const int fl = __ffs(cm) - 1;
        if (lane == fl) {
          double cum = base + (double)(li - ls);
          int tok = -1, lastl = -1;
#pragma unroll
          for (int j = 0; j < EPV; ++j)
            if ((bits >> j) & 1u) {
              cum += (double)wl[j];
              lastl = gid0 + j;
              if (tok < 0 && cum > T) tok = lastl;
            }
          found = (tok >= 0) ? tok : lastl;
        }
        found = __shfl_sync(0xffffffffu, found, fl);
      }
      base += (double)tot;
    }
    if (lane == 0) X.sh->flag[7] = (found >= 0) ? found : lastm;
  }
  __syncthreads();
  return X.sh->flag[7];
}

// Probabilities for a kept set known chunk by chunk (test aid): w / M_p.
template <int DT>
__device__ __forceinline__ void probs_pass(Ctx<DT>& X, uint32_t kB, int nB, bool all, double Mp) {
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE, ITW = ElemT<DT>::ITW;
  float* prow = X.a->probs + (size_t)X.row * X.V;
  const float inv = (float)(1.0 / Mp);
  int tie_base = 0;
  ring_begin(X);
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = ring_wait(X, c);
    int tie_run = 0, ties = 0;
    if (!all) ties = tie_prefix(X, stage, c, kB, tie_base, tie_run);
    for (int it = 0; it < ITW; ++it) {
      const int v = warp_vec<DT>(it);
      const uint4 r = load_masked(X, stage, c, v);
      float x[EPV];
      unpack<DT>(r, x);
      const uint32_t bits = classify<DT>(x, kB, nB, all, tie_run);
      const int gid0 = c * CE + v * EPV;
#pragma unroll
      for (int j = 0; j < EPV; ++j)
        if (gid0 + j < X.V) prow[gid0 + j] = ((bits >> j) & 1u) ? weight(X, x[j]) * inv : 0.f;
    }
    tie_base += ties;
    ring_release(X, c);
  }
}

// ---------------------------------------------------------------------------
// Exact multi-pivot refinement (full-row fallback).  Window [lo, hi] in key
// space over the domain (legal; with a limit, the members of S_k: key > kK or
// one of the first nK copies of kK); one streamed pass counts (and weighs)
// the window against NPIV pivots in registers; the window shrinks to the
// sub-window holding the target.
// ---------------------------------------------------------------------------
struct Win {
  uint32_t lo, hi;
  long long above_cnt;
  double above_mass;
  long long n_in;
};

// Domain bits of one vector inside [lo, hi] (warp-collective when limited).
template <int DT>
__device__ __forceinline__ uint32_t window_bits(const float (&x)[ElemT<DT>::EPV], uint32_t lo,
                                                uint32_t hi, bool limited, uint32_t kK, int nK,
                                                int& tie_run) {
  constexpr int EPV = ElemT<DT>::EPV;
  uint32_t dom = 0u;
  if (limited) {
    dom = classify<DT>(x, kK, nK, false, tie_run);
  } else {
#pragma unroll
    for (int j = 0; j < EPV; ++j)
      if (!is_neg_inf(x[j])) dom |= 1u << j;
  }
  uint32_t wb = 0u;
#pragma unroll
  for (int j = 0; j < EPV; ++j) {
    if (!((dom >> j) & 1u)) continue;
    const uint32_t k = fkey(x[j]);
    if (k >= lo && k <= hi) wb |= 1u << j;
  }
  return wb;
}

template <int DT>
__device__ __forceinline__ void refine_pass(Ctx<DT>& X, Win& Wd, bool mass, long long kneed,
                                            double& target, double target_frac, bool limited,
                                            uint32_t kK, int nK) {
  constexpr int EPV = ElemT<DT>::EPV, ITW = ElemT<DT>::ITW;
  const uint32_t lo = Wd.lo, hi = Wd.hi;
  const unsigned long long span = (unsigned long long)(hi - lo) + 1ull;
  uint32_t piv[NPIV + 1];
  piv[0] = lo;
#pragma unroll
  for (int m = 1; m <= NPIV; ++m) piv[m] = lo + (uint32_t)((span * m) / (NPIV + 1));
  int cnt[NPIV + 1];
  float msum[NPIV + 1];
#pragma unroll
  for (int m = 0; m <= NPIV; ++m) {
    cnt[m] = 0;
    msum[m] = 0.f;
  }
  const float vlo = key_to_float(lo);
  int tie_base = 0;
  ring_begin(X);
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = ring_wait(X, c);
    int tie_run = 0, ties = 0;
    if (limited) ties = tie_prefix(X, stage, c, kK, tie_base, tie_run);
    for (int it = 0; it < ITW; ++it) {
      const uint4 r = load_masked(X, stage, c, warp_vec<DT>(it));
      // vectors below the window hold no window member and (the window starts
      // at kK or above) no copy of kK that a later rank depends on
      if (!__any_sync(0xffffffffu, vmax<DT>(r) >= vlo)) continue;
      float x[EPV];
      unpack<DT>(r, x);
      const uint32_t wb = window_bits<DT>(x, lo, hi, limited, kK, nK, tie_run);
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        if (!((wb >> j) & 1u)) continue;
        const uint32_t k = fkey(x[j]);
        const float w = mass ? fastw(X, x[j]) : 0.f;
#pragma unroll
        for (int m = 0; m <= NPIV; ++m)
          if (k >= piv[m]) {
            ++cnt[m];
            msum[m] += w;
          }
      }
    }
    tie_base += ties;
    ring_release(X, c);
  }
  long long C[NPIV + 2];
  double M[NPIV + 2];
#pragma unroll
  for (int m = 0; m <= NPIV; ++m) {
    C[m] = bsum_i(X, cnt[m], m & 7);
    M[m] = mass ? bsum_d(X, (double)msum[m], m & 7) : 0.0;
    __syncthreads();
  }
  C[NPIV + 1] = 0;
  M[NPIV + 1] = 0.0;
  if (mass && target_frac > 0.0) target = target_frac * (Wd.above_mass + M[0]);
  // sub-window m = [piv[m], piv[m+1]-1] holds the target when the members at
  // or above piv[m] reach it and those at or above piv[m+1] do not
  int sel = -1;
#pragma unroll
  for (int m = NPIV; m >= 0; --m) {
    const bool reach = mass ? (Wd.above_mass + M[m] >= target) : (Wd.above_cnt + C[m] >= kneed);
    if (sel < 0 && reach && (C[m] - C[m + 1]) > 0) sel = m;
  }
  if (sel < 0) sel = 0;
  uint32_t nlo = lo, nhi = hi;
  long long cs = 0, cs1 = 0;
  double ms1 = 0.0;
#pragma unroll
  for (int m = 0; m <= NPIV; ++m)
    if (m == sel) {
      nlo = piv[m];
      nhi = (m == NPIV) ? hi : piv[(m + 1 > NPIV) ? NPIV : m + 1] - 1u;
      cs = C[m];
      cs1 = C[m + 1];
      ms1 = M[m + 1];
    }
  Wd.above_cnt += cs1;
  Wd.above_mass += ms1;
  Wd.n_in = cs - cs1;
  Wd.lo = nlo;
  Wd.hi = max(nlo, nhi);
}

// Gather the window members (same domain as refine_pass) into the candidate
// list in id order; returns the list length.
template <int DT>
__device__ __forceinline__ int gather_window(Ctx<DT>& X, uint32_t lo, uint32_t hi, bool limited,
                                             uint32_t kK, int nK) {
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE, ITW = ElemT<DT>::ITW;
  int tie_base = 0, nlist = 0;
  const float vlo = key_to_float(lo);
  ring_begin(X);
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = ring_wait(X, c);
    int warp_start = 0, ties = 0;
    if (limited) ties = tie_prefix(X, stage, c, kK, tie_base, warp_start);
    int tie_run = warp_start, wcount = 0;
    for (int it = 0; it < ITW; ++it) {
      const uint4 r = load_masked(X, stage, c, warp_vec<DT>(it));
      if (!__any_sync(0xffffffffu, vmax<DT>(r) >= vlo)) continue;
      float x[EPV];
      unpack<DT>(r, x);
      wcount += __popc(window_bits<DT>(x, lo, hi, limited, kK, nK, tie_run));
    }
    int total = 0;
    int pos = list_warp_base(X, wcount, nlist, total);
    tie_run = warp_start;
    for (int it = 0; it < ITW; ++it) {
      const int v = warp_vec<DT>(it);
      const uint4 r = load_masked(X, stage, c, v);
      if (!__any_sync(0xffffffffu, vmax<DT>(r) >= vlo)) continue;
      float x[EPV];
      unpack<DT>(r, x);
      const uint32_t wb = window_bits<DT>(x, lo, hi, limited, kK, nK, tie_run);
      if (__any_sync(0xffffffffu, wb != 0u)) list_emit(X, c * CE + v * EPV, x, wb, pos);
    }
    tie_base += ties;
    nlist += total;
    ring_release(X, c);
  }
  return min(nlist, CAP);
}

// Zero a row's mask words and probabilities (members are written after).
template <int DT>
__device__ __forceinline__ void zero_outputs(const Ctx<DT>& X) {
  const KArgs& a = *X.a;
  if (a.kept_mask)
    for (int w = threadIdx.x; w < a.W; w += NT) a.kept_mask[(size_t)X.row * a.W + w] = 0u;
  if (a.probs)
    for (int e = threadIdx.x; e < a.V; e += NT) a.probs[(size_t)X.row * a.V + e] = 0.f;
  __syncthreads();
}

// Keep the list entries with key >= fk, in order, through the ring scratch.
template <int DT>
__device__ __forceinline__ int filter_list(const Ctx<DT>& X, int n, uint32_t fk) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ch = (n + NT - 1) / NT;
  const int j0 = threadIdx.x * ch, j1 = min(n, j0 + ch);
  int c = 0;
  for (int j = j0; j < j1; ++j) c += (X.ck[j] >= fk) ? 1 : 0;
  const int incl = warp_incl_scan(c);
  if (lane == 31) X.sh->bi[15][warp] = incl;
  __syncthreads();
  int pos = incl - c, tot = 0;
  for (int w = 0; w < NWARP; ++w) {
    if (w < warp) pos += X.sh->bi[15][w];
    tot += X.sh->bi[15][w];
  }
  uint32_t* tk = reinterpret_cast<uint32_t*>(X.ring);
  int* ti = reinterpret_cast<int*>(X.ring + CAP * 4);
  for (int j = j0; j < j1; ++j)
    if (X.ck[j] >= fk) {
      tk[pos] = X.ck[j];
      ti[pos] = X.ci[j];
      ++pos;
    }
  __syncthreads();
  for (int j = threadIdx.x; j < tot; j += NT) {
    X.ck[j] = tk[j];
    X.ci[j] = ti[j];
  }
  __syncthreads();
  return tot;
}

// ---------------------------------------------------------------------------
// One row.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ void process_row(Ctx<DT>& X, const KArgs& a, int row) {
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE, NVEC = ElemT<DT>::NVEC;
  constexpr int ITW = ElemT<DT>::ITW, ES = ElemT<DT>::ES;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  X.row = row;
  X.V = a.V;
  X.W = a.W;
  X.use_tma = a.use_tma;
  X.bm = a.bitmask ? a.bitmask + (size_t)row * a.W : nullptr;
  X.nch = (a.V + CE - 1) / CE;
  X.src = reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)a.ld * ES;
  X.timeout = 0;

  const float t = a.temperature ? a.temperature[row] : 0.f;
  const int kk = a.top_k ? a.top_k[row] : 1;
  const float pp = a.top_p ? a.top_p[row] : 1.f;
  int* rinfo = a.row_info ? a.row_info + (size_t)row * 4 : nullptr;
  const bool sample = a.mode == MODE_SAMPLE;
  if (a.mode != MODE_ARGMAX) {
    const bool bad = isnan(t) || t < 0.f || kk < 1 || isnan(pp) || !(pp > 0.f) || pp > 1.f;
    if (bad) {
      zero_outputs(X);
      if (tid == 0) {
        if (a.tokens) a.tokens[row] = -1;
        a.status[row] = ST_INVALID;
        if (a.kept_count) a.kept_count[row] = 0;
        if (rinfo) rinfo[0] = rinfo[1] = rinfo[2] = rinfo[3] = 0;
      }
      __syncthreads();
      return;
    }
  }
  const bool greedy = (a.mode == MODE_ARGMAX) || (t == 0.f);
  const int K0 = min(kk, a.V);
  const bool predALL = !greedy && K0 >= a.V && pp >= 1.f;
  const bool select = !greedy && !predALL;
  const bool topp_only = select && K0 >= a.V;  // top-k cannot bind: bulk masses needed
  X.temp = t;
  X.c2 = greedy ? 0.f : 1.4426950408889634f / t;
  uint32_t* mrow = a.kept_mask ? a.kept_mask + (size_t)row * a.W : nullptr;

  // legal-token count from the bitmask alone: rows with few legal tokens
  // gather every one of them
  int mask_legal = a.V;
  if (X.bm && select) {
    int cm = 0;
    for (int w = tid; w < a.W; w += NT) {
      uint32_t m = __ldg(X.bm + w);
      if (w == a.W - 1 && (a.V & 31)) m &= (1u << (a.V & 31)) - 1u;
      cm += __popc(m);
    }
    mask_legal = bsum_i(X, cm, 12);
    __syncthreads();
  }
  const bool take_all = select && mask_legal <= CAP;

  // ---- main pass -------------------------------------------------------------
  float bx = -INFINITY;
  int bvi = 0x7fffffff, nl = 0, nonfin = 0;
  int c0 = 0, c1 = 0, c2n = 0, c3 = 0;
  float f0 = 0.f, f1 = 0.f, f2 = 0.f, f3 = 0.f, ftot = 0.f, fref = -INFINITY;
  int nlist = 0, ovf = 0;
  float t0 = -FLT_MAX, t1 = -FLT_MAX, t2 = -FLT_MAX, t3 = -FLT_MAX;
  float aref = -INFINITY;  // all-kept rows: per-thread reference for the chunk masses
  ring_begin(X);
  for (int c = 0; c < X.nch; ++c) {
    const char* stage = ring_wait(X, c);
    // statistics walk (+ a first-chunk sample for mean / deviation)
    {
      const bool samp = (c == 0) && select && !take_all;
      float s = 0.f, s2 = 0.f;
      int ns = 0;
      for (int it = 0; it < ITW; ++it) {
        const int v = warp_vec<DT>(it);
        const uint4 r = load_masked(X, stage, c, v);
        const float mx = vmax_nan<DT>(r);
        if (isnan(mx) || mx == INFINITY) nonfin = 1;
        if (mx > bx) {
          bx = mx;
          bvi = c * NVEC + v;
        }
        const float mn = vmin<DT>(r);
        if (mn > -INFINITY && !samp) {
          nl += EPV;
        } else {
          float x[EPV];
          unpack<DT>(r, x);
#pragma unroll
          for (int j = 0; j < EPV; ++j) {
            if (is_neg_inf(x[j])) continue;
            ++nl;
            if (samp && x[j] < INFINITY && !isnan(x[j])) {
              s += x[j];
              s2 = fmaf(x[j], x[j], s2);
              ++ns;
            }
          }
        }
      }
      if (samp) {
        // thresholds from the first chunk (Qrita key design 1)
        const double ts = bsum_d(X, (double)s, 13);
        const double ts2 = bsum_d(X, (double)s2, 14);
        const int tns = bsum_i(X, ns, 13);
        __syncthreads();
        const double nest = fmax(1.0, (double)mask_legal);
        const double mu = tns ? ts / tns : 0.0;
        const double var = tns ? fmax(ts2 / tns - mu * mu, 0.0) : 0.0;
        const float sigma = (float)sqrt(var);
        const double Kt = topp_only ? fmin(nest, (double)(CAP / 2)) : (double)K0;
        const float q = (float)fmax(fmin(Kt / nest, 1.0), 1e-30);
        float pos = (log2f(q) + 24.f) * 4.f;
        pos = fminf(fmaxf(pos, 0.f), (float)(DTAB - 1));
        const int i0 = min((int)pos, DTAB - 2);
        const float fr = pos - (float)i0;
        const float delta = a.delta[i0] + fr * (a.delta[i0 + 1] - a.delta[i0]);
        const float tz = (float)mu + delta * sigma;
        const float mg = 0.2f * fabsf(tz);
        t0 = tz - mg;
        t1 = tz - 0.5f * mg;
        t2 = tz;
        t3 = tz + 0.5f * mg;
      }
    }
    if (select) {
      // sigma band: counts at four thresholds, then the candidates >= t0
      // written in id order
      int wcount = 0;
      for (int it = 0; it < ITW; ++it) {
        const uint4 r = load_masked(X, stage, c, warp_vec<DT>(it));
        if (topp_only) {
          float x[EPV];
          unpack<DT>(r, x);
#pragma unroll
          for (int j = 0; j < EPV; ++j) {
            if (is_neg_inf(x[j])) continue;
            if (x[j] > fref) {  // per-thread reference: rescale, never overflow
              const float sc = fast_exp2((fref - x[j]) * X.c2);
              ftot *= sc;
              f0 *= sc;
              f1 *= sc;
              f2 *= sc;
              f3 *= sc;
              fref = x[j];
            }
            const float w = fast_exp2((x[j] - fref) * X.c2);
            ftot += w;
            if (x[j] >= t0) {
              ++wcount;
              ++c0;
              f0 += w;
              if (x[j] >= t1) {
                ++c1;
                f1 += w;
              }
              if (x[j] >= t2) {
                ++c2n;
                f2 += w;
              }
              if (x[j] >= t3) {
                ++c3;
                f3 += w;
              }
            }
          }
        } else if (vmax<DT>(r) >= t0) {
          float x[EPV];
          unpack<DT>(r, x);
#pragma unroll
          for (int j = 0; j < EPV; ++j) {
            if (is_neg_inf(x[j]) || x[j] < t0) continue;
            ++wcount;
            ++c0;
            c1 += (x[j] >= t1) ? 1 : 0;
            c2n += (x[j] >= t2) ? 1 : 0;
            c3 += (x[j] >= t3) ? 1 : 0;
          }
        }
      }
      int total = 0;
      int pos = list_warp_base(X, wcount, nlist, total);
      for (int it = 0; it < ITW; ++it) {
        const int v = warp_vec<DT>(it);
        const uint4 r = load_masked(X, stage, c, v);
        if (!__any_sync(0xffffffffu, vmax<DT>(r) >= t0)) continue;
        float x[EPV];
        unpack<DT>(r, x);
        uint32_t bits = 0u;
#pragma unroll
        for (int j = 0; j < EPV; ++j)
          if (!is_neg_inf(x[j]) && x[j] >= t0) bits |= 1u << j;
        list_emit(X, c * CE + v * EPV, x, bits, pos);
      }
      if (nlist + total > CAP) ovf = 1;
      nlist += total;
    } else if (predALL) {
      // every legal token is kept: mask words now, fast mass per chunk
      // relative to a per-thread reference (combined per chunk)
      float acc = 0.f;
      for (int it = 0; it < ITW; ++it) {
        const int v = warp_vec<DT>(it);
        const uint4 r = load_masked(X, stage, c, v);
        float x[EPV];
        unpack<DT>(r, x);
        uint32_t bits = 0u;
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
          if (is_neg_inf(x[j]) || !(x[j] < INFINITY)) continue;
          bits |= 1u << j;
          if (x[j] > aref) {
            acc *= fast_exp2((aref - x[j]) * X.c2);
            aref = x[j];
          }
          acc += fast_exp2((x[j] - aref) * X.c2);
        }
        if (mrow) store_mask_word<DT>(mrow, a.W, c * CE + v * EPV, bits);
      }
      float zmax = aref;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
      const double m =
          warp_sum((aref == -INFINITY) ? 0.0 : (double)acc * (double)fast_exp2((aref - zmax) * X.c2));
      if (lane == 0) {
        X.sh->cpair_m[warp] = m;
        X.sh->cpair_z[warp] = zmax;
      }
      __syncthreads();
      if (tid == 0) {
        float zc = -INFINITY;
        for (int w = 0; w < NWARP; ++w) zc = fmaxf(zc, X.sh->cpair_z[w]);
        double mc = 0.0;
        for (int w = 0; w < NWARP; ++w)
          if (X.sh->cpair_z[w] > -INFINITY)
            mc += X.sh->cpair_m[w] * (double)fast_exp2((X.sh->cpair_z[w] - zc) * X.c2);
        X.sh->chunk_mass[c] = mc;
        X.sh->chunk_zref[c] = zc;
      }
    }
    ring_release(X, c);
  }

  // ---- row statistics --------------------------------------------------------
  float gmax = -INFINITY;
  int gvec;
  {
    float m = bx;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) X.sh->bf[0][warp] = m;
    nl = bsum_i(X, nl, 0);
    for (int w = 0; w < NWARP; ++w) gmax = fmaxf(gmax, X.sh->bf[0][w]);
    const unsigned cand = (bx == gmax) ? (unsigned)bvi : 0xffffffffu;
    gvec = (int)bmin_u(X, cand, 1);
    nonfin = bsum_i(X, nonfin, 2);
    X.timeout = bsum_i(X, X.timeout, 3);
    __syncthreads();
  }
  int status = ST_OK;
  if (X.timeout) status = ST_TIMEOUT;
  else if (nonfin) status = ST_NONFINITE;
  else if (nl == 0) status = ST_EMPTY;
  if (status != ST_OK) {
    zero_outputs(X);
    if (tid == 0) {
      if (a.tokens) a.tokens[row] = -1;
      a.status[row] = status;
      if (a.kept_count) a.kept_count[row] = 0;
      if (rinfo) rinfo[0] = rinfo[1] = rinfo[2] = rinfo[3] = 0;
    }
    __syncthreads();
    return;
  }
  // argmax: the first legal element equal to the max, in the earliest vector
  // holding it (bounded element-wise loads: rows need not be 16-byte aligned)
  int gargmax = 0;
  {
    const int e0 = gvec * EPV;
    const uint32_t lb = X.bm ? mask_bits(X, e0) : ((1u << EPV) - 1u);
    int j = -1;
    for (int q = EPV - 1; q >= 0; --q) {
      const int e = e0 + q;
      if (e >= X.V || !((lb >> q) & 1u)) continue;
      float xv;
      if constexpr (DT == DT_F32) {
        xv = reinterpret_cast<const float*>(X.src)[e];
      } else if constexpr (DT == DT_BF16) {
        xv = __uint_as_float(((uint32_t)reinterpret_cast<const unsigned short*>(X.src)[e]) << 16);
      } else {
        xv = __half2float(__ushort_as_half(reinterpret_cast<const unsigned short*>(X.src)[e]));
      }
      if (xv == gmax) j = q;
    }
    gargmax = e0 + (j < 0 ? 0 : j);
  }
  X.gmax = gmax;
  X.m_z = greedy ? 0.f : __fdiv_rn(gmax, t);
  const double u = (sample && !greedy)
                       ? philox_uniform(a.seed ? a.seed[row] : 0ull, a.offset ? a.offset[row] : 0ull)
                       : 0.0;

  int path = PATH_SIGMA, band_n = 0, sel_rounds = 0, ref_rounds = 0;
  int count = 0, token = -1;
  if (greedy) {
    path = PATH_GREEDY;
    zero_outputs(X);
    if (tid == 0) {
      if (a.kept_mask) atomicOr(&a.kept_mask[(size_t)row * a.W + (gargmax >> 5)], 1u << (gargmax & 31));
      if (a.probs) a.probs[(size_t)row * a.V + gargmax] = 1.f;
    }
    count = 1;
    token = gargmax;
  } else {
    const int K = min(K0, nl);
    const bool need_K = K < nl, need_P = pp < 1.f;
    if (!need_K && !need_P) {
      path = PATH_ALL;
      double Mp = 0.0;
      if (predALL) {
        // masks were written in the main pass; chunk masses relative to the max
        __syncthreads();
        if (tid == 0)
          for (int c = 0; c < X.nch; ++c) {
            const float zc = X.sh->chunk_zref[c];
            X.sh->chunk_mass[c] =
                (zc == -INFINITY) ? 0.0 : X.sh->chunk_mass[c] * (double)fast_exp2((zc - gmax) * X.c2);
          }
        __syncthreads();
        count = nl;
      } else {
        count = member_pass(X, 0u, 0, true);
      }
      for (int c = 0; c < X.nch; ++c) Mp += X.sh->chunk_mass[c];
      if (sample) token = draw_streamed(X, 0u, 0, true, Mp, u);
      if (a.probs) probs_pass(X, 0u, 0, true, Mp);
    } else {
      // ---- select: validate the sigma band -------------------------------------
      long long tc0, tc1, tc2, tc3;
      double tm0 = 0.0, tm1 = 0.0, tm2 = 0.0, tm3 = 0.0, fM = 0.0;
      {
        const float scale = (fref == -INFINITY) ? 0.f : fast_exp2((fref - gmax) * X.c2);
        tc0 = bsum_i(X, c0, 4);
        tc1 = bsum_i(X, c1, 5);
        tc2 = bsum_i(X, c2n, 6);
        tc3 = bsum_i(X, c3, 7);
        ovf = bsum_i(X, ovf, 8);
        if (topp_only) {
          tm0 = bsum_d(X, (double)f0 * scale, 4);
          tm1 = bsum_d(X, (double)f1 * scale, 5);
          tm2 = bsum_d(X, (double)f2 * scale, 6);
          tm3 = bsum_d(X, (double)f3 * scale, 7);
          fM = bsum_d(X, (double)ftot * scale, 8);
        }
        __syncthreads();
      }
      const long long tcnt[NTHR] = {tc0, tc1, tc2, tc3};
      const double tmass[NTHR] = {tm0, tm1, tm2, tm3};
      const float thr[NTHR] = {t0, t1, t2, t3};
      int istar = -1;
      if (!ovf) {
#pragma unroll
        for (int i = NTHR - 1; i >= 0; --i) {
          bool ok = istar < 0 && tcnt[i] <= CAP && tcnt[i] >= 1;
          if (need_K && tcnt[i] < K) ok = false;
          if (need_P && !need_K) {
            const bool all_in = tcnt[i] == nl;
            const bool mass_ok = topp_only && tmass[i] >= (double)pp * fM * (1.0 + 1e-5);
            if (!all_in && !mass_ok) ok = false;
          }
          if (ok) istar = i;
        }
      }
      if (istar >= 0) {
        // ---- the band is complete: select on chip ------------------------------
        int n = min(nlist, CAP);
        float fthr = t0;
        long long tci = tc0;
#pragma unroll
        for (int i = 0; i < NTHR; ++i)
          if (i == istar) {
            fthr = thr[i];
            tci = tcnt[i];
          }
        if (istar > 0) n = filter_list(X, n, fkey(fthr));
        band_n = n;
        float* bw = reinterpret_cast<float*>(X.ring);
        for (int j = tid; j < n; j += NT) bw[j] = weight(X, key_to_float(X.ck[j]));
        __syncthreads();
        int r1 = 0, r2 = 0;
        double Mk;
        if (need_K) {
          int ngt = 0;
          const uint32_t kK = pivot_count(X, n, K, 0, ngt, r1);
          restrict_members(X, n, kK, K - ngt);
          float s = 0.f;
          for (int j = tid; j < n; j += NT)
            if (!(X.ci[j] & NOT_MEMBER)) s += bw[j];
          Mk = bsum_d(X, (double)s, 10);
          __syncthreads();
        } else {
          float s = 0.f;
          for (int j = tid; j < n; j += NT) s += bw[j];
          const double Mband = bsum_d(X, (double)s, 10);
          __syncthreads();
          Mk = (tci == nl) ? Mband : fM;
        }
        if (need_P) {
          const double target = (double)pp * Mk;
          double agt = 0.0;
          int copies = 0;
          const uint32_t kp = pivot_mass(X, bw, n, target, 0.0, agt, copies, r2);
          const int nP = topp_copies(agt, (double)weight(X, key_to_float(kp)), target, copies);
          restrict_members(X, n, kp, nP);
        }
        sel_rounds = r1 + r2;
        // kept set = members; normaliser, count, draw
        float s = 0.f;
        int cc = 0;
        for (int j = tid; j < n; j += NT)
          if (!(X.ci[j] & NOT_MEMBER)) {
            s += bw[j];
            ++cc;
          }
        const double Mp = bsum_d(X, (double)s, 11);
        count = bsum_i(X, cc, 11);
        __syncthreads();
        if (sample) token = sample_members(X, bw, n, u * Mp);
        zero_outputs(X);
        const float inv = (float)(1.0 / Mp);
        for (int j = tid; j < n; j += NT) {
          if (X.ci[j] & NOT_MEMBER) continue;
          const int id = X.ci[j];
          if (mrow) atomicOr(&mrow[id >> 5], 1u << (id & 31));
          if (a.probs) a.probs[(size_t)row * a.V + id] = bw[j] * inv;
        }
      } else {
        // ---- exact multi-pivot refinement ----------------------------------------
        path = PATH_FULL;
        const uint32_t kmax = fkey(gmax);
        uint32_t kK = 0u;
        int nK = 0;
        if (need_K) {
          Win Wd;
          int i = NTHR - 1;
          while (i >= 0 && tcnt[i] < K) --i;
          if (i >= 0) {
            float ti = t0, tn = t0;
            long long cn = 0, ci_ = 0;
#pragma unroll
            for (int q = 0; q < NTHR; ++q) {
              if (q == i) {
                ti = thr[q];
                ci_ = tcnt[q];
              }
              if (q == i + 1) {
                tn = thr[q];
                cn = tcnt[q];
              }
            }
            Wd.lo = fkey(ti);
            Wd.hi = (i < NTHR - 1) ? fkey(tn) - 1u : kmax;
            Wd.above_cnt = (i < NTHR - 1) ? cn : 0;
            Wd.n_in = ci_ - Wd.above_cnt;
          } else {
            Wd.lo = KEY_MIN;
            Wd.hi = (t0 > -FLT_MAX) ? fkey(t0) - 1u : kmax;
            Wd.above_cnt = tc0;
            Wd.n_in = nl - tc0;
          }
          Wd.hi = min(Wd.hi, kmax);
          if (Wd.hi < Wd.lo) Wd.hi = Wd.lo;
          Wd.above_mass = 0.0;
          double no_target = 0.0;
          for (int g = 0; g < 12 && Wd.n_in > CAP && Wd.lo < Wd.hi; ++g) {
            refine_pass(X, Wd, false, (long long)K, no_target, 0.0, false, 0u, 0);
            ++ref_rounds;
          }
          if (Wd.lo < Wd.hi && Wd.n_in <= CAP) {
            const int n = gather_window(X, Wd.lo, Wd.hi, false, 0u, 0);
            band_n = n;
            int ngt = 0, r1 = 0;
            kK = pivot_count(X, n, K, (int)Wd.above_cnt, ngt, r1);
            nK = K - ngt;
            sel_rounds += r1;
          } else {
            kK = Wd.lo;
            nK = K - (int)Wd.above_cnt;
          }
        }
        uint32_t kB = kK;
        int nB = nK;
        if (need_P) {
          Win Wd;
          int i = -1;
          if (!need_K && topp_only) {
#pragma unroll
            for (int q = 0; q < NTHR; ++q)
              if (tmass[q] >= (double)pp * fM * (1.0 + 1e-5)) i = q;
          }
          float ti = t0;
#pragma unroll
          for (int q = 0; q < NTHR; ++q)
            if (q == i) ti = thr[q];
          Wd.lo = need_K ? kK : ((i >= 0) ? fkey(ti) : KEY_MIN);
          Wd.hi = kmax;
          if (Wd.hi < Wd.lo) Wd.lo = Wd.hi;
          Wd.above_cnt = 0;
          Wd.above_mass = 0.0;
          Wd.n_in = 0x7fffffffffffll;
          // the target is p * M_k: the first window's mass when top-k binds or
          // the window covers the row; else the fast whole-row mass
          double target = (double)pp * fM;
          for (int g = 0; g < 12 && (g == 0 || (Wd.n_in > CAP && Wd.lo < Wd.hi)); ++g) {
            const double frac = (g == 0 && (need_K || !topp_only || i < 0)) ? (double)pp : 0.0;
            refine_pass(X, Wd, true, 0, target, frac, need_K, kK, nK);
            ++ref_rounds;
          }
          if (Wd.lo < Wd.hi && Wd.n_in <= CAP) {
            const int n = gather_window(X, Wd.lo, Wd.hi, need_K, kK, nK);
            band_n = n;
            float* bw = reinterpret_cast<float*>(X.ring);
            for (int j = tid; j < n; j += NT) bw[j] = weight(X, key_to_float(X.ck[j]));
            __syncthreads();
            double agt = 0.0;
            int copies = 0, r2 = 0;
            const uint32_t kp = pivot_mass(X, bw, n, target, Wd.above_mass, agt, copies, r2);
            nB = topp_copies(agt, (double)weight(X, key_to_float(kp)), target, copies);
            kB = kp;
            sel_rounds += r2;
          } else {
            const uint32_t kp = Wd.lo;
            const double wv = (double)weight(X, key_to_float(kp));
            const int avail = (need_K && kp == kK) ? nK : (int)min(Wd.n_in, 0x7fffffffll);
            nB = topp_copies(Wd.above_mass, wv, target, avail);
            kB = kp;
          }
        }
        __syncthreads();
        count = member_pass(X, kB, nB, false);
        double Mp = 0.0;
        for (int c = 0; c < X.nch; ++c) Mp += X.sh->chunk_mass[c];
        if (sample) token = draw_streamed(X, kB, nB, false, Mp, u);
        if (a.probs) probs_pass(X, kB, nB, false, Mp);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    if (sample && a.tokens) a.tokens[row] = token;
    if (a.mode == MODE_ARGMAX && a.tokens) a.tokens[row] = gargmax;
    a.status[row] = ST_OK;
    if (a.kept_count) a.kept_count[row] = count;
    if (rinfo) {
      rinfo[0] = path;
      rinfo[1] = band_n;
      rinfo[2] = sel_rounds;
      rinfo[3] = ref_rounds;
    }
  }
  __syncthreads();
}

template <int DT>
__global__ void __launch_bounds__(NT, 2) smp_stream_kernel(const __grid_constant__ KArgs a) {
  extern __shared__ __align__(128) char smem[];
  Ctx<DT> X;
  X.a = &a;
  X.ring = smem;
  X.ck = reinterpret_cast<uint32_t*>(smem + SMEM_RING);
  X.ci = reinterpret_cast<int*>(smem + SMEM_RING + CAP * 4);
  X.sh = reinterpret_cast<Sh*>(smem + SMEM_RING + SMEM_CAND);
  X.parity = 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&X.sh->full[s], 1u);
    fence_mbar_init();
  }
  __syncthreads();
  for (int row = blockIdx.x; row < a.B; row += gridDim.x) process_row(X, a, row);
}

}  // namespace smp
