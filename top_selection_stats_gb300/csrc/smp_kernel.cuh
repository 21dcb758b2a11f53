// smp_kernel.cuh -- fused top-k / top-p truncation and sampling, one
// thread-block cluster per row, the row held once in distributed shared memory.
//
// Per row (contract of the AI Infra KB note M012, sections 02-03):
//   temperature (0 = greedy argmax) -> legal mask -> top-k (earliest ids win
//   ties) -> top-p (shortest prefix whose mass reaches p) -> renormalise ->
//   inverse-CDF draw in token-id order with a Philox4x32-10 uniform.
//
// Data flow (one HBM read of the logits, everything after it on chip):
//   1. every CTA of the cluster bulk-copies its slice of the row into its own
//      shared memory (cp.async.bulk + mbarrier) and loads its bitmask words;
//   2. row statistics in one pass as chunks land: max / argmax, legal count,
//      NaN/+inf flag, sum and sum of squares (Qrita paper notes, key design 1:
//      sample mean and standard deviation); exchanged through DSMEM;
//   3. sigma-truncation (Qrita key design 1): threshold t = mu + delta*sigma
//      lowered by a 0.2|t| margin, delta = Phi^-1(1 - k/V) from a host table;
//      four thresholds are counted in one pass and the tightest one that is
//      valid (holds all of S_k, or enough mass for top-p) and fits the
//      leader's buffer is chosen; its candidates are compacted, in id order,
//      into the leader CTA's shared memory;
//   4. the leader runs the three-pivot search (Qrita key design 2) for the
//      k-th value, the tie quota by prefix count (key design 3), and the same
//      pivot search on probability mass for the top-p boundary;
//   5. when truncation cannot be validated, an exact histogram refinement over
//      the whole row narrows the boundary band first (full-row fallback);
//   6. output stage: every CTA writes its packed kept-mask words, its
//      probabilities, and the CTA holding the draw scans its slice in id order.
#pragma once

#include "smp_device.cuh"

namespace smp {

struct KArgs {
  const void* logits;
  long long ld;
  int B, V, W;
  const uint32_t* bitmask;
  const float* temperature;
  const int* top_k;
  const float* top_p;
  const unsigned long long* seed;
  const unsigned long long* offset;
  int* tokens;
  int* status;
  uint32_t* kept_mask;
  int* kept_count;
  float* probs;
  int* row_info;
  int mode;
  int L;        // slice length in elements (multiple of slice_align(dtype))
  int cap;      // candidate capacity of the leader's gather buffer
  int use_tma;  // rows are 16-byte aligned: stage with bulk copies
  float delta[DTAB];
};

// Exchange record pushed by each CTA into a slot of every CTA of the cluster.
struct XRec {
  double d[6];
  int i[8];
};
enum Xid { X_STATS = 0, X_SIGMA, X_GCNT1, X_RES1, X_TIES, X_GCNT2, X_RES2, X_OUT, NX };

struct Misc {
  uint64_t mbar[NCHUNK];
  double rd[NWARP * 4];
  float rf[NWARP * 4];
  int ri[NWARP * 8];
  uint32_t ru[NWARP * 8];
  int wcnt[NTHR][NWARP];   // per-warp counts of the current band predicate(s)
  int wties[NWARP];        // per-warp count of copies of the tie key
  int wgtc[NWARP];         // output stage: per-warp members above the boundary
  double wgtm[NWARP];      // output stage: per-warp mass above the boundary
  int wlast[NWARP];        // output stage: per-warp last member id
  double scan_d[NBINS];
  int scan_i[NBINS];
  int bflag[8];
};

__host__ __device__ inline int esize_of(int dt) { return dt == DT_F32 ? 4 : 2; }
__host__ __device__ inline int epv_of(int dt) { return 16 / esize_of(dt); }
// Ordered passes give each warp a contiguous range walked 32 lanes x one
// 16-byte vector at a time, so a slice is a multiple of NWARP * 32 vectors.
__host__ __device__ inline int slice_align(int dt) { return NWARP * 32 * epv_of(dt); }

struct Layout {
  int off_data, off_mw, off_gx, off_gid, off_hc, off_hm, off_xch, off_misc, total;
};
__host__ __device__ inline int align_up(int v, int a) { return (v + a - 1) / a * a; }
__host__ __device__ inline Layout make_layout(int L, int dt, int cap, int S) {
  Layout l;
  int o = 0;
  l.off_data = o;
  o = align_up(o + L * esize_of(dt), 128);
  l.off_mw = o;
  o = align_up(o + (L / 32) * 4, 16);
  l.off_gx = o;
  o = align_up(o + cap * 4, 16);
  l.off_gid = o;
  o = align_up(o + cap * 4, 16);
  l.off_hc = o;  // 2 buffers x NBINS int counts
  o = align_up(o + 2 * NBINS * 4, 16);
  l.off_hm = o;  // 2 buffers x NBINS fixed-point masses
  o = align_up(o + 2 * NBINS * 8, 16);
  l.off_xch = o;
  o = align_up(o + NX * S * (int)sizeof(XRec), 16);
  l.off_misc = o;
  o = align_up(o + (int)sizeof(Misc), 128);
  l.total = o;
  return l;
}

// Fixed-point scale for histogram masses: integer atomics keep the merged
// masses independent of the order in which threads add them.
constexpr double MASS_FX = 4398046511104.0;  // 2^42

template <int DT>
struct Row {
  // cluster geometry
  int S, rank, row, L, n_local, base_id, Lw, iters;
  // smem
  char* data;
  uint32_t* mw;
  float* gx;
  int* gid;
  int* hc;
  unsigned long long* hm;
  XRec* xch;
  Misc* ms;
  bool has_mask;
  // row parameters / statistics
  float temp, top_p, m_z;
  int K, n_legal;
  bool need_K, need_P;
};

// ---- element access ------------------------------------------------------
template <int DT>
__device__ __forceinline__ void load_vec(const char* data, int e, float (&x)[16 / (DT == DT_F32 ? 4 : 2)]) {
  const uint4 r = *reinterpret_cast<const uint4*>(data + (size_t)e * esize_of(DT));
  if constexpr (DT == DT_F32) {
    x[0] = __uint_as_float(r.x);
    x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z);
    x[3] = __uint_as_float(r.w);
  } else if constexpr (DT == DT_BF16) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      x[2 * q] = __uint_as_float(w[q] << 16);
      x[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
  } else {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      x[2 * q] = __half2float(__ushort_as_half((unsigned short)(w[q] & 0xffffu)));
      x[2 * q + 1] = __half2float(__ushort_as_half((unsigned short)(w[q] >> 16)));
    }
  }
}
template <int DT>
__device__ __forceinline__ float load_one(const char* data, int e) {
  if constexpr (DT == DT_F32) {
    return reinterpret_cast<const float*>(data)[e];
  } else if constexpr (DT == DT_BF16) {
    return __uint_as_float(((uint32_t)reinterpret_cast<const unsigned short*>(data)[e]) << 16);
  } else {
    return __half2float(__ushort_as_half(reinterpret_cast<const unsigned short*>(data)[e]));
  }
}
// Legal bits of the EPV elements starting at e (e a multiple of EPV).
template <int DT>
__device__ __forceinline__ uint32_t mask_bits(const Row<DT>& R, int e) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  if (!R.has_mask) return (1u << EPV) - 1u;
  return (R.mw[e >> 5] >> (e & 31)) & ((1u << EPV) - 1u);
}
__device__ __forceinline__ bool is_neg_inf(float x) { return __float_as_uint(x) == 0xff800000u; }
__device__ __forceinline__ bool is_finite(float x) {
  return (__float_as_uint(x) & 0x7f800000u) != 0x7f800000u;
}
template <int DT>
__device__ __forceinline__ float weight(const Row<DT>& R, float x) {
  return expf(__fdiv_rn(x, R.temp) - R.m_z);
}
template <int DT>
__device__ __forceinline__ int vec_elem(const Row<DT>& R, int it) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  return warp * R.Lw + it * 32 * EPV + lane * EPV;
}

// ---- cluster exchange ----------------------------------------------------
template <int DT>
__device__ __forceinline__ void push_rec(const Row<DT>& R, int xid, const XRec& rec) {
  // threads 0..S-1 each deliver the record to one CTA (DSMEM stores)
  cg::cluster_group cluster = cg::this_cluster();
  if ((int)threadIdx.x < R.S) {
    XRec* dst = cluster.map_shared_rank(R.xch + xid * R.S + R.rank, (unsigned)threadIdx.x);
    *dst = rec;
  }
}
template <int DT>
__device__ __forceinline__ const XRec& rec_of(const Row<DT>& R, int xid, int r) {
  return R.xch[xid * R.S + r];
}

// --------------------------------------------------------------------------
// Leader-side selection on a gathered band (ids ascending in gid[0..n)).
// Three-pivot search (Qrita key design 2) in the order-preserving key space:
// pivots tau_n = lo + n(hi - lo)/4; one pass counts N = #{key > tau_n}, the
// smallest key above tau_n and its multiplicity; stop as soon as
// N >= K and N - mult < K (then the k-th value is that smallest key).
// gid bit 31 marks a band element that is not a member of the current domain.
// --------------------------------------------------------------------------
constexpr int NOT_MEMBER = (int)0x80000000;

template <int DT>
__device__ void band_minmax(const Row<DT>& R, int n, uint32_t& lo, uint32_t& hi) {
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int j = threadIdx.x; j < n; j += NT) {
    if (R.gid[j] & NOT_MEMBER) continue;
    uint32_t k = fkey(R.gx[j]);
    mn = min(mn, k);
    mx = max(mx, k);
  }
  lo = block_min_u32(mn, R.ms->ru);
  hi = block_max_u32(mx, R.ms->ru);
}

// k-th largest key among members (count target K, `above` members above the band).
template <int DT>
__device__ uint32_t pivot_count(const Row<DT>& R, int n, int K, int above, int& ngt, int& rounds) {
  uint32_t lo, hi;
  band_minmax(R, n, lo, hi);
  Misc* ms = R.ms;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  rounds = 0;
  for (int guard = 0; guard < 64 && lo < hi; ++guard) {
    ++rounds;
    uint32_t tau[3];
    const unsigned long long span = (unsigned long long)(hi - lo);
#pragma unroll
    for (int q = 0; q < 3; ++q) tau[q] = lo + (uint32_t)((span * (q + 1)) / 4);
    int cnt[3] = {0, 0, 0};
    MinCnt mc[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) mc[q] = MinCnt{0xffffffffu, 0};
    for (int j = threadIdx.x; j < n; j += NT) {
      if (R.gid[j] & NOT_MEMBER) continue;
      const uint32_t k = fkey(R.gx[j]);
#pragma unroll
      for (int q = 0; q < 3; ++q)
        if (k > tau[q]) {
          ++cnt[q];
          mc[q] = mc_combine(mc[q], MinCnt{k, 1});
        }
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      cnt[q] = warp_sum(cnt[q]);
      mc[q] = warp_mincnt(mc[q]);
    }
    __syncthreads();
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        ms->ri[q * NWARP + warp] = cnt[q];
        ms->ru[q * NWARP + warp] = mc[q].key;
        ms->ri[(3 + q) * NWARP + warp] = mc[q].cnt;
      }
    }
    __syncthreads();
    bool done = false;
    uint32_t nlo = lo, nhi = hi, found = 0;
    int found_gt = 0;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      int N = above;
      MinCnt m{0xffffffffu, 0};
      for (int w = 0; w < NWARP; ++w) {
        N += ms->ri[q * NWARP + w];
        m = mc_combine(m, MinCnt{ms->ru[q * NWARP + w], ms->ri[(3 + q) * NWARP + w]});
      }
      if (!done && N >= K && N - m.cnt < K) {
        done = true;
        found = m.key;
        found_gt = N - m.cnt;
      }
      if (N >= K) {
        nlo = max(nlo, (N - m.cnt >= K) ? m.key + 1u : tau[q] + 1u);
      } else {
        nhi = min(nhi, tau[q]);
      }
    }
    __syncthreads();
    if (done) {
      ngt = found_gt;
      return found;
    }
    lo = nlo;
    hi = nhi;
  }
  // Interval collapsed to one key: count what lies above it.
  int c = 0;
  for (int j = threadIdx.x; j < n; j += NT)
    if (!(R.gid[j] & NOT_MEMBER) && fkey(R.gx[j]) > lo) ++c;
  ngt = above + block_sum(c, ms->ri);
  return lo;
}

// Top-p boundary among members by mass: the key v with
// above_mass + mass{key > v} < target <= above_mass + mass{key >= v}.
template <int DT>
__device__ uint32_t pivot_mass(const Row<DT>& R, int n, double target, double above,
                               double& a_gt, int& copies, int& rounds) {
  uint32_t lo, hi;
  band_minmax(R, n, lo, hi);
  Misc* ms = R.ms;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  rounds = 0;
  for (int guard = 0; guard < 64 && lo < hi; ++guard) {
    ++rounds;
    uint32_t tau[3];
    const unsigned long long span = (unsigned long long)(hi - lo);
#pragma unroll
    for (int q = 0; q < 3; ++q) tau[q] = lo + (uint32_t)((span * (q + 1)) / 4);
    float ms_[3] = {0.f, 0.f, 0.f};
    MinCnt mc[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) mc[q] = MinCnt{0xffffffffu, 0};
    for (int j = threadIdx.x; j < n; j += NT) {
      if (R.gid[j] & NOT_MEMBER) continue;
      const float x = R.gx[j];
      const uint32_t k = fkey(x);
      const float w = weight(R, x);
#pragma unroll
      for (int q = 0; q < 3; ++q)
        if (k > tau[q]) {
          ms_[q] += w;
          mc[q] = mc_combine(mc[q], MinCnt{k, 1});
        }
    }
    double md[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      md[q] = warp_sum((double)ms_[q]);
      mc[q] = warp_mincnt(mc[q]);
    }
    __syncthreads();
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        ms->rd[q * NWARP + warp] = md[q];
        ms->ru[q * NWARP + warp] = mc[q].key;
        ms->ri[q * NWARP + warp] = mc[q].cnt;
      }
    }
    __syncthreads();
    bool done = false;
    uint32_t nlo = lo, nhi = hi, found = 0;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      double A = above;
      MinCnt m{0xffffffffu, 0};
      for (int w = 0; w < NWARP; ++w) {
        A += ms->rd[q * NWARP + w];
        m = mc_combine(m, MinCnt{ms->ru[q * NWARP + w], ms->ri[q * NWARP + w]});
      }
      const double wm = (m.cnt > 0) ? (double)m.cnt * (double)weight(R, key_to_float(m.key)) : 0.0;
      if (!done && m.cnt > 0 && A >= target && A - wm < target) {
        done = true;
        found = m.key;
      }
      if (A >= target && m.cnt > 0) {
        nlo = max(nlo, (A - wm >= target) ? m.key + 1u : tau[q] + 1u);
      } else {
        nhi = min(nhi, tau[q]);
      }
    }
    __syncthreads();
    if (done) {
      lo = hi = found;
      break;
    }
    if (nlo > nhi) break;  // inconsistent rounding: settle on the lower end
    lo = nlo;
    hi = nhi;
  }
  // The boundary must be a member key; after inconsistent rounding the
  // interval can close on a gap, in which case the next member key up is used.
  uint32_t nxt = 0xffffffffu;
  for (int j = threadIdx.x; j < n; j += NT) {
    if (R.gid[j] & NOT_MEMBER) continue;
    const uint32_t k = fkey(R.gx[j]);
    if (k >= lo) nxt = min(nxt, k);
  }
  nxt = block_min_u32(nxt, ms->ru);
  const uint32_t v = (nxt != 0xffffffffu) ? nxt : hi;
  float s = 0.f;
  int c = 0;
  for (int j = threadIdx.x; j < n; j += NT) {
    if (R.gid[j] & NOT_MEMBER) continue;
    const float x = R.gx[j];
    const uint32_t k = fkey(x);
    if (k > v) s += weight(R, x);
    if (k == v) ++c;
  }
  a_gt = above + block_sum((double)s, ms->rd);
  copies = block_sum(c, ms->ri);
  return v;
}

// Number of copies of the boundary value kept by top-p: copy j (in id order)
// is kept iff a_gt + j * w < target; at least one.
__device__ __forceinline__ int topp_copies(double a_gt, double w, double target, int avail) {
  if (avail <= 0) return 0;
  double need = (target - a_gt) / w;
  long long n = (need <= 0.0) ? 1 : (long long)ceil(need);
  if (n < 1) n = 1;
  if (n > avail) n = avail;
  return (int)n;
}

// Mark members of S_k among the gathered band: key > key_K, or a copy of
// key_K among the first nkeep_K in id order.  Non-members get NOT_MEMBER.
template <int DT>
__device__ void mark_topk(const Row<DT>& R, int n, uint32_t keyK, int nkeepK) {
  // contiguous chunks per thread keep id order for the tie ranks
  const int per = (n + NT - 1) / NT;
  const int j0 = threadIdx.x * per, j1 = min(n, j0 + per);
  int ties = 0;
  for (int j = j0; j < j1; ++j)
    if (fkey(R.gx[j]) == keyK) ++ties;
  // exclusive scan over threads
  int incl = warp_incl_scan(ties);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 31) R.ms->ri[warp] = incl;
  __syncthreads();
  int woff = 0;
  for (int w = 0; w < warp; ++w) woff += R.ms->ri[w];
  int rank = woff + incl - ties;
  for (int j = j0; j < j1; ++j) {
    const uint32_t k = fkey(R.gx[j]);
    bool mem = k > keyK;
    if (k == keyK) {
      mem = rank < nkeepK;
      ++rank;
    }
    if (!mem) R.gid[j] |= NOT_MEMBER;
  }
  __syncthreads();
}

}  // namespace smp

namespace smp {

// --------------------------------------------------------------------------
// Ordered walk over this CTA's slice.  Each warp owns a contiguous range; per
// iteration lane l holds the EPV elements starting at vec_elem(it).  Visits
// elements in increasing id order within a warp, which the compaction, the
// tie ranks and the id-order draw rely on.
// --------------------------------------------------------------------------
struct BandPred {
  int kind;           // 0: x >= thr ; 1: lo <= key <= hi
  float thr;
  uint32_t lo, hi;
  uint32_t tie_key;   // with tie_limit >= 0: copies of tie_key whose CTA-local
  int tie_limit;      // rank (id order) is >= tie_limit are not members
};

template <int DT, class F>
__device__ __forceinline__ void walk_band(const Row<DT>& R, const BandPred& P, int warp_tie_off, F&& f) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  const int lane = threadIdx.x & 31;
  int tie_run = warp_tie_off;
  for (int it = 0; it < R.iters; ++it) {
    const int e = vec_elem(R, it);
    float x[EPV];
    load_vec<DT>(R.data, e, x);
    const uint32_t lb = mask_bits(R, e);
    uint32_t bits = 0u, tbits = 0u;
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      if (!((lb >> j) & 1u) || is_neg_inf(x[j])) continue;
      bool in;
      if (P.kind == 0) {
        in = x[j] >= P.thr;
      } else {
        const uint32_t k = fkey(x[j]);
        in = (k >= P.lo) && (k <= P.hi);
        if (P.tie_limit >= 0 && k == P.tie_key) tbits |= 1u << j;
      }
      if (in) bits |= 1u << j;
    }
    if (P.tie_limit >= 0) {
      const int nt = __popc(tbits);
      const int incl = warp_incl_scan(nt);
      int r = tie_run + incl - nt;
#pragma unroll
      for (int j = 0; j < EPV; ++j)
        if ((tbits >> j) & 1u) {
          if (r >= P.tie_limit) bits &= ~(1u << j);
          ++r;
        }
      tie_run += __shfl_sync(0xffffffffu, incl, 31);
    }
    f(it, e, x, bits);
  }
  (void)lane;
}

// Per-warp member counts of a band predicate -> ms->wcnt[slot][warp]; returns the CTA total.
template <int DT>
__device__ int count_band(const Row<DT>& R, const BandPred& P, int slot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int warp_tie_off = 0;
  if (P.tie_limit >= 0)
    for (int w = 0; w < warp; ++w) warp_tie_off += R.ms->wties[w];
  int c = 0;
  walk_band(R, P, warp_tie_off, [&](int, int, const float*, uint32_t bits) { c += __popc(bits); });
  c = warp_sum(c);
  if (lane == 0) R.ms->wcnt[slot][warp] = c;
  __syncthreads();
  int tot = 0;
  for (int w = 0; w < NWARP; ++w) tot += R.ms->wcnt[slot][w];
  __syncthreads();
  return tot;
}

// Compact the members of P, in id order, into the leader's gx/gid at
// cta_off + (members of earlier warps); per-warp counts from count_band(slot).
template <int DT>
__device__ void gather_band(const Row<DT>& R, const BandPred& P, int slot, int cta_off, int cap) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  cg::cluster_group cluster = cg::this_cluster();
  float* lgx = cluster.map_shared_rank(R.gx, 0u);
  int* lgid = cluster.map_shared_rank(R.gid, 0u);
  const int warp = threadIdx.x >> 5;
  int base = cta_off;
  int warp_tie_off = 0;
  for (int w = 0; w < warp; ++w) {
    base += R.ms->wcnt[slot][w];
    if (P.tie_limit >= 0) warp_tie_off += R.ms->wties[w];
  }
  walk_band(R, P, warp_tie_off, [&](int, int e, const float* x, uint32_t bits) {
    const int c = __popc(bits);
    const int incl = warp_incl_scan(c);
    int pos = base + incl - c;
#pragma unroll
    for (int j = 0; j < EPV; ++j)
      if ((bits >> j) & 1u) {
        if (pos < cap) {
          lgx[pos] = x[j];
          lgid[pos] = R.base_id + e + j;
        }
        ++pos;
      }
    base += __shfl_sync(0xffffffffu, incl, 31);
  });
}

// Per-warp copies of `key` (legal) -> ms->wties; returns the CTA total.
template <int DT>
__device__ int count_ties(const Row<DT>& R, uint32_t key) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int c = 0;
  for (int it = 0; it < R.iters; ++it) {
    const int e = vec_elem(R, it);
    float x[EPV];
    load_vec<DT>(R.data, e, x);
    const uint32_t lb = mask_bits(R, e);
#pragma unroll
    for (int j = 0; j < EPV; ++j)
      if (((lb >> j) & 1u) && !is_neg_inf(x[j]) && fkey(x[j]) == key) ++c;
  }
  c = warp_sum(c);
  if (lane == 0) R.ms->wties[warp] = c;
  __syncthreads();
  int tot = 0;
  for (int w = 0; w < NWARP; ++w) tot += R.ms->wties[w];
  __syncthreads();
  return tot;
}

// --------------------------------------------------------------------------
// Exact histogram refinement (full-row fallback).  One round: every CTA bins
// its members with lo <= key <= hi into NBINS bins of width 2^shift (counts,
// and fixed-point masses when `mass`), the cluster merges the histograms
// through DSMEM, and every CTA picks the same boundary bin.
// --------------------------------------------------------------------------
struct Refine {
  uint32_t lo, hi;
  long long above_cnt;
  unsigned long long above_mfx;  // fixed-point mass above the band
  long long n_in;                // members in the band
  unsigned long long total_mfx;  // round-1 total mass (= M_k)
  int rounds;
};

__device__ __forceinline__ int bin_shift(uint32_t lo, uint32_t hi) {
  const uint32_t span = hi - lo;
  const int bits = span ? 32 - __clz(span) : 0;
  return bits > 8 ? bits - 8 : 0;
}

template <int DT>
__device__ void refine_round(const Row<DT>& R, Refine& F, int buf, bool mass, long long kneed,
                             double p, uint32_t tie_key, int tie_inc, bool first) {
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  const int tid = threadIdx.x;
  int* hc = R.hc + buf * NBINS;
  unsigned long long* hm = R.hm + buf * NBINS;
  const uint32_t lo = F.lo, hi = F.hi;
  const int shift = bin_shift(lo, hi);
  hc[tid] = 0;
  hm[tid] = 0ull;
  __syncthreads();
  for (int it = 0; it < R.iters; ++it) {
    const int e = vec_elem(R, it);
    float x[EPV];
    load_vec<DT>(R.data, e, x);
    const uint32_t lb = mask_bits(R, e);
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      if (!((lb >> j) & 1u) || is_neg_inf(x[j])) continue;
      const uint32_t k = fkey(x[j]);
      if (k < lo || k > hi) continue;
      if (tie_inc >= 0 && k == tie_key) continue;  // added in aggregate below
      const int bin = (int)((k - lo) >> shift);
      atomicAdd(&hc[bin], 1);
      if (mass) atomicAdd(&hm[bin], (unsigned long long)((double)weight(R, x[j]) * MASS_FX + 0.5));
    }
  }
  __syncthreads();
  if (tid == 0 && tie_inc > 0 && tie_key >= lo && tie_key <= hi) {
    const int bin = (int)((tie_key - lo) >> shift);
    hc[bin] += tie_inc;
    if (mass)
      hm[bin] += (unsigned long long)tie_inc *
                 (unsigned long long)((double)weight(R, key_to_float(tie_key)) * MASS_FX + 0.5);
  }
  __syncthreads();
  cluster.sync();
  // Merge: thread t sums bin (NBINS-1-t) over the cluster, so that thread
  // order runs from the highest bin down and an inclusive scan over threads
  // gives the mass / count at or above each bin.
  const int b = NBINS - 1 - tid;
  long long c = 0;
  unsigned long long m = 0ull;
  for (int r = 0; r < R.S; ++r) {
    const int* rc = cluster.map_shared_rank(hc, (unsigned)r);
    const unsigned long long* rm = cluster.map_shared_rank(hm, (unsigned)r);
    c += rc[b];
    m += rm[b];
  }
  // block inclusive scan over threads (c and m)
  const int lane = tid & 31, warp = tid >> 5;
  long long ci = c;
  unsigned long long mi = m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long cn = __shfl_up_sync(0xffffffffu, ci, o);
    unsigned long long mn = __shfl_up_sync(0xffffffffu, mi, o);
    if (lane >= o) {
      ci += cn;
      mi += mn;
    }
  }
  Misc* ms = R.ms;
  long long* wc = reinterpret_cast<long long*>(ms->rd);          // NWARP slots
  unsigned long long* wm = reinterpret_cast<unsigned long long*>(ms->rd + NWARP);
  __syncthreads();
  if (lane == 31) {
    wc[warp] = ci;
    wm[warp] = mi;
  }
  __syncthreads();
  long long cpre = 0, ctot = 0;
  unsigned long long mpre = 0ull, mtot = 0ull;
  for (int w = 0; w < NWARP; ++w) {
    if (w < warp) {
      cpre += wc[w];
      mpre += wm[w];
    }
    ctot += wc[w];
    mtot += wm[w];
  }
  ci += cpre;
  mi += mpre;
  const long long cex = ci - c;
  const unsigned long long mex = mi - m;
  if (first && mass) F.total_mfx = mtot + F.above_mfx;
  // boundary bin
  bool hit;
  if (!mass) {
    hit = (F.above_cnt + cex < kneed) && (kneed <= F.above_cnt + ci);
  } else {
    const double target = p * (double)F.total_mfx;
    hit = ((double)(F.above_mfx + mex) < target) && (target <= (double)(F.above_mfx + mi)) && c > 0;
  }
  __syncthreads();
  if (tid == 0) ms->bflag[0] = -1;
  __syncthreads();
  if (hit) atomicMax(&ms->bflag[0], tid);  // unique in exact arithmetic; take one
  __syncthreads();
  int sel = ms->bflag[0];
  if (sel < 0) {
    // rounding left no bin reaching the target: take the lowest non-empty bin
    if (tid == 0) ms->bflag[1] = -1;
    __syncthreads();
    if (c > 0) atomicMax(&ms->bflag[1], tid);
    __syncthreads();
    sel = ms->bflag[1];
    if (sel < 0) sel = 0;
  }
  if (tid == sel) {
    ms->scan_i[0] = (int)b;
    reinterpret_cast<long long*>(ms->scan_d)[1] = cex;
    reinterpret_cast<long long*>(ms->scan_d)[2] = c;
    reinterpret_cast<unsigned long long*>(ms->scan_d)[3] = mex;
  }
  __syncthreads();
  const int bsel = ms->scan_i[0];
  F.above_cnt += reinterpret_cast<long long*>(ms->scan_d)[1];
  F.n_in = reinterpret_cast<long long*>(ms->scan_d)[2];
  F.above_mfx += reinterpret_cast<unsigned long long*>(ms->scan_d)[3];
  const unsigned long long nlo = (unsigned long long)lo + ((unsigned long long)bsel << shift);
  const unsigned long long nhi = nlo + ((1ull << shift) - 1ull);
  F.lo = (uint32_t)nlo;
  F.hi = (uint32_t)min(nhi, (unsigned long long)hi);
  F.rounds++;
  __syncthreads();
}

// --------------------------------------------------------------------------
// Row statistics pass (chunk-major, overlaps the bulk copies in flight).
// --------------------------------------------------------------------------
struct Stats {
  float bx;
  int bid;
  int nl;
  int nonfin;
  int timeout;
  float s, s2;
};

template <int DT>
__device__ Stats stats_pass(const Row<DT>& R, const KArgs& a, const int* chunk_bulk) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  const int nvec = R.L / EPV, cvec = nvec / NCHUNK;
  Stats st{-INFINITY, 0x7fffffff, 0, 0, 0, 0.f, 0.f};
  for (int c = 0; c < NCHUNK; ++c) {
    if (a.use_tma && chunk_bulk[c] > 0) {
      if (!mbar_wait_bounded(&R.ms->mbar[c], 0u, 4000000000ll)) st.timeout = 1;
    }
    for (int vi = c * cvec + threadIdx.x; vi < (c + 1) * cvec; vi += NT) {
      const int e = vi * EPV;
      float x[EPV];
      load_vec<DT>(R.data, e, x);
      const uint32_t lb = mask_bits(R, e);
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        const float v = x[j];
        if (!((lb >> j) & 1u) || is_neg_inf(v)) continue;
        if (!is_finite(v)) {
          st.nonfin = 1;
          continue;
        }
        st.nl += 1;
        st.s += v;
        st.s2 = fmaf(v, v, st.s2);
        if (v > st.bx) {
          st.bx = v;
          st.bid = R.base_id + e + j;
        }
      }
    }
  }
  return st;
}

__device__ __forceinline__ void argmax_combine(float& bx, int& bid, float ox, int oid) {
  if (ox > bx || (ox == bx && oid < bid)) {
    bx = ox;
    bid = oid;
  }
}

// --------------------------------------------------------------------------
// The kernel: one cluster of S CTAs per row.
// --------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(NT, 2) smp_rows_kernel(const __grid_constant__ KArgs a) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  constexpr int ES = (DT == DT_F32 ? 4 : 2);
  extern __shared__ __align__(128) char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  Row<DT> R;
  R.S = (int)cluster.num_blocks();
  R.rank = (int)cluster.block_rank();
  R.row = blockIdx.x / R.S;
  R.L = a.L;
  R.base_id = R.rank * a.L;
  R.n_local = max(0, min(a.L, a.V - R.base_id));
  R.Lw = a.L / NWARP;
  R.iters = R.Lw / (32 * EPV);
  const Layout lay = make_layout(a.L, DT, a.cap, R.S);
  R.data = smem + lay.off_data;
  R.mw = reinterpret_cast<uint32_t*>(smem + lay.off_mw);
  R.gx = reinterpret_cast<float*>(smem + lay.off_gx);
  R.gid = reinterpret_cast<int*>(smem + lay.off_gid);
  R.hc = reinterpret_cast<int*>(smem + lay.off_hc);
  R.hm = reinterpret_cast<unsigned long long*>(smem + lay.off_hm);
  R.xch = reinterpret_cast<XRec*>(smem + lay.off_xch);
  R.ms = reinterpret_cast<Misc*>(smem + lay.off_misc);
  R.has_mask = a.bitmask != nullptr;
  Misc* ms = R.ms;
  const int row = R.row;
  const bool leader = R.rank == 0;

  // ---- 1. stage the slice: bulk copies in NCHUNK pieces ------------------
  const char* src = reinterpret_cast<const char*>(a.logits) +
                    ((size_t)row * (size_t)a.ld + (size_t)R.base_id) * ES;
  const int chunk_elems = a.L / NCHUNK;
  int chunk_bulk[NCHUNK];
  int bulk_end = 0;  // elements covered by bulk copies
#pragma unroll
  for (int c = 0; c < NCHUNK; ++c) {
    const int c0 = c * chunk_elems;
    const int ne = max(0, min(chunk_elems, R.n_local - c0));
    const int bytes = a.use_tma ? ((ne * ES) & ~15) : 0;
    chunk_bulk[c] = bytes;
    if (bytes > 0) bulk_end = c0 + bytes / ES;
  }
  if (a.use_tma) {
    if (tid == 0) {
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) mbar_init(&ms->mbar[c], 1u);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) {
        if (chunk_bulk[c] > 0) {
          mbar_arrive_expect_tx(&ms->mbar[c], (uint32_t)chunk_bulk[c]);
          bulk_g2s(R.data + (size_t)c * chunk_elems * ES, src + (size_t)c * chunk_elems * ES,
                   (uint32_t)chunk_bulk[c], &ms->mbar[c]);
        }
      }
    }
  }
  // plain loads: everything without TMA, the sub-16-byte tail with it
  {
    const int p0 = a.use_tma ? bulk_end : 0;
    // the tail of the last non-empty chunk starts after its bulk part
    int tail0 = p0;
    if (a.use_tma) {
      tail0 = 0;
      for (int c = 0; c < NCHUNK; ++c) {
        const int c0 = c * chunk_elems;
        const int ne = max(0, min(chunk_elems, R.n_local - c0));
        if (ne > 0) tail0 = c0 + chunk_bulk[c] / ES;
      }
    }
    for (int e = tail0 + tid; e < R.n_local; e += NT) {
      if constexpr (ES == 4) {
        reinterpret_cast<uint32_t*>(R.data)[e] = reinterpret_cast<const uint32_t*>(src)[e];
      } else {
        reinterpret_cast<unsigned short*>(R.data)[e] = reinterpret_cast<const unsigned short*>(src)[e];
      }
    }
    // padding past the row end: -inf, never legal
    for (int e = R.n_local + tid; e < a.L; e += NT) {
      if constexpr (DT == DT_F32) reinterpret_cast<uint32_t*>(R.data)[e] = 0xff800000u;
      else if constexpr (DT == DT_BF16) reinterpret_cast<unsigned short*>(R.data)[e] = 0xff80u;
      else reinterpret_cast<unsigned short*>(R.data)[e] = 0xfc00u;
    }
  }
  if (R.has_mask) {
    const int w0 = R.base_id / 32;
    const uint32_t* mrow = a.bitmask + (size_t)row * (size_t)a.W;
    for (int i = tid; i < a.L / 32; i += NT) R.mw[i] = (w0 + i < a.W) ? mrow[w0 + i] : 0u;
  }
  __syncthreads();

  // ---- 2. row statistics --------------------------------------------------
  Stats st = stats_pass(R, a, chunk_bulk);
  {
    // block reduction of the statistics
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ox = __shfl_xor_sync(0xffffffffu, st.bx, o);
      const int oid = __shfl_xor_sync(0xffffffffu, st.bid, o);
      argmax_combine(st.bx, st.bid, ox, oid);
    }
    const int nl = warp_sum(st.nl);
    const int nf = __reduce_or_sync(0xffffffffu, (unsigned)st.nonfin);
    const int to = __reduce_or_sync(0xffffffffu, (unsigned)st.timeout);
    const float s = warp_sum(st.s), s2 = warp_sum(st.s2);
    if (lane == 0) {
      ms->rf[warp] = st.bx;
      ms->ri[warp] = st.bid;
      ms->ri[NWARP + warp] = nl;
      ms->ri[2 * NWARP + warp] = nf;
      ms->ri[3 * NWARP + warp] = to;
      ms->rd[warp] = s;
      ms->rd[NWARP + warp] = s2;
    }
    __syncthreads();
    if (tid == 0) {
      float bx = ms->rf[0];
      int bid = ms->ri[0], tnl = 0, tnf = 0, tto = 0;
      double ts = 0.0, ts2 = 0.0;
      for (int w = 0; w < NWARP; ++w) {
        argmax_combine(bx, bid, ms->rf[w], ms->ri[w]);
        tnl += ms->ri[NWARP + w];
        tnf |= ms->ri[2 * NWARP + w];
        tto |= ms->ri[3 * NWARP + w];
        ts += ms->rd[w];
        ts2 += ms->rd[NWARP + w];
      }
      XRec rec;
      rec.d[0] = ts;
      rec.d[1] = ts2;
      rec.i[0] = __float_as_int(bx);
      rec.i[1] = bid;
      rec.i[2] = tnl;
      rec.i[3] = tnf;
      rec.i[4] = tto;
      ms->bflag[7] = 0;
      *reinterpret_cast<XRec*>(ms->scan_d) = rec;
    }
    __syncthreads();
    push_rec(R, X_STATS, *reinterpret_cast<const XRec*>(ms->scan_d));
    cluster.sync();
  }
  float gmax = -INFINITY;
  int gargmax = 0x7fffffff, nl = 0, nonfin = 0, timeout = 0;
  double sum = 0.0, sum2 = 0.0;
  for (int r = 0; r < R.S; ++r) {
    const XRec& q = rec_of(R, X_STATS, r);
    argmax_combine(gmax, gargmax, __int_as_float(q.i[0]), q.i[1]);
    nl += q.i[2];
    nonfin |= q.i[3];
    timeout |= q.i[4];
    sum += q.d[0];
    sum2 += q.d[1];
  }

  // ---- 3. parameters and row status --------------------------------------
  const float t = a.temperature ? a.temperature[row] : 0.f;
  const int kk = a.top_k ? a.top_k[row] : 1;
  const float pp = a.top_p ? a.top_p[row] : 1.f;
  int status = ST_OK;
  if (a.mode != MODE_ARGMAX) {
    const bool bad = isnan(t) || t < 0.f || kk < 1 || isnan(pp) || !(pp > 0.f) || pp > 1.f;
    if (bad) status = ST_INVALID;
  }
  if (status == ST_OK) {
    if (timeout) status = ST_TIMEOUT;
    else if (nonfin) status = ST_NONFINITE;
    else if (nl == 0) status = ST_EMPTY;
  }
  const bool greedy = (a.mode == MODE_ARGMAX) || (t == 0.f);
  int* rinfo = a.row_info ? a.row_info + (size_t)row * 4 : nullptr;

  if (a.mode == MODE_ARGMAX || status != ST_OK) {
    if (a.mode != MODE_ARGMAX) {
      // error row: zero mask words and probabilities of this slice
      if (a.kept_mask) {
        const int w0 = R.base_id / 32, w1 = min(a.W, (R.base_id + a.L) / 32);
        for (int w = w0 + tid; w < w1; w += NT) a.kept_mask[(size_t)row * a.W + w] = 0u;
      }
      if (a.probs)
        for (int e = tid; e < R.n_local; e += NT) a.probs[(size_t)row * a.V + R.base_id + e] = 0.f;
    }
    if (leader && tid == 0) {
      if (a.tokens) a.tokens[row] = (status == ST_OK) ? gargmax : -1;
      if (a.status) a.status[row] = status;
      if (a.kept_count) a.kept_count[row] = 0;
      if (rinfo) {
        rinfo[0] = status == ST_OK ? PATH_GREEDY : PATH_ERROR;
        rinfo[1] = rinfo[2] = rinfo[3] = 0;
      }
    }
    if (timeout && a.use_tma && tid == 0)
      for (int c = 0; c < NCHUNK; ++c)
        if (chunk_bulk[c] > 0) mbar_wait_bounded(&ms->mbar[c], 0u, 4000000000ll);
    return;
  }

  // ---- 4. selection --------------------------------------------------------
  uint32_t keyB = 0u;  // boundary key: members are key > keyB, plus ties below
  int nkeepB = 0;      // first nkeepB copies of keyB (id order) are members
  int path = PATH_ALL, band_n = 0, sel_rounds = 0, ref_rounds = 0;
  R.temp = t;
  R.top_p = pp;
  R.n_legal = nl;
  R.m_z = greedy ? 0.f : __fdiv_rn(gmax, t);
  const int K = min(min(kk, a.V), nl);
  R.K = K;
  R.need_K = K < nl;
  R.need_P = pp < 1.f;
  if (greedy) {
    path = PATH_GREEDY;
    keyB = fkey(gmax);
    nkeepB = 1;
  } else if (R.need_K || R.need_P) {
    path = PATH_SIGMA;
    // -- sigma truncation (Qrita key design 1) --
    const double mu = sum / nl;
    const double var = fmax(sum2 / nl - mu * mu, 0.0);
    const float sigma = (float)sqrt(var);
    int istar = -1;
    float thr[NTHR];
    int tcnt[NTHR] = {0, 0, 0, 0};
    double Mtot = 0.0;
    if (!R.need_K || K <= a.cap) {
      const int Kt = R.need_K ? K : min(nl, a.cap / 2);
      const float q = (float)Kt / (float)nl;
      float pos = (log2f(q) + 24.f) * 4.f;
      pos = fminf(fmaxf(pos, 0.f), (float)(DTAB - 1));
      const int i0 = min((int)pos, DTAB - 2);
      const float fr = pos - (float)i0;
      const float delta = a.delta[i0] + fr * (a.delta[i0 + 1] - a.delta[i0]);
      const float t0 = (float)mu + delta * sigma;
      const float mg = 0.2f * fabsf(t0);
      thr[0] = t0 - mg;
      thr[1] = t0 - 0.5f * mg;
      thr[2] = t0;
      thr[3] = t0 + 0.5f * mg;
      // one ordered pass: counts at the four thresholds (+ masses for top-p)
      int c[NTHR] = {0, 0, 0, 0};
      float m4[NTHR] = {0.f, 0.f, 0.f, 0.f};
      float mt = 0.f;
      const bool wmass = !R.need_K;
      for (int it = 0; it < R.iters; ++it) {
        const int e = vec_elem(R, it);
        float x[EPV];
        load_vec<DT>(R.data, e, x);
        const uint32_t lb = mask_bits(R, e);
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
          if (!((lb >> j) & 1u) || is_neg_inf(x[j])) continue;
          float w = 0.f;
          if (wmass) {
            w = weight(R, x[j]);
            mt += w;
          }
#pragma unroll
          for (int i = 0; i < NTHR; ++i)
            if (x[j] >= thr[i]) {
              ++c[i];
              if (wmass) m4[i] += w;
            }
        }
      }
      XRec rec;
#pragma unroll
      for (int i = 0; i < NTHR; ++i) {
        const int wc = warp_sum(c[i]);
        if (lane == 0) ms->wcnt[i][warp] = wc;
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < NTHR; ++i) {
        int tot = 0;
        for (int w = 0; w < NWARP; ++w) tot += ms->wcnt[i][w];
        rec.i[i] = tot;
      }
      if (wmass) {
#pragma unroll
        for (int i = 0; i < NTHR; ++i) rec.d[i] = block_sum((double)m4[i], ms->rd);
        rec.d[4] = block_sum((double)mt, ms->rd);
      } else {
        for (int i = 0; i < 5; ++i) rec.d[i] = 0.0;
      }
      __syncthreads();
      push_rec(R, X_SIGMA, rec);
      cluster.sync();
      double tmass[NTHR] = {0, 0, 0, 0};
      for (int r = 0; r < R.S; ++r) {
        const XRec& qr = rec_of(R, X_SIGMA, r);
        for (int i = 0; i < NTHR; ++i) {
          tcnt[i] += qr.i[i];
          tmass[i] += qr.d[i];
        }
        Mtot += qr.d[4];
      }
      for (int i = NTHR - 1; i >= 0 && istar < 0; --i) {
        bool ok = tcnt[i] >= (R.need_K ? K : 1) && tcnt[i] <= a.cap;
        if (!R.need_K) ok = ok && tmass[i] >= (double)pp * Mtot * (1.0 + 1e-5);
        if (ok) istar = i;
      }
    }
    if (istar >= 0) {
      // -- compact the band into the leader, then select there --
      band_n = tcnt[istar];
      BandPred P{0, thr[istar], 0u, 0u, 0u, -1};
      int cta_off = 0;
      for (int r = 0; r < R.rank; ++r) cta_off += rec_of(R, X_SIGMA, r).i[istar];
      gather_band(R, P, istar, cta_off, a.cap);
      cluster.sync();
      if (leader) {
        int r1 = 0, r2 = 0;
        uint32_t keyK = 0u;
        int nkeepK = 0;
        double Mk = Mtot;
        if (R.need_K) {
          int ngt = 0;
          keyK = pivot_count(R, band_n, K, 0, ngt, r1);
          nkeepK = K - ngt;
          mark_topk(R, band_n, keyK, nkeepK);
          float s = 0.f;
          if (R.need_P)
            for (int j = tid; j < band_n; j += NT)
              if (!(R.gid[j] & NOT_MEMBER)) s += weight(R, R.gx[j]);
          Mk = block_sum((double)s, ms->rd);
        }
        uint32_t kB = keyK;
        int nB = nkeepK;
        if (R.need_P) {
          const double target = (double)pp * Mk;
          double agt = 0.0;
          int copies = 0;
          const uint32_t kp = pivot_mass(R, band_n, target, 0.0, agt, copies, r2);
          const double wv = (double)weight(R, key_to_float(kp));
          kB = kp;
          nB = topp_copies(agt, wv, target, copies);
        }
        if (tid == 0) {
          XRec rec;
          rec.i[0] = (int)kB;
          rec.i[1] = nB;
          rec.i[2] = r1 + r2;
          *reinterpret_cast<XRec*>(ms->scan_d + 128) = rec;
        }
        __syncthreads();
        push_rec(R, X_RES1, *reinterpret_cast<const XRec*>(ms->scan_d + 128));
      }
      cluster.sync();
      const XRec& res = rec_of(R, X_RES1, 0);
      keyB = (uint32_t)res.i[0];
      nkeepB = res.i[1];
      sel_rounds = res.i[2];
    } else {
      // -- full-row refinement (exact) --
      path = PATH_FULL;
      uint32_t keyK = 0u;
      int nkeepK = 0;
      Refine F;
      if (R.need_K) {
        F.lo = 1u;
        if (tcnt[0] >= K) F.lo = fkey(thr[0]);  // at least K members at or above thr[0]
        F.hi = fkey(gmax);
        F.above_cnt = 0;
        F.above_mfx = 0ull;
        F.n_in = nl;
        F.total_mfx = 0ull;
        F.rounds = 0;
        int buf = 0;
        for (int g = 0; g < 6 && F.lo < F.hi; ++g) {
          refine_round(R, F, buf, false, (long long)K, 0.0, 0u, -1, g == 0);
          buf ^= 1;
          if (F.n_in <= a.cap) break;
        }
        ref_rounds += F.rounds;
        if (F.lo == F.hi || F.n_in > a.cap) {
          keyK = F.lo;
          nkeepK = K - (int)F.above_cnt;
        } else {
          BandPred P{1, 0.f, F.lo, F.hi, 0u, -1};
          const int cnt = count_band(R, P, 0);
          XRec rec;
          rec.i[0] = cnt;
          push_rec(R, X_GCNT1, rec);
          cluster.sync();
          int off = 0, tot = 0;
          for (int r = 0; r < R.S; ++r) {
            const int cr = rec_of(R, X_GCNT1, r).i[0];
            if (r < R.rank) off += cr;
            tot += cr;
          }
          gather_band(R, P, 0, off, a.cap);
          cluster.sync();
          band_n = tot;
          if (leader) {
            int ngt = 0, r1 = 0;
            const uint32_t kK = pivot_count(R, tot, K, (int)F.above_cnt, ngt, r1);
            if (tid == 0) {
              XRec rr;
              rr.i[0] = (int)kK;
              rr.i[1] = K - ngt;
              rr.i[2] = r1;
              *reinterpret_cast<XRec*>(ms->scan_d + 128) = rr;
            }
            __syncthreads();
            push_rec(R, X_RES1, *reinterpret_cast<const XRec*>(ms->scan_d + 128));
          }
          cluster.sync();
          const XRec& res = rec_of(R, X_RES1, 0);
          keyK = (uint32_t)res.i[0];
          nkeepK = res.i[1];
          sel_rounds += res.i[2];
        }
      }
      keyB = keyK;
      nkeepB = nkeepK;
      if (R.need_P) {
        // S_k = {key > keyK} plus the first nkeepK copies of keyK (none when !need_K)
        int tie_limit = -1, tie_inc = -1;
        if (R.need_K) {
          const int ties = count_ties(R, keyK);
          XRec rec;
          rec.i[0] = ties;
          push_rec(R, X_TIES, rec);
          cluster.sync();
          int off = 0;
          for (int r = 0; r < R.rank; ++r) off += rec_of(R, X_TIES, r).i[0];
          tie_limit = max(0, min(ties, nkeepK - off));
          tie_inc = tie_limit;
        }
        Refine G;
        G.lo = R.need_K ? keyK : 1u;
        G.hi = fkey(gmax);
        G.above_cnt = 0;
        G.above_mfx = 0ull;
        G.n_in = nl;
        G.total_mfx = 0ull;
        G.rounds = 0;
        int buf = 0;
        for (int g = 0; g < 6; ++g) {
          refine_round(R, G, buf, true, 0, (double)pp, keyK, tie_inc, g == 0);
          buf ^= 1;
          if (G.n_in <= a.cap || G.lo == G.hi) break;
        }
        ref_rounds += G.rounds;
        const double target = (double)pp * (double)G.total_mfx / MASS_FX;
        const double above_m = (double)G.above_mfx / MASS_FX;
        if (G.n_in > a.cap || G.lo == G.hi) {
          // one key holds the boundary: its copies are taken in id order
          const uint32_t kp = G.lo;
          const double wv = (double)weight(R, key_to_float(kp));
          const int avail = (R.need_K && kp == keyK) ? nkeepK : (int)G.n_in;
          keyB = kp;
          nkeepB = topp_copies(above_m, wv, target, avail);
        } else {
          BandPred P{1, 0.f, G.lo, G.hi, keyK, tie_limit};
          const int cnt = count_band(R, P, 1);
          XRec rec;
          rec.i[0] = cnt;
          push_rec(R, X_GCNT2, rec);
          cluster.sync();
          int off = 0, tot = 0;
          for (int r = 0; r < R.S; ++r) {
            const int cr = rec_of(R, X_GCNT2, r).i[0];
            if (r < R.rank) off += cr;
            tot += cr;
          }
          gather_band(R, P, 1, off, a.cap);
          cluster.sync();
          band_n = tot;
          if (leader) {
            double agt = 0.0;
            int copies = 0, r2 = 0;
            const uint32_t kp = pivot_mass(R, tot, target, above_m, agt, copies, r2);
            const double wv = (double)weight(R, key_to_float(kp));
            if (tid == 0) {
              XRec rr;
              rr.i[0] = (int)kp;
              rr.i[1] = topp_copies(agt, wv, target, copies);
              rr.i[2] = r2;
              *reinterpret_cast<XRec*>(ms->scan_d + 128) = rr;
            }
            __syncthreads();
            push_rec(R, X_RES2, *reinterpret_cast<const XRec*>(ms->scan_d + 128));
          }
          cluster.sync();
          const XRec& res = rec_of(R, X_RES2, 0);
          keyB = (uint32_t)res.i[0];
          nkeepB = res.i[1];
          sel_rounds += res.i[2];
        }
      }
    }
  } else {
    path = PATH_ALL;  // every legal token kept
    keyB = 0u;
    nkeepB = 0;
  }

  // ---- 5. output stage -----------------------------------------------------
  // (a) per warp: copies of keyB, members above keyB and their mass
  {
    int ties = 0, gtc = 0, last = -1;
    float gtm = 0.f;
    for (int it = 0; it < R.iters; ++it) {
      const int e = vec_elem(R, it);
      float x[EPV];
      load_vec<DT>(R.data, e, x);
      const uint32_t lb = mask_bits(R, e);
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        if (!((lb >> j) & 1u) || is_neg_inf(x[j])) continue;
        const uint32_t k = fkey(x[j]);
        if (k > keyB) {
          ++gtc;
          if (!greedy) gtm += weight(R, x[j]);
          last = R.base_id + e + j;
        } else if (k == keyB) {
          ++ties;
        }
      }
    }
    ties = warp_sum(ties);
    gtc = warp_sum(gtc);
    const double wm = warp_sum((double)gtm);
    last = __reduce_max_sync(0xffffffffu, (unsigned)(last + 1)) - 1;
    if (lane == 0) {
      ms->wties[warp] = ties;
      ms->wgtc[warp] = gtc;
      ms->wgtm[warp] = wm;
      ms->wlast[warp] = last;
    }
    __syncthreads();
    if (tid == 0) {
      XRec rec;
      int tt = 0, tg = 0, tl = -1;
      double tm = 0.0;
      for (int w = 0; w < NWARP; ++w) {
        tt += ms->wties[w];
        tg += ms->wgtc[w];
        tm += ms->wgtm[w];
        tl = max(tl, ms->wlast[w]);
      }
      rec.i[0] = tt;
      rec.i[1] = tg;
      rec.i[2] = tl;
      rec.d[0] = tm;
      *reinterpret_cast<XRec*>(ms->scan_d + 128) = rec;
    }
    __syncthreads();
    push_rec(R, X_OUT, *reinterpret_cast<const XRec*>(ms->scan_d + 128));
    cluster.sync();
  }
  // (b) cluster-wide combination (identical in every CTA)
  const double wB = (greedy || keyB == 0u) ? 1.0 : (double)weight(R, key_to_float(keyB));
  double Mp = 0.0;
  int count = 0, my_off = 0, my_inc = 0;
  {
    int off = 0;
    for (int r = 0; r < R.S; ++r) {
      const XRec& q = rec_of(R, X_OUT, r);
      const int inc = max(0, min(q.i[0], nkeepB - off));
      if (r == R.rank) {
        my_off = off;
        my_inc = inc;
      }
      off += q.i[0];
      count += q.i[1] + inc;
      Mp += greedy ? 0.0 : q.d[0] + (double)inc * wB;
    }
  }
  const double u = (a.mode == MODE_SAMPLE && !greedy)
                       ? philox_uniform(a.seed ? a.seed[row] : 0ull, a.offset ? a.offset[row] : 0ull)
                       : 0.0;
  const double T = u * Mp;
  int target_cta = -1;
  double P_before = 0.0;
  if (a.mode == MODE_SAMPLE && !greedy) {
    double pre = 0.0;
    int lastnz = -1;
    double pre_last = 0.0;
    int off = 0;
    for (int r = 0; r < R.S; ++r) {
      const XRec& q = rec_of(R, X_OUT, r);
      const int inc = max(0, min(q.i[0], nkeepB - off));
      off += q.i[0];
      const double mr = q.d[0] + (double)inc * wB;
      if (q.i[1] + inc > 0) {
        lastnz = r;
        pre_last = pre;
      }
      if (target_cta < 0 && mr > 0.0 && pre + mr > T) {
        target_cta = r;
        P_before = pre;
      }
      pre += mr;
    }
    if (target_cta < 0) {
      target_cta = lastnz;
      P_before = pre_last;
    }
  }
  // (c) ordered output pass: mask words, probabilities, and the draw
  {
    int warp_tie_off = my_off;
    for (int w = 0; w < warp; ++w) warp_tie_off += ms->wties[w];
    constexpr int LPW = 32 / EPV;  // lanes per 32-bit mask word
    const float inv_mp = greedy ? 1.f : (float)(1.0 / Mp);
    int tie_run = warp_tie_off;
    for (int it = 0; it < R.iters; ++it) {
      const int e = vec_elem(R, it);
      float x[EPV];
      load_vec<DT>(R.data, e, x);
      const uint32_t lb = mask_bits(R, e);
      uint32_t bits = 0u, tbits = 0u;
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        if (!((lb >> j) & 1u) || is_neg_inf(x[j])) continue;
        const uint32_t k = fkey(x[j]);
        if (k > keyB) bits |= 1u << j;
        else if (k == keyB) tbits |= 1u << j;
      }
      const int nt = __popc(tbits);
      const int incl = warp_incl_scan(nt);
      int rr = tie_run + incl - nt;
#pragma unroll
      for (int j = 0; j < EPV; ++j)
        if ((tbits >> j) & 1u) {
          if (rr < nkeepB) bits |= 1u << j;
          ++rr;
        }
      tie_run += __shfl_sync(0xffffffffu, incl, 31);
      if (a.kept_mask) {
        uint32_t word = bits << (EPV * (lane % LPW));
#pragma unroll
        for (int o = 1; o < LPW; o <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, o);
        const int gw = (R.base_id + e) / 32;
        if ((lane % LPW) == 0 && gw < a.W) a.kept_mask[(size_t)row * a.W + gw] = word;
      }
      if (a.probs) {
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
          const int le = e + j;
          if (le < R.n_local) {
            float pr = 0.f;
            if ((bits >> j) & 1u) pr = greedy ? 1.f : weight(R, x[j]) * inv_mp;
            a.probs[(size_t)row * a.V + R.base_id + le] = pr;
          }
        }
      }
    }
  }
  // the draw: the CTA holding T scans its members in id order
  if (a.mode == MODE_SAMPLE && !greedy && R.rank == target_cta) {
    // per-warp member mass (ties split by the CTA-local offsets)
    double wpre = P_before;
    int twarp = -1;
    double tbase = 0.0;
    int lastw = -1;
    {
      int off = my_off;
      for (int w = 0; w < NWARP; ++w) {
        const int inc = max(0, min(ms->wties[w], nkeepB - off));
        off += ms->wties[w];
        const double mw = ms->wgtm[w] + (double)inc * wB;
        if (ms->wgtc[w] + inc > 0) lastw = w;
        if (twarp < 0 && mw > 0.0 && wpre + mw > T) {
          twarp = w;
          tbase = wpre;
        }
        wpre += mw;
      }
      if (twarp < 0) {
        twarp = lastw;
        // base of the last non-empty warp
        double pre = P_before;
        int off2 = my_off;
        for (int w = 0; w < lastw; ++w) {
          const int inc = max(0, min(ms->wties[w], nkeepB - off2));
          off2 += ms->wties[w];
          pre += ms->wgtm[w] + (double)inc * wB;
        }
        tbase = pre;
      }
    }
    if (warp == twarp) {
      int tie_run = my_off;
      for (int w = 0; w < warp; ++w) tie_run += ms->wties[w];
      double base = tbase;
      int found = -1, lastm = -1;
      for (int it = 0; it < R.iters && found < 0; ++it) {
        const int e = vec_elem(R, it);
        float x[EPV];
        load_vec<DT>(R.data, e, x);
        const uint32_t lb = mask_bits(R, e);
        uint32_t bits = 0u, tbits = 0u;
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
          if (!((lb >> j) & 1u) || is_neg_inf(x[j])) continue;
          const uint32_t k = fkey(x[j]);
          if (k > keyB) bits |= 1u << j;
          else if (k == keyB) tbits |= 1u << j;
        }
        const int nt = __popc(tbits);
        const int incl_t = warp_incl_scan(nt);
        int rr = tie_run + incl_t - nt;
#pragma unroll
        for (int j = 0; j < EPV; ++j)
          if ((tbits >> j) & 1u) {
            if (rr < nkeepB) bits |= 1u << j;
            ++rr;
          }
        tie_run += __shfl_sync(0xffffffffu, incl_t, 31);
        float wl[EPV];
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
          wl[j] = ((bits >> j) & 1u) ? weight(R, x[j]) : 0.f;
          ls += wl[j];
        }
        const float li = warp_incl_scan(ls);
        const float tot = __shfl_sync(0xffffffffu, li, 31);
        const bool cross = (base + (double)li > T) && ls > 0.f;
        const unsigned cm = __ballot_sync(0xffffffffu, cross);
        if (bits) lastm = R.base_id + e + (31 - __clz(bits));
        const int lm = (int)__reduce_max_sync(0xffffffffu, (unsigned)(lastm + 1)) - 1;
        lastm = lm;
        if (cm) {
          const int fl = __ffs(cm) - 1;
          if (lane == fl) {
            double c = base + (double)(li - ls);
            int tok = -1, lastl = -1;
#pragma unroll
            for (int j = 0; j < EPV; ++j)
              if ((bits >> j) & 1u) {
                c += (double)wl[j];
                lastl = R.base_id + e + j;
                if (tok < 0 && c > T) tok = lastl;
              }
            if (tok < 0) tok = lastl;
            found = tok;
          }
          found = __shfl_sync(0xffffffffu, found, fl);
        }
        base += (double)tot;
      }
      if (lane == 0) a.tokens[row] = (found >= 0) ? found : lastm;
    }
  }
  if (leader && tid == 0) {
    if (a.mode == MODE_SAMPLE && greedy && a.tokens) a.tokens[row] = gargmax;
    if (a.status) a.status[row] = ST_OK;
    if (a.kept_count) a.kept_count[row] = count;
    if (rinfo) {
      rinfo[0] = path;
      rinfo[1] = band_n;
      rinfo[2] = sel_rounds;
      rinfo[3] = ref_rounds;
    }
  }
}

}  // namespace smp
