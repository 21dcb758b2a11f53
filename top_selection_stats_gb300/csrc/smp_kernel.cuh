// smp_kernel.cuh -- fused top-k / top-p truncation and sampling for sm_103a.
// One thread-block cluster of S CTAs per row; the row is read from HBM once,
// into the CTAs' shared memories, and every later pass runs on chip.
//
// Per row (contract of the AI Infra KB note M012, sections 02-03):
//   temperature (0 = greedy argmax) -> legal mask -> top-k (earliest ids win
//   ties) -> top-p (shortest prefix whose mass reaches p) -> renormalise ->
//   inverse-CDF draw in token-id order with a Philox4x32-10 uniform.
//
// Pipeline:
//  1. each CTA bulk-copies its slice (cp.async.bulk + mbarrier, 4 chunks);
//  2. statistics pass as chunks land: the grammar mask is applied in place
//     (illegal -> -inf), then per 16-byte vector a packed max / min gives the
//     max, the argmax, NaN/+inf detection and the legal count; mean and
//     standard deviation come from a 1-in-8 subsample (Qrita paper notes, key
//     design 1: sample mean and deviation); one DSMEM exchange;
//  3. sigma truncation (Qrita key design 1): t = mu + delta*sigma, lowered by
//     0.2|t|; four thresholds are counted in one pass, and candidates above the
//     lowest are compacted in id order into per-warp buffers in the same pass
//     (vectors whose packed max is below the threshold are skipped);
//  4. the leader CTA pulls the chosen band through DSMEM and one warp runs the
//     three-pivot search for the k-th value (Qrita key design 2), the tie quota
//     (key design 3), the same search on mass for top-p, and the draw;
//  5. when no band validates, an exact multi-pivot refinement: each pass
//     counts (and weighs) the current window against 8 pivots in registers,
//     the cluster merges the counts, and the window shrinks ~9x per pass until
//     it fits the leader's buffer;
//  6. every CTA writes its packed kept-mask words (and probabilities); rows
//     whose kept set was not gathered draw by a cluster-wide prefix of masses
//     and an id-order scan in the CTA that holds the draw.
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
  int cap;      // candidate capacity of the leader's band buffer
  int use_tma;  // rows are 16-byte aligned: stage with bulk copies
  float delta[DTAB];
};

constexpr int CL = 2048;         // local candidate buffer per CTA (entries)
constexpr int CLW = CL / NWARP;  // per warp
constexpr int NPIV = 8;          // pivots per refinement pass
constexpr int NOT_MEMBER = (int)0x80000000;
constexpr uint32_t KEY_MIN = 0x00800000u;  // fkey(-FLT_MAX): the smallest legal key

// Exchange record: each CTA pushes one into a slot of every CTA (DSMEM).
struct XRec {
  double d[10];
  int i[16];
};
enum Xid { X_STATS = 0, X_SIGMA, X_REF0, X_REF1, X_GCNT, X_RES, X_OUT, NX };

struct Misc {
  uint64_t mbar[NCHUNK];
  double rd[NWARP * 10];
  float rf[NWARP];
  int ri[NWARP * 16];
  int wcnt[NPIV + 1][NWARP];  // per-warp counts: sigma thresholds / refinement pivots
  int wst[NWARP];             // per-warp stored candidates
  double wmass[NWARP];        // per-warp member mass (distributed output)
  int wmem[NWARP];            // per-warp member count
  int wlast[NWARP];           // per-warp last member id
  int wties[NWARP];           // per-warp copies of the boundary key
  int seg[MAX_CLUSTER * NWARP + 1];
  XRec tmp;
  int bflag[4];
};

__host__ __device__ inline int esize_of(int dt) { return dt == DT_F32 ? 4 : 2; }
__host__ __device__ inline int epv_of(int dt) { return 16 / esize_of(dt); }
__host__ __device__ inline int slice_align(int dt) { return NWARP * 32 * epv_of(dt); }

struct Layout {
  int off_data, off_mw, off_lk, off_li, off_bk, off_bi, off_xch, off_misc, total;
};
__host__ __device__ inline int align_up(int v, int a) { return (v + a - 1) / a * a; }
__host__ __device__ inline Layout make_layout(int L, int dt, int cap, int S) {
  Layout l;
  int o = 0;
  l.off_data = o;
  o = align_up(o + L * esize_of(dt), 128);
  l.off_mw = o;
  o = align_up(o + (L / 32) * 4, 16);
  l.off_lk = o;
  o = align_up(o + CL * 4, 16);
  l.off_li = o;
  o = align_up(o + CL * 4, 16);
  l.off_bk = o;
  o = align_up(o + cap * 4, 16);
  l.off_bi = o;
  o = align_up(o + cap * 4, 16);
  l.off_xch = o;
  o = align_up(o + NX * S * (int)sizeof(XRec), 16);
  l.off_misc = o;
  o = align_up(o + (int)sizeof(Misc), 128);
  l.total = o;
  return l;
}

template <int DT>
struct Row {
  int S, rank, row, L, n_local, base_id, Lw, iters;
  char* data;
  uint32_t* mw;
  uint32_t* lk;  // local candidate keys
  int* li;       // local candidate ids
  uint32_t* bk;  // leader band keys
  int* bi;       // leader band ids (bit 31: not a member)
  XRec* xch;
  Misc* ms;
  bool has_mask;
  float temp, m_z, gmax;
  float c2;  // log2(e) / T, for the fast bulk weights
};

// ---------------------------------------------------------------------------
// Element access
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ uint4 ld_vec(const Row<DT>& R, int e) {
  return *reinterpret_cast<const uint4*>(R.data + (size_t)e * (DT == DT_F32 ? 4 : 2));
}
template <int DT>
__device__ __forceinline__ void unpack(const uint4 r, float (&x)[16 / (DT == DT_F32 ? 4 : 2)]) {
  if constexpr (DT == DT_F32) {
    x[0] = __uint_as_float(r.x);
    x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z);
    x[3] = __uint_as_float(r.w);
  } else {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if constexpr (DT == DT_BF16) {
        x[2 * q] = __uint_as_float(w[q] << 16);
        x[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
      } else {
        x[2 * q] = __half2float(__ushort_as_half((unsigned short)(w[q] & 0xffffu)));
        x[2 * q + 1] = __half2float(__ushort_as_half((unsigned short)(w[q] >> 16)));
      }
    }
  }
}
// Max over the vector; NaN anywhere gives NaN.
template <int DT>
__device__ __forceinline__ float vmax_nan(const uint4 r) {
  if constexpr (DT == DT_F32) {
    const float a = __uint_as_float(r.x), b = __uint_as_float(r.y), c = __uint_as_float(r.z),
                d = __uint_as_float(r.w);
    const float m = fmaxf(fmaxf(a, b), fmaxf(c, d));
    return (isnan(a) || isnan(b) || isnan(c) || isnan(d)) ? __int_as_float(0x7fffffff) : m;
  } else if constexpr (DT == DT_BF16) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return __bfloat162float(__hmax_nan(__low2bfloat16(m), __high2bfloat16(m)));
  } else {
    const __half2 a = *reinterpret_cast<const __half2*>(&r.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&r.y);
    const __half2 c = *reinterpret_cast<const __half2*>(&r.z);
    const __half2 d = *reinterpret_cast<const __half2*>(&r.w);
    const __half2 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return __half2float(__hmax_nan(__low2half(m), __high2half(m)));
  }
}
// Max over the vector ignoring NaN (used once the row is known finite).
template <int DT>
__device__ __forceinline__ float vmax(const uint4 r) {
  if constexpr (DT == DT_F32) {
    return fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                 fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
  } else if constexpr (DT == DT_BF16) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
    return fmaxf(__low2float(m), __high2float(m));
  } else {
    const __half2 a = *reinterpret_cast<const __half2*>(&r.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&r.y);
    const __half2 c = *reinterpret_cast<const __half2*>(&r.z);
    const __half2 d = *reinterpret_cast<const __half2*>(&r.w);
    const __half2 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
    return fmaxf(__low2float(m), __high2float(m));
  }
}
template <int DT>
__device__ __forceinline__ float vmin(const uint4 r) {
  if constexpr (DT == DT_F32) {
    return fminf(fminf(__uint_as_float(r.x), __uint_as_float(r.y)),
                 fminf(__uint_as_float(r.z), __uint_as_float(r.w)));
  } else if constexpr (DT == DT_BF16) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 m = __hmin2(__hmin2(a, b), __hmin2(c, d));
    return fminf(__low2float(m), __high2float(m));
  } else {
    const __half2 a = *reinterpret_cast<const __half2*>(&r.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&r.y);
    const __half2 c = *reinterpret_cast<const __half2*>(&r.z);
    const __half2 d = *reinterpret_cast<const __half2*>(&r.w);
    const __half2 m = __hmin2(__hmin2(a, b), __hmin2(c, d));
    return fminf(__low2float(m), __high2float(m));
  }
}
// Replace masked-out elements (bit 0) by -inf.
template <int DT>
__device__ __forceinline__ uint4 apply_mask(uint4 r, uint32_t lb) {
  if constexpr (DT == DT_F32) {
    if (!(lb & 1u)) r.x = 0xff800000u;
    if (!(lb & 2u)) r.y = 0xff800000u;
    if (!(lb & 4u)) r.z = 0xff800000u;
    if (!(lb & 8u)) r.w = 0xff800000u;
    return r;
  } else {
    constexpr uint32_t NEG2 = (DT == DT_BF16) ? 0xff80ff80u : 0xfc00fc00u;
    uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t b = (lb >> (2 * q)) & 3u;
      const uint32_t sel = ((b & 1u) ? 0x0000ffffu : 0u) | ((b & 2u) ? 0xffff0000u : 0u);
      w[q] = (w[q] & sel) | (NEG2 & ~sel);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}
__device__ __forceinline__ bool is_neg_inf(float x) { return __float_as_uint(x) == 0xff800000u; }

// Weight of a logit relative to the row maximum, exactly as the contract
// states it: expf(fl32(x / T) - fl32(max / T)).
template <int DT>
__device__ __forceinline__ float weight(const Row<DT>& R, float x) {
  return expf(__fdiv_rn(x, R.temp) - R.m_z);
}
// Cheap weight for bulk sums that only steer band choices:
// 2^((x - max) * log2(e) / T) with the hardware base-2 exponential.
__device__ __forceinline__ float fast_exp2(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
template <int DT>
__device__ __forceinline__ float fast_weight(const Row<DT>& R, float x) {
  return fast_exp2((x - R.gmax) * R.c2);
}

template <int DT>
__device__ __forceinline__ int vec_elem(const Row<DT>& R, int it) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  return (threadIdx.x >> 5) * R.Lw + it * 32 * EPV + (threadIdx.x & 31) * EPV;
}

// ---------------------------------------------------------------------------
// Cluster exchange
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ void push_all(const Row<DT>& R, int xid, const XRec& rec) {
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

// Block reduction of nvi ints and nvd doubles into rec (every thread gets it).
template <int DT>
__device__ void block_reduce_rec(const Row<DT>& R, const int* vi, int nvi, const double* vd,
                                 int nvd, XRec& rec) {
  Misc* ms = R.ms;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  for (int q = 0; q < nvi; ++q) {
    const int s = __reduce_add_sync(0xffffffffu, vi[q]);
    if (lane == 0) ms->ri[q * NWARP + warp] = s;
  }
  for (int q = 0; q < nvd; ++q) {
    const double s = warp_sum(vd[q]);
    if (lane == 0) ms->rd[q * NWARP + warp] = s;
  }
  __syncthreads();
  for (int q = 0; q < nvi; ++q) {
    int s = 0;
    for (int w = 0; w < NWARP; ++w) s += ms->ri[q * NWARP + w];
    rec.i[q] = s;
  }
  for (int q = 0; q < nvd; ++q) {
    double s = 0.0;
    for (int w = 0; w < NWARP; ++w) s += ms->rd[q * NWARP + w];
    rec.d[q] = s;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Leader-side selection on the band (keys bk, ids bi in id order), one warp.
// Lane l owns the contiguous entries [l*ch, min(n, (l+1)*ch)).
// Three-pivot search (Qrita key design 2) in the order-preserving key space:
// pivots tau_q = lo + q(hi - lo)/4; one pass gives N = #{key > tau}, the
// smallest key above tau and its multiplicity; stop when N >= K and
// N - mult < K.
// ---------------------------------------------------------------------------
template <int DT>
__device__ void warp_minmax(const Row<DT>& R, int n, uint32_t& lo, uint32_t& hi) {
  const int lane = threadIdx.x & 31, ch = (n + 31) / 32;
  const int j0 = lane * ch, j1 = min(n, j0 + ch);
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int j = j0; j < j1; ++j) {
    if (R.bi[j] & NOT_MEMBER) continue;
    mn = min(mn, R.bk[j]);
    mx = max(mx, R.bk[j]);
  }
  lo = __reduce_min_sync(0xffffffffu, mn);
  hi = __reduce_max_sync(0xffffffffu, mx);
}

template <int DT>
__device__ uint32_t warp_pivot_count(const Row<DT>& R, int n, int K, int above, int& ngt,
                                     int& rounds) {
  const int lane = threadIdx.x & 31, ch = (n + 31) / 32;
  const int j0 = lane * ch, j1 = min(n, j0 + ch);
  uint32_t lo, hi;
  warp_minmax(R, n, lo, hi);
  rounds = 0;
  for (int guard = 0; guard < 64 && lo < hi; ++guard) {
    ++rounds;
    uint32_t tau[3];
    const unsigned long long span = (unsigned long long)(hi - lo);
#pragma unroll
    for (int q = 0; q < 3; ++q) tau[q] = lo + (uint32_t)((span * (q + 1)) / 4);
    int cnt[3] = {0, 0, 0}, mc[3] = {0, 0, 0};
    uint32_t mk[3] = {0xffffffffu, 0xffffffffu, 0xffffffffu};
    for (int j = j0; j < j1; ++j) {
      if (R.bi[j] & NOT_MEMBER) continue;
      const uint32_t k = R.bk[j];
#pragma unroll
      for (int q = 0; q < 3; ++q)
        if (k > tau[q]) {
          ++cnt[q];
          if (k < mk[q]) {
            mk[q] = k;
            mc[q] = 1;
          } else if (k == mk[q]) {
            ++mc[q];
          }
        }
    }
    bool done = false;
    uint32_t nlo = lo, nhi = hi, found = 0u;
    int found_gt = 0;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int N = above + __reduce_add_sync(0xffffffffu, cnt[q]);
      const uint32_t m = __reduce_min_sync(0xffffffffu, mk[q]);
      const int c = __reduce_add_sync(0xffffffffu, (mk[q] == m) ? mc[q] : 0);
      if (!done && N >= K && N - c < K) {
        done = true;
        found = m;
        found_gt = N - c;
      }
      if (N >= K) nlo = max(nlo, (N - c >= K) ? m + 1u : tau[q] + 1u);
      else nhi = min(nhi, tau[q]);
    }
    if (done) {
      ngt = found_gt;
      return found;
    }
    lo = nlo;
    hi = nhi;
  }
  int c = 0;
  for (int j = j0; j < j1; ++j)
    if (!(R.bi[j] & NOT_MEMBER) && R.bk[j] > lo) ++c;
  ngt = above + __reduce_add_sync(0xffffffffu, c);
  return lo;
}

// Top-p boundary among members by mass: the key v with
// above + mass{key > v} < target <= above + mass{key >= v}.  bw holds weights.
template <int DT>
__device__ uint32_t warp_pivot_mass(const Row<DT>& R, const float* bw, int n, double target,
                                    double above, double& a_gt, int& copies, int& rounds) {
  const int lane = threadIdx.x & 31, ch = (n + 31) / 32;
  const int j0 = lane * ch, j1 = min(n, j0 + ch);
  uint32_t lo, hi;
  warp_minmax(R, n, lo, hi);
  rounds = 0;
  for (int guard = 0; guard < 64 && lo < hi; ++guard) {
    ++rounds;
    uint32_t tau[3];
    const unsigned long long span = (unsigned long long)(hi - lo);
#pragma unroll
    for (int q = 0; q < 3; ++q) tau[q] = lo + (uint32_t)((span * (q + 1)) / 4);
    float ms[3] = {0.f, 0.f, 0.f};
    int mc[3] = {0, 0, 0};
    uint32_t mk[3] = {0xffffffffu, 0xffffffffu, 0xffffffffu};
    for (int j = j0; j < j1; ++j) {
      if (R.bi[j] & NOT_MEMBER) continue;
      const uint32_t k = R.bk[j];
      const float w = bw[j];
#pragma unroll
      for (int q = 0; q < 3; ++q)
        if (k > tau[q]) {
          ms[q] += w;
          if (k < mk[q]) {
            mk[q] = k;
            mc[q] = 1;
          } else if (k == mk[q]) {
            ++mc[q];
          }
        }
    }
    bool done = false;
    uint32_t nlo = lo, nhi = hi, found = 0u;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const double A = above + warp_sum((double)ms[q]);
      const uint32_t m = __reduce_min_sync(0xffffffffu, mk[q]);
      const int c = __reduce_add_sync(0xffffffffu, (mk[q] == m) ? mc[q] : 0);
      const double wm = (c > 0) ? (double)c * (double)weight(R, key_to_float(m)) : 0.0;
      if (!done && c > 0 && A >= target && A - wm < target) {
        done = true;
        found = m;
      }
      if (A >= target && c > 0) nlo = max(nlo, (A - wm >= target) ? m + 1u : tau[q] + 1u);
      else nhi = min(nhi, tau[q]);
    }
    if (done) {
      lo = hi = found;
      break;
    }
    if (nlo > nhi) break;
    lo = nlo;
    hi = nhi;
  }
  // the boundary must be a member key
  uint32_t nxt = 0xffffffffu;
  for (int j = j0; j < j1; ++j)
    if (!(R.bi[j] & NOT_MEMBER) && R.bk[j] >= lo) nxt = min(nxt, R.bk[j]);
  nxt = __reduce_min_sync(0xffffffffu, nxt);
  const uint32_t v = (nxt != 0xffffffffu) ? nxt : hi;
  float s = 0.f;
  int c = 0;
  for (int j = j0; j < j1; ++j) {
    if (R.bi[j] & NOT_MEMBER) continue;
    if (R.bk[j] > v) s += bw[j];
    if (R.bk[j] == v) ++c;
  }
  a_gt = above + warp_sum((double)s);
  copies = __reduce_add_sync(0xffffffffu, c);
  return v;
}

// Copies of the boundary value kept by top-p: copy j (id order) is kept iff
// a_gt + j * w < target; at least one.
__device__ __forceinline__ int topp_copies(double a_gt, double w, double target, int avail) {
  if (avail <= 0) return 0;
  const double need = (target - a_gt) / w;
  long long n = (need <= 0.0) ? 1 : (long long)ceil(need);
  if (n < 1) n = 1;
  if (n > avail) n = avail;
  return (int)n;
}

// Keep members with key > kB and the first nB copies of kB (id order); mark
// the rest NOT_MEMBER.  One warp, contiguous lane chunks.
template <int DT>
__device__ void warp_restrict(const Row<DT>& R, int n, uint32_t kB, int nB) {
  const int lane = threadIdx.x & 31, ch = (n + 31) / 32;
  const int j0 = lane * ch, j1 = min(n, j0 + ch);
  int t = 0;
  for (int j = j0; j < j1; ++j)
    if (!(R.bi[j] & NOT_MEMBER) && R.bk[j] == kB) ++t;
  const int incl = warp_incl_scan(t);
  int rank = incl - t;
  for (int j = j0; j < j1; ++j) {
    if (R.bi[j] & NOT_MEMBER) continue;
    const uint32_t k = R.bk[j];
    bool mem = k > kB;
    if (k == kB) {
      mem = rank < nB;
      ++rank;
    }
    if (!mem) R.bi[j] |= NOT_MEMBER;
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Ordered walk: warp w owns [w*Lw, (w+1)*Lw); per iteration lane l holds the
// EPV elements at vec_elem(it).  Increasing id order within a warp.
// ---------------------------------------------------------------------------

// Write the members flagged in `bits` of this iteration to dst at base + warp-rank.
template <int DT>
__device__ __forceinline__ void warp_emit(const Row<DT>& R, int e, const float* x, uint32_t bits,
                                          int& base, uint32_t* dk, int* di, int limit) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  const int c = __popc(bits);
  const int incl = warp_incl_scan(c);
  int pos = base + incl - c;
#pragma unroll
  for (int j = 0; j < EPV; ++j)
    if ((bits >> j) & 1u) {
      if (pos < limit) {
        dk[pos] = fkey(x[j]);
        di[pos] = R.base_id + e + j;
      }
      ++pos;
    }
  base += __shfl_sync(0xffffffffu, incl, 31);
}

// Per-warp tie copies of key kB in this CTA -> ms->wties; returns the CTA total.
template <int DT>
__device__ int count_ties(const Row<DT>& R, uint32_t kB) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  const float vB = key_to_float(kB);
  int c = 0;
  for (int it = 0; it < R.iters; ++it) {
    const uint4 r = ld_vec(R, vec_elem(R, it));
    if (!__any_sync(0xffffffffu, vmax<DT>(r) >= vB)) continue;
    float x[EPV];
    unpack<DT>(r, x);
#pragma unroll
    for (int j = 0; j < EPV; ++j) c += (fkey(x[j]) == kB && !is_neg_inf(x[j])) ? 1 : 0;
  }
  c = __reduce_add_sync(0xffffffffu, c);
  if ((threadIdx.x & 31) == 0) R.ms->wties[threadIdx.x >> 5] = c;
  __syncthreads();
  int tot = 0;
  for (int w = 0; w < NWARP; ++w) tot += R.ms->wties[w];
  __syncthreads();
  return tot;
}

// ---------------------------------------------------------------------------
// Statistics pass (chunk-major, overlaps the bulk copies in flight).
// ---------------------------------------------------------------------------
struct Stats {
  float bx;
  int bid;
  int nl, nonfin, timeout, ns;
  float s, s2;
};

template <int DT>
__device__ Stats stats_pass(const Row<DT>& R, const KArgs& a, const int* chunk_bulk) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  constexpr uint32_t FULL = (1u << EPV) - 1u;
  const int nvec = R.L / EPV, cvec = nvec / NCHUNK;
  Stats st{-INFINITY, 0x7fffffff, 0, 0, 0, 0, 0.f, 0.f};
  int bestvi = -1;
  for (int c = 0; c < NCHUNK; ++c) {
    if (a.use_tma && chunk_bulk[c] > 0) {
      if (!mbar_wait_bounded(&R.ms->mbar[c], 0u, 4000000000ll)) st.timeout = 1;
    }
    for (int vi = c * cvec + threadIdx.x; vi < (c + 1) * cvec; vi += NT) {
      const int e = vi * EPV;
      uint4 r = ld_vec(R, e);
      if (R.has_mask) {
        const uint32_t lb = (R.mw[e >> 5] >> (e & 31)) & FULL;
        if (lb != FULL) {
          r = apply_mask<DT>(r, lb);
          *reinterpret_cast<uint4*>(R.data + (size_t)e * (DT == DT_F32 ? 4 : 2)) = r;
        }
      }
      const float mx = vmax_nan<DT>(r);
      if (isnan(mx) || mx == INFINITY) st.nonfin = 1;
      if (mx > st.bx) {
        st.bx = mx;
        bestvi = vi;
      }
      const float mn = vmin<DT>(r);
      float x[EPV];
      unpack<DT>(r, x);
      if (mn > -INFINITY) {
        st.nl += EPV;
      } else {
#pragma unroll
        for (int j = 0; j < EPV; ++j) st.nl += is_neg_inf(x[j]) ? 0 : 1;
      }
      const float x0 = x[0];
      if (x0 > -INFINITY && x0 < INFINITY) {
        st.s += x0;
        st.s2 = fmaf(x0, x0, st.s2);
        st.ns += 1;
      }
    }
  }
  if (bestvi >= 0 && !isnan(st.bx)) {
    float x[EPV];
    unpack<DT>(ld_vec(R, bestvi * EPV), x);
    int j = EPV - 1;
#pragma unroll
    for (int q = EPV - 1; q >= 0; --q)
      if (x[q] == st.bx) j = q;
    st.bid = R.base_id + bestvi * EPV + j;
  }
  return st;
}

__device__ __forceinline__ void argmax_combine(float& bx, int& bid, float ox, int oid) {
  if (ox > bx || (ox == bx && oid < bid)) {
    bx = ox;
    bid = oid;
  }
}

// ---------------------------------------------------------------------------
// Multi-pivot refinement (exact full-row fallback).  Window [lo, hi] in key
// space; members above hi are accounted in `above`.  One pass counts (and
// weighs, for top-p) the window against NPIV pivots in registers; the
// cluster merges; the window shrinks to the sub-window holding the target.
// The domain may exclude copies of tie_key beyond a per-CTA quota
// (tie_inc >= 0): those copies are skipped per element and added in
// aggregate (they all have the same value).
// ---------------------------------------------------------------------------
struct Win {
  uint32_t lo, hi;
  long long above_cnt;
  double above_mass;
  long long n_in;
  int sub;  // chosen sub-window index of the last pass (0..NPIV)
};

// With target_frac > 0 the mass target is set after the merge to
// target_frac * (mass above the window + mass of the window).
template <int DT>
__device__ void refine_pass(const Row<DT>& R, Win& Wd, int xid, bool mass, long long kneed,
                            double& target, double target_frac, uint32_t tie_key, int tie_inc,
                            float w_tie, uint32_t (&piv)[NPIV + 1]) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  cg::cluster_group cluster = cg::this_cluster();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lo = Wd.lo, hi = Wd.hi;
  const unsigned long long span = (unsigned long long)(hi - lo) + 1ull;
  piv[0] = lo;
#pragma unroll
  for (int m = 1; m <= NPIV; ++m) piv[m] = lo + (uint32_t)((span * m) / (NPIV + 1));
  const float vlo = key_to_float(lo);
  int cnt[NPIV + 1];
  float msum[NPIV + 1];
#pragma unroll
  for (int m = 0; m <= NPIV; ++m) {
    cnt[m] = 0;
    msum[m] = 0.f;
  }
  for (int it = 0; it < R.iters; ++it) {
    const uint4 r = ld_vec(R, vec_elem(R, it));
    if (!__any_sync(0xffffffffu, vmax<DT>(r) >= vlo)) continue;
    float x[EPV];
    unpack<DT>(r, x);
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      if (is_neg_inf(x[j])) continue;
      const uint32_t k = fkey(x[j]);
      if (k < lo || k > hi) continue;
      if (tie_inc >= 0 && k == tie_key) continue;
      float w = 0.f;
      if (mass) w = weight(R, x[j]);
#pragma unroll
      for (int m = 0; m <= NPIV; ++m)
        if (k >= piv[m]) {
          ++cnt[m];
          if (mass) msum[m] += w;
        }
    }
  }
  // copies of the tie key kept by this CTA, in aggregate
  if (tie_inc > 0 && tie_key >= lo && tie_key <= hi && threadIdx.x == 0) {
#pragma unroll
    for (int m = 0; m <= NPIV; ++m)
      if (tie_key >= piv[m]) {
        cnt[m] += tie_inc;
        if (mass) msum[m] += (float)tie_inc * w_tie;
      }
  }
  // per-warp counts (kept for the gather offsets) and the CTA record
#pragma unroll
  for (int m = 0; m <= NPIV; ++m) {
    const int wc = __reduce_add_sync(0xffffffffu, cnt[m]);
    if (lane == 0) R.ms->wcnt[m][warp] = wc;
  }
  double md[NPIV + 1];
#pragma unroll
  for (int m = 0; m <= NPIV; ++m) md[m] = (double)msum[m];
  XRec rec;
  block_reduce_rec(R, cnt, NPIV + 1, md, mass ? NPIV + 1 : 0, rec);
  if (!mass)
    for (int m = 0; m <= NPIV; ++m) rec.d[m] = 0.0;
  push_all(R, xid, rec);
  cluster.sync();
  long long C[NPIV + 2];
  double M[NPIV + 2];
  for (int m = 0; m <= NPIV; ++m) {
    C[m] = 0;
    M[m] = 0.0;
    for (int q = 0; q < R.S; ++q) {
      C[m] += rec_of(R, xid, q).i[m];
      M[m] += rec_of(R, xid, q).d[m];
    }
  }
  C[NPIV + 1] = 0;
  M[NPIV + 1] = 0.0;
  if (mass && target_frac > 0.0) target = target_frac * (Wd.above_mass + M[0]);
  // sub-window m = [piv[m], piv[m+1]-1] holds the target when the members at
  // or above piv[m] reach it and those at or above piv[m+1] do not
  int sel = 0;
  for (int m = NPIV; m >= 0; --m) {
    const bool reach = mass ? (Wd.above_mass + M[m] >= target) : (Wd.above_cnt + C[m] >= kneed);
    if (reach && (C[m] - C[m + 1]) > 0) {
      sel = m;
      break;
    }
  }
  const uint32_t nlo = piv[sel];
  const uint32_t nhi = (sel == NPIV) ? hi : piv[sel + 1] - 1u;
  Wd.above_cnt += C[sel + 1];
  Wd.above_mass += M[sel + 1];
  Wd.n_in = C[sel] - C[sel + 1];
  Wd.lo = nlo;
  Wd.hi = max(nlo, nhi);
  Wd.sub = sel;
}

}  // namespace smp

#include "smp_kernel_main.cuh"
