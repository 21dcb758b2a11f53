// smp_split.cuh -- the sampler for bf16 / fp16 logits: every row split over a
// small thread-block cluster, every slice streamed once from HBM.
//
// The contract is the one in include/smp.h (AI Infra KB note M012, sections
// 02-03; lecture notes "Decoding: Sampling, Beam Search and Speculative
// Decoding", section 3.3): temperature, legal mask, top-k with the earliest
// ids winning ties, top-p as the shortest prefix reaching p, renormalise, and
// an inverse-CDF draw in token-id order.
//
// Layout on GB300.  The work is one pass over the logits (Qrita paper notes:
// the full-vocabulary passes are the cost), so every row of a launch streams
// at once: a row is split over C CTAs of one cluster (C chosen so that the
// launch has at least two CTAs per SM), and each CTA streams its slice
// through a ring of four 8 KB bulk copies (cp.async.bulk + mbarrier, no
// multicast):
//   sample   the first stage of a slice is also a sample: its maximum, and for
//            top-k rows a fine key histogram, place this CTA's own candidate
//            threshold `lo` (Qrita's sigma truncation, read as a quantile of
//            the sample); no exchange is needed before the stream.
//   stream   per vector: maximum and first id, -inf count, NaN / +inf check
//            (packed bf16x2 / f16x2 max and min), the grammar mask, and by
//            row class: top-k rows mark the vectors holding a value >= lo
//            (their candidates are listed after the stream from L2); flat
//            top-p rows count every key of a 2048-key window below the
//            sample's maximum (one 32-bit counter per 16-bit key) and sum an
//            approximate row mass; keep-all rows accumulate per-(stage, warp)
//            masses and write their kept-mask words.
//   resolve  one cluster barrier exchanges the statistics; every CTA reads
//            all CTAs' per-key counts (distributed shared memory) and finds,
//            identically, the k-th largest key with its tie quota, the kept
//            set's mass and the top-p boundary key with the number of its
//            copies kept (a key's mass is its count times its weight; each
//            CTA's share of the boundary copies follows from the CTAs' rank
//            order, earliest ids first).  A second barrier exchanges the
//            mass each CTA keeps; the CTA holding the draw finds the token.
//   outputs  from the candidate list when it holds the kept set; otherwise a
//            second pass streams the slice through the ring again: mask bits
//            by packed compares, the drawing CTA's per-(stage, warp) kept
//            masses from a table of the kept keys' weights, and boundary
//            copies listed during the pass when their id cut is still open.
// Rows the stream cannot settle (a list or window that misses the boundary,
// keep-all rows whose maximum lies far above the sample's) take the exact
// window search: key windows histogrammed over the slice re-read from global
// memory (L2), sliding down until both boundaries are inside.  Masses that
// decide kept sets are fixed-point integers (units of 2^-40 of the largest
// weight), so sums, prefixes and decisions are exact and equal in every CTA.
#pragma once

#include "smp_device.cuh"

namespace smp {

constexpr int XNT = 128;            // threads per CTA
constexpr int XNW = XNT / 32;       // warps per CTA
constexpr int XSB = 8192;           // bytes per ring stage
constexpr int XNS = 4;              // ring stages
constexpr int XVS = XSB / 16;       // 16-byte vectors per stage (512)
constexpr int XVW = XVS / XNW;      // vectors per warp per stage (128), a contiguous id range
constexpr int XSUB = XVW / 32;      // vectors per lane per stage (4)
constexpr int XMAXST = 64;          // stages per slice, at most (512 KB)
constexpr int XMAXC = 8;            // CTAs per row, at most (portable cluster size)
constexpr int XSW = 128;            // fine sample bins below a stage's maximum (top-k threshold)
constexpr int XMAXWIN = 36;         // windows of one row, at most
constexpr int XWT = XNS * XSB / 16;  // keys whose weight the resolution stores (2048)
constexpr long long XDRAIN = 4000000000ll;  // cycles the drain after an expired wait may take
constexpr int XBL = 1024;     // copies of the boundary value pass C lists for the id cut
constexpr uint32_t XFM = 8;  // flat rows: the counted window reaches cap / XFM keys above the sample

enum XClass { XC_ERROR = 0, XC_GREEDY = 1, XC_ALL = 2, XC_TOPK = 3, XC_FLAT = 4, XC_FLATL = 5 };

struct XArgs {
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
  float* logprob;
  int* row_info;
  int mode;
  int C;            // CTAs per row (the cluster)
  int SL;           // slice length in values, a multiple of 256
  int wf;           // keys per histogram window (2048 or 4096)
  int cap;          // candidate-list capacity per CTA
  int aligned;      // rows start on 16-byte boundaries: bulk copies
  long long wait_limit;  // clock cycles a bounded wait may take
};

// Shared-memory layout (bytes from the dynamic base).
__host__ __device__ inline int xoff_hist() { return XNS * XSB; }
__host__ __device__ inline int xoff_ckey(int wf) { return XNS * XSB + wf * 2; }
__host__ __device__ inline int xoff_cid(int wf, int cap) {
  return xoff_ckey(wf) + ((cap * 2 + 15) & ~15);
}
__host__ __device__ inline int xoff_sh(int wf, int cap) { return xoff_cid(wf, cap) + cap * 4; }

// What each CTA publishes to the cluster after the stream (B2).
struct XPub {
  uint32_t kmax;  // largest legal key seen (0: none)
  int amax;       // smallest id holding it
  int nleg;       // legal values (mask allows, not -inf)
  int flags;      // 1 NaN/+inf legal, 2 wait expired, 4 list overflow, 8 above window,
                  // 16 keep-all reference too low
  int ncand;      // candidates listed
  uint32_t lo, hw;  // this CTA's candidate window: keys [lo, hw]
  uint32_t skey;  // largest key of this CTA's first stage (the local sample)
  float xsv;      // the reference of this CTA's masses: that key's value (0 if none)
  int pad[1];
  double mass;    // flat / keep-all rows: legal mass relative to the local sample's maximum
};
static_assert(sizeof(XPub) % 16 == 0, "published record: whole 16-byte units");
constexpr int XPUBW = (int)sizeof(XPub) / 4;

struct XWin {
  uint32_t hi, lo;
  uint64_t A, MA, myMA;
};

struct XSh {
  uint64_t bar[XNS];
  XPub stage;
  XPub pub2[XMAXC];
  uint64_t km[XMAXC];
  uint64_t uf[XMAXC];
  uint32_t kbelow[XMAXC];   // window search: each CTA's largest legal key below the window
  float rwf[XMAXST][XNW];   // keep-all rows: per-(stage, warp) masses
  XWin win[XMAXWIN];
  uint32_t h64[64];         // radix counters of the tie cut
  uint64_t q[XNW];
  float f[XNW];
  int wi[XNW];
  int bi[24];                // [23]: pass C's expired waits (set remotely)
  uint64_t bq[8];
  double bd[8];
  int ncand;
  int flags;
};

template <int DT>
struct XT;
template <>
struct XT<DT_BF16> {
  typedef __nv_bfloat162 T2;
  static constexpr uint32_t NINF = 0xff80u;   // raw -inf
  static constexpr uint32_t KNINF = 0x0080u;  // key of -inf
  static constexpr int SB = 3;                // sample bins: 8 keys, 1/16 octave
  static constexpr int MB = 7;                // explicit significand bits
  static constexpr int EB = 127 + 7;          // value = significand * 2^(e - EB)
  static __device__ __forceinline__ float f(uint32_t h) { return __uint_as_float(h << 16); }
};
template <>
struct XT<DT_F16> {
  typedef __half2 T2;
  static constexpr uint32_t NINF = 0xfc00u;
  static constexpr uint32_t KNINF = 0x0400u;
  static constexpr int SB = 5;                // 32 keys, 1/32 octave
  static constexpr int MB = 10;
  static constexpr int EB = 15 + 10;
  static __device__ __forceinline__ float f(uint32_t h) {
    return __half2float(__ushort_as_half((unsigned short)h));
  }
};

// Order-preserving 16-bit key of a raw bf16 / fp16 value: 0x8000 + m for
// positive values, 0x8000 - m for negative ones (m = the magnitude bits), so
// -0 and +0 share key 0x8000.  Not used on NaN.
__device__ __forceinline__ uint32_t xkey(uint32_t h) {
  return (h & 0x8000u) ? (0x8000u - (h & 0x7fffu)) : (h | 0x8000u);
}
// Raw value of a key (+0 for key 0x8000).
__device__ __forceinline__ uint32_t xraw(uint32_t k) {
  return (k >= 0x8000u) ? (k & 0x7fffu) : (0x8000u | (0x8000u - k));
}
__device__ __forceinline__ uint32_t xhalf(uint4 q, int e) {
  const uint32_t w = (e < 2) ? q.x : (e < 4) ? q.y : (e < 6) ? q.z : q.w;
  return (e & 1) ? (w >> 16) : (w & 0xffffu);
}
template <int DT>
__device__ __forceinline__ uint32_t xmax2(uint32_t a, uint32_t b) {
  typedef typename XT<DT>::T2 T2;
  const T2 m = __hmax2_nan(*reinterpret_cast<const T2*>(&a), *reinterpret_cast<const T2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&m);
}
template <int DT>
__device__ __forceinline__ uint32_t xmin2(uint32_t a, uint32_t b) {
  typedef typename XT<DT>::T2 T2;
  const T2 m = __hmin2(*reinterpret_cast<const T2*>(&a), *reinterpret_cast<const T2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&m);
}
template <int DT>
__device__ __forceinline__ uint32_t xge2(uint32_t a, uint32_t b) {
  typedef typename XT<DT>::T2 T2;
  return __hge2_mask(*reinterpret_cast<const T2*>(&a), *reinterpret_cast<const T2*>(&b));
}
template <int DT>
__device__ __forceinline__ uint32_t xeq2(uint32_t a, uint32_t b) {
  typedef typename XT<DT>::T2 T2;
  return __heq2_mask(*reinterpret_cast<const T2*>(&a), *reinterpret_cast<const T2*>(&b));
}
template <int DT>
__device__ __forceinline__ uint32_t xgt2(uint32_t a, uint32_t b) {
  typedef typename XT<DT>::T2 T2;
  return __hgt2_mask(*reinterpret_cast<const T2*>(&a), *reinterpret_cast<const T2*>(&b));
}
// One bit per element (element e -> bit e) from four packed compare masks.
__device__ __forceinline__ uint32_t xbits8(uint32_t m0, uint32_t m1, uint32_t m2, uint32_t m3) {
  const uint32_t p0 = __byte_perm(m0, m1, 0x6420) & 0x08040201u;
  const uint32_t p1 = __byte_perm(m2, m3, 0x6420) & 0x08040201u;
  return ((p0 * 0x01010101u) >> 24) | (((p1 * 0x01010101u) >> 24) << 4);
}
template <int DT>
__device__ __forceinline__ uint32_t xvmax(uint4 q) {
  return xmax2<DT>(xmax2<DT>(q.x, q.y), xmax2<DT>(q.z, q.w));
}

// Shared-space loads (the pointers below always point into shared memory).
__device__ __forceinline__ uint4 xlds128(const void* p) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(smem_u32(p)));
  return r;
}
__device__ __forceinline__ float xlds32f(const float* p) {
  float r;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r) : "r"(smem_u32(p)));
  return r;
}

// Fire-and-forget OR into shared memory.
__device__ __forceinline__ void xred_or_shared(uint32_t* p, uint32_t v) {
  asm volatile("red.shared.or.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// floor(w * 2^40) for w in [0, 1], from the float's fields.
__device__ __forceinline__ uint64_t xfx40(float w) {
  const uint32_t b = __float_as_uint(w);
  const int e = (int)(b >> 23);
  if (e == 0 || e > 127) return 0ull;
  const uint64_t m = (uint64_t)((b & 0x7fffffu) | 0x800000u);
  const int sh = e - 110;
  return sh >= 0 ? (m << sh) : (sh > -24 ? (m >> -sh) : 0ull);
}
// A value's weight exp(fl32(x / T) - zmax) in fp32, and as fixed point.  Every
// mass that decides a kept set, or locates a draw among candidates, is a sum
// of these.
__device__ __forceinline__ float xweight(float x, float T, float zmax) {
  return expf(__fdiv_rn(x, T) - zmax);
}
__device__ __forceinline__ uint64_t xwfx(float x, float T, float zmax) {
  return xfx40(xweight(x, T, zmax));
}
// Approximate weight (hardware exp2) for the mass below a flat row's first
// window: it only moves the top-p target, by far less than the 1e-5 band.
__device__ __forceinline__ uint64_t xwfx_fast(float x, float xmax, float c2) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"((x - xmax) * c2));
  return xfx40(r);
}
__device__ __forceinline__ float ex2f(float a) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

// fl32(x / T) of a raw bf16 / fp16 value through a per-row table of the
// significands' quotients: x = S * 2^(e - EB) with S the significand as an
// integer, so x / T rounds exactly like S / T and is scaled by a power of two.
// Subnormal inputs and results near the range limits divide directly.
template <int DT>
__device__ __forceinline__ float xz(uint32_t h, const float* tz, float T) {
  typedef XT<DT> R;
  const int e = (int)((h >> R::MB) & ((DT == DT_BF16) ? 0xffu : 0x1fu));
  const uint32_t f = h & ((1u << R::MB) - 1u);
  const uint32_t t = __float_as_uint(xlds32f(tz + f));
  const int te = (int)((t >> 23) & 0xffu) + e - R::EB;
  if (e == 0 || te <= 0 || te >= 255) return __fdiv_rn(R::f(h), T);
  const uint32_t z = (t & 0x807fffffu) | ((uint32_t)te << 23);
  return __uint_as_float(z | (h & 0x8000u ? 0x80000000u : 0u));
}

// Keep-all rows: the weight of a raw value relative to zref = fl32(xs / T),
// xs the sample's maximum.  Values whose weight is within 2^-10 of the top
// take z = fl32(x / T) exactly (the table) and exp2 of (z - zref) log2(e);
// the rest exp2 of x log2(e) / T - zref log2(e), which differs by at most
// half an ulp of z (6e-8 |z| relative) for values that each weigh less than
// 2^-10 of the top, so the cumulative distribution moves by less than 4e-7.
// -inf weighs 0.
template <int DT>
__device__ __forceinline__ float xall_w(uint32_t h, const float* tz, float T, float zref, float c2,
                                        float zb, float xcf) {
  const float x = XT<DT>::f(h);
  return x >= xcf ? ex2f((xz<DT>(h, tz, T) - zref) * 1.4426950408889634f) : ex2f(fmaf(x, c2, -zb));
}

__device__ __forceinline__ void xcluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void xcluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void xcluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint32_t xcluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
template <class T>
__device__ __forceinline__ T* xremote(T* p, uint32_t rank) {
  return cg::this_cluster().map_shared_rank(p, rank);
}

// Block-wide exclusive scan in thread order; *total receives the sum.
template <class T>
__device__ __forceinline__ T xblock_excl(T v, T* sc, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) sc[warp] = inc;
  __syncthreads();
  T pre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < XNW; ++w) {
    const T s = sc[w];
    pre += (w < warp) ? s : (T)0;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return pre + inc - v;
}
template <class T>
__device__ __forceinline__ T xblock_total(T v, T* sc) {
  T t;
  xblock_excl<T>(v, sc, &t);
  return t;
}
__device__ __forceinline__ uint64_t xwarp_sum64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <class T>
__device__ __forceinline__ T xwarp_incl(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// floor(k * M / 2^24) exactly (k < 2^24, M < 2^64).
__device__ __forceinline__ uint64_t xscale24(uint32_t k, uint64_t M) {
  const uint64_t lo = (uint64_t)k * (M & 0xffffffffull);
  const uint64_t hi = (uint64_t)k * (M >> 32);
  return (lo >> 24) + (hi << 8);
}

// Kept-mask words: lanes 4i..4i+3 of a warp hold the four bytes of one word
// (vector v covers ids 8v..8v+7 of the slice; v % 4 == lane % 4).
__device__ __forceinline__ void xput_mask_byte(uint32_t* out, int v, uint32_t byte, bool in) {
  const int lane = threadIdx.x & 31;
  uint32_t w = byte << ((lane & 3) * 8);
  w |= __shfl_xor_sync(0xffffffffu, w, 1);
  w |= __shfl_xor_sync(0xffffffffu, w, 2);
  if (in && (lane & 3) == 0) out[v >> 2] = w;
}

// First entry of e[0..ne) (in id order) whose inclusive prefix exceeds
// `target` (warp-wide; every lane gets the answer).  *rem: the target left
// within that entry.
template <class T>
__device__ __forceinline__ int xlocate(const T* e, int ne, T target, T* rem) {
  const int lane = threadIdx.x & 31;
  const int per = (ne + 31) / 32;
  T s = 0;
  for (int i = 0; i < per; ++i) {
    const int j = lane * per + i;
    if (j < ne) s += e[j];
  }
  const T inc = xwarp_incl<T>(s);
  const uint32_t hit = __ballot_sync(0xffffffffu, inc > target);
  const int L = hit ? (__ffs(hit) - 1) : 31;
  T before = __shfl_sync(0xffffffffu, inc - s, L);
  int found = -1;
  if (lane == L) {
    for (int i = 0; i < per; ++i) {
      const int j = lane * per + i;
      if (j >= ne) break;
      if (before + e[j] > target) {
        found = j;
        break;
      }
      before += e[j];
    }
    if (found < 0) {  // rounding left the target at the end: the last entry
      found = min(lane * per + per, ne) - 1;
      before -= e[found];
    }
  }
  found = __shfl_sync(0xffffffffu, found, L);
  before = __shfl_sync(0xffffffffu, before, L);
  *rem = target - before;
  return found;
}

// Raw values of vector v read one at a time from global memory (a partial
// last vector, or a row that is not 16-byte aligned); values past n: -inf.
template <int DT>
__device__ __noinline__ uint4 xslow_vec(const uint16_t* gsrc, int v, int n) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = v * 8 + 2 * i;
    const uint32_t lo = e < n ? gsrc[e] : XT<DT>::NINF;
    const uint32_t hi = e + 1 < n ? gsrc[e + 1] : XT<DT>::NINF;
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// The grammar mask of vector v: illegal values become -inf.
template <int DT>
__device__ __noinline__ uint4 xmask_apply(uint4 q, uint32_t m8) {
  uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (!((m8 >> e) & 1u)) {
      const int sh = (e & 1) * 16;
      w[e >> 1] = (w[e >> 1] & ~(0xffffu << sh)) | (XT<DT>::NINF << sh);
    }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
template <int DT>
__device__ __forceinline__ uint4 xmask_vec(uint4 q, const uint32_t* mrow, int v) {
  if (!mrow) return q;
  const uint32_t m8 = (mrow[v >> 2] >> ((v & 3) * 8)) & 0xffu;
  return m8 == 0xffu ? q : xmask_apply<DT>(q, m8);
}
// Vector v of the slice from ring slot `slot` (or from global memory past the
// bulk copies), mask applied.
template <int DT>
__device__ __forceinline__ uint4 xfetch(const unsigned char* ring, int slot, int v, int nfull, int n,
                                        const uint16_t* gsrc, const uint32_t* mrow) {
  const uint4 q = v < nfull ? xlds128(ring + slot * XSB + (v % XVS) * 16)
                            : xslow_vec<DT>(gsrc, v, n);
  return xmask_vec<DT>(q, mrow, v);
}
// The same vector re-read from global memory (an L2 hit after the stream).
template <int DT>
__device__ __forceinline__ uint4 xgfetch(int v, int nfull, int n, const uint16_t* gsrc,
                                         const uint32_t* mrow) {
  const uint4 q = v < nfull ? reinterpret_cast<const uint4*>(gsrc)[v] : xslow_vec<DT>(gsrc, v, n);
  return xmask_vec<DT>(q, mrow, v);
}

// Per-thread statistics of a slice (a8.3): the largest value and its first
// id, a NaN-propagating packed maximum (NaN / +inf detection) and the count
// of -inf values (illegal ones included).
struct XStat {
  float best;
  int bid;
  uint32_t nanacc;
  int ninf;
};
template <int DT>
__device__ __forceinline__ uint32_t xstats(XStat& st, uint4 q, int id0) {
  typedef XT<DT> R;
  const uint32_t vm = xvmax<DT>(q);
  st.nanacc = xmax2<DT>(st.nanacc, vm);
  const uint32_t vn = xmin2<DT>(xmin2<DT>(q.x, q.y), xmin2<DT>(q.z, q.w));
  if ((vn & 0xffffu) == R::NINF || (vn >> 16) == R::NINF) {
#pragma unroll
    for (int e = 0; e < 8; ++e) st.ninf += (xhalf(q, e) == R::NINF) ? 1 : 0;
  }
  const float m = fmaxf(R::f(vm & 0xffffu), R::f(vm >> 16));
  if (m > st.best) {
    int e = 0;
    while (e < 7 && R::f(xhalf(q, e)) != m) ++e;
    st.best = m;
    st.bid = id0 + e;
  }
  return vm;
}
// CTA-wide reduction of the statistics into S.stage (kmax, amax, -inf count
// in nleg, flags).
template <int DT>
__device__ __forceinline__ void xreduce_stats(XSh& S, const XStat& st, int timed_out, int extra) {
  typedef XT<DT> R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int bad;
  {
    const float lo = R::f(st.nanacc & 0xffffu), hi = R::f(st.nanacc >> 16);
    bad = (lo != lo || hi != hi || lo == INFINITY || hi == INFINITY) ? 1 : 0;
  }
  float b = st.best;
  int id = st.bid;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, b, o);
    const int oi = __shfl_xor_sync(0xffffffffu, id, o);
    if (ob > b || (ob == b && oi < id)) {
      b = ob;
      id = oi;
    }
  }
  const int ni = __reduce_add_sync(0xffffffffu, st.ninf);
  bad = (int)__reduce_or_sync(0xffffffffu, (unsigned)bad);
  const int to = (int)__reduce_or_sync(0xffffffffu, (unsigned)timed_out);
  if (lane == 0) {
    S.f[warp] = b;
    S.wi[warp] = id;
    S.bi[warp] = ni;
    S.bi[8 + warp] = bad | (to << 1);
  }
  __syncthreads();
  if (tid == 0) {
    float bb = S.f[0];
    int ii = S.wi[0], nn = S.bi[0], fl = S.bi[8] | extra;
    for (int w = 1; w < XNW; ++w) {
      if (S.f[w] > bb || (S.f[w] == bb && S.wi[w] < ii)) {
        bb = S.f[w];
        ii = S.wi[w];
      }
      nn += S.bi[w];
      fl |= S.bi[8 + w];
    }
    uint32_t km = 0u;
    if (bb > -INFINITY) {
      uint32_t h;
      if constexpr (DT == DT_BF16) h = __float_as_uint(bb) >> 16;
      else h = __half_as_ushort(__float2half_rn(bb));
      km = xkey(h);
    }
    S.stage.kmax = km;
    S.stage.amax = km ? ii : INT_MAX;
    S.stage.nleg = nn;
    S.stage.flags = fl;
  }
  __syncthreads();
}

// What the stream needs of its CTA.
struct XCtx {
  unsigned char* ring;
  XSh* S;
  const uint16_t* gsrc;
  const uint32_t* mrow;
  uint32_t* hist;
  const float* tz;
  uint32_t* mout;
  long long wait_limit;
  int nst, nvec, nfull, n, s0;
  uint32_t lo, hw, lo2;
  float T, zref;
  float xs, c2;  // flat rows: the sample's maximum and log2(e) / T
  float zb;       // keep-all rows: zref log2(e)
  uint32_t xc2;   // keep-all rows: the exact-weight floor, packed twice in the element type
  uint32_t* flagw;  // top-k rows: bitmap of vectors holding candidates
  uint32_t* hcnt;   // flat rows: one 32-bit counter per key of [lo, hw] (bin hw - k)
};
enum { XS_STATS = 0, XS_TOPK = 1, XS_ALL = 2, XS_FLAT = 3 };

// The stream over the slice's stages (a8.2-a8.4): statistics, and by row
// class the top-k candidates (list + window histogram) or the keep-all masses
// and kept-mask words.  Stage 0 is already in slot 0 (masked) and its
// statistics are taken.
template <int DT, int MODE>
__device__ __forceinline__ void xstream(const XCtx cx, XStat& st, int& timed_out, int& issued,
                                        int& xflags, float& fm) {
  typedef XT<DT> R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // every field in a register of its own: stores through the list and mask
  // pointers must not force the context to be reloaded
  unsigned char* const __restrict__ ring = cx.ring;
  XSh* const __restrict__ Sp = cx.S;
  const uint16_t* const __restrict__ gsrc = cx.gsrc;
  const uint32_t* const __restrict__ mrow = cx.mrow;
  const float* const __restrict__ tz = cx.tz;
  uint32_t* const __restrict__ mout = cx.mout;
  const long long wait_limit = cx.wait_limit;
  const int nst = cx.nst, nvec = cx.nvec, nfull = cx.nfull, n = cx.n, s0 = cx.s0;
  const uint32_t lo = cx.lo, lo2 = cx.lo2, xc2 = cx.xc2;
  const float T = cx.T, zref = cx.zref, xs = cx.xs, c2 = cx.c2, zb = cx.zb;
  uint32_t* const __restrict__ flagw = cx.flagw;
  uint32_t* const __restrict__ hcnt = cx.hcnt;
  const uint32_t hw = cx.hw;
  constexpr uint32_t NN = R::NINF | (R::NINF << 16);
  for (int s = 0; s < nst; ++s) {
    const int slot = s % XNS;
    if (!timed_out && s > 0 && s * XVS < nfull &&
        !mbar_wait_bounded(&Sp->bar[slot], (s / XNS) & 1, wait_limit))
      timed_out = 1;
    float am = 0.f;  // keep-all: this lane's mass in this stage
#pragma unroll 1
    for (int r = 0; r < XSUB; ++r) {
      const int v = s * XVS + warp * XVW + r * 32 + lane;
      const bool in = v < nvec;
      uint4 q = make_uint4(NN, NN, NN, NN);
      uint32_t vm = NN;
      if (in) {
        q = (s == 0 && v < nfull) ? xlds128(ring + v * 16)
                                    : xfetch<DT>(ring, slot, v, nfull, n, gsrc, mrow);
        vm = (s > 0) ? xstats<DT>(st, q, s0 + v * 8) : xvmax<DT>(q);
      }
      if (MODE == XS_TOPK) {
        // a vector holding a value >= lo is marked; its candidates are
        // listed after the stream (re-read from L2)
        if (in && xge2<DT>(vm, lo2) != 0u) xred_or_shared(&flagw[v >> 5], 1u << (v & 31));
      } else if (MODE == XS_FLAT) {
        if (in) {
          float f0 = 0.f, f1 = 0.f;  // -inf weighs 0
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            f0 += ex2f((R::f(xhalf(q, e)) - xs) * c2);
            f1 += ex2f((R::f(xhalf(q, e + 1)) - xs) * c2);
          }
          fm += f0 + f1;
          // every key of the window counted (values above it: flag 8)
          if (xge2<DT>(vm, lo2) != 0u) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint32_t k = xkey(xhalf(q, e));
              if (k >= lo) {
                if (k <= hw) atomicAdd(&hcnt[hw - k], 1u);
                else xflags |= 8;
              }
            }
          }
        }
      } else if (MODE == XS_ALL) {
        uint32_t byte = 0;
        if (in) {
          // legal bits from packed -inf tests
          const uint32_t m0 = xeq2<DT>(q.x, NN), m1 = xeq2<DT>(q.y, NN), m2 = xeq2<DT>(q.z, NN),
                         m3 = xeq2<DT>(q.w, NN);
          byte = ~((m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) |
                   ((m2 & 1u) << 4) | ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u)) &
                 0xffu;
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            a0 += ex2f(fmaf(R::f(xhalf(q, e)), c2, -zb));
            a1 += ex2f(fmaf(R::f(xhalf(q, e + 1)), c2, -zb));
          }
          am += a0 + a1;
          if (xge2<DT>(vm, xc2) != 0u) {  // values near the top: exact z
            // one pass per such value (few per lane), in element order
            uint32_t cm = xbits8(xge2<DT>(q.x, xc2), xge2<DT>(q.y, xc2), xge2<DT>(q.z, xc2),
                                 xge2<DT>(q.w, xc2));
#pragma unroll 1
            for (; cm; cm &= cm - 1u) {
              const int e = __ffs(cm) - 1;
              const uint32_t w = e < 4 ? (e < 2 ? q.x : q.y) : (e < 6 ? q.z : q.w);
              const uint32_t h = (e & 1) ? (w >> 16) : (w & 0xffffu);
              am += ex2f((xz<DT>(h, tz, T) - zref) * 1.4426950408889634f) -
                    ex2f(fmaf(R::f(h), c2, -zb));
            }
          }
        }
        if (mout) xput_mask_byte(mout, v, byte, in);
      }
    }
    if (MODE == XS_ALL) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) am += __shfl_xor_sync(0xffffffffu, am, o);
      if (lane == 0) Sp->rwf[s][warp] = am;
    }
    // every warp is done with the slot; after an expired wait no more copies go out
    timed_out = __syncthreads_or(timed_out);
    if (tid == 0 && !timed_out && s + XNS < nst) {
      const int v0 = (s + XNS) * XVS, v1 = min(nfull, v0 + XVS);
      const uint32_t bytes = v1 > v0 ? (uint32_t)(v1 - v0) * 16u : 0u;
      if (s == 0) fence_proxy_async_smem();  // slot 0 may hold the masked copy
      mbar_arrive_expect_tx(&Sp->bar[slot], bytes);
      if (bytes) bulk_g2s(ring + slot * XSB, gsrc + (size_t)v0 * 8, bytes, &Sp->bar[slot]);
      ++issued;
    }
  }
}

// Row outputs written once per row (rank 0, thread 0).
__device__ __forceinline__ void xfinish(const XArgs& a, int row, uint32_t rank, int st, int tok,
                                        int cnt, int path, int i1, int i2, int i3) {
  if (rank == 0 && threadIdx.x == 0) {
    a.status[row] = st;
    if (a.tokens && (st != ST_OK || tok >= 0)) a.tokens[row] = st == ST_OK ? tok : -1;
    if (a.kept_count) a.kept_count[row] = st == ST_OK ? cnt : 0;
    if (a.logprob && st != ST_OK) a.logprob[row] = __uint_as_float(0x7fc00000u);
    if (a.row_info) {
      int* ri = a.row_info + (size_t)row * 4;
      ri[0] = path;
      ri[1] = i1;
      ri[2] = i2;
      ri[3] = i3;
    }
  }
}
// The same over a histogram with one 32-bit counter per bin.
template <int DT>
__device__ __forceinline__ uint64_t xmy_mass32(const uint32_t* hist, uint32_t hi, int upto, float T,
                                               float zmax, uint64_t* sc) {
  uint64_t mine = 0;
  for (int b = threadIdx.x; b < upto; b += XNT) {
    const uint32_t c = hist[b];
    if (c) mine += (uint64_t)c * xwfx(XT<DT>::f(xraw(hi - (uint32_t)b)), T, zmax);
  }
  return xblock_total<uint64_t>(mine, sc);
}
// Count of bin b: 16-bit pairs, or one 32-bit counter per bin.
__device__ __forceinline__ uint32_t xcnt(const uint32_t* h, uint32_t b, bool wide) {
  return wide ? h[b] : (h[b >> 1] >> ((b & 1u) << 4)) & 0xffffu;
}
// Weight of key index i (key gk - i): stored for the first XWT keys.
template <int DT>
__device__ __forceinline__ uint64_t xw_at(const uint64_t* wtab, int i, uint32_t gk, float T,
                                          float zmax) {
  return i < XWT ? wtab[i] : xwfx(XT<DT>::f(xraw(gk - (uint32_t)i)), T, zmax);
}
// The want-th smallest (0-based) of ids[0..nid), ids < 2^18 and distinct:
// radix selection in three rounds of 6-bit digits (block-wide).
__device__ __forceinline__ int xsel_id(const int* ids, int nid, int want, XSh& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0u;
  for (int round = 0; round < 3; ++round) {
    const int sh = 12 - 6 * round;
    if (tid < 64) S.h64[tid] = 0u;
    __syncthreads();
    for (int i = tid; i < nid; i += XNT) {
      const uint32_t id = (uint32_t)ids[i];
      if ((id >> (sh + 6)) == (prefix >> (sh + 6))) atomicAdd(&S.h64[(id >> sh) & 63u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      const uint32_t c0 = S.h64[2 * lane], c1 = S.h64[2 * lane + 1];
      const uint32_t sum = c0 + c1;
      const uint32_t inc = xwarp_incl<uint32_t>(sum);
      const uint32_t hit = __ballot_sync(0xffffffffu, inc > (uint32_t)want);
      const int L = hit ? __ffs(hit) - 1 : 31;
      const uint32_t bef = __shfl_sync(0xffffffffu, inc - sum, L);
      const uint32_t cc0 = __shfl_sync(0xffffffffu, c0, L);
      if (lane == 0) {
        const int d = (bef + cc0 > (uint32_t)want) ? 2 * L : 2 * L + 1;
        S.bi[7] = d;
        S.bi[8] = want - (int)(bef + ((d & 1) ? cc0 : 0u));
      }
    }
    __syncthreads();
    prefix |= (uint32_t)S.bi[7] << sh;
    want = S.bi[8];
    __syncthreads();
  }
  return (int)prefix;
}

// Kept: above the boundary value, or a copy of it with a local id before the cut.
__device__ __forceinline__ bool xkept(float bval, int cut, float x, int id) {
  return x > bval || (x == bval && id < cut);
}

template <int DT>
__global__ void __launch_bounds__(XNT, 4) split_kernel(const XArgs a) {
  typedef XT<DT> R;
  extern __shared__ __align__(128) unsigned char xsm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // B0: this CTA has started (waited on before the first remote store)
  xcluster_arrive_relaxed();

  const int C = a.C;
  const uint32_t rank = xcluster_rank();
  const int row = blockIdx.x / C;
  const int s0 = (int)rank * a.SL;
  const int n = max(0, min(a.SL, a.V - s0));
  const int nvec = (n + 7) >> 3;
  const int nfull = a.aligned ? (n >> 3) : 0;  // vectors the bulk copies bring
  const int nst = (nvec + XVS - 1) / XVS;
  const int wf = a.wf;
  uint32_t* hist = reinterpret_cast<uint32_t*>(xsm + xoff_hist());
  uint16_t* ckey = reinterpret_cast<uint16_t*>(xsm + xoff_ckey(wf));
  int* cid = reinterpret_cast<int*>(xsm + xoff_cid(wf, a.cap));
  XSh& S = *reinterpret_cast<XSh*>(xsm + xoff_sh(wf, a.cap));
  const uint16_t* gsrc =
      reinterpret_cast<const uint16_t*>(a.logits) + (size_t)row * (size_t)a.ld + (size_t)s0;
  const uint32_t* mrow =
      a.bitmask ? a.bitmask + (size_t)row * (size_t)a.W + (size_t)(s0 >> 5) : nullptr;

  // ---- ring: issue the first stages before anything else ----
  int issued = 0;  // stages handed to the copy engine (thread 0's count)
  if (tid == 0) {
#pragma unroll
    for (int p = 0; p < XNS; ++p) mbar_init(&S.bar[p], 1);
    fence_mbar_init();
    for (int s = 0; s < XNS && s < nst; ++s, ++issued) {
      const int v0 = s * XVS, v1 = min(nfull, v0 + XVS);
      const uint32_t bytes = v1 > v0 ? (uint32_t)(v1 - v0) * 16u : 0u;
      mbar_arrive_expect_tx(&S.bar[s], bytes);
      if (bytes) bulk_g2s(xsm + s * XSB, gsrc + (size_t)v0 * 8, bytes, &S.bar[s]);
    }
  }

  // ---- parameters (a8.1) ----
  float T = 0.f, pp = 1.f;
  int kk = 1;
  bool params_ok = true;
  unsigned long long seed = 0, offs = 0;
  if (a.mode != MODE_ARGMAX) {
    T = a.temperature[row];
    kk = a.top_k[row];
    pp = a.top_p[row];
    params_ok = !(T != T || T < 0.f) && kk >= 1 && !(pp != pp) && pp > 0.f && pp <= 1.f;
    if (kk > a.V) kk = a.V;
    if (a.mode == MODE_SAMPLE) {
      seed = a.seed[row];
      offs = a.offset[row];
    }
  }
  // the class the parameters give; the legal count can still change it
  int pcls;
  if (!params_ok) pcls = XC_ERROR;
  else if (a.mode == MODE_ARGMAX || T == 0.f || kk == 1) pcls = XC_GREEDY;
  else if (kk >= a.V) pcls = (pp >= 1.f) ? XC_ALL : XC_FLAT;
  else pcls = XC_TOPK;
  const bool want_samp = pcls == XC_TOPK;

  for (int i = tid; i < (wf >> 1); i += XNT) hist[i] = 0u;
  if (tid == 0) {
    S.ncand = 0;
    S.flags = 0;
  }
  __syncthreads();

  constexpr uint32_t NN4 = R::NINF | (R::NINF << 16);
  XStat st;
  st.best = -INFINITY;
  st.bid = INT_MAX;
  st.nanacc = R::NINF | (R::NINF << 16);
  st.ninf = 0;
  int timed_out = 0;

  // ---- the sample: stage 0 ----
  if (nst > 0 && nfull > 0 && !mbar_wait_bounded(&S.bar[0], 0, a.wait_limit)) timed_out = 1;
#pragma unroll
  for (int r = 0; r < XSUB; ++r) {
    const int v = warp * XVW + r * 32 + lane;
    if (v >= nvec) continue;
    uint4 q = xfetch<DT>(xsm, 0, v, nfull, n, gsrc, mrow);
    if (v < nfull && mrow) reinterpret_cast<uint4*>(xsm)[v] = q;  // masked copy for the stream
    xstats<DT>(st, q, s0 + v * 8);
  }
  // The local sample: this CTA's first stage.  Its maximum is the reference
  // of flat and keep-all masses, and its fine key histogram places this CTA's
  // candidate threshold; no exchange is needed before the stream, because
  // every CTA lists all of its values above its own threshold and the
  // resolution works on the key range that every CTA covers.
  uint32_t sk = 0u;  // this CTA's stage-0 maximum key
  uint32_t lo = 0xffffu, hw = 0xffffu;  // candidate window [lo, hw]
  if (pcls == XC_TOPK || pcls == XC_FLAT || pcls == XC_ALL) {
    xreduce_stats<DT>(S, st, timed_out, 0);
    sk = S.stage.kmax;
  }
  if (want_samp) {
    // every value of stage 0 in the XSW fine bins below the stage's maximum
    const uint32_t kb = sk >> R::SB;
    const uint32_t kfloor = kb >= (uint32_t)(XSW - 1) ? (kb - (XSW - 1)) << R::SB : 0u;
    const uint32_t f2 = xraw(max(kfloor, R::KNINF + 1u)) * 0x10001u;
    for (int i = tid; i < XSW / 2; i += XNT) hist[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < XSUB; ++r) {
      const int v = warp * XVW + r * 32 + lane;
      if (v >= nvec || !sk) continue;
      const uint4 q = v < nfull ? xlds128(xsm + v * 16) : xfetch<DT>(xsm, 0, v, nfull, n, gsrc, mrow);
      if (xge2<DT>(xvmax<DT>(q), f2) == 0u) continue;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t h = xhalf(q, e);
        if (h == R::NINF) continue;
        const uint32_t k = xkey(h);
        if (k < kfloor || k <= R::KNINF || k > sk) continue;  // NaN keys lie above
        const uint32_t b = kb - (k >> R::SB);
        atomicAdd(&hist[b >> 1], 1u << ((b & 1u) << 4));
      }
    }
    __syncthreads();
    // Aim at K + 3 sigma + 4 sampled values, with the sample taken as a
    // sample of the whole row, and start the window at the lower edge of the
    // fine bin that reaches it.
    const float fr = (float)min(n, XVS * 8) / (float)a.V;
    const float kf = (float)kk * fr;
    const int need = max(1, (int)ceilf(kf + 3.f * sqrtf(kf) + 4.f));
    if (warp == 0) {
      uint32_t cb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int b = 4 * lane + i;
        cb[i] = (hist[b >> 1] >> ((b & 1) << 4)) & 0xffffu;
      }
      const uint32_t sum = cb[0] + cb[1] + cb[2] + cb[3];
      const uint32_t inc = xwarp_incl<uint32_t>(sum);
      const uint32_t hit = __ballot_sync(0xffffffffu, inc >= (uint32_t)need);
      int jb = XSW;  // never reached: no threshold from the sample
      if (hit) {
        const int L = __ffs(hit) - 1;
        uint32_t run = __shfl_sync(0xffffffffu, inc - sum, L);
        uint32_t c4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) c4[i] = __shfl_sync(0xffffffffu, cb[i], L);
        jb = 4 * L + 3;
        for (int i = 0; i < 4; ++i) {
          run += c4[i];
          if (run >= (uint32_t)need) {
            jb = 4 * L + i;
            break;
          }
        }
      }
      if (lane == 0) S.bi[16] = jb;
    }
    __syncthreads();
    const int jb = S.bi[16];
    const long long bl = ((long long)kb - jb) << R::SB;
    lo = (uint32_t)max(bl, (long long)R::KNINF);
    if (jb >= XSW || sk == 0u) lo = R::KNINF;  // sample too thin: list every legal value
    hw = min(lo + (uint32_t)wf - 1u, 0xffffu);
  }
  // Flat top-p rows count every key of a window of `cap` keys in the stream,
  // from XFM keys above this CTA's sample maximum down.
  uint32_t* hcnt = reinterpret_cast<uint32_t*>(cid);
  if (pcls == XC_FLAT) {
    const uint32_t WH = (uint32_t)min(a.cap, XNS * XSB / 8);  // the resolution's count array holds as many
    hw = sk ? min(sk + WH / XFM, 0xffffu) : 0xffffu;
    lo = hw >= R::KNINF + WH ? hw - (WH - 1u) : R::KNINF + 1u;
    for (int i = tid; i < (int)WH; i += XNT) hcnt[i] = 0u;
    __syncthreads();
  }
  const uint32_t lo2 = xraw(lo) | (xraw(lo) << 16);

  // keep-all rows: weights relative to the sample's maximum, z from a table
  float* tz = reinterpret_cast<float*>(hist);
  float zref = 0.f;
  const float L2E = 1.4426950408889634f;
  if (pcls == XC_ALL) {
    for (int f = tid; f < (1 << R::MB); f += XNT)
      tz[f] = __fdiv_rn((float)((1u << R::MB) + (uint32_t)f), T);
    zref = sk ? __fdiv_rn(R::f(xraw(sk)), T) : 0.f;
    __syncthreads();
  }
  uint32_t* mout = a.kept_mask ? a.kept_mask + (size_t)row * (size_t)a.W + (size_t)(s0 >> 5)
                               : nullptr;
  float* pout = a.probs ? a.probs + (size_t)row * (size_t)a.V + (size_t)s0 : nullptr;
  int xflags = 0;

  // keep-all rows: the exact-weight floor, 2^-24 below the sample's maximum
  float zb = 0.f, xcf = -INFINITY;  // no sample maximum: every value exact
  uint32_t xc2 = NN4;
  if (pcls == XC_ALL && sk) {
    zb = zref * L2E;
    const float f = R::f(xraw(sk)) - 10.f * 0.6931471805599453f * T;
    uint32_t hb;
    if constexpr (DT == DT_BF16) hb = __bfloat16_as_ushort(__float2bfloat16_rd(f));
    else hb = __half_as_ushort(__float2half_rd(f));
    xcf = R::f(hb);
    xc2 = hb * 0x10001u;
  }
  // top-k and flat rows: the bitmap of vectors holding candidates (histogram area)
  uint32_t* flagw = hist;
  if (want_samp) {
    for (int i = tid; i < (nvec + 31) >> 5; i += XNT) flagw[i] = 0u;
    __syncthreads();
  }

  // ---- the stream (a8.2-a8.4) ----
  timed_out = __syncthreads_or(timed_out);
  float fm = 0.f;  // flat rows: this thread's mass relative to the sample's maximum
  {
    XCtx cx;
    cx.ring = xsm;
    cx.S = &S;
    cx.gsrc = gsrc;
    cx.mrow = mrow;
    cx.hist = hist;
    cx.tz = tz;
    cx.mout = mout;
    cx.wait_limit = a.wait_limit;
    cx.nst = nst;
    cx.nvec = nvec;
    cx.nfull = nfull;
    cx.n = n;
    cx.s0 = s0;
    cx.lo = lo;
    cx.hw = hw;
    cx.lo2 = lo2;
    cx.T = T;
    cx.zref = zref;
    cx.xs = sk ? R::f(xraw(sk)) : 0.f;
    cx.c2 = T > 0.f ? L2E / T : 0.f;
    cx.zb = zb;
    cx.xc2 = xc2;
    cx.flagw = flagw;
    cx.hcnt = hcnt;
    if (pcls == XC_TOPK) xstream<DT, XS_TOPK>(cx, st, timed_out, issued, xflags, fm);
    else if (pcls == XC_FLAT) xstream<DT, XS_FLAT>(cx, st, timed_out, issued, xflags, fm);
    else if (pcls == XC_ALL) xstream<DT, XS_ALL>(cx, st, timed_out, issued, xflags, fm);
    else xstream<DT, XS_STATS>(cx, st, timed_out, issued, xflags, fm);
  }
  // the candidates: the marked vectors re-read (an L2 hit) and their values
  // >= lo listed; then the window histogram of the listed keys (one bin per
  // key; bin b holds key hw - b)
  if (want_samp) {
    constexpr int XVL = XNS * XSB / 4;  // marked vectors the ring area can list
    uint32_t* vlist = reinterpret_cast<uint32_t*>(xsm);
    if (tid == 0) S.bi[13] = 0;
    __syncthreads();
    for (int w = tid; w < (nvec + 31) >> 5; w += XNT) {
      uint32_t bits = flagw[w];
      if (!bits) continue;
      int p = atomicAdd(&S.bi[13], __popc(bits));
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1u;
        if (p < XVL) vlist[p] = (uint32_t)(w * 32 + b);
        ++p;
      }
    }
    __syncthreads();
    const int nfv = S.bi[13];
    if (nfv > XVL) xflags |= 4;
    const int nv = min(nfv, XVL);
    for (int i0 = tid; i0 < nv; i0 += 4 * XNT) {
      uint4 q4[4];
      int v4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * XNT;
        v4[u] = i < nv ? (int)vlist[i] : -1;
        q4[u] = v4[u] >= 0 ? xgfetch<DT>(v4[u], nfull, n, gsrc, mrow) : make_uint4(NN4, NN4, NN4, NN4);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (v4[u] < 0) continue;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t h = xhalf(q4[u], e);
          if (h == R::NINF) continue;
          const uint32_t k = xkey(h);
          if (k < lo) continue;
          const int pos = atomicAdd(&S.ncand, 1);
          if (pos < a.cap) {
            ckey[pos] = (uint16_t)k;
            cid[pos] = v4[u] * 8 + e;
          }
        }
      }
    }
    __syncthreads();
    const int pre = min(S.ncand, a.cap);
    if (S.ncand > a.cap) xflags |= 4;
    for (int i = tid; i < (wf >> 1); i += XNT) hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < pre; i += XNT) {
      const uint32_t k = ckey[i];
      if (k > hw) {
        xflags |= 8;
      } else {
        const uint32_t b = hw - k;
        atomicAdd(&hist[b >> 1], 1u << ((b & 1u) << 4));
      }
    }
  }
  if (pcls == XC_FLAT) {
    double d = (double)fm;
    d = xblock_total<double>(d, S.bd);
    if (tid == 0) {
      S.bd[4] = d;
      if (!(d < 1e300)) S.flags |= 16;  // a value far above the sample's maximum
    }
  }
  // ---- B2: the row's statistics ----
  xflags = (int)__reduce_or_sync(0xffffffffu, (unsigned)xflags);
  if (lane == 0 && xflags) atomicOr(&S.flags, xflags);
  __syncthreads();
  xreduce_stats<DT>(S, st, timed_out, S.flags);
  if (tid == 0) {
    S.stage.nleg = nvec * 8 - S.stage.nleg;
    S.stage.ncand = want_samp ? S.ncand : 0;
    S.stage.lo = lo;
    S.stage.hw = hw;
    S.stage.skey = sk;
    S.stage.xsv = sk ? R::f(xraw(sk)) : 0.f;
    double m = 0.0;
    if (pcls == XC_ALL) {
      for (int s = 0; s < nst; ++s)
        for (int w = 0; w < XNW; ++w) m += (double)S.rwf[s][w];
      if (!(m < 1e300)) S.stage.flags |= 16;  // a value far above the sample's maximum
    }
    if (pcls == XC_FLAT) m = S.bd[4];
    S.stage.mass = m;
  }
  __syncthreads();
  xcluster_wait();  // B0 complete: every CTA of the cluster has started
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&S.stage);
    for (int t = tid; t < C * XPUBW; t += XNT) {
      const int dst = t / XPUBW, w = t % XPUBW;
      xremote(reinterpret_cast<uint32_t*>(&S.pub2[rank]), (uint32_t)dst)[w] = src[w];
    }
  }
  xcluster_sync();

  uint32_t gk = 0u;
  int gid = INT_MAX, nleg = 0, flags = 0, ncand = 0;
  for (int c = 0; c < C; ++c) {
    const XPub& P = S.pub2[c];
    if (P.kmax > gk) {
      gk = P.kmax;
      gid = P.amax;
    }
    nleg += P.nleg;
    flags |= P.flags;
    ncand += P.ncand;
  }
  int status = ST_OK;
  if (!params_ok) status = ST_INVALID;
  else if (flags & 2) status = ST_TIMEOUT;
  else if (flags & 1) status = ST_NONFINITE;
  else if (nleg == 0) status = ST_EMPTY;
  const int K = min(kk, nleg);
  int cls;
  if (status != ST_OK) cls = XC_ERROR;
  else if (pcls == XC_GREEDY || K == 1) cls = XC_GREEDY;
  else if (pcls == XC_ALL) cls = (flags & 16) ? XC_FLAT : XC_ALL;
  else if (pcls == XC_TOPK) {
    // the stream settled it if every boundary candidate is listed
    const bool listed = !(flags & (4 | 8)) && (ncand >= K || ncand == nleg);
    cls = listed ? XC_TOPK : (K < nleg ? -XC_TOPK : XC_FLAT);
  } else {
    // flat top-p: the list settles it when the kept set lies above the threshold
    cls = (flags & (4 | 8 | 16)) ? XC_FLAT : XC_FLATL;
  }
  const bool samp_mode = a.mode == MODE_SAMPLE;
  uint32_t k24 = 0;
  if (samp_mode && cls != XC_ERROR) {
    uint32_t w4[4];
    philox4x32_10(seed, (uint32_t)offs, (uint32_t)(offs >> 32), 0u, 0u, w4);
    k24 = w4[0] >> 8;
  }
  // ---- error and greedy rows (a8.10) ----
  if (cls == XC_ERROR || cls == XC_GREEDY) {
    const bool g = cls == XC_GREEDY;
    if (mout) {
      const int nw = (n + 31) >> 5;
      for (int w = tid; w < nw; w += XNT) {
        const int id0 = s0 + w * 32;
        mout[w] = (g && gid >= id0 && gid < id0 + 32) ? (1u << (gid - id0)) : 0u;
      }
    }
    if (pout)
      for (int e = tid; e < n; e += XNT) pout[e] = (g && s0 + e == gid) ? 1.f : 0.f;
    if (g && a.logprob && rank == 0 && tid == 0) a.logprob[row] = 0.f;
    xfinish(a, row, rank, status, g ? gid : -1, 1, g ? PATH_GREEDY : PATH_ERROR, 0, 0, 0);
    // after an expired wait: wait (bounded again) for every copy still in
    // flight into this CTA's ring before the CTA may exit
    if (timed_out && tid == 0)
      for (int s = max(0, issued - XNS); s < issued; ++s)
        mbar_wait_bounded(&S.bar[s % XNS], (s / XNS) & 1, XDRAIN);
    return;
  }

  const float xmax = XT<DT>::f(xraw(gk));
  const float zmax = __fdiv_rn(xmax, T);
  // Flat and keep-all rows: each CTA's legal mass is relative to its own
  // sample's maximum; scale factors to the row's maximum, and the row's mass
  // in those units (Mflat: in fixed point of the largest weight).
  double xsc[XMAXC];
  double gm = 0.0, sc_me = 1.0;
#pragma unroll
  for (int c = 0; c < XMAXC; ++c) {
    xsc[c] = 0.0;
    if (c < C && (pcls == XC_FLAT || pcls == XC_ALL)) {
      // exp(fl32(xs_c / T) - fl32(xmax / T)): the same z the weights use
      xsc[c] = (double)ex2f((__fdiv_rn(S.pub2[c].xsv, T) - zmax) * L2E);
      gm += S.pub2[c].mass * xsc[c];
    }
    if (c == (int)rank) sc_me = xsc[c];
  }
  const double Mflat = pcls == XC_FLAT ? gm * 1099511627776.0 : 0.0;

  // ---- keep-all rows: the masses came with the stream ----
  if (cls == XC_ALL) {
    const double M = gm;
    if (pout) {
      for (int v = tid; v < nvec; v += XNT) {
        const uint4 q = xgfetch<DT>(v, nfull, n, gsrc, mrow);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (v * 8 + e >= n) break;
          const uint32_t h = xhalf(q, e);
          pout[v * 8 + e] =
              h != R::NINF ? (float)((double)xall_w<DT>(h, tz, T, zref, L2E / T, zb, xcf) * sc_me / M)
                           : 0.f;
        }
      }
    }
    if (samp_mode) {
      const double tgt = (double)k24 * 0x1p-24 * M;
      double before = 0.0;
      int cs = C - 1;
      for (int c = 0; c < C; ++c) {
        const double mc = S.pub2[c].mass * xsc[c];
        if (before + mc > tgt) {
          cs = c;
          break;
        }
        before += mc;
      }
      if ((int)rank == cs && warp == 0) {
        // per-(stage, warp) masses of this slice, in id order
        const int ne = nst * XNW;
        const int per = (ne + 31) / 32;
        double sacc = 0.0;
        for (int i = 0; i < per; ++i) {
          const int j = lane * per + i;
          if (j < ne) sacc += (double)S.rwf[j / XNW][j % XNW];
        }
        const double inc = xwarp_incl<double>(sacc);
        const double t2 = sc_me > 0.0 ? (tgt - before) / sc_me : 0.0;  // in this CTA's units
        const uint32_t hit = __ballot_sync(0xffffffffu, inc > t2);
        const int L = hit ? __ffs(hit) - 1 : 31;
        double bef = __shfl_sync(0xffffffffu, inc - sacc, L);
        int piece = -1;
        if (lane == L) {
          for (int i = 0; i < per; ++i) {
            const int j = lane * per + i;
            if (j >= ne) break;
            const double x = (double)S.rwf[j / XNW][j % XNW];
            if (bef + x > t2) {
              piece = j;
              break;
            }
            bef += x;
          }
          if (piece < 0) {
            piece = min(lane * per + per, ne) - 1;
            bef -= (double)S.rwf[piece / XNW][piece % XNW];
          }
        }
        piece = __shfl_sync(0xffffffffu, piece, L);
        bef = __shfl_sync(0xffffffffu, bef, L);
        double rr = t2 - bef;
        // re-read the piece: four sub-rounds of 32 consecutive vectors
        uint4 qs[XSUB];
        float ls[XSUB];
        double tot[XSUB];
#pragma unroll
        for (int r = 0; r < XSUB; ++r) {
          const int v = (piece / XNW) * XVS + (piece % XNW) * XVW + r * 32 + lane;
          ls[r] = 0.f;
          qs[r] = make_uint4(R::NINF | (R::NINF << 16), R::NINF | (R::NINF << 16),
                             R::NINF | (R::NINF << 16), R::NINF | (R::NINF << 16));
          if (v < nvec) {
            qs[r] = xgfetch<DT>(v, nfull, n, gsrc, mrow);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint32_t h = xhalf(qs[r], e);
              if (h != R::NINF) ls[r] += xall_w<DT>(h, tz, T, zref, L2E / T, zb, xcf);
            }
          }
          double t = (double)ls[r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
          tot[r] = t;
        }
        int rs = -1;
        double cum = 0.0;
#pragma unroll
        for (int r = 0; r < XSUB; ++r) {
          if (rs < 0 && cum + tot[r] > rr) rs = r;
          else if (rs < 0) cum += tot[r];
        }
        if (rs < 0) {  // rounding left the target at the end: the last sub-round with mass
          rs = XSUB - 1;
          while (rs > 0 && tot[rs] <= 0.0) --rs;
          cum -= tot[rs];
        }
        const double rr2 = rr - cum;
        float lsr = 0.f;
        uint4 qr = qs[0];
#pragma unroll
        for (int r = 0; r < XSUB; ++r)
          if (r == rs) {
            lsr = ls[r];
            qr = qs[r];
          }
        const double li = xwarp_incl<double>((double)lsr);
        const uint32_t hh = __ballot_sync(0xffffffffu, li > rr2);
        const uint32_t any = __ballot_sync(0xffffffffu, lsr > 0.f);
        const int L2 = hh ? __ffs(hh) - 1 : (any ? 31 - __clz(any) : 0);
        if (lane == L2) {
          const int v = (piece / XNW) * XVS + (piece % XNW) * XVW + rs * 32 + lane;
          double c = li - (double)lsr;
          int tok = -1;
          float wt = 0.f;
          for (int e = 0; e < 8; ++e) {
            const uint32_t h = xhalf(qr, e);
            if (h == R::NINF) continue;
            const float w = xall_w<DT>(h, tz, T, zref, L2E / T, zb, xcf);
            c += (double)w;
            tok = s0 + v * 8 + e;
            wt = w;
            if (c > rr2) break;
          }
          S.bi[17] = tok;
          S.f[0] = wt;
        }
      }
      __syncthreads();
      if ((int)rank == cs && tid == 0) {
        a.tokens[row] = S.bi[17];
        if (a.logprob) a.logprob[row] = fminf((float)(log((double)S.f[0] * sc_me) - log(M)), 0.f);
      }
    }
    xfinish(a, row, rank, ST_OK, -1, nleg, PATH_ALL, 0, nst, 0);
    return;
  }

  // ---- top-k rows settled by the stream: resolve on the candidates ----
  uint32_t beta = 0u;  // the boundary key: kept = keys > beta, plus the first nb copies of beta
  int nb = 0;
  uint64_t Abeta = 0;  // kept values above beta
  uint64_t KMme = 0;   // the mass this CTA keeps
  int share = 0, Nme = 0;
  int path = PATH_SIGMA, passes = 1, nwin = 0, band = 0;
  bool failed = false;
  uint32_t whi = 0, wlo = 0;  // the window the boundary was resolved in
  uint32_t* cntA = reinterpret_cast<uint32_t*>(xsm);  // the row's per-key counts (ring area)
  uint64_t* wtab = reinterpret_cast<uint64_t*>(xsm + XNS * XSB / 2);  // weights of the first XWT keys

  bool sync_first = false;  // the window search must first wait for this pull
  if (cls == XC_TOPK || cls == XC_FLATL) {
    // Every CTA listed all of its values >= its own threshold, so the key
    // range [LO, gk] with LO the largest threshold is complete.  Key index
    // i stands for key gk - i; CTA c counts key k in bin hw_c - k.  The
    // row's counts go to shared memory (ring area), with the weights of the
    // first XWT keys beside them.
    uint32_t LO = 0u;
    for (int c = 0; c < C; ++c) LO = max(LO, S.pub2[c].lo);
    const bool wide = cls == XC_FLATL;  // the stream's own window counts
    const uint32_t* hc = wide ? hcnt : hist;
    const int nk = gk >= LO ? (int)(gk - LO) + 1 : 0;
    band = nk;
    for (int i = tid; i < nk; i += XNT) {
      const uint32_t k = gk - (uint32_t)i;
      uint32_t cnt = 0;
#pragma unroll
      for (int c = 0; c < XMAXC; ++c) {
        if (c < C) {
          const uint32_t hwc = S.pub2[c].hw;
          if (k <= hwc) {
            const uint32_t bq = hwc - k;
            cnt += xcnt(xremote(hc, (uint32_t)c), bq, wide);
          }
        }
      }
      cntA[i] = cnt;
      if (i < XWT) wtab[i] = cnt ? xwfx(XT<DT>::f(xraw(k)), T, zmax) : 0ull;
    }
    __syncthreads();
    const int cpt = (nk + XNT - 1) / XNT;
    const int t0 = min(tid * cpt, nk), t1 = min(t0 + cpt, nk);  // this thread's contiguous keys
    uint32_t ct = 0;
    for (int i = t0; i < t1; ++i) ct += cntA[i];
    uint32_t ctot;
    const uint32_t cpre = xblock_excl<uint32_t>(ct, reinterpret_cast<uint32_t*>(S.wi), &ctot);
    // the listed keys must hold the k-th largest value (or every legal one)
    const bool short_list = cls == XC_TOPK && ctot < (uint32_t)K && ctot != (uint32_t)nleg;
    if (short_list) {
      sync_first = true;
      cls = K < nleg ? -XC_TOPK : XC_FLAT;
    } else {
      // the k-th largest key and its quota (a8.5, a8.6); flat rows, and
      // top-k rows whose every legal value is listed, keep every key
      if (tid == 0) {
        S.bi[18] = (cls == XC_FLATL || ctot < (uint32_t)K) ? nk : -1;
        S.bi[19] = 0;
      }
      __syncthreads();
      if (cls == XC_TOPK && ctot >= (uint32_t)K && cpre < (uint32_t)K && cpre + ct >= (uint32_t)K) {
        uint32_t c = cpre;
        for (int i = t0; i < t1; ++i) {
          if (c + cntA[i] >= (uint32_t)K) {
            S.bi[18] = i;
            S.bi[19] = (int)((uint32_t)K - c);
            break;
          }
          c += cntA[i];
        }
      }
      __syncthreads();
      const int kbin = S.bi[18];
      const int quota = S.bi[19];
      if (kbin < 0) {
        failed = true;
      } else {
        uint64_t mt = 0;
        for (int i = t0; i < min(t1, kbin + 1); ++i) {
          const uint32_t cnt = (i == kbin) ? (uint32_t)quota : cntA[i];
          if (cnt) mt += (uint64_t)cnt * xw_at<DT>(wtab, i, gk, T, zmax);
        }
        uint64_t Mk;
        const uint64_t mpre = xblock_excl<uint64_t>(mt, S.q, &Mk);
        if (cls == XC_TOPK && pp >= 1.f) {
          if (kbin >= nk) {  // every legal value is kept
            beta = 0u;
            nb = 0;
            Abeta = ctot;
          } else {
            beta = gk - (uint32_t)kbin;
            nb = quota;
            Abeta = (uint64_t)(K - quota);
          }
        } else if (cls == XC_FLATL && (double)Mk < (double)pp * Mflat) {
          sync_first = true;  // the boundary lies below the listed values
          cls = XC_FLAT;
        } else {
          // top-p (a8.7): the first key whose prefix reaches ceil(p * Mk)
          const uint64_t P64 =
              (uint64_t)ceil((double)pp * (cls == XC_FLATL ? Mflat : (double)Mk));
          if (tid == 0) S.bi[20] = -1;
          __syncthreads();
          if (mpre < P64 && mpre + mt >= P64) {
            uint64_t c = mpre;
            uint64_t cc = cpre;
            for (int i = t0; i < min(t1, kbin + 1); ++i) {
              const uint64_t avail = (i == kbin) ? (uint64_t)quota : (uint64_t)cntA[i];
              if (!avail) continue;
              const uint64_t w = xw_at<DT>(wtab, i, gk, T, zmax);
              if (c + avail * w >= P64) {
                uint64_t need = w ? (P64 - c + w - 1) / w : avail;
                need = min(max(need, (uint64_t)1), avail);
                S.bi[20] = i;
                S.bi[21] = (int)need;
                S.bq[0] = cc;
                break;
              }
              c += avail * w;
              cc += avail;
            }
          }
          __syncthreads();
          if (S.bi[20] < 0) {
            failed = true;
          } else {
            beta = gk - (uint32_t)S.bi[20];
            nb = S.bi[21];
            Abeta = S.bq[0];
          }
        }
      }
      if (!failed && cls != XC_FLAT) {
        // this CTA's share of beta's copies (ids before this slice come first)
        // and the mass it keeps
        const int ib = beta ? (int)(gk - beta) : nk;  // keys above beta: indices [0, ib)
        if (beta) {
          const uint32_t bq = hw - beta;
          Nme = beta <= hw ? (int)xcnt(hc, bq, wide) : 0;
          if (warp == 0) {
            uint32_t c = 0;
            if (lane < C && lane < (int)rank) {
              const uint32_t hwc = S.pub2[lane].hw;
              if (beta <= hwc) {
                const uint32_t bc2 = hwc - beta;
                c = xcnt(xremote(hc, (uint32_t)lane), bc2, wide);
              }
            }
            c = __reduce_add_sync(0xffffffffu, c);
            if (lane == 0) S.bi[22] = (int)c;
          }
          __syncthreads();
          share = min(max(nb - S.bi[22], 0), Nme);
        }
        uint64_t mine = 0;
        for (int i = tid; i < ib; i += XNT) {
          const uint32_t k = gk - (uint32_t)i;
          if (k > hw) continue;
          const uint32_t c = xcnt(hc, hw - k, wide);
          if (c) mine += (uint64_t)c * xw_at<DT>(wtab, i, gk, T, zmax);
        }
        mine = xblock_total<uint64_t>(mine, S.q);
        KMme = mine + (beta ? (uint64_t)share * xw_at<DT>(wtab, ib, gk, T, zmax) : 0ull);
      }
      whi = gk;
      wlo = LO;
    }
  }
  if (cls == -XC_TOPK || cls == XC_FLAT) {
    // ---- the exact window search over the slice re-read from global ----
    // Windows of WB keys (one 32-bit counter per key).  Each warp counts into
    // its own copy in the ring area (fewer atomic conflicts); the copies are
    // summed into this CTA's histogram, which every CTA then reads.
    failed = false;
    beta = 0u;
    nb = 0;
    Abeta = 0;
    KMme = 0;
    share = 0;
    Nme = 0;
    path = PATH_FULL;
    const int WB = wf >> 1;
    uint32_t* wh = reinterpret_cast<uint32_t*>(xsm);  // XNW copies of WB counters
    const float c2 = L2E / T;
    const uint32_t floor_key = R::KNINF + 1u;
    uint32_t hi = gk;
    uint32_t wl = hi >= floor_key + (uint32_t)(WB - 1) ? hi - (uint32_t)(WB - 1) : floor_key;
    const int ccls = (cls == -XC_TOPK) ? XC_TOPK : XC_FLAT;
    // flat rows that streamed their mass need no pass below the first window
    const bool have_mflat = pcls == XC_FLAT && !(flags & 16);
    enum { FIND_K = 0, FIND_P = 1 };
    int phase = (ccls == XC_TOPK) ? FIND_K : FIND_P;
    uint64_t A = 0, MA = 0, myMA = 0, Mk = 0, P64 = 0;
    uint32_t kap = 0u;
    int quota = 0;
    bool first = true, resolved = false, all_legal = false;
    passes = 0;
    for (int guard = 0; guard < 2 * XMAXWIN; ++guard) {
      ++passes;
      if (!first || sync_first) xcluster_sync();  // every CTA is done reading the previous histograms
      sync_first = false;
      for (int i = tid; i < XNW * WB; i += XNT) wh[i] = 0u;
      __syncthreads();
      const uint32_t l2 = xraw(wl) | (xraw(wl) << 16);
      uint64_t ufm = 0;
      const bool want_uf = first && ccls == XC_FLAT && !have_mflat;
      uint32_t* myh = wh + warp * WB;
      uint32_t kbl = 0u;  // this thread's largest legal key below the window
      for (int v0 = tid; v0 < nvec; v0 += 4 * XNT) {
        uint4 q4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int v = v0 + u * XNT;
          q4[u] = v < nvec ? xgfetch<DT>(v, nfull, n, gsrc, mrow) : make_uint4(NN4, NN4, NN4, NN4);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 q = q4[u];
          const uint32_t vm = xvmax<DT>(q);
          if (xge2<DT>(vm, l2) != 0u || want_uf) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint32_t h = xhalf(q, e);
              if (h == R::NINF) continue;
              const uint32_t k = xkey(h);
              if (k >= wl) {
                if (k <= hi) atomicAdd(&myh[hi - k], 1u);
              } else {
                kbl = max(kbl, k);
                if (want_uf) ufm += xwfx_fast(R::f(h), xmax, c2);
              }
            }
          } else {  // the whole vector lies below the window
            kbl = max(kbl, max(xkey(vm & 0xffffu), xkey(vm >> 16)));
          }
        }
      }
      __syncthreads();
      const int nbins = (int)(hi - wl) + 1;
      for (int bq = tid; bq < nbins; bq += XNT) {
        uint32_t c = 0;
#pragma unroll
        for (int w = 0; w < XNW; ++w) c += wh[w * WB + bq];
        hist[bq] = c;
      }
      if (want_uf) {
        ufm = xblock_total<uint64_t>(ufm, S.q);
        for (int c = tid; c < C; c += XNT) *xremote(&S.uf[rank], (uint32_t)c) = ufm;
      }
      kbl = __reduce_max_sync(0xffffffffu, kbl);
      if (lane == 0) S.wi[warp] = (int)kbl;
      __syncthreads();
      if (tid < C) {
        uint32_t kb = 0u;
        for (int w = 0; w < XNW; ++w) kb = max(kb, (uint32_t)S.wi[w]);
        *xremote(&S.kbelow[rank], (uint32_t)tid) = kb;
      }
      __syncthreads();
      xcluster_sync();  // every CTA's window histogram is complete
      // the next window starts at the largest legal key below this one (empty
      // key ranges are skipped); none below: this window is the last
      uint32_t nxt = 0u;
      for (int c = 0; c < C; ++c) nxt = max(nxt, S.kbelow[c]);
      const bool none_below = nxt < floor_key;
      uint64_t uf_total = 0;
      if (want_uf)
        for (int c = 0; c < C; ++c) uf_total += S.uf[c];
      constexpr int PB = 16;  // bins per thread (WB <= 2048)
      uint32_t cnt[PB];
#pragma unroll
      for (int i = 0; i < PB; ++i) cnt[i] = 0u;
      const int cpt = (nbins + XNT - 1) / XNT;
      const int t0 = tid * cpt;
      {
        const int nw = min(cpt, max(0, nbins - t0));
#pragma unroll
        for (int c = 0; c < XMAXC; ++c) {
          if (c >= C) break;
          const uint32_t* rh = xremote(hist, (uint32_t)c) + t0;
#pragma unroll
          for (int i = 0; i < PB; ++i)
            if (i < nw) cnt[i] += rh[i];
        }
      }
      uint32_t ct = 0;
#pragma unroll
      for (int i = 0; i < PB; ++i) ct += (i < cpt && t0 + i < nbins) ? cnt[i] : 0u;
      uint32_t ctot;
      const uint32_t cpre = xblock_excl<uint32_t>(ct, reinterpret_cast<uint32_t*>(S.wi), &ctot);
      int kbin = -1;
      if (phase == FIND_K) {
        if (A + ctot >= (uint64_t)K) {
          if (A + cpre < (uint64_t)K && A + cpre + ct >= (uint64_t)K) {
            uint64_t c = A + cpre;
#pragma unroll
            for (int i = 0; i < PB; ++i) {
              if (i < cpt && t0 + i < nbins && c < (uint64_t)K && c + cnt[i] >= (uint64_t)K) {
                S.bi[1] = t0 + i;
                S.bi[2] = (int)((uint64_t)K - c);
              }
              c += (i < cpt && t0 + i < nbins) ? cnt[i] : 0u;
            }
          }
          __syncthreads();
          kbin = S.bi[1];
          quota = S.bi[2];
          kap = hi - (uint32_t)kbin;
          __syncthreads();
        }
      } else if (kap != 0u && kap >= wl && kap <= hi) {
        kbin = (int)(hi - kap);
      }
      uint64_t mt = 0;
#pragma unroll
      for (int i = 0; i < PB; ++i) {
        const int b = t0 + i;
        if (i >= cpt || b >= nbins || !cnt[i]) continue;
        if (kbin >= 0 && b > kbin) continue;
        const uint64_t nn = (b == kbin) ? (uint64_t)quota : (uint64_t)cnt[i];
        mt += nn * xwfx(R::f(xraw(hi - (uint32_t)b)), T, zmax);
      }
      uint64_t mtot;
      const uint64_t mpre = xblock_excl<uint64_t>(mt, S.q, &mtot);
      if (phase == FIND_K) {
        if (kbin < 0) {
          if (tid == 0) S.win[nwin] = XWin{hi, wl, A, MA, myMA};
          const uint64_t mine = xmy_mass32<DT>(hist, hi, nbins, T, zmax, S.q);
          ++nwin;
          A += ctot;
          MA += mtot;
          myMA += mine;
          first = false;
          if (wl <= floor_key || none_below || nwin >= XMAXWIN - 1) {
            failed = true;
            break;
          }
          hi = min(wl - 1u, nxt);
          wl = hi >= floor_key + (uint32_t)(WB - 1) ? hi - (uint32_t)(WB - 1) : floor_key;
          continue;
        }
        Mk = MA + mtot;
        if (pp >= 1.f) {
          beta = kap;
          nb = quota;
          Abeta = (uint64_t)K - (uint64_t)quota;
          resolved = true;
        } else {
          P64 = (uint64_t)ceil((double)pp * (double)Mk);
          phase = FIND_P;
        }
      } else if (first) {
        // flat row: the whole legal mass, from the stream or from this pass.
        // top_p = 1 keeps every legal value (a top-k row whose k covers the
        // legal set): no target is reached, the windows walk to the last
        // legal key and sum the exact masses on the way.
        const double m = have_mflat ? Mflat : (double)(mtot + uf_total);
        P64 = pp >= 1.f ? ~0ull : (uint64_t)ceil((double)pp * m);
      }
      if (!resolved && phase == FIND_P) {
        if (MA >= P64 && nwin > 0) {
          int wsel = 0;
          for (int w = 0; w < nwin; ++w)
            if (S.win[w].MA < P64) wsel = w;
          const XWin W0 = S.win[wsel];
          hi = W0.hi;
          wl = W0.lo;
          A = W0.A;
          MA = W0.MA;
          myMA = W0.myMA;
          nwin = wsel;
          first = false;
          __syncthreads();
          continue;
        }
        if (MA + mtot < P64) {
          if (tid == 0) S.win[nwin] = XWin{hi, wl, A, MA, myMA};
          const uint64_t mine =
              xmy_mass32<DT>(hist, hi, kbin >= 0 ? kbin + 1 : nbins, T, zmax, S.q);
          ++nwin;
          A += ctot;
          MA += mtot;
          myMA += mine;
          first = false;
          if (wl <= floor_key || none_below || nwin >= XMAXWIN - 1) {
            beta = 0u;  // no prefix reaches p after rounding: keep every legal value
            nb = 0;
            Abeta = A;
            all_legal = true;
            resolved = true;
            break;
          }
          hi = min(wl - 1u, nxt);
          wl = hi >= floor_key + (uint32_t)(WB - 1) ? hi - (uint32_t)(WB - 1) : floor_key;
          continue;
        }
        if (tid == 0) S.bi[3] = -1;
        __syncthreads();
        if (MA + mpre < P64 && MA + mpre + mt >= P64) {
          uint64_t c = MA + mpre;
          uint64_t cc = A + cpre;
          bool done = false;
#pragma unroll
          for (int i = 0; i < PB; ++i) {
            const int b = t0 + i;
            if (done || i >= cpt || b >= nbins || !cnt[i] || (kbin >= 0 && b > kbin)) continue;
            const uint64_t avail = (b == kbin) ? (uint64_t)quota : (uint64_t)cnt[i];
            const uint64_t w = xwfx(R::f(xraw(hi - (uint32_t)b)), T, zmax);
            if (c + avail * w >= P64) {
              uint64_t need = w ? (P64 - c + w - 1) / w : avail;
              need = min(max(need, (uint64_t)1), avail);
              S.bi[3] = b;
              S.bi[4] = (int)need;
              S.bq[2] = cc;
              done = true;
            }
            c += avail * w;
            cc += avail;
          }
        }
        __syncthreads();
        if (S.bi[3] < 0) {
          failed = true;
          break;
        }
        beta = hi - (uint32_t)S.bi[3];
        nb = S.bi[4];
        Abeta = S.bq[2];
        __syncthreads();
        resolved = true;
      }
      if (resolved) break;
      first = false;
    }
    if (!resolved) failed = true;
    band = (int)(hi - wl) + 1;
    whi = hi;
    wlo = wl;
    if (!failed) {
      const int bb = (int)(hi - beta);
      const bool beta_in = beta != 0u && beta >= wl && beta <= hi;
      if (beta_in) {
        Nme = (int)hist[bb];
        if (warp == 0) {
          uint32_t c = 0;
          if (lane < C && lane < (int)rank) c = xremote(hist, (uint32_t)lane)[bb];
          c = __reduce_add_sync(0xffffffffu, c);
          if (lane == 0) S.bi[6] = (int)c;
        }
        __syncthreads();
        share = min(max(nb - S.bi[6], 0), Nme);
      }
      const int nbins = (int)(hi - wl) + 1;
      const int top = all_legal ? 0 : (beta_in ? bb : nbins);
      const uint64_t mine = xmy_mass32<DT>(hist, hi, top, T, zmax, S.q);
      KMme = myMA + mine;
      if (beta_in) KMme += (uint64_t)share * xwfx(R::f(xraw(beta)), T, zmax);
    }
  }

  // ---- B3: every CTA's kept mass ----
  if (tid == 0) S.bi[23] = 0;  // pass C's expired waits, set by any CTA of the row
  for (int c = tid; c < C; c += XNT) *xremote(&S.km[rank], (uint32_t)c) = KMme;
  __syncthreads();
  xcluster_sync();  // the kept masses are in place
  uint64_t Mp = 0;
  for (int c = 0; c < C; ++c) Mp += S.km[c];
  if (failed || Mp == 0) {
    // no exact resolution (should not happen): an error status, never a token
    if (mout)
      for (int w = tid; w < ((n + 31) >> 5); w += XNT) mout[w] = 0u;
    if (pout)
      for (int e = tid; e < n; e += XNT) pout[e] = 0.f;
    xfinish(a, row, rank, ST_TIMEOUT, -1, 0, PATH_ERROR, __LINE__, passes, nwin);
    return;
  }
  const float Mf = (float)Mp * 0x1p-40f;
  const float bval = beta ? XT<DT>::f(xraw(beta)) : -INFINITY;
  const uint32_t bv2 = beta ? (xraw(beta) | (xraw(beta) << 16)) : 0u;
  const bool from_list = cls == XC_TOPK;
  const int nc = from_list ? min(S.ncand, a.cap) : 0;
  // Outside the list a partial tie (some of this CTA's copies of beta kept)
  // is settled after pass C from the copies' ids, which the pass lists, when
  // they fit the id list; otherwise by a selection over the slice first.
  const bool dtie = !from_list && beta && share > 0 && share < Nme && Nme <= XBL;

  // ---- the id cut among the copies of beta kept here (earliest ids) ----
  int cut = INT_MAX;  // copies of beta with local id < cut are kept
  if (beta && share < Nme && !dtie) {
    if (share == 0) {
      cut = -1;
    } else {
      // radix selection of the share-th smallest local id among the copies:
      // three rounds of 6-bit digits over ids < 2^18
      uint32_t* h64 = S.h64;  // 64 counters
      int want = share - 1;  // 0-based rank
      uint32_t prefix = 0u;
      for (int round = 0; round < 3; ++round) {
        const int sh = 12 - 6 * round;
        if (tid < 64) h64[tid] = 0u;
        __syncthreads();
        if (from_list) {
          for (int i = tid; i < nc; i += XNT) {
            const int id = cid[i];
            if (ckey[i] == beta && ((uint32_t)id >> (sh + 6)) == (prefix >> (sh + 6)))
              atomicAdd(&h64[(id >> sh) & 63], 1u);
          }
        } else {
          for (int v0 = tid; v0 < nvec; v0 += 4 * XNT) {
            uint4 q4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int v = v0 + u * XNT;
              q4[u] = v < nvec ? xgfetch<DT>(v, nfull, n, gsrc, mrow) : make_uint4(NN4, NN4, NN4, NN4);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int v = v0 + u * XNT;
              const uint4 q = q4[u];
              if (!(xeq2<DT>(q.x, bv2) | xeq2<DT>(q.y, bv2) | xeq2<DT>(q.z, bv2) |
                    xeq2<DT>(q.w, bv2)))
                continue;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int id = v * 8 + e;
                if (R::f(xhalf(q, e)) == bval && ((uint32_t)id >> (sh + 6)) == (prefix >> (sh + 6)))
                  atomicAdd(&h64[(id >> sh) & 63], 1u);
              }
            }
          }
        }
        __syncthreads();
        if (warp == 0) {
          const uint32_t c0 = h64[2 * lane], c1 = h64[2 * lane + 1];
          const uint32_t s = c0 + c1;
          const uint32_t inc = xwarp_incl<uint32_t>(s);
          const uint32_t hit = __ballot_sync(0xffffffffu, inc > (uint32_t)want);
          const int L = hit ? __ffs(hit) - 1 : 31;
          const uint32_t bef = __shfl_sync(0xffffffffu, inc - s, L);
          const uint32_t cc0 = __shfl_sync(0xffffffffu, c0, L);
          if (lane == 0) {
            const int d = (bef + cc0 > (uint32_t)want) ? 2 * L : 2 * L + 1;
            S.bi[7] = d;
            S.bi[8] = want - (int)(bef + (d & 1 ? cc0 : 0u));
          }
        }
        __syncthreads();
        prefix |= (uint32_t)S.bi[7] << sh;
        want = S.bi[8];
        __syncthreads();
      }
      cut = (int)prefix + 1;
    }
  }

  // ---- draw target and the CTA that holds it (a8.8) ----
  uint64_t tgt = 0, before = 0;
  int cs = -1;
  if (samp_mode) {
    tgt = xscale24(k24, Mp);
    cs = C - 1;
    for (int c = 0; c < C; ++c) {
      if (before + S.km[c] > tgt) {
        cs = c;
        break;
      }
      before += S.km[c];
    }
  }
  const bool drawer = (int)rank == cs;

  if (from_list) {
    // ---- outputs from the candidate list ----
    if (mout)
      for (int w = tid; w < ((n + 31) >> 5); w += XNT) mout[w] = 0u;
    if (pout)
      for (int e = tid; e < n; e += XNT) pout[e] = 0.f;
    __syncthreads();
    for (int i = tid; i < nc; i += XNT) {
      const uint32_t k = ckey[i];
      const int id = cid[i];
      const float x = XT<DT>::f(xraw(k));
      if ((unsigned)id >= (unsigned)n || !xkept(bval, cut, x, id)) continue;
      if (mout) red_or_global(&mout[id >> 5], 1u << (id & 31));
      if (pout) pout[id] = xweight(x, T, zmax) / Mf;
    }
    if (drawer) {
      // id buckets (the histogram area as 64-bit masses), the bucket that
      // holds the target, then the kept candidates of that bucket in id order
      uint64_t* bkt = reinterpret_cast<uint64_t*>(hist);
      const int nbk = wf / 4;
      const int bw = (n + nbk - 1) / nbk;
      for (int i = tid; i < nbk; i += XNT) bkt[i] = 0ull;
      __syncthreads();
      for (int i = tid; i < nc; i += XNT) {
        const uint32_t k = ckey[i];
        const int id = cid[i];
        if ((unsigned)id >= (unsigned)n || k > gk || !xkept(bval, cut, XT<DT>::f(xraw(k)), id))
          continue;
        smem_add_u64(&bkt[id / bw], xw_at<DT>(wtab, (int)(gk - k), gk, T, zmax));
      }
      __syncthreads();
      if (warp == 0) {
        uint64_t rem;
        const int b = xlocate<uint64_t>(bkt, nbk, tgt - before, &rem);
        if (lane == 0) {
          S.bi[9] = b;
          S.bq[4] = rem;
          S.bi[10] = 0;
        }
      }
      __syncthreads();
      const int b = S.bi[9];
      const uint64_t rem = S.bq[4];
      uint2* g = reinterpret_cast<uint2*>(hist);  // (id, key) of the bucket's kept candidates
      for (int i = tid; i < nc; i += XNT) {
        const uint32_t k = ckey[i];
        const int id = cid[i];
        if ((unsigned)id >= (unsigned)n || k > gk || id / bw != b ||
            !xkept(bval, cut, XT<DT>::f(xraw(k)), id))
          continue;
        const int p = atomicAdd(&S.bi[10], 1);
        if (p < nbk) g[p] = make_uint2((uint32_t)id, k);
      }
      __syncthreads();
      const int ng = min(S.bi[10], nbk);
      if (tid == 0) S.bi[11] = 0;
      __syncthreads();
      for (int i = tid; i < ng; i += XNT) {
        const int id = (int)g[i].x;
        const uint64_t w = xw_at<DT>(wtab, (int)(gk - g[i].y), gk, T, zmax);
        uint64_t cum = 0;
        for (int j = 0; j < ng; ++j)
          if ((int)g[j].x < id) cum += xw_at<DT>(wtab, (int)(gk - g[j].y), gk, T, zmax);
        if (cum <= rem && rem < cum + w) {
          S.bi[11] = id;
          S.bi[12] = (int)g[i].y;
        }
      }
      __syncthreads();
      if (tid == 0) {
        a.tokens[row] = s0 + S.bi[11];
        if (a.logprob) {
          const float wt = xweight(XT<DT>::f(xraw((uint32_t)S.bi[12])), T, zmax);
          a.logprob[row] = fminf(logf(wt) - logf(Mf), 0.f);
        }
      }
    }
  } else {
    // ---- pass C: the slice streamed through the ring again ----
    // Kept: above beta, or a copy of beta before the id cut (an open cut:
    // the copies are listed and settled after the pass).  The drawer sums
    // the kept weights per (stage, warp) cell, the cells being consecutive
    // id ranges of XVW vectors.
    unsigned char* reg = xsm + xoff_hist();
    uint64_t* pq = reinterpret_cast<uint64_t*>(reg);  // per-cell kept masses
    int* blist = reinterpret_cast<int*>(reg + XMAXST * XNW * 8);  // copies of beta
    uint64_t* wt = reinterpret_cast<uint64_t*>(reg + XMAXST * XNW * 8 + XBL * 4);
    const int tcap = (xoff_sh(wf, a.cap) - xoff_hist() - XMAXST * XNW * 8 - XBL * 4) / 8;
    const int ntab = drawer ? (beta ? min((int)(gk - beta) + 1, tcap) : tcap) : 0;
    const uint32_t kv2 = beta ? bv2 : NN4;  // kept: above this (every legal value when beta = 0)
    const bool run = mout || pout || drawer;
    int tfail = 0;
    if (run) {
      for (int i = tid; i < ntab; i += XNT) {
        const uint32_t k = gk - (uint32_t)i;
        wt[i] = k > R::KNINF ? xwfx(R::f(xraw(k)), T, zmax) : 0ull;
      }
      if (tid == 0) S.bi[13] = 0;
      __syncthreads();  // the ring area is free, the table ready
      // slot j finished (nst - j + XNS - 1) / XNS phases in the first stream
      int issued2 = 0;
      if (tid == 0) {
        fence_proxy_async_smem();
        for (int t = 0; t < XNS && t < nst; ++t, ++issued2) {
          const int v0 = t * XVS, v1 = min(nfull, v0 + XVS);
          const uint32_t bytes = v1 > v0 ? (uint32_t)(v1 - v0) * 16u : 0u;
          mbar_arrive_expect_tx(&S.bar[t], bytes);
          if (bytes) bulk_g2s(xsm + t * XSB, gsrc + (size_t)v0 * 8, bytes, &S.bar[t]);
        }
      }
      const bool ties = beta && (dtie || cut >= 0);  // copies of beta may be kept
      for (int st2 = 0; st2 < nst; ++st2) {
        const int slot = st2 % XNS;
        const int par = (((nst - slot + XNS - 1) / XNS) + st2 / XNS) & 1;
        if (!tfail && st2 * XVS < nfull && !mbar_wait_bounded(&S.bar[slot], par, a.wait_limit))
          tfail = 1;
        uint64_t sw = 0;
        // the warp's XSUB vectors of this stage, loaded together
        uint4 q4[XSUB];
#pragma unroll
        for (int r = 0; r < XSUB; ++r) {
          const int v = st2 * XVS + warp * XVW + r * 32 + lane;
          q4[r] = (v < nvec && !tfail) ? xfetch<DT>(xsm, slot, v, nfull, n, gsrc, mrow)
                                       : make_uint4(NN4, NN4, NN4, NN4);
        }
#pragma unroll
        for (int r = 0; r < XSUB; ++r) {
          const int v = st2 * XVS + warp * XVW + r * 32 + lane;
          const bool in = v < nvec && !tfail;
          uint32_t byte = 0;
          const uint4 q = q4[r];
          if (in) {
            byte = xbits8(xgt2<DT>(q.x, kv2), xgt2<DT>(q.y, kv2), xgt2<DT>(q.z, kv2),
                          xgt2<DT>(q.w, kv2));
            if (ties) {
              const uint32_t eb = xbits8(xeq2<DT>(q.x, bv2), xeq2<DT>(q.y, bv2),
                                         xeq2<DT>(q.z, bv2), xeq2<DT>(q.w, bv2));
              if (eb) {
#pragma unroll 1
                for (uint32_t m = eb; m; m &= m - 1u) {
                  const int id = v * 8 + (__ffs(m) - 1);
                  if (dtie) {
                    const int pos = atomicAdd(&S.bi[13], 1);
                    if (pos < XBL) blist[pos] = id;
                  } else if (id < cut) {
                    byte |= 1u << (__ffs(m) - 1);
                  }
                }
              }
            }
          }
          if (mout) xput_mask_byte(mout, v, byte, in);
          if (drawer && byte) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (!((byte >> e) & 1u)) continue;
              const uint32_t h = xhalf(q, e);
              const int i = (int)(gk - xkey(h));
              sw += i < ntab ? wt[i] : xwfx(R::f(h), T, zmax);
            }
          }
          if (pout && in) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (v * 8 + e < n)
                pout[v * 8 + e] = ((byte >> e) & 1u) ? xweight(R::f(xhalf(q, e)), T, zmax) / Mf : 0.f;
          }
        }
        if (drawer) {
          sw = xwarp_sum64(sw);
          if (lane == 0) pq[st2 * XNW + warp] = sw;
        }
        // every warp is done with the slot; after an expired wait no more copies go out
        tfail = __syncthreads_or(tfail);
        if (tid == 0 && !tfail && st2 + XNS < nst) {
          const int v0 = (st2 + XNS) * XVS, v1 = min(nfull, v0 + XVS);
          const uint32_t bytes = v1 > v0 ? (uint32_t)(v1 - v0) * 16u : 0u;
          mbar_arrive_expect_tx(&S.bar[slot], bytes);
          if (bytes) bulk_g2s(xsm + slot * XSB, gsrc + (size_t)v0 * 8, bytes, &S.bar[slot]);
          ++issued2;
        }
      }
      if (tfail && tid == 0) {
        // wait (bounded again) for every copy still in flight into the ring
        for (int t = max(0, issued2 - XNS); t < issued2; ++t) {
          const int sl = t % XNS;
          mbar_wait_bounded(&S.bar[sl], (((nst - sl + XNS - 1) / XNS) + t / XNS) & 1, XDRAIN);
        }
      }
      if (dtie && !tfail) {
        // the share-th earliest copy of beta here; then the kept copies' bits,
        // probabilities and masses
        const int nbl = min(S.bi[13], XBL);
        cut = xsel_id(blist, nbl, share - 1, S) + 1;
        const uint64_t wb = drawer ? xwfx(bval, T, zmax) : 0ull;
        for (int i = tid; i < nbl; i += XNT) {
          const int id = blist[i];
          if (id >= cut) continue;
          if (mout) atomicOr(&mout[id >> 5], 1u << (id & 31));
          if (pout) pout[id] = xweight(bval, T, zmax) / Mf;
          if (drawer) smem_add_u64(&pq[(id >> 3) / XVW], wb);
        }
        __syncthreads();
      }
      if (drawer && !tfail) {
        if (warp == 0) {
          uint64_t rem;
          const int e = xlocate<uint64_t>(pq, nst * XNW, tgt - before, &rem);
          if (lane == 0) {
            S.bi[12] = e;
            S.bq[5] = rem;
          }
        }
        __syncthreads();
        if (warp == 0) {
          // the cell's XVW vectors, 32 at a time, in id order
          const int e = S.bi[12];
          uint64_t rem = S.bq[5];
          const int vb = (e / XNW) * XVS + (e % XNW) * XVW;
          uint4 q4[XSUB];
#pragma unroll
          for (int r = 0; r < XSUB; ++r) {
            const int v = vb + r * 32 + lane;
            q4[r] = v < nvec ? xgfetch<DT>(v, nfull, n, gsrc, mrow) : make_uint4(NN4, NN4, NN4, NN4);
          }
          bool done = false;
#pragma unroll
          for (int r = 0; r < XSUB; ++r) {
            if (done) break;
            const int v = vb + r * 32 + lane;
            uint64_t sv = 0;
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) {
              const uint32_t h = xhalf(q4[r], e8);
              if (h == R::NINF || !xkept(bval, cut, R::f(h), v * 8 + e8)) continue;
              const int i = (int)(gk - xkey(h));
              sv += i < ntab ? wt[i] : xwfx(R::f(h), T, zmax);
            }
            const uint64_t inc = xwarp_incl<uint64_t>(sv);
            const uint64_t tot = __shfl_sync(0xffffffffu, inc, 31);
            if (rem >= tot && r + 1 < XSUB) {
              rem -= tot;
              continue;
            }
            done = true;
            const uint32_t hit = __ballot_sync(0xffffffffu, inc > rem);
            const int L = hit ? __ffs(hit) - 1 : 31;
            if (lane == L) {
              uint64_t c = inc - sv;
              int tok = -1;
              float wx = 0.f;
              for (int e8 = 0; e8 < 8; ++e8) {
                const uint32_t h = xhalf(q4[r], e8);
                if (h == R::NINF || !xkept(bval, cut, R::f(h), v * 8 + e8)) continue;
                const int i = (int)(gk - xkey(h));
                c += i < ntab ? wt[i] : xwfx(R::f(h), T, zmax);
                tok = s0 + v * 8 + e8;
                wx = R::f(h);
                if (c > rem) break;
              }
              a.tokens[row] = tok;
              if (a.logprob) a.logprob[row] = fminf(logf(xweight(wx, T, zmax)) - logf(Mf), 0.f);
            }
          }
        }
      }
    }
    // ---- the row's pass C statuses: every CTA learns of any expired wait ----
    if (tfail && tid < C) atomicOr(xremote(&S.bi[23], (uint32_t)tid), 1);
    __syncthreads();
    xcluster_sync();  // no remote access follows
    if (S.bi[23]) {
      if (mout)
        for (int w = tid; w < ((n + 31) >> 5); w += XNT) mout[w] = 0u;
      if (pout)
        for (int e = tid; e < n; e += XNT) pout[e] = 0.f;
      xfinish(a, row, rank, ST_TIMEOUT, -1, 0, PATH_ERROR, __LINE__, passes, nwin);
      return;
    }
  }
  xfinish(a, row, rank, ST_OK, -1, (int)(Abeta + (uint64_t)nb), path, band, passes, nwin);
  (void)whi;
  (void)wlo;
}

}  // namespace smp
