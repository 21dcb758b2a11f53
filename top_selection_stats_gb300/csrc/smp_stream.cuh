// smp_stream.cuh -- fused top-k / top-p truncation and sampling for sm_103a.
//
// One CTA per row.  The row streams once from HBM through a ring of NSTAGE
// shared-memory stages filled by 1-D bulk TMA copies (cp.async.bulk +
// mbarrier); two CTAs share an SM, so a B=256 batch is in flight at once on
// 152 SMs and the HBM stream is never interrupted by a wave boundary.
//
// Per row (contract of the AI Infra KB note M012, sections 02-03):
//   temperature (0 = greedy argmax) -> legal mask -> top-k (earliest ids win
//   ties) -> top-p (shortest prefix whose mass reaches p) -> renormalise ->
//   inverse-CDF draw in token-id order with a Philox4x32-10 uniform.
//
// Main pass, per 16-byte vector of each chunk as it lands:
//   * the grammar mask is applied in place (illegal -> -inf);
//   * packed bf16x2 / f16x2 max and min give the row max, the argmax, the
//     NaN / +inf flag and the legal count (statistics, Qrita paper notes key
//     design 1);
//   * sigma truncation (Qrita key design 1): thresholds t = mu + delta*sigma,
//     lowered by a 0.2|t| margin, with mean and deviation from the first chunk
//     (a sample of the row) and delta = Phi^-1(1 - k/V) from a host table;
//     four thresholds are counted and the candidates above the lowest are
//     compacted in id order, a vector at a time only when its packed max
//     reaches the threshold;
//   * rows whose kept set is every legal token accumulate their mass chunk
//     by chunk and write the kept mask on the fly.
// After the pass the tightest valid band is selected on chip: three-pivot
// search for the k-th value (Qrita key design 2), the tie quota by prefix
// counts (key design 3), the same pivot search on probability mass for
// top-p, and the id-order draw.  Rows whose band does not validate (very flat
// rows under top-p, k beyond the band buffer) take an exact multi-pivot
// refinement that re-reads the row (from L2) a few times.
#pragma once

#include "smp_device.cuh"

namespace smp {

constexpr int NSTAGE = 3;            // ring stages
constexpr int STAGE_BYTES = 16384;   // bytes per stage (one chunk)
constexpr int CAP = 4096;            // candidate list capacity
constexpr int MAXCH = 128;           // chunks per row, at most
constexpr int NPIV = 8;              // pivots per refinement pass
constexpr int NOT_MEMBER = (int)0x80000000;
constexpr uint32_t KEY_MIN = 0x00800000u;  // fkey(-FLT_MAX): the smallest legal key

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
  int use_tma;  // rows are 16-byte aligned: stage with bulk copies
  float delta[DTAB];
};

// Block-level scratch (after the ring, the candidate list and the staging).
struct Sh {
  uint64_t full[NSTAGE];
  double rd[2][3][NWARP];
  uint32_t ru[2][3][NWARP];
  int ri[2][3][NWARP];
  double bd[16][NWARP];
  int bi[16][NWARP];
  float bf[4][NWARP];
  int wst[NWARP];
  double chunk_mass[MAXCH];
  float chunk_zref[MAXCH];
  int chunk_ties[MAXCH];
  double cpair_m[NWARP];
  float cpair_z[NWARP];
  float thr[NTHR];
  int flag[8];
  int sel_thread;
  double sel_base;
};

__host__ __device__ inline int esize_of(int dt) { return dt == DT_F32 ? 4 : 2; }

constexpr int SMEM_RING = NSTAGE * STAGE_BYTES;
constexpr int SMEM_CAND = CAP * 8;
constexpr int SMEM_TOTAL = SMEM_RING + SMEM_CAND + (int)sizeof(Sh) + 128;

template <int DT>
struct ElemT {
  static constexpr int ES = (DT == DT_F32) ? 4 : 2;
  static constexpr int EPV = 16 / ES;
  static constexpr int CE = STAGE_BYTES / ES;  // elements per chunk
  static constexpr int NVEC = CE / EPV;        // vectors per chunk
  static constexpr int VW = NVEC / NWARP;      // vectors per warp per chunk
  static constexpr int ITW = VW / 32;          // warp iterations per chunk
};

template <int DT>
struct Ctx {
  const KArgs* a;
  const uint32_t* bm;  // this row's bitmask words, or null
  int W, use_tma;
  char* ring;
  uint32_t* ck;  // candidate keys (id order)
  int* ci;       // candidate ids (bit 31: not a member)
  Sh* sh;
  int row, V, nch;
  const char* src;
  uint32_t parity;  // per-stage mbarrier parity bits
  int timeout;
  float temp, m_z, gmax, c2;
};

// ---------------------------------------------------------------------------
// Element helpers (16-byte vectors: 8 bf16 / 8 fp16 / 4 fp32)
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ void unpack(const uint4 r, float (&x)[ElemT<DT>::EPV]) {
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
// Max ignoring NaN (rows are known finite when this is used).
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

// The contract's weight: expf(fl32(x / T) - fl32(max / T)).
template <int DT>
__device__ __forceinline__ float weight(const Ctx<DT>& X, float x) {
  return expf(__fdiv_rn(x, X.temp) - X.m_z);
}
// The contract's weight relative to an arbitrary reference zr (= fl32(ref / T)).
template <int DT>
__device__ __forceinline__ float weight_rel(const Ctx<DT>& X, float x, float zr) {
  return expf(__fdiv_rn(x, X.temp) - zr);
}
// Cheap weight for bulk sums that only steer band choices: the hardware
// base-2 exponential of (x - ref) * log2(e) / T.
__device__ __forceinline__ float fast_exp2(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// ---------------------------------------------------------------------------
// Row streaming through the TMA ring.  ring_begin issues the first NSTAGE
// chunks; ring_wait(c) returns the stage holding chunk c once it landed
// (elements past V are -inf); ring_release(c) frees the stage after a block
// barrier and issues chunk c + NSTAGE into it.  mbarrier waits are bounded
// (~2 s): a timeout is recorded and the pass continues.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ void issue_chunk(Ctx<DT>& X, int c, int s) {
  constexpr int ES = ElemT<DT>::ES, CE = ElemT<DT>::CE;
  const int ne = min(CE, X.V - c * CE);
  const uint32_t bytes = X.use_tma ? (uint32_t)((ne * ES) & ~15) : 0u;
  uint64_t* bar = &X.sh->full[s];
  // order earlier generic-proxy stores to the stage before the async copy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_arrive_expect_tx(bar, bytes);
  if (bytes > 0)
    bulk_g2s(X.ring + (size_t)s * STAGE_BYTES, X.src + (size_t)c * CE * ES, bytes, bar);
}

template <int DT>
__device__ __forceinline__ void ring_begin(Ctx<DT>& X) {
  __syncthreads();
  if (threadIdx.x == 0)
    for (int s = 0; s < NSTAGE && s < X.nch; ++s) issue_chunk(X, s, s);
}

template <int DT>
__device__ __forceinline__ char* ring_wait(Ctx<DT>& X, int c) {
  constexpr int ES = ElemT<DT>::ES, CE = ElemT<DT>::CE;
  const int s = c % NSTAGE;
  char* stage = X.ring + (size_t)s * STAGE_BYTES;
  const uint32_t par = (X.parity >> s) & 1u;
  if (!mbar_wait_bounded(&X.sh->full[s], par, 4000000000ll)) X.timeout = 1;
  X.parity ^= 1u << s;
  // elements not covered by the bulk copy (misaligned rows, the sub-16-byte
  // tail) by plain loads, and -inf past the end of the row
  const int ne = min(CE, X.V - c * CE);
  const int nb = X.use_tma ? ((ne * ES) & ~15) / ES : 0;
  if (nb < CE) {
    const char* g = X.src + (size_t)c * CE * ES;
    for (int e = nb + (int)threadIdx.x; e < CE; e += NT) {
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
  return stage;
}

template <int DT>
__device__ __forceinline__ void ring_release(Ctx<DT>& X, int c) {
  __syncthreads();
  if (threadIdx.x == 0 && c + NSTAGE < X.nch) issue_chunk(X, c + NSTAGE, c % NSTAGE);
}

// Bitmask word for element index e (global in the row); 0 past V.
template <int DT>
__device__ __forceinline__ uint32_t mask_bits(const Ctx<DT>& X, int e) {
  constexpr int EPV = ElemT<DT>::EPV;
  const int w = e >> 5;
  if (w >= X.W) return 0u;
  return (__ldg(X.bm + w) >> (e & 31)) & ((1u << EPV) - 1u);
}

// Lane l of warp w holds vector (w * VW + it * 32 + l) of a chunk.
template <int DT>
__device__ __forceinline__ int warp_vec(int it) {
  return (threadIdx.x >> 5) * ElemT<DT>::VW + it * 32 + (threadIdx.x & 31);
}

// Ordered compaction into the candidate list.  A chunk is compacted in two
// walks: the first counts each warp's members (warp totals -> sh->wst), the
// second writes them at nlist + (members of earlier warps) + warp rank, so
// the list stays in id order (warps own contiguous ranges of the chunk).
// list_emit writes one iteration's members; `pos` is the warp's running
// position.  Entries past CAP are counted but not stored.
template <int DT>
__device__ __forceinline__ void list_emit(const Ctx<DT>& X, int gid0, const float* x,
                                          uint32_t bits, int& pos) {
  constexpr int EPV = ElemT<DT>::EPV;
  const int c = __popc(bits);
  const int incl = warp_incl_scan(c);
  int p = pos + incl - c;
#pragma unroll
  for (int j = 0; j < EPV; ++j)
    if ((bits >> j) & 1u) {
      if (p < CAP) {
        X.ck[p] = fkey(x[j]);
        X.ci[p] = gid0 + j;
      }
      ++p;
    }
  pos += __shfl_sync(0xffffffffu, incl, 31);
}

// After the counting walk: publish warp totals, return this warp's start
// position and (via total) the chunk's member count.
template <int DT>
__device__ __forceinline__ int list_warp_base(const Ctx<DT>& X, int warp_count, int nlist,
                                              int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wc = __reduce_add_sync(0xffffffffu, warp_count);
  if (lane == 0) X.sh->wst[warp] = wc;
  __syncthreads();
  int base = nlist;
  total = 0;
  for (int w = 0; w < NWARP; ++w) {
    if (w < warp) base += X.sh->wst[w];
    total += X.sh->wst[w];
  }
  __syncthreads();  // wst is reused by the next walk
  return base;
}

// ---------------------------------------------------------------------------
// Block reductions (NT threads).  Each uses slot parity `par` so that
// consecutive calls need one __syncthreads each.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ double bsum_d(const Ctx<DT>& X, double v, int slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) X.sh->bd[slot][warp] = v;
  __syncthreads();
  double r = 0.0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r += X.sh->bd[slot][w];
  return r;
}
template <int DT>
__device__ __forceinline__ int bsum_i(const Ctx<DT>& X, int v, int slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_add_sync(0xffffffffu, v);
  if (lane == 0) X.sh->bi[slot][warp] = v;
  __syncthreads();
  int r = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r += X.sh->bi[slot][w];
  return r;
}
template <int DT>
__device__ __forceinline__ uint32_t bmin_u(const Ctx<DT>& X, uint32_t v, int slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_min_sync(0xffffffffu, v);
  if (lane == 0) X.sh->bi[slot][warp] = (int)v;
  __syncthreads();
  uint32_t r = 0xffffffffu;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r = min(r, (uint32_t)X.sh->bi[slot][w]);
  return r;
}
template <int DT>
__device__ __forceinline__ uint32_t bmax_u(const Ctx<DT>& X, uint32_t v, int slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_max_sync(0xffffffffu, v);
  if (lane == 0) X.sh->bi[slot][warp] = (int)v;
  __syncthreads();
  uint32_t r = 0u;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r = max(r, (uint32_t)X.sh->bi[slot][w]);
  return r;
}

// ---------------------------------------------------------------------------
// Selection on the candidate list (n entries, id order).  Three-pivot search
// (Qrita key design 2) in the order-preserving key space: pivots
// tau_q = lo + q(hi - lo)/4; one pass gives N = #{key > tau}, the smallest
// key above tau and its multiplicity (warp REDUX + one block combine per
// round); stop when N >= K and N - mult < K.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ uint32_t pivot_count(const Ctx<DT>& X, int n, int K, int above, int& ngt, int& rounds) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int j = threadIdx.x; j < n; j += NT) {
    if (X.ci[j] & NOT_MEMBER) continue;
    mn = min(mn, X.ck[j]);
    mx = max(mx, X.ck[j]);
  }
  uint32_t lo = bmin_u(X, mn, 0), hi = bmax_u(X, mx, 1);
  rounds = 0;
  int par = 0;
  for (int guard = 0; guard < 64 && lo < hi; ++guard) {
    ++rounds;
    uint32_t tau[3];
    const unsigned long long span = (unsigned long long)(hi - lo);
#pragma unroll
    for (int q = 0; q < 3; ++q) tau[q] = lo + (uint32_t)((span * (q + 1)) / 4);
    int cnt[3] = {0, 0, 0}, mc[3] = {0, 0, 0};
    uint32_t mk[3] = {0xffffffffu, 0xffffffffu, 0xffffffffu};
    for (int j = threadIdx.x; j < n; j += NT) {
      if (X.ci[j] & NOT_MEMBER) continue;
      const uint32_t k = X.ck[j];
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
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int c = __reduce_add_sync(0xffffffffu, cnt[q]);
      const uint32_t m = __reduce_min_sync(0xffffffffu, mk[q]);
      const int cm = __reduce_add_sync(0xffffffffu, (mk[q] == m) ? mc[q] : 0);
      if (lane == 0) {
        X.sh->ri[par][q][warp] = c;
        X.sh->ru[par][q][warp] = m;
        X.sh->bi[8 + q + 3 * par][warp] = cm;
      }
    }
    __syncthreads();
    bool done = false;
    uint32_t nlo = lo, nhi = hi, found = 0u;
    int found_gt = 0;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      int N = above;
      uint32_t m = 0xffffffffu;
      for (int w = 0; w < NWARP; ++w) {
        N += X.sh->ri[par][q][w];
        m = min(m, X.sh->ru[par][q][w]);
      }
      int c = 0;
      for (int w = 0; w < NWARP; ++w)
        if (X.sh->ru[par][q][w] == m) c += X.sh->bi[8 + q + 3 * par][w];
      if (!done && N >= K && N - c < K) {
        done = true;
        found = m;
        found_gt = N - c;
      }
      if (N >= K) nlo = max(nlo, (N - c >= K) ? m + 1u : tau[q] + 1u);
      else nhi = min(nhi, tau[q]);
    }
    par ^= 1;
    if (done) {
      ngt = found_gt;
      return found;
    }
    lo = nlo;
    hi = nhi;
  }
  int c = 0;
  for (int j = threadIdx.x; j < n; j += NT)
    if (!(X.ci[j] & NOT_MEMBER) && X.ck[j] > lo) ++c;
  ngt = above + bsum_i(X, c, 2);
  return lo;
}

// Top-p boundary among members by mass: the key v with
// above + mass{key > v} < target <= above + mass{key >= v}; bw holds weights.
template <int DT>
__device__ __forceinline__ uint32_t pivot_mass(const Ctx<DT>& X, const float* bw, int n, double target,
                               double above, double& a_gt, int& copies, int& rounds) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int j = threadIdx.x; j < n; j += NT) {
    if (X.ci[j] & NOT_MEMBER) continue;
    mn = min(mn, X.ck[j]);
    mx = max(mx, X.ck[j]);
  }
  uint32_t lo = bmin_u(X, mn, 3), hi = bmax_u(X, mx, 4);
  rounds = 0;
  int par = 0;
  for (int guard = 0; guard < 64 && lo < hi; ++guard) {
    ++rounds;
    uint32_t tau[3];
    const unsigned long long span = (unsigned long long)(hi - lo);
#pragma unroll
    for (int q = 0; q < 3; ++q) tau[q] = lo + (uint32_t)((span * (q + 1)) / 4);
    float ms[3] = {0.f, 0.f, 0.f};
    int mc[3] = {0, 0, 0};
    uint32_t mk[3] = {0xffffffffu, 0xffffffffu, 0xffffffffu};
    for (int j = threadIdx.x; j < n; j += NT) {
      if (X.ci[j] & NOT_MEMBER) continue;
      const uint32_t k = X.ck[j];
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
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const double s = warp_sum((double)ms[q]);
      const uint32_t m = __reduce_min_sync(0xffffffffu, mk[q]);
      const int cm = __reduce_add_sync(0xffffffffu, (mk[q] == m) ? mc[q] : 0);
      if (lane == 0) {
        X.sh->rd[par][q][warp] = s;
        X.sh->ru[par][q][warp] = m;
        X.sh->ri[par][q][warp] = cm;
      }
    }
    __syncthreads();
    bool done = false;
    uint32_t nlo = lo, nhi = hi, found = 0u;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      double A = above;
      uint32_t m = 0xffffffffu;
      for (int w = 0; w < NWARP; ++w) {
        A += X.sh->rd[par][q][w];
        m = min(m, X.sh->ru[par][q][w]);
      }
      int c = 0;
      for (int w = 0; w < NWARP; ++w)
        if (X.sh->ru[par][q][w] == m) c += X.sh->ri[par][q][w];
      const double wm = (c > 0) ? (double)c * (double)weight(X, key_to_float(m)) : 0.0;
      if (!done && c > 0 && A >= target && A - wm < target) {
        done = true;
        found = m;
      }
      if (A >= target && c > 0) nlo = max(nlo, (A - wm >= target) ? m + 1u : tau[q] + 1u);
      else nhi = min(nhi, tau[q]);
    }
    par ^= 1;
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
  for (int j = threadIdx.x; j < n; j += NT)
    if (!(X.ci[j] & NOT_MEMBER) && X.ck[j] >= lo) nxt = min(nxt, X.ck[j]);
  nxt = bmin_u(X, nxt, 5);
  const uint32_t v = (nxt != 0xffffffffu) ? nxt : hi;
  float s = 0.f;
  int c = 0;
  for (int j = threadIdx.x; j < n; j += NT) {
    if (X.ci[j] & NOT_MEMBER) continue;
    if (X.ck[j] > v) s += bw[j];
    if (X.ck[j] == v) ++c;
  }
  a_gt = above + bsum_d(X, (double)s, 6);
  copies = bsum_i(X, c, 7);
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
// the rest NOT_MEMBER.  Contiguous chunks per thread keep id order.
template <int DT>
__device__ __forceinline__ void restrict_members(const Ctx<DT>& X, int n, uint32_t kB, int nB) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ch = (n + NT - 1) / NT;
  const int j0 = threadIdx.x * ch, j1 = min(n, j0 + ch);
  int t = 0;
  for (int j = j0; j < j1; ++j)
    if (!(X.ci[j] & NOT_MEMBER) && X.ck[j] == kB) ++t;
  const int incl = warp_incl_scan(t);
  if (lane == 31) X.sh->bi[9][warp] = incl;
  __syncthreads();
  int rank = incl - t;
  for (int w = 0; w < warp; ++w) rank += X.sh->bi[9][w];
  for (int j = j0; j < j1; ++j) {
    if (X.ci[j] & NOT_MEMBER) continue;
    const uint32_t k = X.ck[j];
    bool mem = k > kB;
    if (k == kB) {
      mem = rank < nB;
      ++rank;
    }
    if (!mem) X.ci[j] |= NOT_MEMBER;
  }
  __syncthreads();
}

// Draw among members in id order: the first member whose cumulative weight
// exceeds T (the last member if rounding leaves none).  Returns the id.
template <int DT>
__device__ __forceinline__ int sample_members(const Ctx<DT>& X, const float* bw, int n, double T) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ch = (n + NT - 1) / NT;
  const int j0 = threadIdx.x * ch, j1 = min(n, j0 + ch);
  double ls = 0.0;
  int lc = 0;
  for (int j = j0; j < j1; ++j)
    if (!(X.ci[j] & NOT_MEMBER)) {
      ls += (double)bw[j];
      ++lc;
    }
  // block exclusive scan of ls (thread order = id order)
  double incl = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) X.sh->bd[10][warp] = incl;
  const int anyc = __reduce_add_sync(0xffffffffu, lc);
  if (lane == 0) X.sh->bi[10][warp] = anyc;
  if (threadIdx.x == 0) {
    X.sh->sel_thread = -1;
    X.sh->flag[5] = -1;
  }
  __syncthreads();
  double pre = 0.0;
  for (int w = 0; w < warp; ++w) pre += X.sh->bd[10][w];
  const double ex = pre + incl - ls;
  const bool cross = lc > 0 && ex + ls > T;
  if (cross) atomicMin(reinterpret_cast<unsigned*>(&X.sh->sel_thread), (unsigned)threadIdx.x);
  if (lc > 0) atomicMax(&X.sh->flag[5], (int)threadIdx.x);
  __syncthreads();
  int sel = X.sh->sel_thread;
  if (sel < 0 || sel >= NT) sel = X.sh->flag[5];  // rounding: the last member
  int tok = -1;
  if ((int)threadIdx.x == sel) {
    double c = ex;
    int last = -1;
    for (int j = j0; j < j1; ++j)
      if (!(X.ci[j] & NOT_MEMBER)) {
        c += (double)bw[j];
        last = X.ci[j];
        if (tok < 0 && c > T) tok = X.ci[j];
      }
    if (tok < 0) tok = last;
    X.sh->flag[6] = tok;
  }
  __syncthreads();
  return X.sh->flag[6];
}

}  // namespace smp

#include "smp_stream_main.cuh"
