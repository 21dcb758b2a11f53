// smp_list.cuh -- the candidate list: warp-aggregated appends during a pass,
// radix selection on it (k-th value, tie quota by id, top-p boundary by mass)
// and the id-order inverse-CDF draw over the kept entries.
//
// The list holds, in no particular order, every legal element whose key lies
// in a band of the rank order.  Order-dependent rules -- earliest ids win
// ties, the draw scans ids upward -- are evaluated on ids, never on list
// positions, and every mass is a fixed-point integer, so results do not depend
// on the append order.
//
// The selection runs on a thread group of G threads: one warp (G = 32,
// warp-synchronous, no block barrier) for lists of up to GSMALL entries, the
// whole CTA (G = NT) beyond that.
#pragma once

#include "smp_core.cuh"

namespace smp {

constexpr int GSMALL = 0;  // lists up to this size are resolved by one warp

// After a pass the ring is idle; its bytes hold the list weights and the
// selection scratch (histogram bins, id-segment masses, the gathered segment
// of the draw).
template <int DT>
__device__ __forceinline__ float* list_w(const Ctx<DT>& X) {
  return reinterpret_cast<float*>(X.ring);
}
template <int DT>
__device__ __forceinline__ uint64_t* list_scratch(const Ctx<DT>& X) {
  return reinterpret_cast<uint64_t*>(X.ring + CAP * 4);
}

__device__ __forceinline__ bool in_set(uint32_t k, int id, uint32_t v, int idv) {
  return k > v || (k == v && id <= idv);
}

// Raw bits of element j (0 <= j < EPV, any j) of a vector, without indexing
// a local array.
template <int DT>
__device__ __forceinline__ uint32_t elem_bits_dyn(const uint4 r, int j) {
  if constexpr (DT == DT_F32) {
    const uint32_t lo = (j & 1) ? r.y : r.x, hi = (j & 1) ? r.w : r.z;
    return (j & 2) ? hi : lo;
  } else {
    const int q = j >> 1;
    const uint32_t lo = (q & 1) ? r.y : r.x, hi = (q & 1) ? r.w : r.z;
    const uint32_t w = (q & 2) ? hi : lo;
    return (j & 1) ? (w >> 16) : (w & 0xffffu);
  }
}

// Appends the elements flagged in cm (bit j = element j of this lane's
// vector, ids id0 + j).  Called by all lanes of a warp.  Entries past CAP are
// dropped; sh->n keeps counting, so n > CAP flags the overflow.  Returns the
// largest key appended by this lane (0 if none).
template <int DT>
__device__ __forceinline__ uint32_t list_append(Ctx<DT>& X, const uint4 r, int id0, uint32_t cm) {
  const int lane = threadIdx.x & 31;
  const int cnt = __popc(cm);
  const int inc = warp_incl_scan(cnt);
  const int tot = __shfl_sync(0xffffffffu, inc, 31);
  uint32_t kmax = 0u;
  if (tot == 0) return kmax;
  int base = 0;
  if (lane == 31) base = atomicAdd(&X.sh->n, tot);
  base = __shfl_sync(0xffffffffu, base, 31);
  int pos = base + inc - cnt;
  while (cm) {
    const int j = __ffs(cm) - 1;
    cm &= cm - 1u;
    const uint32_t k = bits_key<DT>(elem_bits_dyn<DT>(r, j));
    kmax = max(kmax, k);
    if (pos < CAP) {
      X.lk[pos] = k;
      X.li[pos] = id0 + j;
    }
    ++pos;
  }
  return kmax;
}


// Bits of the elements >= t (packed compares; NaN compares false); a NaN in
// the vector raises nf (+inf is kept and caught by the list's largest key).
template <int DT>
__device__ __forceinline__ uint32_t ge_mask(const uint4 r, uint32_t t2, float tf, int& nf) {
  if constexpr (DT == DT_F32) {
    const float a = __uint_as_float(r.x), b = __uint_as_float(r.y), c = __uint_as_float(r.z),
                d = __uint_as_float(r.w);
    if (a != a || b != b || c != c || d != d) nf = 1;
    return (a >= tf ? 1u : 0u) | (b >= tf ? 2u : 0u) | (c >= tf ? 4u : 0u) | (d >= tf ? 8u : 0u);
  } else {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint32_t cm = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t m;
      if constexpr (DT == DT_BF16)
        m = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[q]),
                        *reinterpret_cast<const __nv_bfloat162*>(&t2));
      else
        m = __hge2_mask(*reinterpret_cast<const __half2*>(&w[q]),
                        *reinterpret_cast<const __half2*>(&t2));
      cm |= ((m & 1u) | ((m >> 15) & 2u)) << (2 * q);
    }
    const float mx = p2f_max<DT>(vmax2<DT>(r));
    if (mx != mx) nf = 1;
    return cm;
  }
}

// Warp-cooperative append of the elements >= t of a staged chunk's hit
// vectors.  hits (per lane): bit it marks vector (warp base + 32 it + lane)
// as holding an element >= t or a NaN.  The warp's hit vectors are dealt out
// one per lane, so the element tests and list writes run on all lanes at once
// rather than on the few lanes that hold a hit, with one list reservation per
// 32 hit vectors.  MASS: lm adds the appended elements' weights 2^(x c2 +
// nref).  Called by all lanes; returns the largest key this lane appended.
template <int DT, bool MASS>
__device__ __forceinline__ uint32_t warp_append_hits(Ctx<DT>& X, const char* stage, int c,
                                                     uint32_t hits, uint32_t t2, float tf,
                                                     int& nf, float c2, float nref, float& lm) {
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE, VW = ElemT<DT>::VW;
  const int lane = threadIdx.x & 31;
  const int vbase = (threadIdx.x >> 5) * VW;
  uint32_t bal[ITW];
  int H = 0;
#pragma unroll
  for (int it = 0; it < ITW; ++it) {
    bal[it] = __ballot_sync(0xffffffffu, (hits >> it) & 1u);
    H += __popc(bal[it]);
  }
  uint32_t kmax = 0u;
#pragma unroll 1
  for (int k0 = 0; k0 < H; k0 += 32) {
    // this lane's hit vector: the (k0 + lane)-th in (it, lane) order
    int rem = k0 + lane, vi = -1;
#pragma unroll
    for (int it = 0; it < ITW; ++it) {
      const int pc = __popc(bal[it]);
      if (rem >= 0 && rem < pc) vi = vbase + 32 * it + (int)__fns(bal[it], 0u, rem + 1);
      rem -= pc;
    }
    uint32_t cm = 0u;
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
    if (vi >= 0) {
      r = load_vec(X, stage, c, vi);
      cm = ge_mask<DT>(r, t2, tf, nf);
    }
    const int cnt = __popc(cm);
    const int inc = warp_incl_scan(cnt);
    const int tot = __shfl_sync(0xffffffffu, inc, 31);
    int base = 0;
    if (lane == 31 && tot) base = atomicAdd(&X.sh->n, tot);
    base = __shfl_sync(0xffffffffu, base, 31);
    int pos = base + inc - cnt;
    const int id0 = c * CE + vi * EPV;
    while (cm) {
      const int j = __ffs(cm) - 1;
      cm &= cm - 1u;
      const uint32_t b = elem_bits_dyn<DT>(r, j);
      const uint32_t k = bits_key<DT>(b);
      kmax = max(kmax, k);
      if (MASS) lm += fast_exp2(fmaf(bits_value<DT>(b), c2, nref));
      if (pos < CAP) {
        X.lk[pos] = k;
        X.li[pos] = id0 + j;
      }
      ++pos;
    }
  }
  return kmax;
}


// ---------------------------------------------------------------------------
// Thread groups
// ---------------------------------------------------------------------------
template <int G>
__device__ __forceinline__ int gtid() {
  return G == 32 ? (int)(threadIdx.x & 31) : (int)threadIdx.x;
}
template <int G>
__device__ __forceinline__ void gsync() {
  if (G == 32) __syncwarp();
  else __syncthreads();
}
template <int G>
__device__ __forceinline__ uint64_t gsum_q(uint64_t v, uint64_t* s) {
  if (G == 32) return warp_sum(v);
  return bsum_q(v, s);
}
template <int G>
__device__ __forceinline__ uint32_t gmax_u(uint32_t v, uint32_t* s) {
  if (G == 32) return __reduce_max_sync(0xffffffffu, v);
  return bmax_u(v, s);
}
template <int G, class T>
__device__ __forceinline__ T gscan_excl(T v, T* s, T& total) {
  if (G == 32) {
    const T inc = warp_incl_scan(v);
    total = __shfl_sync(0xffffffffu, inc, 31);
    return inc - v;
  }
  return bscan_excl<T>(v, s, total);
}

// ---------------------------------------------------------------------------
// Radix selection over list entries, 8-bit digits from the top.
//   SEL_COUNT : key = entry key, every entry, weight 1
//   SEL_MASS  : key = entry key, members of S_k, weight = fixed-point mass
//   SEL_TIEID : key = 2^24 - 1 - id, members of S_k whose key is `at`, weight 1
// Finds the largest key value v whose weight at-or-above reaches target;
// above = weight strictly above v, at_w / at_n = weight / count at v.  With
// p_rel > 0 the target is ceil(p_rel * total weight) (the first round's sum).
// ---------------------------------------------------------------------------
enum { SEL_COUNT = 0, SEL_MASS = 1, SEL_TIEID = 2 };

struct SelOut {
  uint32_t v;
  uint64_t above, at_w, total, target;
  int above_n;  // entries strictly above v
  int at_n;
  int ok;
};

template <int G, int DT, int KIND>
__device__ __noinline__ SelOut list_select(Ctx<DT>& Xr, int n, uint64_t target, float p_rel,
                                           uint32_t vK, int idK, uint32_t at) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  // Digits are taken over the list's own key range [kbase, kbase + 2^SIGB):
  // the keys of a candidate list cluster, and digits of the full key width
  // would pile them onto a few bins (serialised shared atomics).
  const uint32_t kbase = (KIND == SEL_TIEID) ? 0u : X.sh->bu[4];
  const int SIGB = (KIND == SEL_TIEID) ? 24 : max(8, 32 - __clz((int)(X.sh->bu[5] - kbase)));
  const int ROUNDS = (SIGB + 7) / 8;
  uint64_t* bw = list_scratch(X);                                // [2][256] weights
  uint32_t* bc = reinterpret_cast<uint32_t*>(bw + 512);          // [2][256] counts
  const float* wq = list_w(X);
  const int t = gtid<G>();
  const int lane = threadIdx.x & 31;
  const bool scanner = (G == 32) || (threadIdx.x < 32);
  uint32_t prefix = 0u;
  uint64_t above = 0;
  int above_n = 0;
  SelOut o;
  o.ok = 1;
  o.at_w = 0;
  o.at_n = 0;
  o.total = 0;
  gsync<G>();
  for (int b = t; b < 256; b += G) {
    bw[b] = 0;
    bc[b] = 0u;
  }
  gsync<G>();
#pragma unroll 1
  for (int rd = 0; rd < ROUNDS; ++rd) {
    const int shift = max(SIGB - 8 * (rd + 1), 0);  // = SIGB - 8 rd - wr
    // round rd takes the next wr bits below the prefix (the last round the
    // remaining low bits)
    const int wr = min(8, SIGB - 8 * rd);
    const uint32_t dmask = (1u << wr) - 1u;
    uint64_t* w = bw + (rd & 1) * 256;
    uint32_t* c = bc + (rd & 1) * 256;
    uint64_t* w2 = bw + ((rd + 1) & 1) * 256;
    uint32_t* c2 = bc + ((rd + 1) & 1) * 256;
    for (int b = t; b < 256; b += G) {  // the other buffer, for the next round
      w2[b] = 0;
      c2[b] = 0u;
    }
#pragma unroll 1
    for (int i = t; i < n; i += G) {
      const uint32_t k0 = X.lk[i];
      const int id = X.li[i];
      bool f = true;
      uint32_t key = k0 - kbase;
      if constexpr (KIND == SEL_MASS) f = in_set(k0, id, vK, idK);
      if constexpr (KIND == SEL_TIEID) {
        f = (k0 == at) && in_set(k0, id, vK, idK);
        key = 0xffffffu - (uint32_t)id;
      }
      if (!f) continue;
      if (rd > 0 && (key >> (shift + wr)) != prefix) continue;
      const int d = (key >> shift) & dmask;
      // counts and (SEL_MASS) fixed-point masses; the other kinds weigh by count
      if constexpr (KIND == SEL_MASS) smem_add_u64(&w[d], to_fx(wq[i]));
      atomicAdd(&c[d], 1u);
    }
    gsync<G>();
    if (scanner) {
      // lane l reads digits 255 - 8l ... 248 - 8l (descending)
      uint64_t v[8];
      uint32_t cv[8];
      uint64_t loc = 0;
      uint32_t locc = 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        cv[q] = c[255 - 8 * lane - q];
        v[q] = (KIND == SEL_MASS) ? w[255 - 8 * lane - q] : (uint64_t)cv[q];
        loc += v[q];
        locc += cv[q];
      }
      const uint64_t inc = warp_incl_scan(loc);
      uint32_t cumc = (uint32_t)above_n + warp_incl_scan(locc) - locc;
      const uint64_t tot = __shfl_sync(0xffffffffu, inc, 31);
      if (rd == 0) {
        o.total = tot;
        if (p_rel > 0.f) {
          target = (uint64_t)ceil((double)p_rel * (double)tot);
          if (target == 0) target = 1;
        }
      }
      uint64_t cum = above + inc - loc;
      int hit = -1;
      uint64_t hb = 0, hv = 0;
      uint32_t hc = 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (hit < 0 && v[q] > 0 && cum < target && cum + v[q] >= target) {
          hit = 255 - 8 * lane - q;
          hb = cum;
          hv = v[q];
          hc = cumc;
        }
        cum += v[q];
        cumc += cv[q];
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, hit >= 0);
      const int src = bal ? (__ffs(bal) - 1) : 0;
      const int d = __shfl_sync(0xffffffffu, hit, src);
      const uint64_t hb2 = __shfl_sync(0xffffffffu, hb, src);
      const uint64_t hv2 = __shfl_sync(0xffffffffu, hv, src);
      const uint32_t hc2 = __shfl_sync(0xffffffffu, hc, src);
      if (G == 32) {
        if (bal == 0u) {
          o.ok = 0;
        } else {
          prefix = (prefix << wr) | (uint32_t)d;
          above = hb2;
          above_n = (int)hc2;
          o.at_w = hv2;
          o.at_n = (int)c[d];
        }
      } else if (lane == 0) {
        X.sh->bi[0] = bal ? d : -1;
        X.sh->bq[0] = hb2;
        X.sh->bq[1] = hv2;
        X.sh->bq[2] = tot;
        X.sh->bq[3] = target;
        X.sh->bi[1] = bal ? (int)c[d] : 0;
        X.sh->bi[3] = (int)hc2;
      }
    }
    if (G != 32) {
      __syncthreads();
      const int d = X.sh->bi[0];
      if (d < 0) {
        o.ok = 0;
      } else {
        prefix = (prefix << wr) | (uint32_t)d;
        above = X.sh->bq[0];
        above_n = X.sh->bi[3];
        o.at_w = X.sh->bq[1];
        o.at_n = X.sh->bi[1];
        if (rd == 0) {
          o.total = X.sh->bq[2];
          target = X.sh->bq[3];
        }
      }
    }
    if (!o.ok) break;
  }
  o.v = (KIND == SEL_TIEID) ? prefix : prefix + kbase;
  o.above = above;
  o.above_n = above_n;
  o.target = target;
  return o;
}

// Key range of the list entries (sh->bu[4], sh->bu[5]): the radix digits of
// list_select are taken inside it.  All threads of the CTA call it.
template <int DT>
__device__ __noinline__ void list_range(Ctx<DT>& Xr, int n) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint32_t k = X.lk[i];
    lo = min(lo, k);
    hi = max(hi, k);
  }
  lo = bmin_u(lo, X.sh->ru[0]);
  hi = bmax_u(hi, X.sh->ru[1]);
  if (threadIdx.x == 0) {
    X.sh->bu[4] = (n > 0) ? lo : 0u;
    X.sh->bu[5] = (n > 0) ? hi : 0u;
  }
  __syncthreads();
}

// Weight of a value relative to the row maximum.  Precise: the contract's
// expf(fl32(x / T) - fl32(max / T)) (m_z = fl32(max / T)).  FAST: the base-2
// hardware exponential of the row passes (nm = -max * log2(e) / T), so a band
// list weighs its elements exactly as the pass that chose it.
template <int DT, bool FAST>
__device__ __forceinline__ float rel_weight(const Ctx<DT>& X, float x, float m_z, float nm) {
  if (FAST) return fast_exp2(fmaf(x, X.c2, nm));
  return expf(__fdiv_rn(x, X.temp) - m_z);
}

// Resolution of a kept set inside a list (targets already net of the part
// of the row above the list).
struct Res {
  uint32_t vK;
  int idK;  // S_k = {key > vK} + {key == vK, id <= idK}
  uint32_t vP;
  int idP;  // S_p = S_k restricted to {key > vP} + {key == vP, id <= idP}
};

// ---------------------------------------------------------------------------
// Selection on 16-bit keys by one count histogram.  A bf16 / fp16 value is
// one of 2^16 keys, so when the
// list's keys span fewer than NB16 values a histogram with one bin per key
// gives the k-th key by suffix counts in one round, instead of radix rounds.
// The tie quota by id comes from a gather of the boundary key's copies,
// ranked by id when there are at most NT of them.
// ---------------------------------------------------------------------------
constexpr int NB16 = 4096;        // key bins
constexpr int TG16 = 2048;        // ids gathered for a tie quota
static_assert(CAP * 4 + NB16 * 4 + TG16 * 4 <= SMEM_RING, "16-bit selection scratch lives in the ring");

template <int DT>
__device__ __forceinline__ uint32_t* hist16(const Ctx<DT>& X) {
  return reinterpret_cast<uint32_t*>(X.ring + CAP * 4);
}
template <int DT>
__device__ __forceinline__ int* tie16(const Ctx<DT>& X) {
  return reinterpret_cast<int*>(X.ring + CAP * 4 + NB16 * 4);
}

// Counts per key (bin key - kbase) of the list entries, of S_k members only
// when sk is set.
template <int DT>
__device__ void hist16_build(Ctx<DT>& X, int n, uint32_t kbase, bool sk, uint32_t vK, int idK) {
  uint32_t* hc = hist16(X);
  __syncthreads();
  for (int b = threadIdx.x; b < NB16; b += NT) hc[b] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint32_t k = X.lk[i];
    if (sk && !in_set(k, X.li[i], vK, idK)) continue;
    atomicAdd(&hc[k - kbase], 1u);
  }
  __syncthreads();
}

// j-th smallest (1-based) of the m distinct ids g[0..m), NT < m <= TG16: a
// count of the ids in NT bins of consecutive ids (one bin per thread), a block
// scan to the bin that holds the j-th, then ranks among that bin's ids.  -2
// when that bin holds more than NT ids.  Scratch: the 16-bit key histogram's
// area (its counts are no longer needed when a tie quota is taken).
template <int DT>
__device__ int nth_id_bins(Ctx<DT>& X, const int* g, int m, int j) {
  uint32_t* bc = hist16(X);             // NT bin counts
  int* gb = reinterpret_cast<int*>(bc + NT);  // the chosen bin's ids
  uint32_t* bs = bc + 2 * NT;           // chosen bin, rank in it, gathered, result
  const int t = threadIdx.x;
  int sh = 0;
  while (((X.V - 1) >> sh) >= NT) ++sh;  // bin of id: id >> sh, below NT
  bc[t] = 0u;
  if (t == 0) {
    bs[0] = (uint32_t)NT;  // no bin yet
    bs[2] = 0u;
    bs[3] = 0xffffffffu;
  }
  __syncthreads();
  for (int i = t; i < m; i += NT) atomicAdd(&bc[min(g[i] >> sh, NT - 1)], 1u);
  __syncthreads();
  const uint32_t c = bc[t];
  uint32_t tot;
  const uint32_t cum = bscan_excl<uint32_t>(c, X.sh->ru[0], tot);
  if (cum < (uint32_t)j && cum + c >= (uint32_t)j) {
    bs[0] = (uint32_t)t;
    bs[1] = (uint32_t)j - cum;
  }
  __syncthreads();
  const int b = (int)bs[0];
  if (b >= NT) return -1;  // j beyond the ids (every thread: the same answer)
  const int jb = (int)bs[1];
  const int cb = (int)bc[b];
  if (cb > NT) return -2;
  for (int i = t; i < m; i += NT) {
    const int id = g[i];
    if (min(id >> sh, NT - 1) == b) gb[atomicAdd(&bs[2], 1u)] = id;
  }
  __syncthreads();
  if (t < cb) {
    const int ida = gb[t];
    int r = 0;
#pragma unroll 4
    for (int q = 0; q < cb; ++q) r += (gb[q] < ida) ? 1 : 0;
    if (r == jb - 1) bs[3] = (uint32_t)ida;
  }
  __syncthreads();
  const int id = (int)bs[3];
  __syncthreads();  // the scratch may be reused once every thread has read it
  return id;
}

// The j-th smallest id (j >= 1) among the entries with key v that are S_k
// members: up to NT entries ranked directly, up to TG16 through nth_id_bins;
// -2 beyond that, or when one bin of ids holds more than NT of them (the
// caller then ranks them by radix selection on ids).
template <int DT>
__device__ int nth_id16(Ctx<DT>& X, int n, uint32_t v, int j, uint32_t vK, int idK) {
  int* g = tie16(X);
  __syncthreads();
  if (threadIdx.x == 0) {
    X.sh->gn = 0;
    X.sh->bi[3] = -1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += NT) {
    if (X.lk[i] != v) continue;
    const int id = X.li[i];
    if (!in_set(v, id, vK, idK)) continue;
    const int slot = atomicAdd(&X.sh->gn, 1);
    if (slot < TG16) g[slot] = id;
  }
  __syncthreads();
  const int m = X.sh->gn;
  if (m > TG16) return -2;
  if (m > NT) return nth_id_bins(X, g, m, j);
  if ((int)threadIdx.x < m) {
    const int ida = g[threadIdx.x];
    int r0 = 0, r1 = 0, r2 = 0, r3 = 0;  // ids are distinct
    int b = 0;
#pragma unroll 2
    for (; b + 4 <= m; b += 4) {
      r0 += (g[b] < ida) ? 1 : 0;
      r1 += (g[b + 1] < ida) ? 1 : 0;
      r2 += (g[b + 2] < ida) ? 1 : 0;
      r3 += (g[b + 3] < ida) ? 1 : 0;
    }
    for (; b < m; ++b) r0 += (g[b] < ida) ? 1 : 0;
    if (r0 + r1 + r2 + r3 == j - 1) X.sh->bi[3] = ida;
  }
  __syncthreads();
  return X.sh->bi[3];
}

// k-th largest key: 1 = found (vK, idK), 0 = not found, -1 = the key range
// does not fit the bins.
template <int DT>
__device__ __noinline__ int hsel_k16(Ctx<DT>& Xr, int n, int K, uint32_t& vK, int& idK) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  const uint32_t kbase = X.sh->bu[4];
  const uint32_t top = X.sh->bu[5] - kbase;
  if (X.sh->bu[5] < kbase || top >= (uint32_t)NB16) return -1;
  hist16_build(X, n, kbase, false, 0u, -1);
  const uint32_t* hc = hist16(X);
  const int t = threadIdx.x;
  // this thread's bins b0, b0 - 1, ..., b0 - bpt + 1 (as few per thread as
  // the key range allows, so a narrow range spreads over many threads)
  const int bpt = ((int)top + NT) / NT;
  const int b0 = (int)top - t * bpt;
  uint32_t s = 0u;
#pragma unroll 1
  for (int e = 0; e < bpt; ++e) s += (b0 - e >= 0) ? hc[b0 - e] : 0u;
  uint32_t tot;
  uint32_t cum = bscan_excl<uint32_t>(s, X.sh->ru[0], tot);
  if (t == 0) X.sh->bi[0] = -1;
  __syncthreads();
  if (cum < (uint32_t)K && cum + s >= (uint32_t)K) {
#pragma unroll 1
    for (int e = 0; e < bpt; ++e) {
      const uint32_t c = (b0 - e >= 0) ? hc[b0 - e] : 0u;
      if (c > 0u && cum + c >= (uint32_t)K) {
        X.sh->bi[0] = b0 - e;
        X.sh->bi[1] = (int)cum;
        X.sh->bi[2] = (int)c;
        break;
      }
      cum += c;
    }
  }
  __syncthreads();
  const int bK = X.sh->bi[0];
  if (bK < 0) return 0;
  const int above = X.sh->bi[1], atn = X.sh->bi[2];
  vK = kbase + (uint32_t)bK;
  idK = NOID;
  const int keep = K - above;  // ties at vK kept, earliest ids first
  if (keep < atn) {
    idK = nth_id16(X, n, vK, keep, 0u, -1);
    if (idK == -2) {
      const SelOut ti = list_select<NT, DT, SEL_TIEID>(X, n, (uint64_t)keep, 0.f, 0u, NOID, vK);
      if (!ti.ok) return 0;
      idK = (int)(0xffffffu - ti.v);
    }
    if (idK < 0) return 0;
  }
  return 1;
}

// Top-p boundary among the S_k members of a list (as list_resolve_p): every
// copy of a key has the same weight, so each bin's fixed-point mass is count *
// the key's weight (the same integer as summing the copies).  1 = found, 0 =
// not found, -1 = the key range does not fit the bins.
template <int DT, bool FAST>
__device__ __noinline__ int hsel_p16(Ctx<DT>& Xr, int n, uint64_t target, float p, float m_z,
                                     float nm, Res& R, uint64_t& kept_mass, int* kept_n) {
  LocalCtx<DT> lc_(Xr);
  Ctx<DT>& X = lc_.v;
  const uint32_t kbase = X.sh->bu[4];
  const uint32_t top = X.sh->bu[5] - kbase;
  if (X.sh->bu[5] < kbase || top >= (uint32_t)NB16) return -1;
  hist16_build(X, n, kbase, true, R.vK, R.idK);
  const uint32_t* hc = hist16(X);
  const int t = threadIdx.x;
  // this thread's bins b0, b0 - 1, ..., b0 - bpt + 1 (as few per thread as
  // the key range allows, so a narrow range spreads over many threads)
  const int bpt = ((int)top + NT) / NT;
  const int b0 = (int)top - t * bpt;
  uint64_t s = 0;
#pragma unroll 1
  for (int e = 0; e < bpt; ++e) {
    const int b = b0 - e;
    const uint32_t c = (b >= 0) ? hc[b] : 0u;
    if (c) s += (uint64_t)c * to_fx(rel_weight<DT, FAST>(X, key_value<DT>(kbase + (uint32_t)b), m_z, nm));
  }
  uint64_t tot;
  uint64_t cum = bscan_excl<uint64_t>(s, X.sh->rq[0], tot);
  if (!target) {
    target = (uint64_t)ceil((double)p * (double)tot);
    if (target == 0) target = 1;
  }
  if (t == 0) X.sh->bi[0] = -1;
  __syncthreads();
  if (cum < target && cum + s >= target) {
#pragma unroll 1
    for (int e = 0; e < bpt; ++e) {
      const int b = b0 - e;
      const uint32_t c = (b >= 0) ? hc[b] : 0u;
      if (!c) continue;
      const uint64_t mb =
          (uint64_t)c * to_fx(rel_weight<DT, FAST>(X, key_value<DT>(kbase + (uint32_t)b), m_z, nm));
      if (mb > 0 && cum + mb >= target) {
        X.sh->bi[0] = b;
        X.sh->bq[0] = cum;
        break;
      }
      cum += mb;
    }
  }
  __syncthreads();
  const int bP = X.sh->bi[0];
  if (bP < 0) return 0;
  const uint64_t above = X.sh->bq[0];
  // S_k members strictly above the boundary key, and its copies
  int an = 0;
#pragma unroll 1
  for (int e = 0; e < bpt; ++e) {
    const int b = b0 - e;
    if (b > bP) an += (int)hc[b];
  }
  an = bsum_i(an, X.sh->ri[0]);
  const int at_n = (int)hc[bP];
  R.vP = kbase + (uint32_t)bP;
  const uint64_t qv = to_fx(rel_weight<DT, FAST>(X, key_value<DT>(R.vP), m_z, nm));
  if (qv == 0) return 0;
  const uint64_t need = target - above;  // > 0 by the selection
  int j = (int)((need + qv - 1) / qv);
  if (j > at_n) j = at_n;
  R.idP = (R.vP == R.vK) ? R.idK : NOID;
  if (j < at_n) {
    int id = nth_id16(X, n, R.vP, j, R.vK, R.idK);
    if (id == -2) {
      const SelOut ti = list_select<NT, DT, SEL_TIEID>(X, n, (uint64_t)j, 0.f, R.vK, R.idK, R.vP);
      if (!ti.ok) return 0;
      id = (int)(0xffffffu - ti.v);
    }
    if (id < 0) return 0;
    R.idP = id;
  }
  kept_mass = above + (uint64_t)j * qv;
  if (kept_n) *kept_n = an + j;
  return 1;
}

// k-th largest key inside the list (K counted from the top of the list).
template <int G, int DT>
__device__ bool list_resolve_k(Ctx<DT>& X, int n, int K, uint32_t& vK, int& idK) {
  if constexpr (DT != DT_F32 && G == NT) {
    const int r = hsel_k16(X, n, K, vK, idK);
    if (r >= 0) return r == 1;
  }
  const SelOut s = list_select<G, DT, SEL_COUNT>(X, n, (uint64_t)K, 0.f, 0u, NOID, 0u);
  if (!s.ok) return false;
  vK = s.v;
  const int keep = K - (int)s.above;  // ties at vK kept, earliest ids first
  idK = NOID;
  if (keep < s.at_n) {
    const SelOut ti = list_select<G, DT, SEL_TIEID>(X, n, (uint64_t)keep, 0.f, 0u, NOID, vK);
    if (!ti.ok) return false;
    idK = (int)(0xffffffu - ti.v);
  }
  return true;
}

// Weights of the S_k members (others 0) into the list weight array.
template <int G, int DT, bool FAST>
__device__ void list_weights(Ctx<DT>& X, int n, float m_z, float nm, uint32_t vK, int idK) {
  float* wq = list_w(X);
  const uint32_t* lk = X.lk;
  const int* li = X.li;
  const float temp = X.temp, c2 = X.c2;
  for (int i = gtid<G>(); i < n; i += G) {
    const uint32_t k = lk[i];
    float w = 0.f;
    if (in_set(k, li[i], vK, idK)) {
      const float x = key_value<DT>(k);
      w = FAST ? fast_exp2(fmaf(x, c2, nm)) : expf(__fdiv_rn(x, temp) - m_z);
    }
    wq[i] = w;
  }
  gsync<G>();
}

// Top-p boundary inside the list: the shortest prefix (value descending, id
// ascending) of S_k members whose mass reaches the target.  target > 0: that
// fixed-point mass (net of the mass above the list); otherwise p times the
// list's S_k mass.  kept_mass receives the mass of S_p inside the list.
template <int G, int DT, bool FAST>
__device__ bool list_resolve_p(Ctx<DT>& X, int n, uint64_t target, float p, float m_z, float nm,
                               Res& R, uint64_t& kept_mass, int* kept_n = nullptr) {
  // bf16 / fp16 lists: one count histogram
  if constexpr (DT != DT_F32 && G == NT) {
    const int r = hsel_p16<DT, FAST>(X, n, target, p, m_z, nm, R, kept_mass, kept_n);
    if (r >= 0) return r == 1;
  }
  const SelOut s = list_select<G, DT, SEL_MASS>(X, n, target, target ? 0.f : p, R.vK, R.idK, 0u);
  if (!s.ok) return false;
  R.vP = s.v;
  const uint64_t qv = to_fx(rel_weight<DT, FAST>(X, key_value<DT>(s.v), m_z, nm));
  if (qv == 0) return false;
  const uint64_t need = s.target - s.above;  // > 0 by the selection
  int j = (int)((need + qv - 1) / qv);
  if (j > s.at_n) j = s.at_n;
  R.idP = (s.v == R.vK) ? R.idK : NOID;
  if (j < s.at_n) {
    const SelOut ti = list_select<G, DT, SEL_TIEID>(X, n, (uint64_t)j, 0.f, R.vK, R.idK, s.v);
    if (!ti.ok) return false;
    R.idP = (int)(0xffffffu - ti.v);
  }
  kept_mass = s.above + (uint64_t)j * qv;
  if (kept_n) *kept_n = s.above_n + j;
  return true;
}

// ---------------------------------------------------------------------------
// Id-order draw over the kept entries {key > vP} + {key == vP, id <= idP}:
// fixed-point masses summed per id segment (2^sshift ids), the segment holding
// u * Mp found by a scan, and that segment's kept entries ranked by id.
// ---------------------------------------------------------------------------
template <int G, int DT>
__device__ int list_draw(Ctx<DT>& X, int n, uint32_t vP, int idP, uint64_t Mp, double u) {
  const float* wq = list_w(X);
  uint64_t* seg = list_scratch(X);
  const uint32_t* lk = X.lk;
  const int* li = X.li;
  Sh* sh = X.sh;
  const int t = gtid<G>();
  int sshift = 8;
  while (((X.V - 1) >> sshift) + 1 > SEG_MAX) ++sshift;
  const int nseg = ((X.V - 1) >> sshift) + 1;
  // T = floor(u * Mp) exactly (u = k * 2^-24): integer compares below
  const uint64_t T = __umul64hi(Mp, ((uint64_t)(u * 16777216.0)) << 40);
  gsync<G>();
  for (int s = t; s < nseg; s += G) seg[s] = 0;
  gsync<G>();
  // contiguous runs of entries per thread (list order follows the row, so a
  // run mostly stays in one segment): a segment's sum is added when the run
  // leaves it, instead of one contended 64-bit add per entry
  int lastk = -1;
  {
    const int per = (n + G - 1) / G;
    const int i0 = t * per, i1 = min(n, i0 + per);
    int sc = -1;
    uint64_t acc = 0;
#pragma unroll 1
    for (int i = i0; i < i1; ++i) {
      const int id = li[i];
      if (!in_set(lk[i], id, vP, idP)) continue;
      const int sg = id >> sshift;
      if (sg != sc) {
        if (sc >= 0) smem_add_u64(&seg[sc], acc);
        sc = sg;
        acc = 0;
      }
      acc += to_fx(wq[i]);
      lastk = max(lastk, id);
    }
    if (sc >= 0) smem_add_u64(&seg[sc], acc);
  }
  const int last = (int)gmax_u<G>((uint32_t)(lastk + 1), sh->ru[0]) - 1;
  gsync<G>();
  const int spt = (nseg + G - 1) / G;
  const int s0 = t * spt, s1 = min(nseg, s0 + spt);
  uint64_t loc = 0;
  for (int s = s0; s < s1; ++s) loc += seg[s];
  uint64_t tot;
  uint64_t cum = gscan_excl<G, uint64_t>(loc, sh->rq[0], tot);
  int hit = -1;
  uint64_t before = 0;
  for (int s = s0; s < s1; ++s) {
    const uint64_t v = seg[s];
    if (hit < 0 && v > 0 && cum <= T && cum + v > T) {
      hit = s;
      before = cum;
    }
    cum += v;
  }
  // the (unique) crossing segment
  int ss;
  uint64_t bf;
  if (G == 32) {
    const uint32_t bal = __ballot_sync(0xffffffffu, hit >= 0);
    const int src = bal ? __ffs(bal) - 1 : 0;
    ss = bal ? __shfl_sync(0xffffffffu, hit, src) : -1;
    bf = __shfl_sync(0xffffffffu, before, src);
  } else {
    if (threadIdx.x == 0) sh->bi[0] = -1;
    __syncthreads();
    if (hit >= 0) {
      sh->bi[0] = hit;
      sh->bq[0] = before;
    }
    __syncthreads();
    ss = sh->bi[0];
    bf = sh->bq[0];
  }
  if (ss < 0) return last;
  // gather the kept entries of segment ss (the segment sums are no longer needed)
  gsync<G>();
  uint64_t* gq = seg;
  int* gid = reinterpret_cast<int*>(seg + GMAX);
  if (t == 0) sh->gn = 0;
  gsync<G>();
#pragma unroll 1
  for (int i = t; i < n; i += G) {
    const int id = li[i];
    if ((id >> sshift) == ss && in_set(lk[i], id, vP, idP)) {
      const int slot = atomicAdd(&sh->gn, 1);
      if (slot < GMAX) {
        gid[slot] = id;
        gq[slot] = to_fx(wq[i]);
      }
    }
  }
  gsync<G>();
  const int gn = min(sh->gn, GMAX);
  int tok = -1;
#pragma unroll 1
  for (int q = t; q < gn; q += G) {
    const int my = gid[q];
    uint64_t pre = bf;
    for (int r = 0; r < gn; ++r)
      if (gid[r] < my) pre += gq[r];
    if (gq[q] > 0 && pre <= T && pre + gq[q] > T) tok = my;
  }
  tok = (int)gmax_u<G>((uint32_t)(tok + 1), sh->ru[1]) - 1;
  return tok >= 0 ? tok : last;
}

// Id-order draw over a short kept set (at most NT entries): the kept entries
// are compacted, ranked by id, laid out in id order and prefix-summed.
template <int DT>
__device__ int list_draw_small(Ctx<DT>& X, int n, uint32_t vP, int idP, uint64_t Mp, double u) {
  const float* wq = list_w(X);
  const uint32_t* lk = X.lk;
  const int* li = X.li;
  Sh* sh = X.sh;
  uint64_t* gq = list_scratch(X);            // compacted masses   [NT]
  uint64_t* sq = gq + NT;                    // id-ordered masses  [NT]
  int* gid = reinterpret_cast<int*>(sq + NT);  // compacted ids  [NT]
  int* sid = gid + NT;                         // id-ordered ids [NT]
  const int t = threadIdx.x;
  // T = floor(u * Mp) exactly (u = k * 2^-24): integer compares below
  const uint64_t T = __umul64hi(Mp, ((uint64_t)(u * 16777216.0)) << 40);
  __syncthreads();
  if (t == 0) {
    sh->gn = 0;
    sh->bi[6] = -1;
  }
  __syncthreads();
  for (int i = t; i < n; i += NT) {
    const int id = li[i];
    if (in_set(lk[i], id, vP, idP)) {
      const int slot = atomicAdd(&sh->gn, 1);
      if (slot < NT) {
        gid[slot] = id;
        gq[slot] = to_fx(wq[i]);
      }
    }
  }
  __syncthreads();
  const int m = min(sh->gn, NT);
  if (t < m) {
    const int my = gid[t];
    int r = 0;
    for (int j = 0; j < m; ++j) r += (gid[j] < my) ? 1 : 0;
    sq[r] = gq[t];
    sid[r] = my;
  }
  __syncthreads();
  const uint64_t v = (t < m) ? sq[t] : 0;
  uint64_t tot;
  const uint64_t ex = bscan_excl<uint64_t>(v, sh->rq[0], tot);
  if (t < m && v > 0 && ex <= T && ex + v > T) sh->bi[6] = sid[t];
  __syncthreads();
  const int tok = sh->bi[6];
  return tok >= 0 ? tok : ((m > 0) ? sid[m - 1] : -1);
}

}  // namespace smp
