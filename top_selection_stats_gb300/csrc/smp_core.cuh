// smp_core.cuh -- shared definitions of the sampling kernel (sm_103a): launch
// arguments, the shared-memory layout, 16-byte element vectors, order-preserving
// keys, deterministic block reductions and the bulk-copy row ring.
//
// One CTA owns a row.  Rows stream from HBM through a ring of NSTAGE shared-
// memory stages filled by 1-D bulk copies (cp.async.bulk + mbarrier).  Lane l
// of warp w reads 16-byte vector (w * VW + it * 32 + l) of a chunk for it <
// ITW, so a warp covers VW consecutive vectors and the element order inside a
// chunk is (warp, it, lane, element).
#pragma once

#include "smp_device.cuh"

namespace smp {

constexpr int NSTAGE = 2;           // ring stages
constexpr int STAGE_BYTES = 24576;  // bytes per stage (one chunk)
constexpr int CAP = 6144;           // candidate list capacity (key, id pairs)
constexpr int MAXCH = 128;          // chunks per row, at most
constexpr int ITW = 6;              // vectors per thread per chunk
constexpr int FX = 40;              // fraction bits of fixed-point masses
constexpr int KLIST = 4096;         // top_k served by the sigma-truncated list
constexpr int HB = 11;              // digit bits of the descent histograms
constexpr int HBINS = 1 << HB;
constexpr int SEG_MAX = 3072;       // id segments of the list sampler
constexpr int GMAX = 512;           // ids per segment, at most
constexpr int NOID = 0x7fffffff;

// Weight histogram of the mass stream: bin = floor(HOFF - HS * a) with a =
// (x - ref) * log2(e) / T, clamped to [0, WBINS): HS bins per factor of two.
constexpr int WBINS = 2048;
constexpr int WHS = 16;
constexpr int WHOFF = 256;

// Job board (device workspace owned by the handle).  A row that would pass
// over its chunks on its own for long publishes the pass as a job: the mass
// stream of a row whose kept set is predicted to be large (kind JOB_STREAM),
// and the band pass over a weight-histogram bracket (JOB_BAND).  The owner
// keeps streaming the row from the front through its ring; CTAs without a row
// of their own, or done with theirs, take chunks from the back, one claim at a
// time, and stay on the job while chunks are left.  One
// 64-bit word holds both ends (front << 32 | back + ENDS_OFF): the owner adds
// 1 << 32 and owns chunk `front` if front < back; a helper adds -1 and owns
// chunk back - 1 if that is >= front.  Once the owner's claim fails, chunks
// [front, nch) are exactly the helpers' ones, and it waits (bounded) until
// the helpers report that many chunks done.  ENDS_OFF keeps failed helper claims from borrowing into
// the front half; bit ENDS_KIND of the back half holds the job's kind.  The
// word is written last when a job is published (after the header and a
// fence), so a claim that succeeds sees the whole header, and a helper finds
// open jobs with one load per slot.
constexpr int MAXJOBS = 32;
constexpr int JOB_BAND = 0, JOB_STREAM = 1;
constexpr uint32_t ENDS_OFF = 1u << 20;
constexpr uint32_t ENDS_KIND = 1u << 30;
struct JobHdr {
  unsigned long long ends;
  int pad, row, kind, nch;
  int b_lo, b_hi, done, list_n;
  float nref, nm, c2;
  int above_n;
  uint32_t mxk;  // stream: largest key of the helpers' chunks
  int nleg, nf;
  float xa, xb;  // band: value thresholds of the bracket (above: x >= xa; band: xb <= x < xa)
  int bad;  // a helper's bounded wait expired on a chunk of this job
};
static_assert(sizeof(JobHdr) % 16 == 0, "job headers keep the board's arrays aligned");
struct Board {
  int njobs, ctas_done, exits;
  int next_row;  // the next row a CTA takes (rows are handed out as CTAs free up)
  JobHdr hdr[MAXJOBS];
  float cmass[MAXJOBS][MAXCH * NWARP];  // per-(chunk, warp) masses of the helpers' chunks
  uint32_t lk[MAXJOBS][CAP];            // band: the helpers' bracket elements (key, id)
  int li[MAXJOBS][CAP];
  uint32_t wh[MAXJOBS][WBINS];          // stream: weight histogram of the helpers' chunks
};

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
  float* logprob;  // natural log of the drawn token's final probability, or null
  int* row_info;
  int mode;
  int use_tma;  // rows are 16-byte aligned: stage them with bulk copies
  Board* board;  // job board (zeroed between launches), or null
  long long wait_limit;  // SM clock cycles a bounded wait may take
  float delta[DTAB];
};

// Block scratch that lives beside the ring and the list.
struct Sh {
  uint64_t full[NSTAGE];
  uint64_t rq[2][NWARP];
  double rd[2][NWARP];
  float rf[3][NWARP];
  float r5[5][NWARP];         // the first chunk's statistics (one reduction)
  uint32_t ru[2][NWARP];
  int ri[2][NWARP];
  float cmass[MAXCH][NWARP];  // per-chunk, per-warp masses of the keep-all stream
  int ctie[MAXCH];            // per-chunk tie counts of the tie pass
  int done[NSTAGE];           // warps done with each stage in the current pass
  int n;                      // list entries appended (may exceed CAP: overflow)
  int nf;                     // NaN / +inf seen in a legal slot
  int timeout;                // a bounded wait expired: no copy is issued after it
  int niss[NSTAGE];           // bulk copies issued into each stage (for the final drain)
  int gn;                     // gathered entries of the sampled segment
  int bi[8];                  // broadcast ints
  int row_next;               // the row this CTA takes next (from the board)
  int primed;                 // chunks 0.. of the row are in flight for its first pass
  uint32_t bu[8];             // broadcast keys
  uint64_t bq[4];             // broadcast masses
  double bd[4];               // broadcast doubles
};

constexpr int SMEM_RING = NSTAGE * STAGE_BYTES;
constexpr int SMEM_LIST = CAP * 8;
constexpr int SMEM_HIST = WBINS * 4;
constexpr int SMEM_TOTAL = SMEM_RING + SMEM_LIST + SMEM_HIST + (int)sizeof(Sh) + 128;
static_assert(HBINS * 12 <= SMEM_LIST, "descent histograms live in the list area");
static_assert(CAP * 4 + SEG_MAX * 8 <= SMEM_RING, "list weights + segment sums live in the ring");
static_assert(STAGE_BYTES / 16 == ITW * NT, "a chunk is ITW vectors per thread");

__host__ __device__ inline int esize_of(int dt) { return dt == DT_F32 ? 4 : 2; }

template <int DT>
struct ElemT {
  static constexpr int ES = (DT == DT_F32) ? 4 : 2;
  static constexpr int EPV = 16 / ES;           // elements per 16-byte vector
  static constexpr int CE = STAGE_BYTES / ES;   // elements per chunk
  static constexpr int NVEC = CE / EPV;         // vectors per chunk (1536)
  static constexpr int VW = NVEC / NWARP;       // vectors per warp per chunk (192)
  static constexpr int SIG = (DT == DT_F32) ? 32 : 16;  // significant key bits
  static constexpr uint32_t NEG2 = (DT == DT_BF16) ? 0xff80ff80u : 0xfc00fc00u;
  // native keys of -inf, the lowest finite value and +inf
  static constexpr uint32_t KNINF = (DT == DT_F32) ? 0x007fffffu : (DT == DT_BF16 ? 0x007fu : 0x03ffu);
  static constexpr uint32_t KLOW = KNINF + 1u;
  static constexpr uint32_t KPINF = (DT == DT_F32) ? 0xff800000u : (DT == DT_BF16 ? 0xff80u : 0xfc00u);
};

template <int DT>
struct Ctx {
  const KArgs* a;
  char* ring;
  uint32_t* lk;  // list keys (native order-preserving keys)
  int* li;       // list ids
  uint32_t* wh;  // weight histogram (WBINS counts)
  Sh* sh;
  const char* src;
  const uint32_t* bm;  // this row's bitmask words, or null
  int row, V, W, nch, use_tma;
  uint32_t parity;  // per-stage mbarrier phase bits
  float temp, c2;   // temperature, log2(e) / temperature
};

// Register copy of a context for a function that streams: the caller's copy
// sits in local memory (its address is passed), so a leaf function works on
// its own copy and hands the ring phase bits back when it returns.
template <int DT>
struct LocalCtx {
  Ctx<DT>& ref;
  Ctx<DT> v;
  __device__ __forceinline__ explicit LocalCtx(Ctx<DT>& r) : ref(r), v(r) {}
  __device__ __forceinline__ ~LocalCtx() { ref.parity = v.parity; }
};

// ---------------------------------------------------------------------------
// Keys.  A native key is the order-preserving unsigned image of the stored
// value: 16 bits for bf16 / fp16, 32 bits for fp32; -0 folds onto +0.  Every
// legal finite value has key >= KLOW > 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t key16(uint32_t b) {
  b &= 0xffffu;
  if ((b & 0x7fffu) == 0u) b = 0u;
  return (b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u);
}
template <int DT>
__device__ __forceinline__ float bits_value(uint32_t b) {
  if constexpr (DT == DT_F32) return __uint_as_float(b);
  else if constexpr (DT == DT_BF16) return __uint_as_float(b << 16);
  else return __half2float(__ushort_as_half((unsigned short)b));
}
template <int DT>
__device__ __forceinline__ uint32_t bits_key(uint32_t b) {
  if constexpr (DT == DT_F32) return fkey(__uint_as_float(b));
  else return key16(b);
}
template <int DT>
__device__ __forceinline__ float key_value(uint32_t k) {
  if constexpr (DT == DT_F32) return key_to_float(k);
  else {
    const uint32_t b = (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
    return bits_value<DT>(b);
  }
}
// Raw bits of element j of a vector.
template <int DT>
__device__ __forceinline__ uint32_t elem_bits(const uint4 r, int j) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
  if constexpr (DT == DT_F32) return w[j];
  else return (w[j >> 1] >> ((j & 1) * 16)) & 0xffffu;
}
template <int DT>
__device__ __forceinline__ void unpack(const uint4 r, float (&x)[ElemT<DT>::EPV]) {
#pragma unroll
  for (int j = 0; j < ElemT<DT>::EPV; ++j) x[j] = bits_value<DT>(elem_bits<DT>(r, j));
}
// The stored value rounded toward -inf into the element type, packed twice.
template <int DT>
__device__ __forceinline__ uint32_t pack_down(float t) {
  if constexpr (DT == DT_BF16) {
    const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rd(t));
    return b | (b << 16);
  } else if constexpr (DT == DT_F16) {
    const uint32_t b = __half_as_ushort(__float2half_rd(t));
    return b | (b << 16);
  } else {
    return __float_as_uint(t);
  }
}

// ---------------------------------------------------------------------------
// Vector tests.  any_ge: some element >= t or NaN.  any_gt: some element > t
// or NaN.  t2 is t packed in the element type (pack_down), tf the float value.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ bool any_ge(const uint4 r, uint32_t t2, float tf) {
  if constexpr (DT == DT_F32) {
    return !(__uint_as_float(r.x) < tf && __uint_as_float(r.y) < tf && __uint_as_float(r.z) < tf &&
             __uint_as_float(r.w) < tf);
  } else if constexpr (DT == DT_BF16) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return !__hblt2(m, *reinterpret_cast<const __nv_bfloat162*>(&t2));
  } else {
    const __half2 a = *reinterpret_cast<const __half2*>(&r.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&r.y);
    const __half2 c = *reinterpret_cast<const __half2*>(&r.z);
    const __half2 d = *reinterpret_cast<const __half2*>(&r.w);
    const __half2 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return !__hblt2(m, *reinterpret_cast<const __half2*>(&t2));
  }
}
template <int DT>
__device__ __forceinline__ bool any_gt(const uint4 r, uint32_t t2, float tf) {
  if constexpr (DT == DT_F32) {
    return !(__uint_as_float(r.x) <= tf && __uint_as_float(r.y) <= tf &&
             __uint_as_float(r.z) <= tf && __uint_as_float(r.w) <= tf);
  } else if constexpr (DT == DT_BF16) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return !__hble2(m, *reinterpret_cast<const __nv_bfloat162*>(&t2));
  } else {
    const __half2 a = *reinterpret_cast<const __half2*>(&r.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&r.y);
    const __half2 c = *reinterpret_cast<const __half2*>(&r.z);
    const __half2 d = *reinterpret_cast<const __half2*>(&r.w);
    const __half2 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return !__hble2(m, *reinterpret_cast<const __half2*>(&t2));
  }
}
// Maximum of the vector as a float; NaN anywhere gives NaN.
template <int DT>
__device__ __forceinline__ float vmax_nan_f(const uint4 r) {
  if constexpr (DT == DT_F32) {
    const float a = __uint_as_float(r.x), b = __uint_as_float(r.y), c = __uint_as_float(r.z),
                d = __uint_as_float(r.w);
    const float m = fmaxf(fmaxf(a, b), fmaxf(c, d));
    return (a != a || b != b || c != c || d != d) ? __uint_as_float(0x7fc00000u) : m;
  } else if constexpr (DT == DT_BF16) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    const uint32_t u = *reinterpret_cast<const uint32_t*>(&m);
    const float lo = __uint_as_float(u << 16), hi = __uint_as_float(u & 0xffff0000u);
    return (lo != lo || hi != hi) ? __uint_as_float(0x7fc00000u) : fmaxf(lo, hi);
  } else {
    const __half2 a = *reinterpret_cast<const __half2*>(&r.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&r.y);
    const __half2 c = *reinterpret_cast<const __half2*>(&r.z);
    const __half2 d = *reinterpret_cast<const __half2*>(&r.w);
    const __half2 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    const float lo = __low2float(m), hi = __high2float(m);
    return (lo != lo || hi != hi) ? __uint_as_float(0x7fc00000u) : fmaxf(lo, hi);
  }
}
// Packed vector extrema (NaN-propagating) and their running accumulation:
// two bf16 / fp16 lanes in a 32-bit word, or one fp32 value.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float fmin_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
template <int DT>
__device__ __forceinline__ uint32_t pmax(uint32_t a, uint32_t b) {
  if constexpr (DT == DT_F32) {
    return __float_as_uint(fmax_nan(__uint_as_float(a), __uint_as_float(b)));
  } else if constexpr (DT == DT_BF16) {
    const __nv_bfloat162 m = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                         *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&m);
  } else {
    const __half2 m = __hmax2_nan(*reinterpret_cast<const __half2*>(&a),
                                  *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&m);
  }
}
template <int DT>
__device__ __forceinline__ uint32_t pmin(uint32_t a, uint32_t b) {
  if constexpr (DT == DT_F32) {
    return __float_as_uint(fmin_nan(__uint_as_float(a), __uint_as_float(b)));
  } else if constexpr (DT == DT_BF16) {
    const __nv_bfloat162 m = __hmin2_nan(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                         *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&m);
  } else {
    const __half2 m = __hmin2_nan(*reinterpret_cast<const __half2*>(&a),
                                  *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&m);
  }
}
template <int DT>
__device__ __forceinline__ uint32_t vmax2(const uint4 r) {
  return pmax<DT>(pmax<DT>(r.x, r.y), pmax<DT>(r.z, r.w));
}
template <int DT>
__device__ __forceinline__ uint32_t vmin2(const uint4 r) {
  return pmin<DT>(pmin<DT>(r.x, r.y), pmin<DT>(r.z, r.w));
}
// Largest lane of a packed value as a float (NaN if either lane is NaN).
template <int DT>
__device__ __forceinline__ float p2f_max(uint32_t m) {
  if constexpr (DT == DT_F32) return __uint_as_float(m);
  else return fmax_nan(bits_value<DT>(m & 0xffffu), bits_value<DT>(m >> 16));
}
template <int DT>
__device__ __forceinline__ float p2f_min(uint32_t m) {
  if constexpr (DT == DT_F32) return __uint_as_float(m);
  else return fmin_nan(bits_value<DT>(m & 0xffffu), bits_value<DT>(m >> 16));
}
// Some lane of a packed maximum is >= t (t2 = t packed), or NaN.
template <int DT>
__device__ __forceinline__ bool p_any_ge(uint32_t m, uint32_t t2, float tf) {
  if constexpr (DT == DT_F32) return !(__uint_as_float(m) < tf);
  else if constexpr (DT == DT_BF16)
    return !__hblt2(*reinterpret_cast<const __nv_bfloat162*>(&m),
                    *reinterpret_cast<const __nv_bfloat162*>(&t2));
  else
    return !__hblt2(*reinterpret_cast<const __half2*>(&m), *reinterpret_cast<const __half2*>(&t2));
}
// Packed -inf of the element type: the identity of pmax.
template <int DT>
__device__ __forceinline__ uint32_t p_ninf() {
  return DT == DT_F32 ? 0xff800000u : ElemT<DT>::NEG2;
}
template <int DT>
__device__ __forceinline__ uint32_t p_pinf() {
  return DT == DT_F32 ? 0x7f800000u : (DT == DT_BF16 ? 0x7f807f80u : 0x7c007c00u);
}

template <int DT>
__device__ __forceinline__ uint32_t ninf2() {
  return DT == DT_F32 ? 0xff800000u : ElemT<DT>::NEG2;
}
// Replace masked-out elements (bit 0 in lb) by -inf.
template <int DT>
__device__ __forceinline__ uint4 apply_mask(uint4 r, uint32_t lb) {
  if constexpr (DT == DT_F32) {
    if (!(lb & 1u)) r.x = 0xff800000u;
    if (!(lb & 2u)) r.y = 0xff800000u;
    if (!(lb & 4u)) r.z = 0xff800000u;
    if (!(lb & 8u)) r.w = 0xff800000u;
    return r;
  } else {
    constexpr uint32_t NEG2 = ElemT<DT>::NEG2;
    uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t lo = 0u - ((lb >> (2 * q)) & 1u);
      const uint32_t hi = 0u - ((lb >> (2 * q + 1)) & 1u);
      const uint32_t sel = (lo & 0x0000ffffu) | (hi & 0xffff0000u);
      w[q] = (w[q] & sel) | (NEG2 & ~sel);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Hardware base-2 exponential (bulk masses, never an output on its own).
__device__ __forceinline__ float fast_exp2(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
// Fixed-point mass of a weight in [0, 1]: w * 2^FX, truncated.
// Built from the float's fields with integer operations (the float -> 64-bit
// integer conversion runs on a slow pipe); equal to truncating w * 2^FX.
__device__ __forceinline__ uint64_t to_fx(float w) {
  const uint32_t b = __float_as_uint(w);
  const int ex = (int)(b >> 23) - (127 + 23 - FX);  // weight of the significand's unit bit
  const uint64_t m = (uint64_t)((b & 0x7fffffu) | 0x800000u);
  if ((b >> 31) || (b >> 23) == 0u) return 0ull;  // negative, zero or subnormal
  if (ex > 63 - 24) return ~0ull;                  // beyond 2^64 (never a weight)
  return ex >= 0 ? (m << ex) : (ex > -24 ? (m >> -ex) : 0ull);
}
// floor(w * 2^s) for 0 <= w with a result below 2^63, by integer operations.
__device__ __forceinline__ uint64_t fx_scaled(float w, int s) {
  const uint32_t b = __float_as_uint(w);
  if ((b >> 31) || (b >> 23) == 0u) return 0ull;
  const int ex = (int)(b >> 23) - 150 + s;  // weight of the significand's unit bit
  const uint64_t m = (uint64_t)((b & 0x7fffffu) | 0x800000u);
  if (ex > 39) return ~0ull >> 1;
  return ex >= 0 ? (m << ex) : (ex > -24 ? (m >> -ex) : 0ull);
}
// floor(max(y, -1)) as an int for y < 2^22 by one round-down add of 1.5 *
// 2^23 (no float -> int conversion, which runs at an eighth of the ALU rate);
// y >= 2^22 (or +inf) gives at least 2^22, NaN gives -1, so callers that clamp
// to [0, n) with n <= 2^22 get the clamped floor.
__device__ __forceinline__ int floor_small(float y) {
  return __float_as_int(__fadd_rd(fmaxf(y, -1.f), 12582912.0f)) - 0x4B400000;
}

// ---------------------------------------------------------------------------
// Deterministic block reductions: warp trees, then every thread adds the
// NWARP partials in warp order.  Each call begins with a barrier, so scratch
// slots can be reused by the next call.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bsum_f(float v, float* s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s[warp] = v;
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r += s[w];
  return r;
}
__device__ __forceinline__ double bsum_d(double v, double* s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s[warp] = v;
  __syncthreads();
  double r = 0.0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r += s[w];
  return r;
}
__device__ __forceinline__ uint64_t bsum_q(uint64_t v, uint64_t* s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s[warp] = v;
  __syncthreads();
  uint64_t r = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r += s[w];
  return r;
}
__device__ __forceinline__ int bsum_i(int v, int* s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_add_sync(0xffffffffu, v);
  __syncthreads();
  if (lane == 0) s[warp] = v;
  __syncthreads();
  int r = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r += s[w];
  return r;
}
__device__ __forceinline__ uint32_t bmax_u(uint32_t v, uint32_t* s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_max_sync(0xffffffffu, v);
  __syncthreads();
  if (lane == 0) s[warp] = v;
  __syncthreads();
  uint32_t r = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r = max(r, s[w]);
  return r;
}
__device__ __forceinline__ uint32_t bmin_u(uint32_t v, uint32_t* s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_min_sync(0xffffffffu, v);
  __syncthreads();
  if (lane == 0) s[warp] = v;
  __syncthreads();
  uint32_t r = 0xffffffffu;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r = min(r, s[w]);
  return r;
}
__device__ __forceinline__ float bmax_f(float v, float* s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) s[warp] = v;
  __syncthreads();
  float r = -INFINITY;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) r = fmaxf(r, s[w]);
  return r;
}
// Exclusive scan in thread order; `total` receives the block sum.
template <class T>
__device__ __forceinline__ T bscan_excl(T v, T* s, T& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T inc = warp_incl_scan(v);
  __syncthreads();
  if (lane == 31) s[warp] = inc;
  __syncthreads();
  T off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    const T x = s[w];
    if (w < warp) off += x;
    tot += x;
  }
  total = tot;
  return off + inc - v;
}

// ---------------------------------------------------------------------------
// Row ring.  ring_begin issues the first NSTAGE chunks of the row; ring_wait(c)
// returns the stage holding chunk c once it landed (elements past V read as
// -inf); ring_release(c) frees the stage after a block barrier and issues
// chunk c + NSTAGE into it.  mbarrier waits are bounded (about 2 s at 2 GHz):
// an expired wait is recorded and the pass carries on.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ void issue_chunk(Ctx<DT>& X, int c, int s) {
  constexpr int ES = ElemT<DT>::ES, CE = ElemT<DT>::CE;
  const int ne = min(CE, X.V - c * CE);
  const uint32_t bytes = X.use_tma ? (uint32_t)((ne * ES) & ~15) : 0u;
  uint64_t* bar = &X.sh->full[s];
  // after an expired wait the stages' phases are unknown: nothing more goes out
  if (X.sh->timeout) return;
  ++X.sh->niss[s];
  // order earlier generic-proxy accesses of the stage before the async copy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_arrive_expect_tx(bar, bytes);
  if (bytes > 0)
    bulk_g2s(X.ring + (size_t)s * STAGE_BYTES, X.src + (size_t)c * CE * ES, bytes, bar);
}

template <int DT>
__device__ __forceinline__ void ring_begin(Ctx<DT>& X, int first = 0) {
  if (threadIdx.x == 0)
    for (int s = 0; s < NSTAGE; ++s) X.sh->done[s] = 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    if (X.sh->primed && first == 0) {
      X.sh->primed = 0;  // the row's first pass: its chunks were issued with the row
    } else {
      for (int s = 0; s < NSTAGE && first + s < X.nch; ++s)
        issue_chunk(X, first + s, (first + s) % NSTAGE);
    }
  }
}

// The first chunks of a row, issued as soon as the row is known (before its
// parameters are read) for the first pass to take over in ring_begin.
template <int DT>
__device__ __forceinline__ void ring_prime(Ctx<DT>& X) {
  if (threadIdx.x == 0 && !X.sh->timeout) {
    for (int s = 0; s < NSTAGE; ++s) X.sh->done[s] = 0;
    for (int s = 0; s < NSTAGE && s < X.nch; ++s) issue_chunk(X, s, s);
    X.sh->primed = 1;
  }
}

// Per-warp consumption of a pass (no block barrier inside the loop): each warp
// waits for chunk c itself, reads only its own VW vectors of the stage, and
// the last warp to release a stage issues the chunk NSTAGE ahead into it.
// Warps may drift apart by up to NSTAGE - 1 chunks.
template <int DT>
__device__ __forceinline__ const char* warp_wait(Ctx<DT>& X, int c) {
  constexpr int ES = ElemT<DT>::ES, CE = ElemT<DT>::CE, EPV = ElemT<DT>::EPV, VW = ElemT<DT>::VW;
  const int s = c % NSTAGE;
  char* stage = X.ring + (size_t)s * STAGE_BYTES;
  const uint32_t par = (X.parity >> s) & 1u;
  if (!X.sh->timeout && !mbar_wait_bounded(&X.sh->full[s], par, X.a->wait_limit)) X.sh->timeout = 1;
  X.parity ^= 1u << s;
  const int ne = min(CE, X.V - c * CE);
  const int nb = X.use_tma ? ((ne * ES) & ~15) / ES : 0;
  if (nb < CE) {
    // this warp's elements the bulk copy did not cover: plain loads, -inf past V
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = w * VW * EPV, e1 = e0 + VW * EPV;
    const char* g = X.src + (size_t)c * CE * ES;
    for (int e = max(e0, nb) + lane; e < e1; e += 32) {
      if constexpr (ES == 4) {
        reinterpret_cast<uint32_t*>(stage)[e] =
            (e < ne) ? reinterpret_cast<const uint32_t*>(g)[e] : 0xff800000u;
      } else {
        constexpr unsigned short NEG = (unsigned short)(ElemT<DT>::NEG2 & 0xffffu);
        reinterpret_cast<unsigned short*>(stage)[e] =
            (e < ne) ? reinterpret_cast<const unsigned short*>(g)[e] : NEG;
      }
    }
    __syncwarp();
  }
  return stage;
}
template <int DT>
__device__ __forceinline__ void warp_release(Ctx<DT>& X, int c) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    const int s = c % NSTAGE;
    __threadfence_block();
    const int old = atomicAdd(&X.sh->done[s], 1);
    if (old == (c / NSTAGE + 1) * NWARP - 1 && c + NSTAGE < X.nch) issue_chunk(X, c + NSTAGE, s);
  }
}

template <int DT>
__device__ __forceinline__ const char* ring_wait_at(Ctx<DT>& X, int c, int s) {
  constexpr int ES = ElemT<DT>::ES, CE = ElemT<DT>::CE;
  char* stage = X.ring + (size_t)s * STAGE_BYTES;
  const uint32_t par = (X.parity >> s) & 1u;
  if (!X.sh->timeout && !mbar_wait_bounded(&X.sh->full[s], par, X.a->wait_limit)) X.sh->timeout = 1;
  X.parity ^= 1u << s;
  const int ne = min(CE, X.V - c * CE);
  const int nb = X.use_tma ? ((ne * ES) & ~15) / ES : 0;
  if (nb < CE) {
    const char* g = X.src + (size_t)c * CE * ES;
    for (int e = nb + (int)threadIdx.x; e < CE; e += NT) {
      if constexpr (ES == 4) {
        reinterpret_cast<uint32_t*>(stage)[e] =
            (e < ne) ? reinterpret_cast<const uint32_t*>(g)[e] : 0xff800000u;
      } else {
        constexpr unsigned short NEG = (unsigned short)(ElemT<DT>::NEG2 & 0xffffu);
        reinterpret_cast<unsigned short*>(stage)[e] =
            (e < ne) ? reinterpret_cast<const unsigned short*>(g)[e] : NEG;
      }
    }
    __syncthreads();
  }
  return stage;
}
template <int DT>
__device__ __forceinline__ const char* ring_wait(Ctx<DT>& X, int c) {
  return ring_wait_at(X, c, c % NSTAGE);
}

// A helper's next chunk of job j, claimed from the back (see JobHdr) by
// thread 0 while the current chunk is processed: -1 when none is left or the
// CTA stopped streaming after an expired wait.
__device__ __forceinline__ int helper_claim(Board* bd, int j, int timeout) {
  if (timeout) return -1;
  const unsigned long long old = atomicAdd(&bd->hdr[j].ends, ~0ull);
  const int d = (int)((uint32_t)old & (ENDS_KIND - 1u)) - (int)ENDS_OFF - 1;
  return (d >= (int)(old >> 32)) ? d : -1;
}

template <int DT>
__device__ __forceinline__ void ring_release(Ctx<DT>& X, int c) {
  __syncthreads();
  if (threadIdx.x == 0 && c + NSTAGE < X.nch) issue_chunk(X, c + NSTAGE, c % NSTAGE);
}


// Register-resident iterator of a per-warp pass: stage index, pass round and
// the last chunk fully covered by bulk copies, kept incrementally so the
// per-chunk bookkeeping is a handful of instructions.
template <int DT>
struct RingIt {
  int c, s, rnd, nfull;
  __device__ __forceinline__ explicit RingIt(const Ctx<DT>& X)
      : c(0), s(0), rnd(0), nfull(X.use_tma ? X.V / ElemT<DT>::CE : 0) {}
  __device__ __forceinline__ const char* wait(Ctx<DT>& X) {
    constexpr int ES = ElemT<DT>::ES, CE = ElemT<DT>::CE, EPV = ElemT<DT>::EPV, VW = ElemT<DT>::VW;
    char* stage = X.ring + s * STAGE_BYTES;
    if (!X.sh->timeout &&
        !mbar_wait_bounded(&X.sh->full[s], (X.parity >> s) & 1u, X.a->wait_limit))
      X.sh->timeout = 1;
    X.parity ^= 1u << s;
    if (c >= nfull) {
      // this warp's elements the bulk copy did not cover: plain loads, -inf past V
      const int ne = min(CE, X.V - c * CE);
      const int nb = X.use_tma ? ((ne * ES) & ~15) / ES : 0;
      const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
      const int e0 = w * VW * EPV, e1 = e0 + VW * EPV;
      const char* g = X.src + (size_t)c * CE * ES;
      for (int e = max(e0, nb) + lane; e < e1; e += 32) {
        if constexpr (ES == 4) {
          reinterpret_cast<uint32_t*>(stage)[e] =
              (e < ne) ? reinterpret_cast<const uint32_t*>(g)[e] : 0xff800000u;
        } else {
          constexpr unsigned short NEG = (unsigned short)(ElemT<DT>::NEG2 & 0xffffu);
          reinterpret_cast<unsigned short*>(stage)[e] =
              (e < ne) ? reinterpret_cast<const unsigned short*>(g)[e] : NEG;
        }
      }
      __syncwarp();
    }
    return stage;
  }
  __device__ __forceinline__ void release(Ctx<DT>& X) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      __threadfence_block();
      const int old = atomicAdd(&X.sh->done[s], 1);
      if (old == rnd * NWARP + NWARP - 1 && c + NSTAGE < X.nch) issue_chunk(X, c + NSTAGE, s);
    }
    ++c;
    if (++s == NSTAGE) {
      s = 0;
      ++rnd;
    }
  }
};

// Vector index of lane l of warp w in iteration it.
template <int DT>
__device__ __forceinline__ int warp_vec(int it) {
  return (threadIdx.x >> 5) * ElemT<DT>::VW + it * 32 + (threadIdx.x & 31);
}
// Legal-mask bits for the EPV elements starting at row element e (a multiple
// of EPV); all ones without a bitmask; 0 past V.
template <int DT>
__device__ __forceinline__ uint32_t mask_bits(const Ctx<DT>& X, int e) {
  constexpr int EPV = ElemT<DT>::EPV;
  if (!X.bm) return (1u << EPV) - 1u;
  const int w = e >> 5;
  if (w >= X.W) return 0u;
  return (__ldg(X.bm + w) >> (e & 31)) & ((1u << EPV) - 1u);
}
template <int DT>
__device__ __forceinline__ uint4 load_vec(const Ctx<DT>& X, const char* stage, int c, int vi) {
  constexpr int EPV = ElemT<DT>::EPV, CE = ElemT<DT>::CE;
  uint4 r = reinterpret_cast<const uint4*>(stage)[vi];
  if (X.bm) {
    const uint32_t lb = mask_bits(X, c * CE + vi * EPV);
    if (lb != (1u << EPV) - 1u) r = apply_mask<DT>(r, lb);
  }
  return r;
}

}  // namespace smp
