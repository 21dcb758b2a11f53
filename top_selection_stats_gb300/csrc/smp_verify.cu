// smp_verify.cu -- speculative-decoding verification with the exact
// accept / reject rule (lecture notes "Decoding: Sampling, Beam Search and
// Speculative Decoding", section 5.2, after Leviathan et al. 2023 and Chen et
// al. 2023), for a batch of sequences that each carry G draft tokens:
//   for i = 0, 1, ...: accept d_i iff u_acc(i) * q_i(d_i) < p_i(d_i), that is
//   with probability min(1, p/q); at the first rejection draw a token from
//   norm(max(0, p_i - q_i)) and stop; after G acceptances draw one more token
//   from the target's distribution p_G.
// The acceptance tests read two numbers per draft token; the cost is the one
// drawn row (two rows, p_j and q_j, after a rejection), streamed once from HBM.
//
// Layout on GB300: a thread-block cluster of NC CTAs per sequence splits the
// drawn row into NC segments of whole 512-element blocks, each CTA's four
// warps into contiguous slabs walked in 128-element steps (one float4 per
// lane).  Small CTAs, eight per SM, keep the per-CTA latencies (acceptance
// tests, cluster barriers, the final re-read) overlapped with other CTAs'
// streaming; each lane keeps four steps of loads in flight.  Weights are fixed-point integers, floor(w * 2^42), so the row sum
// and every prefix are exact and independent of the order of summation.  Each
// warp keeps its per-step sums in shared memory; after one cluster barrier
// every CTA reads the NC segment sums through distributed shared memory, and
// the CTA whose segment holds the drawn position finds the step from its
// stored sums and re-reads only that step's 128 elements.  No global scratch,
// no atomics, no waits other than two cluster barriers.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/smp.h"
#include "smp_philox.cuh"

namespace cg = cooperative_groups;

namespace smp {

constexpr int VT = 128;             // threads per CTA
constexpr int VWARPS = VT / 32;
constexpr int VSTEP = 128;          // elements per warp step (32 lanes x float4)
constexpr int VBLOCK = VSTEP * VWARPS;  // segment granule: 512 elements
constexpr int VMAXSTEPS = 256;      // steps per warp slab: segments of <= 131072
constexpr int VMAXC = 8;            // CTAs per cluster (portable size)
constexpr int VMAXG = 31;           // draft tokens per sequence (lanes 0..G of a warp)

struct VerifyArgs {
  const float* p;       // [B][G+1][ld]
  const float* q;       // [B][G][ld] (unused when G == 0)
  const int32_t* d;     // [B][G]
  const uint64_t* seed;
  const uint64_t* offset;
  int32_t* out_tokens;  // [B][G+1]
  int32_t* n_acc;       // [B]
  int32_t* status;      // [B]
  int64_t ld;
  int B, G, V;
  int nc;               // CTAs per cluster = per sequence
  int seg;              // elements per CTA segment, a multiple of VBLOCK
};

// floor(w * 2^42) for a float w in [0, 1], from the float's fields (no float
// to 64-bit integer conversion, which is slow on this GPU).  Zero, subnormal
// and negative inputs give 0.
__device__ __forceinline__ uint64_t fx42(float w) {
  const uint32_t b = __float_as_uint(w);
  const int e = (int)(b >> 23);  // biased exponent; the sign bit makes e >= 256
  if (e == 0 || e > 127) return 0ull;  // also every input above 2 (flagged bad)
  const uint64_t m = (uint64_t)((b & 0x7fffffu) | 0x800000u);
  const int sh = e - 108;  // the significand's unit bit weighs 2^(e - 150 + 42)
  return sh >= 0 ? (m << sh) : (sh > -24 ? (m >> -sh) : 0ull);
}

__device__ __forceinline__ bool prob_ok(float v) { return v >= 0.f && v <= 1.f; }

// Words 0 and 1 of the Philox4x32-10 block at key (lo32 seed, hi32 seed),
// counter (lo32 ctr, hi32 ctr, 0, 0).
__device__ __forceinline__ void philox_w01(uint64_t seed, uint64_t ctr, uint32_t& w0,
                                           uint32_t& w1) {
  uint32_t w[4];
  philox4x32_10(seed, (uint32_t)ctr, (uint32_t)(ctr >> 32), 0u, 0u, w);
  w0 = w[0];
  w1 = w[1];
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The four fixed-point weights of one float4 of the drawn row at element idx
// (elements at or past V weigh 0); `bad` collects out-of-range probabilities.
__device__ __forceinline__ void step_weights(float4 pv, float4 qv, bool residual, int idx, int V,
                                             uint64_t (&w)[4], bool& bad) {
  const float pa[4] = {pv.x, pv.y, pv.z, pv.w};
  const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const bool in = idx + e < V;
    float r = pa[e];
    bool ok = prob_ok(pa[e]);
    if (residual) {
      ok = ok && prob_ok(qa[e]);
      r = __fsub_rn(pa[e], qa[e]);
      r = r > 0.f ? r : 0.f;
    }
    bad |= in && !ok;
    w[e] = in ? fx42(r) : 0ull;
  }
}

__global__ void __launch_bounds__(VT, 8) spec_verify_kernel(const VerifyArgs a) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int s = blockIdx.x / a.nc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G, V = a.V;

  __shared__ uint64_t step_sum[VWARPS][VMAXSTEPS];
  __shared__ uint64_t warp_tot[VWARPS];
  __shared__ uint64_t cta_tot;     // read by the cluster's other CTAs
  __shared__ int cta_bad;          // read by the cluster's other CTAs
  __shared__ uint64_t all_tot[VMAXC];
  __shared__ int all_bad[VMAXC];
  __shared__ int sh_j, sh_bad;
  __shared__ uint32_t sh_k;

  // 1. the acceptance tests, one draft position per lane of warp 0; lane G
  //    also draws the bonus position's block
  if (warp == 0) {
    bool bad = false, rej = false;
    uint32_t w1 = 0u;
    if (lane <= G) {
      uint32_t w0;
      philox_w01(a.seed[s], a.offset[s] + (uint64_t)lane, w0, w1);
      if (lane < G) {
        const int x = a.d[(size_t)s * G + lane];
        if (x < 0 || x >= V) {
          bad = true;
        } else {
          const float pa = __ldg(a.p + ((size_t)s * (G + 1) + lane) * a.ld + x);
          const float qa = __ldg(a.q + ((size_t)s * G + lane) * a.ld + x);
          bad = !prob_ok(pa) || !prob_ok(qa);
          // u * q < p, exact in double: u = k * 2^-24 and q carry 24 bits each
          const double u = (double)(w0 >> 8) * (1.0 / 16777216.0);
          rej = !(u * (double)qa < (double)pa);
        }
      }
    }
    const uint32_t badm = __ballot_sync(0xffffffffu, bad);
    const uint32_t rejm = __ballot_sync(0xffffffffu, rej);
    const int j = rejm ? __ffs(rejm) - 1 : G;
    const uint32_t k = __shfl_sync(0xffffffffu, w1 >> 8, j);
    if (lane == 0) {
      sh_j = j;
      sh_k = k;
      sh_bad = badm != 0u;
      cta_bad = 0;
    }
  }
  __syncthreads();
  const int j = sh_j;
  int32_t* out = a.out_tokens + (size_t)s * (G + 1);
  if (sh_bad) {  // no cluster-shared memory is touched on this path
    if (rank == 0) {
      for (int i = threadIdx.x; i <= G; i += VT) out[i] = -1;
      if (threadIdx.x == 0) {
        a.n_acc[s] = 0;
        a.status[s] = SMP_ERR_INVALID_PARAM;
      }
    }
    return;
  }

  // 2. this CTA's segment of the drawn row: residual max(0, p_j - q_j) after a
  //    rejection, the target row p_G after G acceptances
  const bool residual = j < G;
  const float* prow = a.p + ((size_t)s * (G + 1) + j) * a.ld;
  const float* qrow = residual ? a.q + ((size_t)s * G + j) * a.ld : prow;
  const int wseg = a.seg / VWARPS;
  const int slab0 = rank * a.seg + warp * wseg;
  const int slab1 = min(slab0 + wseg, V);
  const int nsteps = slab1 > slab0 ? (slab1 - slab0 + VSTEP - 1) / VSTEP : 0;
  bool bad = false;
  uint64_t wtot = 0;
  constexpr int UNR = 4;
  for (int st = 0; st < nsteps; st += UNR) {
    float4 pv[UNR], qv[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int idx = slab0 + (st + u) * VSTEP + lane * 4;
      pv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      qv[u] = pv[u];
      if (st + u < nsteps && idx < V) {
        pv[u] = __ldg(reinterpret_cast<const float4*>(prow + idx));
        if (residual) qv[u] = __ldg(reinterpret_cast<const float4*>(qrow + idx));
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (st + u < nsteps) {
        const int idx = slab0 + (st + u) * VSTEP + lane * 4;
        uint64_t w[4];
        step_weights(pv[u], qv[u], residual, idx, V, w, bad);
        const uint64_t tot = warp_sum_u64(w[0] + w[1] + w[2] + w[3]);
        if (lane == 0) step_sum[warp][st + u] = tot;
        wtot += tot;
      }
    }
  }
  if (lane == 0) warp_tot[warp] = wtot;
  if (__syncthreads_or(bad) && threadIdx.x == 0) cta_bad = 1;
  if (threadIdx.x == 0) {
    uint64_t t = 0;
    for (int w = 0; w < VWARPS; ++w) t += warp_tot[w];
    cta_tot = t;
  }

  // 3. every CTA reads the cluster's segment sums (distributed shared memory)
  cluster.sync();
  if (threadIdx.x < a.nc) {
    all_tot[threadIdx.x] = *cluster.map_shared_rank(&cta_tot, threadIdx.x);
    all_bad[threadIdx.x] = *cluster.map_shared_rank(&cta_bad, threadIdx.x);
  }
  cluster.sync();  // no remote read follows: CTAs may leave after this

  uint64_t S = 0, before = 0;
  int any_bad = 0;
  for (int c = 0; c < a.nc; ++c) {
    S += all_tot[c];
    if (c < rank) before += all_tot[c];
    any_bad |= all_bad[c];
  }
  if (any_bad || S == 0ull) {
    if (rank == 0) {
      for (int i = threadIdx.x; i <= G; i += VT) out[i] = -1;
      if (threadIdx.x == 0) {
        a.n_acc[s] = 0;
        a.status[s] = any_bad ? SMP_ERR_INVALID_PARAM : SMP_ERR_EMPTY;
      }
    }
    return;
  }
  // draw target T = floor(u * S) with u = k * 2^-24: the token is the first
  // id whose inclusive prefix exceeds T (T < S, so one exists)
  const uint64_t T = __umul64hi(S, (uint64_t)sh_k << 40);
  if (T < before || T - before >= all_tot[rank]) return;  // not in this segment

  // 4. this CTA holds the drawn token: the warp, then the step, from the
  //    stored sums; then one re-read of that step's 128 elements
  uint64_t T1 = T - before;
  int w = 0;
  while (w < VWARPS - 1 && T1 >= warp_tot[w]) T1 -= warp_tot[w++];
  if (warp != w) return;
  const int ws0 = rank * a.seg + w * wseg;
  const int wsteps = min(ws0 + wseg, V) > ws0 ? (min(ws0 + wseg, V) - ws0 + VSTEP - 1) / VSTEP : 0;
  int st = 0;
  while (st < wsteps - 1 && T1 >= step_sum[w][st]) T1 -= step_sum[w][st++];
  const int idx = ws0 + st * VSTEP + lane * 4;
  float4 pv = make_float4(0.f, 0.f, 0.f, 0.f), qv = pv;
  if (idx < V) {
    pv = __ldg(reinterpret_cast<const float4*>(prow + idx));
    if (residual) qv = __ldg(reinterpret_cast<const float4*>(qrow + idx));
  }
  uint64_t wt[4];
  bool dummy = false;
  step_weights(pv, qv, residual, idx, V, wt, dummy);
  const uint64_t mine = wt[0] + wt[1] + wt[2] + wt[3];
  uint64_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t hit = __ballot_sync(0xffffffffu, incl > T1);
  // the last lane's prefix is the step's sum, which exceeds T1
  const int hl = hit ? __ffs(hit) - 1 : 31;
  if (lane == hl) {
    uint64_t r = T1 - (incl - mine);
    int e = 0;
    while (e < 3 && r >= wt[e]) r -= wt[e++];
    const int token = idx + e;
    for (int i = 0; i < j; ++i) out[i] = a.d[(size_t)s * G + i];
    out[j] = token;
    for (int i = j + 1; i <= G; ++i) out[i] = -1;
    a.n_acc[s] = j;
    a.status[s] = SMP_OK;
  }
}

const void* verify_kernel_ptr() { return reinterpret_cast<const void*>(spec_verify_kernel); }

// Cluster size and segment length for V: whole 512-element blocks per CTA, at
// least 8 K elements each, at most VMAXC CTAs and VMAXSTEPS steps per warp.
void verify_plan(int V, int& nc, int& seg) {
  const int blocks = (V + VBLOCK - 1) / VBLOCK;
  nc = (blocks + 15) / 16;
  nc = nc < 1 ? 1 : (nc > VMAXC ? VMAXC : nc);
  seg = ((blocks + nc - 1) / nc) * VBLOCK;
}

int verify_max_vocab() { return VMAXC * VMAXSTEPS * VSTEP * VWARPS; }
int verify_max_g() { return VMAXG; }

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * a.nc));
  cfg.blockDim = dim3(VT);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, spec_verify_kernel, a);
}

}  // namespace smp

namespace smp {

// Host side: argument checks are done by the caller (smp_spec_verify);
// returns SMP_OK, SMP_ERR_CAPACITY or SMP_ERR_CUDA.
int verify_enqueue(const float* p, const float* q, const int32_t* d, int B, int G, int V,
                   int64_t ld, const uint64_t* seed, const uint64_t* offset, int32_t* out_tokens,
                   int32_t* n_acc, int32_t* status, cudaStream_t st) {
  if (G > VMAXG || V > verify_max_vocab()) return SMP_ERR_CAPACITY;
  if (B == 0) return SMP_OK;
  VerifyArgs a;
  a.p = p;
  a.q = q;
  a.d = d;
  a.seed = seed;
  a.offset = offset;
  a.out_tokens = out_tokens;
  a.n_acc = n_acc;
  a.status = status;
  a.ld = ld;
  a.B = B;
  a.G = G;
  a.V = V;
  verify_plan(V, a.nc, a.seg);
  if ((long long)B * a.nc > 0x7fffffffLL) return SMP_ERR_CAPACITY;
  return launch_verify(a, st) == cudaSuccess ? SMP_OK : SMP_ERR_CUDA;
}

}  // namespace smp
