// smp_gumbel.cu -- Gumbel-max sampling over a kept set, the sort-free second
// sampler family (lecture notes "Decoding: Sampling, Beam Search and
// Speculative Decoding", section 3.2: the argmax of z_i + g_i, with
// g_i = -log(-log(u_i)) independent Gumbel noise, is a draw from softmax(z)).
// With the kept mask of smp_topk_topp_mask it draws from the exact top-k /
// top-p distribution in one pass over the row and no prefix sum; it is kept
// beside the inverse-CDF sampler for distribution and timing comparisons.
//
// Per row: candidates are the tokens whose kept-mask bit is set (no mask: all)
// and whose logit is not -inf; z_i = fl32(x_i / T); u_i is word (i mod 4) of
// the Philox4x32-10 block at key (lo32 seed, hi32 seed) and counter (lo32
// offset, hi32 offset, i / 4, 0x47554D42), as ((w >> 8) + 1/2) * 2^-24;
// T == 0 takes the argmax of x.  Ties go to the smallest id.
//
// Layout: a cluster of up to 8 CTAs of 128 threads per row, each CTA a
// segment of the row, each thread four consecutive elements per step (one
// Philox block).  The CTAs' best candidates meet through distributed shared
// memory.  The noise is evaluated in fp32: -log(u) as -logf(u) for u < 1/2 and
// as -log1pf(-(1 - u)) above, both on exact arguments, so that u close to 1
// keeps its (large) perturbation.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/smp.h"
#include "smp_philox.cuh"

namespace cg = cooperative_groups;

namespace smp {

constexpr int GT = 128;      // threads per CTA
constexpr int GWARPS = GT / 32;
constexpr int GMAXC = 8;     // CTAs per cluster

struct GumbelArgs {
  const void* logits;
  long long ld;
  const uint32_t* kept;  // [B][W] or null
  const float* temperature;
  const uint64_t* seed;
  const uint64_t* offset;
  int32_t* tokens;
  int32_t* status;
  int B, V, W;
  int nc, seg;  // CTAs per row, elements per CTA (a multiple of 4)
  int vec;      // rows are aligned for vector loads
};

struct Best {
  float v;
  int id;
};

__device__ __forceinline__ bool better(float v, int id, float bv, int bid) {
  return v > bv || (v == bv && id < bid);
}

// -log(-log(u)) for u = (k + 1/2) * 2^-24, k = w >> 8 in [0, 2^24).
__device__ __forceinline__ float gumbel_noise(uint32_t w) {
  const uint32_t k = w >> 8;
  float e;
  if (k < (1u << 23)) {
    e = -logf(((float)k + 0.5f) * 5.9604644775390625e-08f);  // exact argument
  } else {
    const float v = ((float)((1u << 24) - 1u - k) + 0.5f) * 5.9604644775390625e-08f;  // 1 - u
    e = -log1pf(-v);
  }
  return -logf(e);
}

template <int DT>
__device__ __forceinline__ float load_x(const void* row, int i) {
  if constexpr (DT == SMP_F32) return __ldg(reinterpret_cast<const float*>(row) + i);
  else if constexpr (DT == SMP_BF16)
    return __bfloat162float(__ushort_as_bfloat16(__ldg(reinterpret_cast<const unsigned short*>(row) + i)));
  else return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(row) + i)));
}

// Four consecutive elements starting at i (a multiple of 4); entries at or
// past V are -inf.
template <int DT>
__device__ __forceinline__ void load4(const void* row, int i, int V, bool vec, float (&x)[4]) {
  if (vec && i + 3 < V) {
    if constexpr (DT == SMP_F32) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(row) + i));
      x[0] = f.x;
      x[1] = f.y;
      x[2] = f.z;
      x[3] = f.w;
    } else {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const unsigned short*>(row) + i));
      const unsigned short h[4] = {(unsigned short)(u.x & 0xffffu), (unsigned short)(u.x >> 16),
                                   (unsigned short)(u.y & 0xffffu), (unsigned short)(u.y >> 16)};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        x[e] = (DT == SMP_BF16) ? __bfloat162float(__ushort_as_bfloat16(h[e]))
                                : __half2float(__ushort_as_half(h[e]));
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = (i + e < V) ? load_x<DT>(row, i + e) : -INFINITY;
}

template <int DT>
__global__ void __launch_bounds__(GT, 8) gumbel_kernel(const GumbelArgs a) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int r = blockIdx.x / a.nc;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ Best wbest[GWARPS];
  __shared__ int wflag[GWARPS];
  __shared__ Best cbest;  // read by rank 0
  __shared__ int cflag;   // read by rank 0: 1 = NaN or +inf among the candidates

  const float T = a.temperature[r];
  const bool tok_ok = T >= 0.f;  // also rejects NaN
  const bool greedy = T == 0.f;
  const uint64_t seed = a.seed ? a.seed[r] : 0ull, off = a.offset ? a.offset[r] : 0ull;
  const char* row = reinterpret_cast<const char*>(a.logits) +
                    (size_t)r * (size_t)a.ld * (DT == SMP_F32 ? 4 : 2);
  const uint32_t* km = a.kept ? a.kept + (size_t)r * a.W : nullptr;
  float bv = -INFINITY;
  int bid = 0x7fffffff, bad = 0;
  if (tok_ok) {
    const int i0 = rank * a.seg, i1 = min(a.V, i0 + a.seg);
#pragma unroll 1
    for (int i = i0 + 4 * (int)threadIdx.x; i < i1; i += 4 * GT) {
      const uint32_t kw = km ? __ldg(km + (i >> 5)) >> (i & 31) : 0xfu;
      if ((kw & 0xfu) == 0u) continue;  // no kept token among the four
      float x[4];
      load4<DT>(row, i, a.V, a.vec != 0, x);
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      if (!greedy) philox4x32_10(seed, (uint32_t)off, (uint32_t)(off >> 32), (uint32_t)(i >> 2),
                                 0x47554D42u, w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (!((kw >> e) & 1u) || i + e >= i1) continue;
        const float xe = x[e];
        if (xe == -INFINITY) continue;
        if (!(xe < INFINITY)) {  // NaN or +inf
          bad = 1;
          continue;
        }
        const float v = greedy ? xe : __fadd_rn(__fdiv_rn(xe, T), gumbel_noise(w[e]));
        if (better(v, i + e, bv, bid)) {
          bv = v;
          bid = i + e;
        }
      }
    }
  }
  // CTA: warps, then the warps' bests
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oid = __shfl_xor_sync(0xffffffffu, bid, o);
    if (better(ov, oid, bv, bid)) {
      bv = ov;
      bid = oid;
    }
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    wbest[warp] = Best{bv, bid};
    wflag[warp] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Best b = wbest[0];
    int f = wflag[0];
    for (int q = 1; q < GWARPS; ++q) {
      if (better(wbest[q].v, wbest[q].id, b.v, b.id)) b = wbest[q];
      f |= wflag[q];
    }
    cbest = b;
    cflag = f;
  }
  // cluster: rank 0 reads every CTA's best, then all leave together
  cluster.sync();
  if (rank == 0 && threadIdx.x == 0) {
    Best b = cbest;
    int f = cflag;
    for (int c = 1; c < a.nc; ++c) {
      const Best o = *cluster.map_shared_rank(&cbest, c);
      if (better(o.v, o.id, b.v, b.id)) b = o;
      f |= *cluster.map_shared_rank(&cflag, c);
    }
    int st = SMP_OK, tok = -1;
    if (!tok_ok) st = SMP_ERR_INVALID_PARAM;
    else if (f) st = SMP_ERR_NONFINITE;
    else if (b.id == 0x7fffffff) st = SMP_ERR_EMPTY;
    else tok = b.id;
    a.status[r] = st;
    a.tokens[r] = tok;
  }
  cluster.sync();
}

int gumbel_enqueue(const void* logits, int dtype, int B, int V, long long ld,
                   const uint32_t* kept, const float* temperature, const uint64_t* seed,
                   const uint64_t* offset, int32_t* tokens, int32_t* status, cudaStream_t st) {
  if (B == 0) return SMP_OK;
  GumbelArgs a;
  a.logits = logits;
  a.ld = ld;
  a.kept = kept;
  a.temperature = temperature;
  a.seed = seed;
  a.offset = offset;
  a.tokens = tokens;
  a.status = status;
  a.B = B;
  a.V = V;
  a.W = (V + 31) / 32;
  const int groups = (V + 3) / 4;
  int nc = (V + 8191) / 8192;
  nc = nc < 1 ? 1 : (nc > GMAXC ? GMAXC : nc);
  a.nc = nc;
  a.seg = ((groups + nc - 1) / nc) * 4;
  const size_t es = dtype == SMP_F32 ? 4 : 2;
  const size_t va = dtype == SMP_F32 ? 16 : 8;
  a.vec = ((reinterpret_cast<uintptr_t>(logits) % va) == 0 && ((size_t)ld * es) % va == 0) ? 1 : 0;
  if ((long long)B * nc > 0x7fffffffLL) return SMP_ERR_CAPACITY;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * nc));
  cfg.blockDim = dim3(GT);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  switch (dtype) {
    case SMP_F32: e = cudaLaunchKernelEx(&cfg, gumbel_kernel<SMP_F32>, a); break;
    case SMP_BF16: e = cudaLaunchKernelEx(&cfg, gumbel_kernel<SMP_BF16>, a); break;
    default: e = cudaLaunchKernelEx(&cfg, gumbel_kernel<SMP_F16>, a); break;
  }
  return e == cudaSuccess ? SMP_OK : SMP_ERR_CUDA;
}

}  // namespace smp
