// smp_toplp.cu -- top logprobs: the n most likely tokens of each row's kept
// set with their log-probabilities ("Sampling system design" post, section on
// logprobs: besides the selected token's logprob an API may return the top
// candidates and theirs, under the distribution it states).  The
// distribution is the processed one smp_sample_logprob uses: temperature,
// mask, top-k and top-p, renormalised over the kept set.  Two kept tokens'
// log-probabilities differ by the difference of their scaled logits, so with
// the drawn token's logprob known,
//     logprob_j = logprob_tok + (fl32(x_j / T) - fl32(x_tok / T)),
// and the kept set's normaliser is never needed again.
//
// One cluster of up to 8 CTAs of 128 threads per row.  A warp reads 32 kept-
// mask words at a time, one per lane (coalesced), so a lane owns 32
// consecutive tokens; a lane whose word has a kept bit loads those 32 logits
// as 16-byte vectors, all lanes' loads in flight together.  The warp keeps
// the 32 best (logit descending, id ascending) kept tokens it has seen as
// 64-bit order keys, one per lane, sorted across the lanes; unless some
// lane's best new key beats the warp's 32nd best (after the first steps,
// rare), the 32 tokens of each lane are skipped at once; otherwise batches of
// 32 candidates (bit j of every lane) are merged (a bitonic sort of the batch
// and a bitonic merge).  The warps' lists, then the CTAs' lists (through
// distributed shared memory), are merged the same way.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/smp.h"

namespace cg = cooperative_groups;

namespace smp {

constexpr int LT = 128;  // threads per CTA
constexpr int LWARPS = LT / 32;
constexpr int LMAXC = 8;
constexpr int LMAXN = 32;

struct TopArgs {
  const void* logits;
  long long ld;
  const uint32_t* kept;
  const float* temperature;
  const int32_t* tokens;
  const float* logprobs;
  int32_t* out_ids;   // [B][n]
  float* out_lp;      // [B][n]
  int B, V, W, n;
  int nc, seg;
  int vec;  // rows 16-byte aligned: logits read as 16-byte vectors
};

// Order key: larger is better (larger logit, then smaller id); 0 = empty.
__device__ __forceinline__ uint64_t order_key(float x, int id) {
  uint32_t b = __float_as_uint(x + 0.f);  // -0 folds onto +0
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)b << 32) | (uint64_t)(0xffffffffu - (uint32_t)id);
}
__device__ __forceinline__ float key_value(uint64_t k) {
  uint32_t b = (uint32_t)(k >> 32);
  b = (b & 0x80000000u) ? (b & 0x7fffffffu) : ~b;
  return __uint_as_float(b);
}
__device__ __forceinline__ int key_id(uint64_t k) { return (int)(0xffffffffu - (uint32_t)k); }

// Sort the warp's 32 keys (one per lane) descending across the lanes.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool up = (lane & k) == 0;         // this k-block sorts descending
      const bool low = (lane & j) == 0;        // lower index of the pair
      const bool take_max = (low == up);
      v = take_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// a: sorted descending across the lanes; b: any 32 keys.  Returns the 32
// largest of both, sorted descending.
__device__ __forceinline__ uint64_t warp_merge_top(uint64_t a, uint64_t b, int lane) {
  b = warp_sort_desc(b, lane);
  // a descending, b descending -> max(a_i, b_{31-i}) holds the 32 largest as a
  // bitonic sequence
  const uint64_t br = __shfl_sync(0xffffffffu, b, 31 - lane);
  uint64_t v = a > br ? a : br;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
    const bool low = (lane & j) == 0;
    v = low ? (v > o ? v : o) : (v < o ? v : o);
  }
  return v;
}

template <int DT>
__device__ __forceinline__ float load_logit(const char* row, int i) {
  if constexpr (DT == SMP_F32) return __ldg(reinterpret_cast<const float*>(row) + i);
  else if constexpr (DT == SMP_BF16)
    return __bfloat162float(__ushort_as_bfloat16(__ldg(reinterpret_cast<const unsigned short*>(row) + i)));
  else return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(row) + i)));
}

template <int DT>
__global__ void __launch_bounds__(LT, 8) toplp_kernel(const TopArgs a) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int r = blockIdx.x / a.nc;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ uint64_t wl[LWARPS][32];
  __shared__ uint64_t cl[32];  // this CTA's list, read by rank 0
  const char* row = reinterpret_cast<const char*>(a.logits) +
                    (size_t)r * (size_t)a.ld * (DT == SMP_F32 ? 4 : 2);
  const uint32_t* km = a.kept + (size_t)r * a.W;
  const bool live = a.tokens[r] >= 0;

  // this CTA's segment (a multiple of 32 tokens), 32 mask words per warp step
  constexpr int ES = DT == SMP_F32 ? 4 : 2;
  constexpr int NV = 32 * ES / 16;  // 16-byte vectors per lane's 32 tokens
  __shared__ unsigned long long tau;  // the best 32nd-best key any warp here holds
  if (threadIdx.x == 0) tau = 0ull;
  __syncthreads();
  uint64_t top = 0ull;
  if (live) {
    const int c0 = rank * a.seg, c1 = min(a.V, c0 + a.seg);
    const int w0 = c0 >> 5, w1 = (c1 + 31) >> 5;
#pragma unroll 1
    for (int wb = w0 + warp * 32; wb < w1; wb += LWARPS * 32) {
      const int w = wb + lane;
      uint32_t bits = w < w1 ? __ldg(km + w) : 0u;
      if (w == w1 - 1 && (c1 & 31)) bits &= (1u << (c1 & 31)) - 1u;  // ids >= c1 belong elsewhere
      if (!__any_sync(0xffffffffu, bits != 0u)) continue;
      // this lane's 32 tokens as order values (0: not kept or not finite)
      uint32_t u[32];
      if (a.vec && (w + 1) * 32 <= a.V) {  // a whole word of tokens inside the row
        uint4 q[NV];
        const uint4* src = reinterpret_cast<const uint4*>(row + (size_t)w * 32 * ES);
#pragma unroll
        for (int v = 0; v < NV; ++v) q[v] = bits ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const uint32_t word = reinterpret_cast<const uint32_t*>(q)[j * ES / 4];
          float x;
          if constexpr (DT == SMP_F32) x = __uint_as_float(word);
          else {
            const unsigned short h = (unsigned short)((j & 1) ? (word >> 16) : (word & 0xffffu));
            x = DT == SMP_BF16 ? __bfloat162float(__ushort_as_bfloat16(h))
                               : __half2float(__ushort_as_half(h));
          }
          u[j] = (((bits >> j) & 1u) && x > -INFINITY && x < INFINITY)
                     ? (uint32_t)(order_key(x, 0) >> 32) : 0u;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x = ((bits >> j) & 1u) ? load_logit<DT>(row, w * 32 + j) : -INFINITY;
          u[j] = (x > -INFINITY && x < INFINITY) ? (uint32_t)(order_key(x, 0) >> 32) : 0u;
        }
      }
      // rounds: every lane offers its best token not yet offered; those above
      // the threshold are merged; until no lane has one above it
      uint32_t offered = 0u;
#pragma unroll 1
      while (true) {
        uint64_t thr = __shfl_sync(0xffffffffu, top, 31);
        const uint64_t tc = *reinterpret_cast<volatile unsigned long long*>(&tau);
        thr = tc > thr ? tc : thr;
        uint32_t bu = 0u;
        int bj = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const bool take = !((offered >> j) & 1u) && u[j] > bu;  // the earliest of equals
          bu = take ? u[j] : bu;
          bj = take ? j : bj;
        }
        const uint64_t k = bu ? (((uint64_t)bu << 32) | (uint64_t)(0xffffffffu - (uint32_t)(w * 32 + bj)))
                              : 0ull;
        const bool sub = k > thr;
        if (!__any_sync(0xffffffffu, sub)) break;
        if (sub) offered |= 1u << bj;
        top = warp_merge_top(top, sub ? k : 0ull, lane);
        if (lane == 31 && top) atomicMax(&tau, (unsigned long long)top);
      }
    }
  }
  wl[warp][lane] = top;
  __syncthreads();
  if (warp == 0) {
    uint64_t t = wl[0][lane];
#pragma unroll 1
    for (int w = 1; w < LWARPS; ++w) t = warp_merge_top(t, wl[w][lane], lane);
    cl[lane] = t;
  }
  cluster.sync();
  if (rank == 0 && warp == 0) {
    uint64_t t = cl[lane];
#pragma unroll 1
    for (int c = 1; c < a.nc; ++c) t = warp_merge_top(t, *cluster.map_shared_rank(&cl[lane], c), lane);
    if (lane < a.n) {
      int32_t* oid = a.out_ids + (size_t)r * a.n;
      float* olp = a.out_lp + (size_t)r * a.n;
      if (!live) {
        oid[lane] = -1;
        olp[lane] = __int_as_float(0x7fffffff);
      } else if (t == 0ull) {
        oid[lane] = -1;
        olp[lane] = -INFINITY;
      } else {
        const int id = key_id(t);
        const float x = key_value(t);
        const float T = a.temperature[r];
        const int tok = a.tokens[r];
        const float lpt = a.logprobs[r];
        float lp;
        if (T == 0.f) {
          lp = (id == tok) ? 0.f : -INFINITY;  // the kept set is {argmax}
        } else {
          const float zt = __fdiv_rn(load_logit<DT>(row, tok), T);
          lp = fminf(__fadd_rn(lpt, __fsub_rn(__fdiv_rn(x, T), zt)), 0.f);
        }
        oid[lane] = id;
        olp[lane] = lp;
      }
    }
  }
  cluster.sync();
}

int toplp_enqueue(const void* logits, int dtype, int B, int V, long long ld, const uint32_t* kept,
                  const float* temperature, const int32_t* tokens, const float* logprobs, int n,
                  int32_t* out_ids, float* out_lp, cudaStream_t st) {
  if (n < 1 || n > LMAXN) return SMP_ERR_CAPACITY;
  if (B == 0) return SMP_OK;
  TopArgs a;
  a.logits = logits;
  a.ld = ld;
  a.kept = kept;
  a.temperature = temperature;
  a.tokens = tokens;
  a.logprobs = logprobs;
  a.out_ids = out_ids;
  a.out_lp = out_lp;
  a.B = B;
  a.V = V;
  a.W = (V + 31) / 32;
  a.n = n;
  int nc = (V + 8191) / 8192;
  nc = nc < 1 ? 1 : (nc > LMAXC ? LMAXC : nc);
  a.nc = nc;
  a.seg = ((V + nc * 32 - 1) / (nc * 32)) * 32;
  const size_t es = dtype == SMP_F32 ? 4 : 2;
  a.vec = ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && ((size_t)ld * es) % 16 == 0) ? 1 : 0;
  if ((long long)B * nc > 0x7fffffffLL) return SMP_ERR_CAPACITY;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * nc));
  cfg.blockDim = dim3(LT);
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
    case SMP_F32: e = cudaLaunchKernelEx(&cfg, toplp_kernel<SMP_F32>, a); break;
    case SMP_BF16: e = cudaLaunchKernelEx(&cfg, toplp_kernel<SMP_BF16>, a); break;
    default: e = cudaLaunchKernelEx(&cfg, toplp_kernel<SMP_F16>, a); break;
  }
  return e == cudaSuccess ? SMP_OK : SMP_ERR_CUDA;
}

}  // namespace smp
