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
// One cluster of up to 8 CTAs of 128 threads per row.  A warp keeps the 32
// best (logit descending, id ascending) kept tokens it has seen as 64-bit
// order keys, one per lane, sorted across the lanes; a batch of 32 new
// candidates is merged only when one of them beats the warp's 32nd best (a
// bitonic sort of the batch and a bitonic merge), which after the first
// steps is rare.  The warps' lists, then the CTAs' lists (through
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

  // this warp's slab of the CTA's segment, 32 elements per step
  uint64_t top = 0ull;
  if (live) {
    const int c0 = rank * a.seg, c1 = min(a.V, c0 + a.seg);
    const int per = (c1 - c0 + LWARPS - 1) / LWARPS;
    const int s0 = c0 + warp * per, s1 = min(c1, s0 + per);
#pragma unroll 1
    for (int i = s0; i < s1; i += 32) {
      const int id = i + lane;
      uint64_t k = 0ull;
      if (id < s1 && ((__ldg(km + (id >> 5)) >> (id & 31)) & 1u)) {
        const float x = load_logit<DT>(row, id);
        if (x > -INFINITY && x < INFINITY) k = order_key(x, id);
      }
      const uint64_t thr = __shfl_sync(0xffffffffu, top, 31);
      if (__any_sync(0xffffffffu, k > thr)) top = warp_merge_top(top, k, lane);
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
