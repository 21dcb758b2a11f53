// smp_penalty.cu -- repetition penalty as an in-place logits processor
// ("Sampling system design" post, section on the repetition penalty: a
// state-dependent processor that reads the sequence's history tokens and
// lowers the logits of tokens already seen, placed before the sampler).  The
// post leaves the formula open; the rule here is CTRL's (Keskar et al. 2019):
// for every distinct token t of the row's history, x_t / theta if x_t > 0,
// else x_t * theta, in binary32 with correct rounding, stored back in the
// logits' format with round-to-nearest-even.
//
// One CTA per row.  Only the history's tokens are touched (a read and a write
// each), so the row itself is never streamed: the pass costs B * H index
// loads and at most B * H scattered element updates.  A token that appears
// several times in the history is penalised once: the CTA keeps a bitmap of
// the row's vocabulary in shared memory and the thread whose atomicOr sets a
// token's bit owns that token's update.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/smp.h"

namespace smp {

constexpr int PT = 256;                   // threads per CTA
constexpr int PEN_MAX_VOCAB = 1572864;    // bitmap of 49,152 words = 192 KB of shared memory
constexpr int PEN_SMEM_MAX = PEN_MAX_VOCAB / 32 * 4;

template <int DT>
__global__ void __launch_bounds__(PT) penalty_kernel(void* logits, int V, long long ld,
                                                     const int32_t* history, int H,
                                                     long long hld, const float* penalty,
                                                     int32_t* status) {
  extern __shared__ uint32_t seen[];
  const int r = blockIdx.x;
  const float th = penalty[r];
  const bool ok = th > 0.f && th < INFINITY;  // also rejects NaN
  if (threadIdx.x == 0) status[r] = ok ? SMP_OK : SMP_ERR_INVALID_PARAM;
  if (!ok) return;
  const int W = (V + 31) >> 5;
  for (int w = threadIdx.x; w < W; w += PT) seen[w] = 0u;
  __syncthreads();
  const int32_t* hrow = history + (size_t)r * (size_t)hld;
#pragma unroll 1
  for (int i = threadIdx.x; i < H; i += PT) {
    const int t = __ldg(hrow + i);
    if (t < 0 || t >= V) continue;  // padding
    const uint32_t bit = 1u << (t & 31);
    if (atomicOr(&seen[t >> 5], bit) & bit) continue;  // another entry owns this token
    const size_t at = (size_t)r * (size_t)ld + (size_t)t;
    if constexpr (DT == SMP_F32) {
      float* p = reinterpret_cast<float*>(logits) + at;
      const float x = *p;
      *p = (x > 0.f) ? __fdiv_rn(x, th) : __fmul_rn(x, th);
    } else if constexpr (DT == SMP_BF16) {
      __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(logits) + at;
      const float x = __bfloat162float(*p);
      *p = __float2bfloat16_rn((x > 0.f) ? __fdiv_rn(x, th) : __fmul_rn(x, th));
    } else {
      __half* p = reinterpret_cast<__half*>(logits) + at;
      const float x = __half2float(*p);
      *p = __float2half_rn((x > 0.f) ? __fdiv_rn(x, th) : __fmul_rn(x, th));
    }
  }
}

// Shared-memory limit of the three instantiations (once per device, from
// smp_create).
cudaError_t penalty_setup() {
  cudaError_t e = cudaFuncSetAttribute(penalty_kernel<SMP_F32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, PEN_SMEM_MAX);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(penalty_kernel<SMP_BF16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, PEN_SMEM_MAX);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(penalty_kernel<SMP_F16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, PEN_SMEM_MAX);
  return e;
}

int penalty_max_vocab() { return PEN_MAX_VOCAB; }

// Host side; arguments were checked by smp_repetition_penalty.  Returns
// SMP_OK, SMP_ERR_CAPACITY or SMP_ERR_CUDA.
int penalty_enqueue(void* logits, int dtype, int B, int V, long long ld, const int32_t* history,
                    int H, long long hld, const float* penalty, int32_t* status,
                    cudaStream_t st) {
  if (V > PEN_MAX_VOCAB) return SMP_ERR_CAPACITY;
  if (B == 0) return SMP_OK;
  const size_t smem = (size_t)((V + 31) / 32) * 4;
  switch (dtype) {
    case SMP_F32:
      penalty_kernel<SMP_F32><<<B, PT, smem, st>>>(logits, V, ld, history, H, hld, penalty,
                                                   status);
      break;
    case SMP_BF16:
      penalty_kernel<SMP_BF16><<<B, PT, smem, st>>>(logits, V, ld, history, H, hld, penalty,
                                                    status);
      break;
    default:
      penalty_kernel<SMP_F16><<<B, PT, smem, st>>>(logits, V, ld, history, H, hld, penalty,
                                                   status);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? SMP_OK : SMP_ERR_CUDA;
}

}  // namespace smp
