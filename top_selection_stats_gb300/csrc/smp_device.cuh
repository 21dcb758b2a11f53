// smp_device.cuh -- device helpers for the sampling kernels (sm_103a):
// mbarrier + bulk-TMA staging, thread-block-cluster exchange, order-preserving
// float keys, Philox4x32-10 and block-level reductions.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "smp_philox.cuh"

namespace smp {
namespace cg = cooperative_groups;

constexpr int NT = 256;           // threads per CTA
constexpr int NWARP = NT / 32;    // warps per CTA
constexpr int NBINS = 256;        // refinement histogram bins (one per thread)
constexpr int NCHUNK = 4;         // bulk-copy chunks per slice (one mbarrier each)
constexpr int MAX_CLUSTER = 16;   // CTAs per row, at most
constexpr int DTAB = 97;          // sigma-truncation table: log2(q) in [-24, 0], step 1/4
constexpr int NTHR = 4;           // sigma thresholds probed in one counting pass

enum Dtype { DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2 };
enum Mode { MODE_SAMPLE = 0, MODE_MASK = 1, MODE_ARGMAX = 2 };
enum Status { ST_OK = 0, ST_EMPTY = 1, ST_NONFINITE = 2, ST_INVALID = 3, ST_TIMEOUT = 4 };
enum Path { PATH_ERROR = 0, PATH_GREEDY = 1, PATH_ALL = 2, PATH_SIGMA = 3, PATH_FULL = 4 };

// --------------------------------------------------------------------------
// Order-preserving keys.  Finite floats map to uint32 so that unsigned order
// equals numeric order; -0 is folded onto +0 so that equal values share a key.
// Every legal finite value has a key >= 0x00800000; key 0 is never legal.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b << 1) == 0u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(b);
}

// --------------------------------------------------------------------------
// Shared-memory addressing, mbarriers and bulk copies (inline PTX).
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses (after a
// barrier: the block's) before bulk copies it issues next into the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// try_wait with a suspend-time hint: a thread whose phase is not complete is
// parked by the hardware (up to ~hint ns) instead of re-issuing the poll.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000u)
      : "memory");
  return ok != 0u;
}
// Bounded wait: gives up after `limit` SM clock cycles and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// 64-bit add into shared memory as two native 32-bit atomics: the low word's
// wrap-around (seen by exactly the add that caused it) carries into the high
// word, so after a barrier the pair reads as the exact 64-bit sum.  (A 64-bit
// shared atomicAdd is a compare-and-swap loop, which serialises badly when
// many lanes hit one bin.)
__device__ __forceinline__ void smem_add_u64(uint64_t* p, uint64_t v) {
  uint32_t* q = reinterpret_cast<uint32_t*>(p);
  const uint32_t lo = (uint32_t)v;
  const uint32_t hi = (uint32_t)(v >> 32);
  const uint32_t old = atomicAdd(q, lo);
  const uint32_t up = hi + ((old + lo < old) ? 1u : 0u);
  if (up) atomicAdd(q + 1, up);
}

// Fire-and-forget OR into global memory (a reduction: the issuing thread does
// not wait for the old value).
__device__ __forceinline__ void red_or_global(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.or.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// --------------------------------------------------------------------------
// The sampler's uniform: Philox4x32-10 (smp_philox.cuh) at key (lo32 seed,
// hi32 seed), counter (lo32 offset, hi32 offset, 0, 0); u = (word0 >> 8) *
// 2^-24 in [0, 1).
// --------------------------------------------------------------------------
__device__ __forceinline__ double philox_uniform(uint64_t seed, uint64_t offset) {
  uint32_t w[4];
  philox4x32_10(seed, (uint32_t)offset, (uint32_t)(offset >> 32), 0u, 0u, w);
  return (double)(w[0] >> 8) * (1.0 / 16777216.0);
}

// --------------------------------------------------------------------------
// Warp reductions and scans.
// --------------------------------------------------------------------------
template <class T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Inclusive warp scan (lane order).
template <class T>
__device__ __forceinline__ T warp_incl_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

}  // namespace smp
