// smp_k_bf16.cu -- the sampling kernel instantiated for bf16 logits (one
// translation unit per element type, so the three compile in parallel).
#include "smp_kernel.cuh"

namespace smp {
const void* kernel_bf16() { return reinterpret_cast<const void*>(&smp_kernel<DT_BF16>); }
cudaError_t launch_bf16(const KArgs& a, int grid, cudaStream_t st) {
  smp_kernel<DT_BF16><<<grid, NT, SMEM_TOTAL, st>>>(a);
  return cudaGetLastError();
}
}  // namespace smp
