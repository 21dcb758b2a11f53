// smp_k_f16.cu -- the sampling kernel instantiated for f16 logits (one
// translation unit per element type, so the three compile in parallel).
#include "smp_kernel.cuh"

namespace smp {
const void* kernel_f16() { return reinterpret_cast<const void*>(&smp_kernel<DT_F16>); }
cudaError_t launch_f16(const KArgs& a, int grid, cudaStream_t st) {
  smp_kernel<DT_F16><<<grid, NT, SMEM_TOTAL, st>>>(a);
  return cudaGetLastError();
}
}  // namespace smp
