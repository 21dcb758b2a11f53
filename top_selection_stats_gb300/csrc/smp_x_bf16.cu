// smp_x_bf16.cu -- the split-row streaming sampler (smp_split.cuh) instantiated
// for bf16 logits, with its cluster launch (one cluster of a.C CTAs per row).
#include "smp_split.cuh"

namespace smp {
const void* split_kernel_bf16() { return reinterpret_cast<const void*>(&split_kernel<DT_BF16>); }
cudaError_t split_launch_bf16(const XArgs& a, int smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * a.C), 1, 1);
  cfg.blockDim = dim3(XNT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_kernel<DT_BF16>, a);
}
}  // namespace smp
