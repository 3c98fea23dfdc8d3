// The row-wise top-k kernel and the fused path's planner.
#include <cuda_runtime.h>

#include "launch.h"
#include "plan_kernel.cuh"
#include "topk_kernel.cuh"

namespace dsa {

cudaError_t launch_topk_rows(int grid, size_t smem, cudaStream_t stream, const TopkParams& p) {
  cudaError_t e =
      cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  topk_rows_kernel<<<grid, kTopkThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_plan(cudaStream_t stream, const PlanArgs& a) {
  const size_t smem = a.stage_windows ? static_cast<size_t>(a.T) * sizeof(int2) : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  plan_kernel<<<1, kPlanThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
