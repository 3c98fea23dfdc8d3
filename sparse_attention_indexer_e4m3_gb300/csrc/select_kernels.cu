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
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
