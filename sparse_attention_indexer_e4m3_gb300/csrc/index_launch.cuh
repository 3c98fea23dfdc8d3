// Instantiation and launch of the index kernel for one head dimension D (included by the
// per-D translation units).
#pragma once

#include <cuda_runtime.h>

#include "index_kernel.cuh"
#include "launch.h"

namespace dsa {

// The fused kernel is launched as a programmatic dependent of the planner (it may start while
// the planner finishes and waits for it with griddepcontrol.wait before reading the plan).
template <int H, int D, bool FUSED>
cudaError_t launch_index_one(int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                             const CUtensorMap& qmap, const IndexParams& p) {
  auto kern = index_kernel<H, D, FUSED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kIndexThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = FUSED ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, kmap, qmap, p);
}

template <int D>
cudaError_t launch_index_for_d(int H, bool fused, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                               const CUtensorMap& qmap, const IndexParams& p) {
#define DSA_CASE(HH)                                                                    \
  case HH:                                                                              \
    return fused ? launch_index_one<HH, D, true>(grid, smem, stream, kmap, qmap, p)     \
                 : launch_index_one<HH, D, false>(grid, smem, stream, kmap, qmap, p);
  switch (H) {
    DSA_CASE(4)
    DSA_CASE(8)
    DSA_CASE(16)
    DSA_CASE(32)
    DSA_CASE(64)
    default:
      return cudaErrorInvalidValue;
  }
#undef DSA_CASE
}

}  // namespace dsa
