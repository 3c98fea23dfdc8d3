// Instantiation and launch of the K-resident scorer for one head dimension D (included by the
// per-D translation units): the window pass, then the scorer as its programmatic dependent.
#pragma once

#include <cuda_runtime.h>

#include "kres_kernel.cuh"
#include "launch.h"

namespace dsa {

template <int H, int D>
cudaError_t launch_kres_one(int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                            const CUtensorMap& qmap, const KresParams& p) {
  auto kern = kres_kernel<H, D>;
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
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, kmap, qmap, p);
}

template <int D>
cudaError_t launch_kres_for_d(int H, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                              const CUtensorMap& qmap, const KresParams& p, const int32_t* ks, const int32_t* ke) {
  kres_windows_kernel<<<(p.nblocks + 255) / 256, 256, 0, stream>>>(
      ks, ke, p.T, p.N, p.ntok, p.nblocks, const_cast<int2*>(p.blk_win), const_cast<int2*>(p.tok_win), p.queue);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  switch (H) {
    case 4:
      return launch_kres_one<4, D>(grid, smem, stream, kmap, qmap, p);
    case 8:
      return launch_kres_one<8, D>(grid, smem, stream, kmap, qmap, p);
    case 16:
      return launch_kres_one<16, D>(grid, smem, stream, kmap, qmap, p);
    case 32:
      return launch_kres_one<32, D>(grid, smem, stream, kmap, qmap, p);
    case 64:
      return launch_kres_one<64, D>(grid, smem, stream, kmap, qmap, p);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
