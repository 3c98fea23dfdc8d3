// Index kernels for D = 128 (128-byte rows, 128-byte TMA / MMA swizzle).
#include "index_launch.cuh"

namespace dsa {
cudaError_t launch_index_d128(int H, bool fused, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                              const CUtensorMap& qmap, const IndexParams& p) {
  return launch_index_for_d<128>(H, fused, grid, smem, stream, kmap, qmap, p);
}
}  // namespace dsa
