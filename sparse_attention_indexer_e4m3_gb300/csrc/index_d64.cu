// Index kernels for D = 64 (64-byte rows, 64-byte TMA / MMA swizzle).
#include "index_launch.cuh"

namespace dsa {
cudaError_t launch_index_d64(int H, bool fused, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                             const CUtensorMap& qmap, const IndexParams& p) {
  return launch_index_for_d<64>(H, fused, grid, smem, stream, kmap, qmap, p);
}
}  // namespace dsa
