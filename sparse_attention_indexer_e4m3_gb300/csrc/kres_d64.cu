// K-resident scorer for D = 64 (64-byte rows, 64-byte TMA / MMA swizzle).
#include "kres_launch.cuh"

namespace dsa {
cudaError_t launch_kres_d64(int H, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                            const CUtensorMap& qmap, const KresParams& p, const int32_t* ks, const int32_t* ke) {
  return launch_kres_for_d<64>(H, grid, smem, stream, kmap, qmap, p, ks, ke);
}
}  // namespace dsa
