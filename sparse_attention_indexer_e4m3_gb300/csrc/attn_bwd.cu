// Gradients of the sparse attention: launcher (its own translation unit).
#include <cuda_runtime.h>

#include "attn_bwd_kernel.cuh"
#include "launch.h"

namespace dsa {

namespace {

static_assert(kTcAttnHeads == kTcMaxHeads, "head capacity of the tensor-core attention");

template <int D>
cudaError_t launch_attn_bwd_d(int grid, const AttnBwdParams& p, unsigned* err, cudaStream_t stream) {
  if (p.H < 1 || p.H > kTcMaxHeads || p.hs < p.H) return cudaErrorInvalidValue;
  constexpr int smem = TcBwdLayout<D>::kSmem;
  cudaError_t e =
      cudaFuncSetAttribute(sparse_attn_bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  sparse_attn_bwd_tc_kernel<D><<<grid, kTcAttnThreads, smem, stream>>>(p, err);
  return cudaGetLastError();
}

}  // namespace

int sparse_attn_bwd_tc_smem(int D) {
  switch (D) {
    case 128: return TcBwdLayout<128>::kSmem;
    case 256: return TcBwdLayout<256>::kSmem;
    default: return 0;
  }
}

cudaError_t launch_sparse_attn_bwd_tc(int D, int grid, const AttnBwdParams& p, unsigned* err, cudaStream_t stream) {
  switch (D) {
    case 128: return launch_attn_bwd_d<128>(grid, p, err, stream);
    case 256: return launch_attn_bwd_d<256>(grid, p, err, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
