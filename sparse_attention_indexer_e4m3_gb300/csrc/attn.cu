// Sparse attention over the selected keys: launcher (its own translation unit, compiled in
// parallel with the others).
#include <cuda_runtime.h>

#include "attn_kernel.cuh"
#include "attn_tc_kernel.cuh"
#include "launch.h"

namespace dsa {

namespace {

template <int D>
cudaError_t launch_attn_d(const AttnParams& p, cudaStream_t stream) {
  const size_t smem = attn_smem_bytes(D);
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(p.T), static_cast<unsigned>((p.H + kAttnHeads - 1) / kAttnHeads));
  sparse_attn_kernel<D><<<grid, kAttnThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

static_assert(kTcAttnHeads == kTcMaxHeads, "head capacity of the tensor-core attention");

template <int D>
cudaError_t launch_attn_tc_d(int grid, const AttnParams& p, unsigned* err, cudaStream_t stream) {
  if (p.H < 1 || p.H > kTcMaxHeads || p.hs < p.H) return cudaErrorInvalidValue;
  constexpr int smem = TcAttnLayout<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  sparse_attn_tc_kernel<D><<<grid, kTcAttnThreads, smem, stream>>>(p, err);
  return cudaGetLastError();
}

}  // namespace

int sparse_attn_tc_smem(int D) {
  switch (D) {
    case 128: return TcAttnLayout<128>::kSmem;
    case 256: return TcAttnLayout<256>::kSmem;
    case 512: return TcAttnLayout<512>::kSmem;
    default: return 0;
  }
}

cudaError_t launch_sparse_attn_tc(int D, int grid, const AttnParams& p, unsigned* err, cudaStream_t stream) {
  switch (D) {
    case 128: return launch_attn_tc_d<128>(grid, p, err, stream);
    case 256: return launch_attn_tc_d<256>(grid, p, err, stream);
    case 512: return launch_attn_tc_d<512>(grid, p, err, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_sparse_attn(int D, const AttnParams& p, cudaStream_t stream) {
  switch (D) {
    case 64: return launch_attn_d<64>(p, stream);
    case 128: return launch_attn_d<128>(p, stream);
    case 256: return launch_attn_d<256>(p, stream);
    case 512: return launch_attn_d<512>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
