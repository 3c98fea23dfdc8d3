// The row-wise top-k kernels, the fused path's planner, the key quantiser and the bounded-wait
// self-check.
#include <cuda_runtime.h>

#include <algorithm>

#include "launch.h"
#include "plan_kernel.cuh"
#include "quant_kernel.cuh"
#include "topk_kernel.cuh"

namespace dsa {

cudaError_t launch_topk_rows(int grid, size_t smem, cudaStream_t stream, const TopkParams& p) {
  cudaError_t e =
      cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  topk_rows_kernel<<<grid, kTopkThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

// Self-check of the bounded wait that every pipeline wait of the library goes through.  Warp 0
// waits on an mbarrier that nothing ever arrives on: the wait must give up after kWaitLimitNs,
// record a timeout in the error word and raise the CTA's abort flag.  Warp 1 waits (bounded)
// for that flag and then starts a wait on a second such barrier, which must return at once
// without recording anything.  Each lane-0 writes how long its mbar_wait took (ns).
__global__ void wait_check_kernel(unsigned* err, unsigned long long* took_ns) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) != 0) return;
  if (warp == 0) {
    const uint64_t t0 = global_timer_ns();
    const bool done = mbar_wait(&bars[0], 0, abort_flag, err, kSiteWaitCheck);
    took_ns[0] = done ? 0ull : global_timer_ns() - t0;
  } else {
    const uint64_t t0 = global_timer_ns();
    while (!*abort_flag && global_timer_ns() - t0 < 2 * kWaitLimitNs) {
    }
    const uint64_t t1 = global_timer_ns();
    const bool done = mbar_wait(&bars[1], 0, abort_flag, err, kSiteWaitCheck + 1);
    took_ns[1] = done ? ~0ull : global_timer_ns() - t1;
  }
}

cudaError_t launch_wait_check(cudaStream_t stream, unsigned* err, unsigned long long* took_ns) {
  wait_check_kernel<<<1, 64, 0, stream>>>(err, took_ns);
  return cudaGetLastError();
}

cudaError_t launch_topk_stream(int max_grid, size_t smem, cudaStream_t stream, const TopkParams& p) {
  cudaError_t e = cudaFuncSetAttribute(topk_rows_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_rows_stream_kernel, kTopkStreamThreads, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int grid = std::max(1, std::min(max_grid, std::max(1, per_sm) * sms));
  topk_rows_stream_kernel<<<grid, kTopkStreamThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quantize(int D, const uint16_t* x, int64_t N, uint8_t* codes, float* scale, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t per_block = static_cast<int64_t>(kQuantThreads / 32) * kRowsPerWarp;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((N + per_block - 1) / per_block,
                                                                           16LL * sms)));
  if (D == 128) {
    quantize_rows_kernel<128><<<grid, kQuantThreads, 0, stream>>>(x, N, codes, scale);
  } else {
    quantize_rows_kernel<64><<<grid, kQuantThreads, 0, stream>>>(x, N, codes, scale);
  }
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
