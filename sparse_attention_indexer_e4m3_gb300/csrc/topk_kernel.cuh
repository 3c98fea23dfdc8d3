// Row-wise exact top-k over a logits buffer (TileLang deepseek_v32 README, "Top-k Selector").
//
// One CTA of kTopkThreads threads per query row (grid-strided over rows).  The row's window is
// read once from HBM with coalesced loads; while it is read, each value is mapped to its
// order-preserving uint32 key, parked in shared memory, and counted in the most-significant-digit
// histogram, so the remaining radix passes and the ordered emit run out of shared memory.  Rows
// longer than the shared-memory cache are re-read from global memory on every pass instead.
// Rows whose window holds at most k keys need no selection at all: the output is the window
// itself (ascending) followed by -1, and the logits are not read.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"
#include "select.cuh"
#include "types.cuh"

namespace dsa {

struct SmemKeys {
  const uint32_t* keys;
  int n;
  int base;
  __device__ __forceinline__ int segments() const { return 1; }
  __device__ __forceinline__ int seg_len(int) const { return n; }
  __device__ __forceinline__ uint32_t key(int, int i) const { return keys[i]; }
  __device__ __forceinline__ int32_t index(int, int i) const { return base + i; }
};

struct GlobalKeys {
  const float* row;  // logits of the window's first key
  int n;
  int base;
  __device__ __forceinline__ int segments() const { return 1; }
  __device__ __forceinline__ int seg_len(int) const { return n; }
  __device__ __forceinline__ uint32_t key(int, int i) const { return score_key(__ldg(row + i)); }
  __device__ __forceinline__ int32_t index(int, int i) const { return base + i; }
};

__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectScratch* sc = reinterpret_cast<SelectScratch*>(smem_raw);
  uint32_t* cache = reinterpret_cast<uint32_t*>(smem_raw + ((sizeof(SelectScratch) + 15) & ~size_t(15)));
  const int gtid = threadIdx.x;
  const int lane = gtid & 31;

  for (int row = blockIdx.x; row < p.T; row += gridDim.x) {
    const int lo = static_cast<int>(clamp_i64(p.ks[row], 0, p.N));
    const int hi = static_cast<int>(clamp_i64(p.ke[row], 0, p.N));
    const int n = hi > lo ? hi - lo : 0;
    int32_t* out = p.idx + static_cast<int64_t>(row) * p.topk;
    if (n <= p.topk) {
      for (int i = gtid; i < p.topk; i += kTopkThreads) out[i] = i < n ? lo + i : -1;
      continue;
    }
    const float* rp = p.logits + static_cast<int64_t>(row) * p.N + lo;
    if (n <= p.cache_keys) {
      for (int b = gtid; b < 256; b += kTopkThreads) sc->hist[b] = 0;
      group_sync<kTopkThreads>(0);
      // load + key map + top-digit histogram (warp-aggregated), 4 loads in flight per thread
      for (int i0 = 0; i0 < n; i0 += 4 * kTopkThreads) {
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * kTopkThreads + gtid;
          v[u] = i < n ? __ldg(rp + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * kTopkThreads + gtid;
          uint32_t bin = 256;
          if (i < n) {
            const uint32_t key = score_key(v[u]);
            cache[i] = key;
            bin = key >> 24;
          }
          const unsigned m = __match_any_sync(0xffffffffu, bin);
          if (bin < 256 && lane == __ffs(m) - 1) atomicAdd(&sc->hist[bin], static_cast<uint32_t>(__popc(m)));
        }
      }
      const SmemKeys src{cache, n, lo};
      const SelectResult res = group_select<kTopkThreads>(src, n, p.topk, gtid, sc, 0, true);
      group_emit<kTopkThreads, 4>(src, res, gtid, sc, 0, [&](int q, int s, int j) { out[q] = src.index(s, j); });
    } else {
      const GlobalKeys src{rp, n, lo};
      const SelectResult res = group_select<kTopkThreads>(src, n, p.topk, gtid, sc, 0, false);
      group_emit<kTopkThreads, 4>(src, res, gtid, sc, 0, [&](int q, int s, int j) { out[q] = src.index(s, j); });
    }
    group_sync<kTopkThreads>(0);  // shared memory is reused by the next row
  }
}

}  // namespace dsa
