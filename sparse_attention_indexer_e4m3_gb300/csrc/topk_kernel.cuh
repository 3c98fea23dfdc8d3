// Row-wise exact top-k over a logits buffer (TileLang deepseek_v32 README, "Top-k Selector").
//
// One CTA of kTopkThreads threads per query row (grid-strided over rows).  The row's window is
// read once from HBM with coalesced loads; while it is read, each value is mapped to its
// order-preserving uint32 key, parked in shared memory, and counted in the most-significant-digit
// histogram, so the selection (row_topk: one refinement sweep, one selection sweep into a
// bitmap, and the ordered emit) runs out of shared memory.  Rows longer than the shared-memory
// cache run the general radix select re-reading global memory on every pass instead.
// Rows whose window holds at most k keys need no selection at all: the output is the window
// itself (ascending) followed by -1, and the logits are not read.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"
#include "select.cuh"
#include "types.cuh"

namespace dsa {

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
  uint32_t* bitmap = cache + ((p.cache_keys + 3) & ~3);  // one bit per cached key
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
          hist_add_warp(sc->hist, bin, lane);
        }
      }
      group_sync<kTopkThreads>(0);
      const RowKeys src{cache, 0, n, lo};
      row_topk<kTopkThreads>(src, p.topk, sc->hist, 24, 0u, bitmap, gtid, sc, 0, [&](int q, int j) { out[q] = lo + j; });
    } else {
      const GlobalKeys src{rp, n, lo};
      const SelectResult res = group_select<kTopkThreads>(src, n, p.topk, gtid, sc, 0, nullptr);
      group_emit_row<kTopkThreads>(src, res, gtid, sc, 0, [&](int q, int j) {
        if (q < p.topk) out[q] = lo + j;  // never past the row
      });
    }
    group_sync<kTopkThreads>(0);  // shared memory is reused by the next row
  }
}

}  // namespace dsa
