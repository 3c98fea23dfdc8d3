// Row-wise exact top-k over a logits buffer (TileLang deepseek_v32 README, "Top-k Selector").
// Two kernels: topk_rows_stream_kernel (below) when every row fits a small CTA's shared-memory
// buffers, and topk_rows_kernel otherwise.
//
// topk_rows_kernel: one CTA of kTopkThreads threads per query row (grid-strided over rows).  The row's window is
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
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  SelectScratch* sc = reinterpret_cast<SelectScratch*>(smem_raw);
  uint32_t* cache = reinterpret_cast<uint32_t*>(smem_raw + ((sizeof(SelectScratch) + 15) & ~size_t(15)));
  uint32_t* bitmap = cache + ((p.cache_keys + 3) & ~3);  // one bit per cached key
  const int gtid = threadIdx.x;

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
      // load + key map + top-digit histogram, 4 loads in flight per thread
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
          if (i < n) {
            const uint32_t key = score_key(v[u]);
            cache[i] = key;
            atomicAdd(&sc->hist[key >> 24], 1u);
          }
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

// Streaming variant for rows of at most kTopkStreamMaxKeys keys: CTAs of kTopkStreamThreads
// threads with one row buffer each, as many per SM as shared memory allows (six at 8192 keys).
// Thread 0 brings a row in with a bulk copy of the 16-byte aligned interior of its window (the at
// most 3 + 3 keys outside it are read with plain loads), issuing the next row's copy as soon as
// the buffer is free; the copied logits are turned into keys in place, counting the top-digit
// histogram, and the 4-warp team selects.  The selection, not the HBM read, bounds this kernel,
// and small teams select more rows per SM at once (measured: six single-buffered CTAs per SM
// beat three double-buffered ones, whose next row's copy overlapped the selection, by 1.4x).
__global__ void __launch_bounds__(kTopkStreamThreads, 6) topk_rows_stream_kernel(const TopkParams p) {
  constexpr int NT = kTopkStreamThreads;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  SelectScratch* sc = reinterpret_cast<SelectScratch*>(smem_raw);
  const int bw = p.cache_keys + 8;  // row-buffer words
  // the row being selected (its window starts up to 3 words into the buffer), then its bitmap
  uint32_t* rb = reinterpret_cast<uint32_t*>(smem_raw + ((sizeof(SelectScratch) + 15) & ~size_t(15)));
  uint32_t* bitmap = rb + bw;  // one bit per key
  uint64_t* bar = reinterpret_cast<uint64_t*>(bitmap + (((p.cache_keys + 31) / 32 + 3) & ~3));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 1);
  const int tid = threadIdx.x;

  auto window = [&](int row, int& lo, int& n) {
    lo = static_cast<int>(clamp_i64(p.ks[row], 0, p.N));
    const int hi = static_cast<int>(clamp_i64(p.ke[row], 0, p.N));
    n = hi > lo ? hi - lo : 0;
  };
  auto staged = [&](int n) { return n > p.topk && n <= p.cache_keys; };
  // aligned interior [e0, e1) (element indices into logits) of a staged row's window
  auto interior = [&](int row, int lo, int n, int64_t& g0, int64_t& e0, int64_t& e1) {
    g0 = static_cast<int64_t>(row) * p.N + lo;
    e0 = (g0 + 3) & ~int64_t(3);
    e1 = (g0 + n) & ~int64_t(3);
  };
  uint32_t parity = 0u;  // phase parity to wait for next (every thread)
  bool pending = false;  // a copy issued and not waited for yet (thread 0)
  auto issue = [&](int row) {
    int lo, n;
    window(row, lo, n);
    if (!staged(n) || *abort_flag) return;  // after an expired wait no new copy is started
    int64_t g0, e0, e1;
    interior(row, lo, n, g0, e0, e1);
    if (e1 > e0) {
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>((e1 - e0) * 4));
      bulk_load_1d(rb + (e0 - (g0 & ~int64_t(3))), p.logits + e0, static_cast<uint32_t>((e1 - e0) * 4), bar);
    } else {
      mbar_arrive(bar);  // no aligned interior: complete the phase without a copy
    }
    pending = true;
  };

  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0 && static_cast<int>(blockIdx.x) < p.T) issue(blockIdx.x);

  for (int row = blockIdx.x; row < p.T; row += gridDim.x) {
    int lo, n;
    window(row, lo, n);
    int32_t* out = p.idx + static_cast<int64_t>(row) * p.topk;
    if (n <= p.topk) {
      for (int i = tid; i < p.topk; i += NT) out[i] = i < n ? lo + i : -1;
    } else if (n <= p.cache_keys) {
      for (int i = tid; i < 256; i += NT) sc->hist[i] = 0u;
      if (mbar_wait(bar, parity, abort_flag, p.err, 0x40)) {
        parity ^= 1u;
        pending = false;
      }
      int64_t g0, e0, e1;
      interior(row, lo, n, g0, e0, e1);
      const int lead = static_cast<int>(g0 & 3);
      // the keys outside the copied interior: at most 3 before it and 3 after it
      const int head = static_cast<int>(min(static_cast<int64_t>(n), e0 - g0));
      const int tail0 = static_cast<int>(max(e1, e0) - g0);
      if (tid < 4 && tid < head) rb[lead + tid] = __float_as_uint(__ldg(p.logits + g0 + tid));
      if (tid >= 4 && tid < 8 && tail0 + tid - 4 < n)
        rb[lead + tail0 + tid - 4] = __float_as_uint(__ldg(p.logits + g0 + tail0 + tid - 4));
      __syncthreads();
      if (!*abort_flag) {  // (read after the barrier: the same decision in every thread)
        // logits -> keys in place, with the top-digit histogram: the 4-key vectors wholly inside
        // the window without per-key bounds tests, two in flight per thread, then the at most two
        // partial vectors at its ends (the same vector when the window lies inside one)
        const int end = lead + n;
        const int vbeg = lead ? 4 : 0;  // first whole vector
        const int vend = end & ~3;      // end of the whole vectors
        auto convert4 = [&](uint4& v) {
          v.x = score_key(__uint_as_float(v.x));
          v.y = score_key(__uint_as_float(v.y));
          v.z = score_key(__uint_as_float(v.z));
          v.w = score_key(__uint_as_float(v.w));
          atomicAdd(&sc->hist[v.x >> 24], 1u);
          atomicAdd(&sc->hist[v.y >> 24], 1u);
          atomicAdd(&sc->hist[v.z >> 24], 1u);
          atomicAdd(&sc->hist[v.w >> 24], 1u);
        };
        for (int j = vbeg + 4 * tid; j < vend; j += 8 * NT) {
          const int j2 = j + 4 * NT;
          uint4 a = *reinterpret_cast<const uint4*>(rb + j);
          uint4 b = make_uint4(0u, 0u, 0u, 0u);
          if (j2 < vend) b = *reinterpret_cast<const uint4*>(rb + j2);
          convert4(a);
          *reinterpret_cast<uint4*>(rb + j) = a;
          if (j2 < vend) {
            convert4(b);
            *reinterpret_cast<uint4*>(rb + j2) = b;
          }
        }
        if (tid < 2) {
          const int j = tid == 0 ? 0 : vend;
          if (tid == 0 ? lead > 0 : (vend < end && vend >= vbeg)) {
            for (int q = 0; q < 4; ++q) {
              if (j + q >= lead && j + q < end) {
                const uint32_t e = score_key(__uint_as_float(rb[j + q]));
                rb[j + q] = e;
                atomicAdd(&sc->hist[e >> 24], 1u);
              }
            }
          }
        }
        __syncthreads();
        const RowKeys src{rb, lead, n, lo};
        row_topk<NT>(src, p.topk, sc->hist, 24, 0u, bitmap, tid, sc, 1, [&](int q, int j) { out[q] = lo + j; });
      }
    } else {
      const GlobalKeys src{p.logits + static_cast<int64_t>(row) * p.N + lo, n, lo};
      const SelectResult res = group_select<NT>(src, n, p.topk, tid, sc, 1, nullptr);
      group_emit_row<NT>(src, res, tid, sc, 1, [&](int q, int j) {
        if (q < p.topk) out[q] = lo + j;  // never past the row
      });
    }
    // this row's generic accesses to the buffer come before the bulk copy that reuses it
    fence_proxy_async_shared();
    __syncthreads();
    if (tid == 0 && row + static_cast<int>(gridDim.x) < p.T) issue(row + gridDim.x);
  }
  if (tid == 0 && pending) mbar_wait_drain(bar, parity);  // after an expired wait: let the copy land
}

}  // namespace dsa
