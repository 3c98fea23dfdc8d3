// Exact, deterministic top-k selection by radix select on order-preserving uint32 keys,
// executed cooperatively by a group of NT threads (a whole CTA, or one epilogue warpgroup).
//
// Method (TileLang README, "Top-k Selector"): histogram the most significant 8 bits of every
// key, find the bin that holds the k-th largest key from the cumulative counts, then refine
// that bin with the next 8 bits, and so on.  Here the key is the full 32-bit image of the fp32
// score (score_key), so at most 4 passes (one 8-bit pass and up to 3 refinements) pin the exact
// k-th key.  A pass stops the descent early when the whole threshold bin is taken.
//
// The result is expressed as (prefix, shift, take_eq): a key u is selected iff
//     (u >> shift) > prefix,  or  (u >> shift) == prefix and it is among the first take_eq such
//     keys in ascending key-index order.
// That is exactly "larger score first, then lower key index".  The emit step walks the keys in
// ascending index order and compacts the selected ones with a group-wide prefix scan, so the
// output is in ascending key order and independent of thread scheduling (the page's version
// appends with atomics, whose order is not deterministic).
//
// A Source describes the keys as an ordered list of segments (segment s holds seg_len(s) keys;
// the keys of all segments, in order, are in ascending key-index order):
//   int segments() const;  int seg_len(int s) const;
//   uint32_t key(int s, int i) const;  int32_t index(int s, int i) const;
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"
#include "types.cuh"

namespace dsa {

template <int NT>
__device__ __forceinline__ void group_sync(int bar_id) {
  named_bar_sync(bar_id, NT);
}

// Exclusive prefix sum of v over the NT threads of the group (thread order = gtid).
// Returns the exclusive sum; *total receives the group total.
template <int NT>
__device__ __forceinline__ uint32_t group_excl_scan(uint32_t v, int gtid, SelectScratch* sc, int bar_id,
                                                    uint32_t* total) {
  constexpr int kWarps = NT / 32;
  const int lane = gtid & 31, warp = gtid >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    uint32_t t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) sc->warp_tot[warp] = incl;
  group_sync<NT>(bar_id);
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    uint32_t x = sc->warp_tot[w];
    if (w < warp) before += x;
    tot += x;
  }
  group_sync<NT>(bar_id);  // warp_tot may be rewritten by the next scan
  *total = tot;
  return before + incl - v;
}

// One histogram pass: counts, for every key whose bits above `shift + 8` equal `prefix`, the
// 8-bit digit at `shift`.  `first` = the most significant digit (no prefix condition).
template <int NT, class Src>
__device__ __forceinline__ void histogram_pass(const Src& src, int gtid, SelectScratch* sc, bool first,
                                               uint32_t prefix, int shift) {
  const int lane = gtid & 31;
  const int nseg = src.segments();
  for (int s = 0; s < nseg; ++s) {
    const int len = src.seg_len(s);
    for (int i0 = 0; i0 < len; i0 += NT) {
      const int i = i0 + gtid;
      uint32_t bin = 256;
      if (i < len) {
        const uint32_t u = src.key(s, i);
        if (first || (u >> (shift + 8)) == prefix) bin = (u >> shift) & 0xFFu;
      }
      if (first) {
        // warp-aggregated: the top digit concentrates in few bins (sign and high exponent bits)
        const unsigned m = __match_any_sync(0xffffffffu, bin);
        if (bin < 256 && lane == __ffs(m) - 1) atomicAdd(&sc->hist[bin], static_cast<uint32_t>(__popc(m)));
      } else if (bin < 256) {
        atomicAdd(&sc->hist[bin], 1u);
      }
    }
  }
}

// Finds the bin holding the k_rem-th largest counted key (warp 0 of the group) and broadcasts
// (bin, count strictly above it, count in it) through sc->bcast.
template <int NT>
__device__ __forceinline__ void find_threshold_bin(int gtid, SelectScratch* sc, int k_rem) {
  if (gtid < 32) {
    const int lane = gtid;
    uint32_t c[8];
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = sc->hist[8 * lane + j];
      sum += c[j];
    }
    uint32_t incl = sum;  // suffix sum over lanes >= lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      uint32_t t = __shfl_down_sync(0xffffffffu, incl, off);
      if (lane + off < 32) incl += t;
    }
    uint32_t above = incl - sum;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (above < static_cast<uint32_t>(k_rem) && above + c[j] >= static_cast<uint32_t>(k_rem)) {
        sc->bcast[0] = 8 * lane + j;
        sc->bcast[1] = static_cast<int>(above);
        sc->bcast[2] = static_cast<int>(c[j]);
      }
      above += c[j];
    }
  }
}

// Radix select of the k largest of n keys.  If hist_ready, sc->hist already holds the
// most-significant-digit histogram of all n keys (built while loading them).
template <int NT, class Src>
__device__ SelectResult group_select(const Src& src, int n, int k, int gtid, SelectScratch* sc, int bar_id,
                                     bool hist_ready) {
  SelectResult r;
  if (n <= k) {
    r.prefix = 0;
    r.shift = 0;
    r.take_eq = 0;
    r.all = 1;
    return r;
  }
  r.all = 0;
  uint32_t prefix = 0;
  int k_rem = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (!(pass == 0 && hist_ready)) {
      for (int b = gtid; b < 256; b += NT) sc->hist[b] = 0;
      group_sync<NT>(bar_id);
      histogram_pass<NT>(src, gtid, sc, pass == 0, prefix, shift);
    }
    group_sync<NT>(bar_id);
    find_threshold_bin<NT>(gtid, sc, k_rem);
    group_sync<NT>(bar_id);
    const int bin = sc->bcast[0];
    const int above = sc->bcast[1];
    const int in_bin = sc->bcast[2];
    group_sync<NT>(bar_id);  // bcast / hist are reused by the next pass
    k_rem -= above;
    prefix = (pass == 0) ? static_cast<uint32_t>(bin) : ((prefix << 8) | static_cast<uint32_t>(bin));
    if (in_bin == k_rem || shift == 0) {
      r.prefix = prefix;
      r.shift = shift;
      r.take_eq = k_rem;
      return r;
    }
  }
  r.prefix = prefix;  // not reached
  r.shift = 0;
  r.take_eq = k_rem;
  return r;
}

// Walks the keys in order and calls out(pos, s, i) for every selected key, pos being its rank
// in ascending key-index order.  Returns the number of selected keys (min(n, k)).
template <int NT, int V, class Src, class Out>
__device__ int group_emit(const Src& src, const SelectResult& r, int gtid, SelectScratch* sc, int bar_id,
                          Out&& out) {
  uint32_t gt_run = 0, eq_run = 0;
  const int nseg = src.segments();
  for (int s = 0; s < nseg; ++s) {
    const int len = src.seg_len(s);
    for (int i0 = 0; i0 < len; i0 += NT * V) {
      const int ib = i0 + gtid * V;
      uint32_t flags_gt = 0, flags_eq = 0;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int i = ib + v;
        if (i < len) {
          if (r.all) {
            flags_gt |= 1u << v;
          } else {
            const uint32_t kk = r.shift >= 32 ? 0u : (src.key(s, i) >> r.shift);
            if (kk > r.prefix) flags_gt |= 1u << v;
            else if (kk == r.prefix) flags_eq |= 1u << v;
          }
        }
      }
      const uint32_t packed = static_cast<uint32_t>(__popc(flags_gt)) | (static_cast<uint32_t>(__popc(flags_eq)) << 16);
      uint32_t total;
      const uint32_t before = group_excl_scan<NT>(packed, gtid, sc, bar_id, &total);
      uint32_t gt_pos = gt_run + (before & 0xFFFFu);
      uint32_t eq_rank = eq_run + (before >> 16);
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const bool gt = (flags_gt >> v) & 1u;
        const bool eq = (flags_eq >> v) & 1u;
        const uint32_t take = static_cast<uint32_t>(r.take_eq);
        if (gt) {
          out(static_cast<int>(gt_pos + (eq_rank < take ? eq_rank : take)), s, ib + v);
          ++gt_pos;
        } else if (eq) {
          if (eq_rank < take) out(static_cast<int>(gt_pos + eq_rank), s, ib + v);
          ++eq_rank;
        }
      }
      gt_run += total & 0xFFFFu;
      eq_run += total >> 16;
    }
  }
  const uint32_t take = static_cast<uint32_t>(r.take_eq);
  return static_cast<int>(gt_run + (eq_run < take ? eq_run : take));
}

}  // namespace dsa
