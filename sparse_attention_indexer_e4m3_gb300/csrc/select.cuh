// Exact, deterministic top-k selection by radix select on order-preserving uint32 keys,
// executed cooperatively by a group of NT threads (a whole CTA, or one epilogue group of 4 warps).
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
// ascending index order and compacts the selected ones with prefix sums, so the output is in
// ascending key order and independent of thread scheduling (the page's version appends with
// atomics, whose order is not deterministic).
//
// Sources.  A single-row source in shared memory (RowKeys) is read 16 bytes at a time; any
// other source provides the ordered-segment interface
//   int segments() const;  int seg_len(int s) const;
//   uint32_t key(int s, int i) const;  int32_t index(int s, int i) const;
// (the keys of all segments, in order, are in ascending key-index order).
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

// One row of keys in shared memory: key i (0 <= i < n) is base[lead + i]; base is 16-byte
// aligned; the key's index is index0 + i.
struct RowKeys {
  const uint32_t* base;
  int lead;
  int n;
  int index0;
  __device__ __forceinline__ int segments() const { return 1; }
  __device__ __forceinline__ int seg_len(int) const { return n; }
  __device__ __forceinline__ uint32_t key(int, int i) const { return base[lead + i]; }
  __device__ __forceinline__ int32_t index(int, int i) const { return index0 + i; }
};

template <class Src>
struct IsRowKeys {
  static constexpr bool value = false;
};
template <>
struct IsRowKeys<RowKeys> {
  static constexpr bool value = true;
};

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

__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t u, bool first, uint32_t prefix, int shift) {
  if (first || (u >> (shift + 8)) == prefix) atomicAdd(&hist[(u >> shift) & 0xFFu], 1u);
}

// One histogram pass: counts, for every key whose bits above `shift + 8` equal `prefix`, the
// 8-bit digit at `shift`.  `first` = the most significant digit (no prefix condition).
template <int NT, class Src>
__device__ __forceinline__ void histogram_pass(const Src& src, int gtid, uint32_t* hist, bool first, uint32_t prefix,
                                               int shift) {
  if constexpr (IsRowKeys<Src>::value) {
    // 16-byte loads over the aligned span that covers [lead, lead + n)
    const int a0 = src.lead & ~3;
    const int end = src.lead + src.n;
    for (int j = a0 + 4 * gtid; j < end; j += 4 * NT) {
      const uint4 v = *reinterpret_cast<const uint4*>(src.base + j);
      const uint32_t e[4] = {v.x, v.y, v.z, v.w};
      if (first) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = j + q;
          const uint32_t bin = (i >= src.lead && i < end) ? (e[q] >> 24) : 256u;
          if (bin < 256) atomicAdd(&hist[bin], 1u);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = j + q;
          if (i >= src.lead && i < end) hist_add(hist, e[q], false, prefix, shift);
        }
      }
    }
  } else {
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
        if (bin < 256) atomicAdd(&hist[bin], 1u);
      }
    }
  }
}

// Finds the bin holding the k_rem-th largest counted key (warp 0 of the group) and broadcasts
// (bin, count strictly above it, count in it) through sc->bcast.
__device__ __forceinline__ void find_threshold_bin(int gtid, const uint32_t* hist, SelectScratch* sc, int k_rem) {
  if (gtid < 32) {
    const int lane = gtid;
    uint32_t c[8];
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[8 * lane + j];
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

// Radix select of the k largest of n keys.  hist0, if not null, already holds the
// most-significant-digit histogram of exactly these n keys (built while they were produced).
template <int NT, class Src>
__device__ SelectResult group_select(const Src& src, int n, int k, int gtid, SelectScratch* sc, int bar_id,
                                     const uint32_t* hist0) {
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
    const uint32_t* hist = sc->hist;
    if (pass == 0 && hist0 != nullptr) {
      hist = hist0;
    } else {
      for (int b = gtid; b < 256; b += NT) sc->hist[b] = 0;
      group_sync<NT>(bar_id);
      histogram_pass<NT>(src, gtid, sc->hist, pass == 0, prefix, shift);
    }
    group_sync<NT>(bar_id);
    find_threshold_bin(gtid, hist, sc, k_rem);
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

// Ordered emit for a single-row source: calls out(pos, i) for every selected key i (pos = its
// rank in ascending key-index order).  Each warp of the group owns one contiguous quarter (or
// 1/W-th) of the row: a counting sweep gives every warp its starting ranks (one group barrier),
// then a second sweep ranks its keys with warp shuffles only.  Returns min(n, k).
template <int NT, class Src, class Out>
__device__ int group_emit_row(const Src& src, const SelectResult& r, int gtid, SelectScratch* sc, int bar_id,
                              Out&& out) {
  constexpr int W = NT / 32;
  constexpr int V = 4;
  const int n = src.seg_len(0);
  if (r.all) {
    for (int i = gtid; i < n; i += NT) out(i, i);
    return n;
  }
  const int lane = gtid & 31, warp = gtid >> 5;
  const int span = 32 * V;
  const int chunk = ((n + W - 1) / W + span - 1) / span * span;
  const int beg = min(n, warp * chunk);
  const int end = min(n, beg + chunk);
  auto flags = [&](int i0, uint32_t& fgt, uint32_t& feq) {
    fgt = feq = 0;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int i = i0 + lane * V + v;
      if (i < end) {
        const uint32_t kk = src.key(0, i) >> r.shift;
        if (kk > r.prefix) fgt |= 1u << v;
        else if (kk == r.prefix) feq |= 1u << v;
      }
    }
  };
  // sweep 1: this warp's counts
  uint32_t cgt = 0, ceq = 0;
  for (int i0 = beg; i0 < end; i0 += span) {
    uint32_t fgt, feq;
    flags(i0, fgt, feq);
    cgt += __popc(fgt);
    ceq += __popc(feq);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    cgt += __shfl_xor_sync(0xffffffffu, cgt, off);
    ceq += __shfl_xor_sync(0xffffffffu, ceq, off);
  }
  if (lane == 0) {
    sc->warp_tot[warp] = cgt;
    sc->warp_eq[warp] = ceq;
  }
  group_sync<NT>(bar_id);
  uint32_t gt_run = 0, eq_run = 0, gt_all = 0, eq_all = 0;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    const uint32_t a = sc->warp_tot[w], b = sc->warp_eq[w];
    if (w < warp) {
      gt_run += a;
      eq_run += b;
    }
    gt_all += a;
    eq_all += b;
  }
  group_sync<NT>(bar_id);  // warp_tot / warp_eq are reused by the next call
  // sweep 2: ranks inside the warp by shuffles
  const uint32_t take = static_cast<uint32_t>(r.take_eq);
  for (int i0 = beg; i0 < end; i0 += span) {
    uint32_t fgt, feq;
    flags(i0, fgt, feq);
    const uint32_t packed = static_cast<uint32_t>(__popc(fgt)) | (static_cast<uint32_t>(__popc(feq)) << 16);
    uint32_t incl = packed;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
    const uint32_t ex = incl - packed;
    uint32_t gpos = gt_run + (ex & 0xFFFFu);
    uint32_t erank = eq_run + (ex >> 16);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int i = i0 + lane * V + v;
      if ((fgt >> v) & 1u) {
        out(static_cast<int>(gpos + (erank < take ? erank : take)), i);
        ++gpos;
      } else if ((feq >> v) & 1u) {
        if (erank < take) out(static_cast<int>(gpos + erank), i);
        ++erank;
      }
    }
    gt_run += tot & 0xFFFFu;
    eq_run += tot >> 16;
  }
  return static_cast<int>(gt_all + (eq_all < take ? eq_all : take));
}

// Bitmap -> ordered output: bit i of bitmap[0 .. ceil(n/32)) marks key i as selected.  Each
// warp takes a contiguous run of words; a group scan of the warps' popcounts gives their
// starting ranks; inside a word, lane l writes key 32w + l at its rank among the word's set
// bits, so every store instruction covers consecutive output positions.  Calls out(pos, i) for
// pos < limit.  Returns min(number of set bits, limit).
template <int NT, class Out>
__device__ __forceinline__ int emit_bitmap(const uint32_t* bitmap, int n, int limit, int gtid, SelectScratch* sc,
                                           int bar_id, Out&& out) {
  constexpr int W = NT / 32;
  const int lane = gtid & 31, warp = gtid >> 5;
  const int words = (n + 31) >> 5;
  const int wpw = (words + W - 1) / W;
  const int w0 = min(words, warp * wpw), w1 = min(words, w0 + wpw);
  uint32_t cnt = 0;
  for (int w = w0 + lane; w < w1; w += 32) cnt += __popc(bitmap[w]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
  if (lane == 0) sc->warp_tot[warp] = cnt;
  group_sync<NT>(bar_id);
  uint32_t pos = 0, total = 0;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    const uint32_t x = sc->warp_tot[w];
    if (w < warp) pos += x;
    total += x;
  }
  group_sync<NT>(bar_id);  // warp_tot is reused by the next call
  const uint32_t below = (1u << lane) - 1u;
  for (int w = w0; w < w1; w += 8) {
    uint32_t b[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) b[q] = (w + q < w1) ? bitmap[w + q] : 0u;
    uint32_t r[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      r[q] = pos + __popc(b[q] & below);
      pos += __popc(b[q]);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const bool take = ((b[q] >> lane) & 1u) && r[q] < static_cast<uint32_t>(limit);  // never past the row
      if (take) out(static_cast<int>(r[q]), 32 * (w + q) + lane);
    }
  }
  return min(static_cast<int>(total), limit);
}

// Exact top-k of one row in shared memory, in two sweeps over the row (TileLang README, "Top-k
// Selector": an 8-bit histogram, then refinement of the threshold bin).
//   hist0   the 256-bin histogram of the keys' digit at bits [shift0, shift0 + 8), already built
//           (while the scores were produced, or while candidate lists were staged): it gives the
//           threshold bin without reading the row.  Every key's bits above shift0 + 8 equal
//           prefix0 (shift0 = 24 and prefix0 = 0 for the plain top-byte histogram; a larger
//           common prefix lets a row of close keys start at a digit where they differ);
//   sweep 1 while the threshold bin holds more than kCandCap keys, histograms the next 8 bits
//           of the keys in it (fewer at the bottom) -> a narrower threshold bin;
//   sweep 2 records every key above the threshold bin as selected (one ballot per 32 keys into
//           a bitmap) and collects the keys inside it (at most kCandCap);
// the collected keys are ranked exactly under (larger score, then lower index) and the best
// k_rem of them are added to the bitmap, which is then emitted in key order.  If more than
// kCandCap keys equal the threshold key itself, the general radix select runs instead.
// Calls out(pos, i) for every selected key i; returns min(n, k).
template <int NT, class Out>
__device__ int row_topk(const RowKeys& src, int k, uint32_t* hist0, int shift0, uint32_t prefix0, uint32_t* bitmap,
                        int gtid, SelectScratch* sc, int bar_id, Out&& out) {
  constexpr int W = NT / 32;
  const int n = src.n;
  if (n <= k) {
    for (int i = gtid; i < n; i += NT) out(i, i);
    return n;
  }
  const int lane = gtid & 31, warp = gtid >> 5;
  const int words = (n + 31) >> 5;
  const uint32_t* keys = src.base + src.lead;
  // threshold bin of the first digit, from the prebuilt histogram
  find_threshold_bin(gtid, hist0, sc, k);
  group_sync<NT>(bar_id);
  uint32_t prefix = (prefix0 << 8) | static_cast<uint32_t>(sc->bcast[0]);  // threshold bin's top bits
  int shift = shift0;                                                      // ... are key >> shift
  int k_rem = k - sc->bcast[1];
  int in_bin = sc->bcast[2];
  if (gtid == 0) sc->cand_n = 0;  // sweep 2's candidate count
  group_sync<NT>(bar_id);
  bool take_bin = in_bin == k_rem;
  // sweep 1: while the threshold bin holds more keys than can be ranked one against another,
  // refine it by the next (up to) 8 bits, counted in the consumed first-digit histogram's array
  uint32_t* h1 = hist0;
  while (!take_bin && in_bin > kCandCap && shift > 0) {
    const int next = shift > 8 ? shift - 8 : 0;
    const uint32_t dmask = (1u << (shift - next)) - 1u;
    for (int b = gtid; b < 256; b += NT) h1[b] = 0u;
    group_sync<NT>(bar_id);
    // The 4-key vectors wholly inside [lead, lead + n) are swept without per-key bounds tests,
    // the next step's two loaded before this step's histogram atomics are issued (a load issued
    // after them would wait behind them in the shared-memory pipe); the at most 3 + 3 keys of
    // the partial vectors at the two ends are counted one per thread.
    const int end = src.lead + n;
    const int vbeg = (src.lead + 3) & ~3;
    const int vend = max(vbeg, end & ~3);
    auto count = [&](uint32_t e) {
      if ((e >> shift) == prefix) atomicAdd(&h1[(e >> next) & dmask], 1u);
    };
    auto load = [&](int j) {
      return j < vend ? *reinterpret_cast<const uint4*>(src.base + j) : make_uint4(0u, 0u, 0u, 0u);
    };
    auto count4 = [&](const uint4& v) {
      count(v.x);
      count(v.y);
      count(v.z);
      count(v.w);
    };
    uint4 v0 = load(vbeg + 4 * gtid), v1 = load(vbeg + 4 * gtid + 4 * NT);
    for (int j0 = vbeg + 4 * gtid; j0 < vend; j0 += 8 * NT) {
      const uint4 n0 = load(j0 + 8 * NT), n1 = load(j0 + 12 * NT);
      count4(v0);
      if (j0 + 4 * NT < vend) count4(v1);
      v0 = n0;
      v1 = n1;
    }
    if (gtid < 8) {
      const int i = gtid < 4 ? src.lead + gtid : vend + gtid - 4;
      if (i < (gtid < 4 ? min(vbeg, end) : end)) count(src.base[i]);
    }
    group_sync<NT>(bar_id);
    find_threshold_bin(gtid, h1, sc, k_rem);
    group_sync<NT>(bar_id);
    prefix = (prefix << (shift - next)) | static_cast<uint32_t>(sc->bcast[0]);
    shift = next;
    k_rem -= sc->bcast[1];
    in_bin = sc->bcast[2];
    group_sync<NT>(bar_id);
    take_bin = in_bin == k_rem;
  }
  if (!take_bin && in_bin > kCandCap) {
    // more than kCandCap keys equal the threshold key itself (exact ties, broken by index):
    // the general radix select (it rebuilds its own first digit)
    const SelectResult r = group_select<NT>(src, n, k, gtid, sc, bar_id, nullptr);
    return group_emit_row<NT>(src, r, gtid, sc, bar_id, [&](int q, int i) {
      if (q < k) out(q, i);  // never past the row
    });
  }
  // sweep 2: keys above the threshold bin -> bitmap; keys inside it -> candidates.  A warp takes
  // 8 consecutive words per step (8 independent loads in flight); a step that holds candidates
  // reserves their slots with one shared atomic (a warp-uniform branch, at most once per step).
  const uint32_t below = (1u << lane) - 1u;
  for (int w0 = 8 * warp; w0 < words; w0 += 8 * W) {
    uint32_t u[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 32 * (w0 + q) + lane;
      u[q] = i < n ? keys[i] : 0u;
    }
    uint32_t bq = 0, cm[8];
    int ctot = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 32 * (w0 + q) + lane;
      const bool valid = i < n;
      const uint32_t hi = u[q] >> shift;
      const uint32_t b = __ballot_sync(0xffffffffu, valid && hi > prefix);
      cm[q] = __ballot_sync(0xffffffffu, valid && hi == prefix);
      const uint32_t sel = take_bin ? (b | cm[q]) : b;
      bq = (lane == q) ? sel : bq;
      ctot += __popc(cm[q]);
    }
    if (lane < 8 && w0 + lane < words) bitmap[w0 + lane] = bq;
    if (!take_bin && ctot != 0) {  // warp-uniform
      int base = 0;
      if (lane == 0) base = atomicAdd(&sc->cand_n, ctot);
      base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int pos = base + __popc(cm[q] & below);
        if (((cm[q] >> lane) & 1u) && pos < kCandCap) {
          sc->cand_u[pos] = u[q];
          sc->cand_i[pos] = 32 * (w0 + q) + lane;
        }
        base += __popc(cm[q]);
      }
    }
  }
  group_sync<NT>(bar_id);
  if (!take_bin) {
    const int m = min(sc->cand_n, kCandCap);  // == in_bin <= kCandCap by construction
    // rank each candidate: it is selected iff fewer than k_rem candidates beat it
    for (int c = gtid; c < m; c += NT) {
      const uint32_t uc = sc->cand_u[c];
      const int ic = sc->cand_i[c];
      int rank = 0;
      for (int j = 0; j < m; ++j) {
        const uint32_t uj = sc->cand_u[j];
        const int ij = sc->cand_i[j];
        rank += (uj > uc || (uj == uc && ij < ic)) ? 1 : 0;
      }
      if (rank < k_rem) atomicOr(&bitmap[ic >> 5], 1u << (ic & 31));
    }
    group_sync<NT>(bar_id);
  }
  return emit_bitmap<NT>(bitmap, n, k, gtid, sc, bar_id, out);
}

// Ordered emit over a multi-segment source (candidate lists of several chunks): calls
// out(pos, s, i) for every selected key.  Uses a group-wide scan per NT * V keys.
template <int NT, int V, class Src, class Out>
__device__ int group_emit_segments(const Src& src, const SelectResult& r, int gtid, SelectScratch* sc, int bar_id,
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
            const uint32_t kk = src.key(s, i) >> r.shift;
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
      const uint32_t take = static_cast<uint32_t>(r.take_eq);
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const bool gt = (flags_gt >> v) & 1u;
        const bool eq = (flags_eq >> v) & 1u;
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
  return r.all ? static_cast<int>(gt_run) : static_cast<int>(gt_run + (eq_run < take ? eq_run : take));
}

}  // namespace dsa
