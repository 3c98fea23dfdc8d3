// Work planner of the fused indexer + top-k path (one CTA, runs on the device so the host never
// reads ks / ke).
//
// 1. Tokens are taken in groups of `ntok_max` consecutive tokens (fewer when there are fewer
//    than ntok_max tokens per SM: down to T / SMs, so that every SM gets a unit).  A group whose
//    windows overlap strongly (causal prefill: twice the sum of window lengths is at least (nonempty + 1) times
//    the span of their union) becomes one or more units of consecutive tokens that are scored
//    together over the union of their windows (the key-range skip of the TileLang README,
//    "Lightning Indexer").  The unit size halves until the union fits the shared-memory row
//    buffer.  A group whose windows are (nearly) disjoint -- packed decode requests -- becomes one
//    unit per token, so no token's MMA columns are spent on another token's keys.  One pass over
//    the groups (a block-wide scan per 1024 groups) writes the units; when there are at least
//    `target_items` units and each fits its row buffer, every unit is one item and the plan is
//    complete.
// 2. Otherwise units are cut into chunks.  Fewer units than SMs (few, long rows): chunks of one
//    split length x (at least `cl_min` keys, just above the mean work per SM) plus one shorter
//    last chunk per unit, the x-long chunks listed first and the short ones after them, longest
//    first.  A unit longer than its row-buffer capacity (with enough units): chunks of equal
//    length (to a key tile), none over the capacity.  A cut unit's chunks write candidate lists
//    to workspace slots and the last chunk to finish merges them.
// 3. Otherwise items (unit, chunk) are listed from the last unit to the first: for causal prefill
//    the last tokens have the longest windows, so the longest items are scheduled first.
// Tokens with an empty window are listed; the run kernel writes their all -1 rows.  A plan
// depends only on (ks, ke, T, N, H, D, topk) and may be reused by any number of runs.
#pragma once

#include <climits>
#include <cstdint>

#include "common.cuh"
#include "index_kernel.cuh"
#include "types.cuh"

namespace dsa {

// Exclusive prefix sum over the 1024 threads of the CTA; *total gets the sum (every thread).
// sh holds 33 slots: the warps' sums are scanned by warp 0, and slot 32 receives the total.
__device__ __forceinline__ long long plan_scan(long long v, long long* sh, long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const long long x = sh[lane];
    long long wi = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += t;
    }
    sh[lane] = wi - x;
    if (lane == 31) sh[32] = wi;
  }
  __syncthreads();
  const long long before = sh[warp];
  *total = sh[32];
  __syncthreads();
  return before + incl - v;
}

// Records a token whose window is empty; the run kernel writes its all -1 output row.
__device__ __forceinline__ void note_empty(const PlanArgs& a, int* n_empty, int tok) {
  a.empty[atomicAdd(n_empty, 1)] = tok;
}

// Union of the non-empty clamped windows of tokens [t0, t1); returns false if all are empty.
template <class Win>
__device__ __forceinline__ bool window_union(const Win& win, int t0, int t1, int* lo, int* hi, long long* sum,
                                             int* nonempty) {
  int l = INT_MAX, h = INT_MIN, ne = 0;
  long long s = 0;
  for (int t = t0; t < t1; ++t) {
    const int2 wt = win(t);
    const int x = wt.x, e = wt.y;
    if (e > x) {
      l = min(l, x);
      h = max(h, e);
      s += e - x;
      ++ne;
    }
  }
  *lo = l;
  *hi = h;
  *sum = s;
  *nonempty = ne;
  return ne > 0;
}

__device__ __forceinline__ int unit_chunk_len(const PlanArgs& a, int ntok, long long cl_par) {
  long long cap = row_stride_keys(a.row_keys, ntok);
  if (cap < kKeysPerTile) cap = kKeysPerTile;
  long long cl = cl_par < cap ? cl_par : cap;
  cl = cl / kKeysPerTile * kKeysPerTile;
  if (cl < kKeysPerTile) cl = kKeysPerTile;
  return static_cast<int>(cl);
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanArgs a) {
  __shared__ long long sh[kPlanThreads / 32 + 1];
  __shared__ int n_empty;
  extern __shared__ int2 staged_windows[];
  // the run kernel may be scheduled now; it waits for this grid to finish before reading the plan
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Token groups of gsz tokens: ntok_max, or with few tokens (fewer than ntok_max per SM) the
  // power of two at most T / target_items, so that the grid gets about one unit per SM.
  int gsz = 1;
  while (2 * gsz <= a.ntok_max && 2LL * gsz * a.target_items <= a.T) gsz *= 2;
  if (a.T >= static_cast<long long>(a.ntok_max) * a.target_items) gsz = a.ntok_max;
  const int G = ceil_div(a.T, gsz);
  if (threadIdx.x == 0) n_empty = 0;
  // clamped windows, staged in shared memory when they fit (else read from global memory)
  if (a.stage_windows) {
    for (int t = threadIdx.x; t < a.T; t += kPlanThreads)
      staged_windows[t] = make_int2(clamp_key(a.ks[t], a.N), clamp_key(a.ke[t], a.N));
    __syncthreads();
  }
  auto win = [&](int t) -> int2 {
    if (a.stage_windows) return staged_windows[t];
    return make_int2(clamp_key(a.ks[t], a.N), clamp_key(a.ke[t], a.N));
  };

  // ---- 1. units, one pass over the groups: each group's unit count (grouped with a sub-unit
  //         size, or one unit per token), an exclusive scan for the unit ids, the unit records
  //         (as one chunk each); empty tokens are listed for their -1 rows
  long long carry = 0, r_local = 0;
  int over_cap = 0;  // a unit longer than its row buffer: it must be cut
  for (int g0 = 0; g0 < G; g0 += kPlanThreads) {
    const int g = g0 + threadIdx.x;
    const int t0 = g * gsz, t1 = min(a.T, t0 + gsz);
    int count = 0, ntu = 0;
    int glo = 0, ghi = 0;  // the group's window union
    if (g < G) {
      int lo, hi, ne;
      long long sum;
      window_union(win, t0, t1, &lo, &hi, &sum, &ne);
      glo = lo;
      ghi = hi;
      if (ne >= 2 && 2 * sum >= static_cast<long long>(ne + 1) * (hi - lo)) {
        ntu = gsz;
        while (ntu > 1 && (hi - lo) > row_stride_keys(a.row_keys, ntu)) ntu >>= 1;  // (the units' capacity)
        if (ntu == gsz) {
          count = 1;
        } else {
          for (int s0 = t0; s0 < t1; s0 += ntu) {
            int l2, h2, ne2;
            long long s2;
            if (window_union(win, s0, min(t1, s0 + ntu), &l2, &h2, &s2, &ne2)) ++count;
          }
        }
      } else {
        count = ne;
      }
    }
    long long tot;
    const long long base = carry + plan_scan(count, sh, &tot);
    if (g < G) {
      int u = static_cast<int>(base);
      auto put = [&](int tok, int ntok, int lo, int hi) {
        const int len = hi - lo;
        const int cl = (len + kKeysPerTile - 1) / kKeysPerTile * kKeysPerTile;
        if (u < a.max_units) a.units[u] = PlanUnit{tok, ntok, lo, hi, cl, 1, -1, 0};
        r_local += len;
        over_cap |= len > row_stride_keys(a.row_keys, ntok) ? 1 : 0;
        ++u;
      };
      if (ntu == gsz) {
        put(t0, t1 - t0, glo, ghi);  // the group is one unit (its union is non-empty)
      } else if (ntu > 0) {
        for (int s0 = t0; s0 < t1; s0 += ntu) {
          const int s1 = min(t1, s0 + ntu);
          int l2, h2, ne2;
          long long s2;
          if (window_union(win, s0, s1, &l2, &h2, &s2, &ne2)) {
            put(s0, s1 - s0, l2, h2);
          } else {
            for (int t = s0; t < s1; ++t) note_empty(a, &n_empty, t);
          }
        }
      } else {
        for (int t = t0; t < t1; ++t) {
          const int2 wt = win(t);
          if (wt.y > wt.x) {
            put(t, 1, wt.x, wt.y);
          } else {
            note_empty(a, &n_empty, t);
          }
        }
      }
    }
    carry += tot;
  }
  const int n_units = static_cast<int>(carry);
  if (n_units > a.max_units) {
    if (threadIdx.x == 0) {
      a.hdr->n_items = 0;
      a.hdr->n_units = 0;
      a.hdr->n_slots = 0;
      a.hdr->status = 1;
      a.hdr->n_empty = 0;
      a.hdr->next_item = 0;
      record_error(a.err, kErrPlan);
    }
    return;
  }
  const bool split = n_units < a.target_items || __syncthreads_or(over_cap) != 0;
  if (!split) {
    // ---- every unit is one item; items from the last unit to the first
    for (int u = threadIdx.x; u < n_units; u += kPlanThreads) a.items[n_units - 1 - u] = PlanItem{u, 0};
    __syncthreads();  // n_empty is final
    if (threadIdx.x == 0) {
      a.hdr->n_items = n_units;
      a.hdr->n_units = n_units;
      a.hdr->n_slots = 0;
      a.hdr->status = 0;
      a.hdr->n_empty = n_empty;
      a.hdr->next_item = 0;
    }
    return;
  }
  __syncthreads();  // unit records written by other threads are read below

  // ---- 2. chunk length: split only when the units alone cannot fill the machine, or when a
  //         unit exceeds its row-buffer capacity; grow the split length until the slots fit
  long long r_total;
  plan_scan(r_local, sh, &r_total);
  long long cl_par = LLONG_MAX / 4;
  // Few, long units: cut them into chunks of one split length x (a key-tile multiple just above
  // the mean work per SM, 1.05 x total / SMs) plus one shorter last chunk per unit.  The x-long
  // chunks are listed first and the last chunks after them, longest first, so the run kernel's
  // item queue (longest first, the next item to whichever SM is free) packs the short ones
  // around the long ones.
  const bool rem_mode = n_units < a.target_items;
  if (rem_mode) {
    constexpr long long kT = kKeysPerTile;
    const long long tiles = (r_total + kT - 1) / kT;
    long long x = (tiles * 21 + 20LL * a.target_items - 1) / (20LL * a.target_items);
    const long long x_min = (a.cl_min + kT - 1) / kT;
    cl_par = (x > x_min ? x : x_min) * kT;
  }
  long long slots_total = 0, items_total = 0;
  for (int attempt = 0; attempt < 40; ++attempt) {
    long long s_local = 0, i_local = 0;
    for (int u = threadIdx.x; u < n_units; u += kPlanThreads) {
      const PlanUnit un = a.units[u];
      const int cl = unit_chunk_len(a, un.ntok, cl_par);
      const long long nch = (un.hi - un.lo + cl - 1) / cl;
      i_local += nch;
      if (nch > 1) s_local += nch * un.ntok;
    }
    plan_scan(s_local, sh, &slots_total);
    plan_scan(i_local, sh, &items_total);
    if (slots_total <= a.max_slots && items_total <= a.max_items) break;
    if (cl_par >= LLONG_MAX / 8) break;
    cl_par *= 2;
  }
  if (slots_total > a.max_slots || items_total > a.max_items) {
    if (threadIdx.x == 0) {
      a.hdr->n_items = 0;
      a.hdr->n_units = n_units;
      a.hdr->n_slots = 0;
      a.hdr->status = 2;
      a.hdr->n_empty = 0;
      a.hdr->next_item = 0;
      record_error(a.err, kErrPlan);
    }
    return;
  }

  if (rem_mode) {
    // ---- 3'. (fewer units than SMs, so fewer than kPlanThreads: one unit per thread)
    const int u = threadIdx.x;
    PlanUnit un{};
    int cl = 0;
    long long nch = 0, full = 0, rem = 0;
    if (u < n_units) {
      un = a.units[u];
      cl = unit_chunk_len(a, un.ntok, cl_par);
      const long long len = un.hi - un.lo;
      nch = (len + cl - 1) / cl;
      full = len / cl;
      rem = len - full * cl;
    }
    // rank of this unit's short last chunk: longer ones first, ties by unit
    __shared__ int rem_s[kPlanThreads];
    if (u < n_units) rem_s[u] = static_cast<int>(rem);
    __syncthreads();
    int rank = 0;
    if (u < n_units && rem > 0) {
      for (int v = 0; v < n_units; ++v) {
        const int rv = rem_s[v];
        rank += (rv > rem || (rv == rem && v < u)) ? 1 : 0;
      }
    }
    long long full_tot, sl_tot;
    const long long fb = plan_scan(full, sh, &full_tot);
    const long long sb = plan_scan(nch > 1 ? nch * un.ntok : 0, sh, &sl_tot);  // (syncs: reads done)
    if (u < n_units) {
      un.chunk_len = cl;
      un.nchunks = static_cast<int>(nch);
      un.slot_base = nch > 1 ? static_cast<int>(sb) : -1;
      a.units[u] = un;
      for (long long c = 0; c < full; ++c) a.items[fb + c] = PlanItem{u, static_cast<int>(c)};
      if (rem > 0) a.items[full_tot + rank] = PlanItem{u, static_cast<int>(full)};
      if (nch > 1)
        for (int t = 0; t < un.ntok; ++t) a.counters[sb + static_cast<long long>(t) * nch] = 0u;
    }
    __syncthreads();  // n_empty is final
    if (threadIdx.x == 0) {
      a.hdr->n_items = static_cast<int>(items_total);
      a.hdr->n_units = n_units;
      a.hdr->n_slots = static_cast<int>(slots_total);
      a.hdr->status = 0;
      a.hdr->n_empty = n_empty;
      a.hdr->next_item = 0;
    }
    return;
  }

  // ---- 3. slot bases, items (last unit first), zeroed merge counters
  long long item_carry = 0, slot_carry = 0;
  for (int u0 = 0; u0 < n_units; u0 += kPlanThreads) {
    const int u = u0 + threadIdx.x;
    long long nch = 0, ns = 0;
    PlanUnit un{};
    int cl = 0;
    if (u < n_units) {
      un = a.units[u];
      cl = unit_chunk_len(a, un.ntok, cl_par);
      nch = (un.hi - un.lo + cl - 1) / cl;
      ns = nch > 1 ? nch * un.ntok : 0;
      // equal chunks: the same count, each a whole number of key tiles, none longer than cl
      const long long eq = (un.hi - un.lo + nch - 1) / nch;
      cl = static_cast<int>((eq + kKeysPerTile - 1) / kKeysPerTile * kKeysPerTile);
    }
    long long it_tot, sl_tot;
    const long long ib = item_carry + plan_scan(nch, sh, &it_tot);
    const long long sb = slot_carry + plan_scan(ns, sh, &sl_tot);
    if (u < n_units) {
      un.chunk_len = cl;
      un.nchunks = static_cast<int>(nch);
      un.slot_base = nch > 1 ? static_cast<int>(sb) : -1;
      a.units[u] = un;
      for (long long cidx = 0; cidx < nch; ++cidx) {
        const long long pos = items_total - 1 - (ib + cidx);
        a.items[pos] = PlanItem{u, static_cast<int>(cidx)};
      }
      if (nch > 1)
        for (int t = 0; t < un.ntok; ++t) a.counters[sb + static_cast<long long>(t) * nch] = 0u;
    }
    item_carry += it_tot;
    slot_carry += sl_tot;
  }
  if (threadIdx.x == 0) {
    a.hdr->n_items = static_cast<int>(items_total);
    a.hdr->n_units = n_units;
    a.hdr->n_slots = static_cast<int>(slots_total);
    a.hdr->status = 0;
    a.hdr->n_empty = n_empty;
    a.hdr->next_item = 0;
  }
}

}  // namespace dsa
