// The FP8 lightning-indexer kernel for sm_103a, in two modes sharing one pipeline:
//   SCORE  (FUSED = false): writes fp32 logits for every in-window (token, key) pair;
//   FUSED  (FUSED = true) : keeps each token's scores on chip and selects its top-k keys.
//
// What it computes (Modular "sparse_index_fp8_sm100_prefill", the per-(token, key) logit; TileLang
// deepseek_v32 README, "Lightning Indexer"):
//     score[t, j] = k_scale[j] * sum_h relu(q[t,h,:] . k[j,:]) * w[t,h],   ks[t] <= j < ke[t].
//
// Layout of the work (the Q-resident / K-streaming orientation of the Modular page, rebuilt for
// tcgen05): a work item owns a block of up to `ntok` consecutive query tokens and a contiguous key
// range.  The item's Q rows, [ntok * H, D] e4m3, stay in shared memory as the B operand; 128-key
// tiles of K, [128, D] e4m3, stream through a TMA ring as the A operand.  One tcgen05 MMA chain
// per tile computes S^T = K . Q^T = [128 keys, ntok * H columns] in fp32 in tensor memory, so
// thread i of an epilogue warp reads key row i and owns all of that key's (token, head) scores:
// relu, head weight and head sum need no cross-thread reduction.
//
// Roles (640 threads):
//   warps 0,2,3 TMA producers: warp 0 claims items and loads each item's Q block; the three
//               share the K tiles of the item's key range (stage st is filled by producer
//               st % 3).
//   warp 1      MMA issuer and tensor-memory owner (512 columns = 2 accumulator stages of 256).
//   warps 4-19  epilogue, four groups of 4 warps (one warp per 32-lane tensor-memory quarter);
//               group g reads accumulator columns [64g, 64g + 64) of each stage.
// A 256-column accumulator stage holds one key tile of an item whose ntok * H columns exceed
// 128; for narrower items it stacks 2 (<= 128 columns) or 4 (<= 64 columns, e.g. one decode
// token at H = 64) consecutive key tiles side by side, so all four groups have work.  The
// per-(key, token) arithmetic is the same in every layout.  In the fused mode the tokens of an
// item are then selected by teams of 128 * (tiles per stage) threads.
// Hand-offs use mbarriers: k_full / k_empty (K ring), q_full / q_empty (Q buffer),
// acc_full / acc_empty (tensor-memory accumulator stages).  Every wait is bounded.
//
// Key-range skip (TileLang README, "Lightning Indexer": only keys in [min ks, max ke) of a token
// block are processed): an item's key range is the union of its tokens' clamped windows, and
// per-token guards restrict what is written or ranked.
#pragma once

#include <cuda.h>

#include <climits>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"
#include "select.cuh"
#include "types.cuh"

namespace dsa {

struct ItemInfo {
  int tok0;
  int ntok;
  int k_lo;  // first key of the item
  int k_hi;  // one past the last key of the item
  int ntiles;
  int chunk;
  int nchunks;
  int slot_base;
};

__device__ __forceinline__ int clamp_key(int32_t x, int N) { return x < 0 ? 0 : (x > N ? N : x); }

// Row-buffer keys per token for an item of ntok tokens (a multiple of 128, so that per-token
// rows and their selection bitmaps stay 16-byte aligned).  The planner's chunk length never
// exceeds it.
__host__ __device__ __forceinline__ int row_stride_keys(int row_keys, int ntok) {
  return (row_keys / ntok) / 128 * 128;
}

// Item `pos` of the work list.  In SCORE mode the item is block b (from the last block, so the
// longest causal blocks start first) and split s of that block's key range.  All threads that
// call this get the same answer; `lane`/`nl` let a warp share the window scan.
template <bool FUSED>
__device__ __forceinline__ ItemInfo item_info(const IndexParams& p, int pos, int lane, int nl) {
  ItemInfo it;
  if constexpr (FUSED) {
    const PlanItem pi = p.items[pos];
    const PlanUnit u = p.units[pi.unit];
    it.tok0 = u.tok0;
    it.ntok = u.ntok;
    it.chunk = pi.chunk;
    it.nchunks = u.nchunks;
    it.slot_base = u.slot_base;
    it.k_lo = u.lo + pi.chunk * u.chunk_len;
    it.k_hi = min(u.hi, it.k_lo + u.chunk_len);
  } else {
    const int b = p.nblocks - 1 - pos / p.nsplit;
    const int s = pos % p.nsplit;
    it.tok0 = b * p.ntok_max;
    it.ntok = min(p.ntok_max, p.T - it.tok0);
    int lo = INT_MAX, hi = INT_MIN;
    for (int t = lane; t < it.ntok; t += nl) {
      const int a = clamp_key(p.ks[it.tok0 + t], p.N);
      const int e = clamp_key(p.ke[it.tok0 + t], p.N);
      if (e > a) {
        lo = min(lo, a);
        hi = max(hi, e);
      }
    }
    if (nl == 32) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
      }
    }
    it.chunk = 0;
    it.nchunks = 1;
    it.slot_base = -1;
    if (hi <= lo) {
      it.k_lo = it.k_hi = 0;
    } else {
      const int tiles_total = ceil_div(hi - lo, kKeysPerTile);
      const int t0 = static_cast<int>(static_cast<int64_t>(s) * tiles_total / p.nsplit);
      const int t1 = static_cast<int>(static_cast<int64_t>(s + 1) * tiles_total / p.nsplit);
      it.k_lo = lo + t0 * kKeysPerTile;
      it.k_hi = min(hi, lo + t1 * kKeysPerTile);
    }
  }
  it.ntiles = it.k_hi > it.k_lo ? ceil_div(it.k_hi - it.k_lo, kKeysPerTile) : 0;
  return it;
}

// Position of this CTA's r-th item: a snake over the (ordered) item list, so that a CTA that
// took a long item in one round takes a short one in the next.
__device__ __forceinline__ int item_pos(int r, int G, int c) { return r * G + ((r & 1) ? (G - 1 - c) : c); }

// relu(x) doubled, exactly: x + |x| is 2x for x >= 0 and +0 otherwise (no rounding for the
// finite, far-from-overflow dot products of e4m3 rows).  One add on the FMA pipe instead of a
// max on the integer / logic pipe, which the rest of the epilogue keeps busy.
__device__ __forceinline__ float relu2x(float x) { return __fadd_rn(x, fabsf(x)); }

// Weighted head sum of one (key, token): sum_h relu(s[h]) * w[h] in a fixed order: head pairs
// accumulate with packed fp32 FMAs into 4 partial sums (pair p -> partial p mod 4), which are
// then added in a fixed tree.  Both modes sum in this order (at H = 64 the epilogue runs the
// same steps over 16-column quarters), so their scores are bit-identical.  The products are
// formed from 2 relu(s[h]) and the total halved at the end: every product, partial sum and the
// total are then exactly twice the plain ones (scaling by 2 commutes with rounding), so the
// result equals the plain evaluation bit for bit.
template <int H>
__device__ __forceinline__ float head_sum(const float* s, const float* w) {
  float2 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
  for (int h = 0; h < H; h += 4) {
    const float4 wv = *reinterpret_cast<const float4*>(w + h);
    const float2 r0 = make_float2(relu2x(s[h]), relu2x(s[h + 1]));
    const float2 r1 = make_float2(relu2x(s[h + 2]), relu2x(s[h + 3]));
    acc[(h / 2) % 4] = __ffma2_rn(r0, make_float2(wv.x, wv.y), acc[(h / 2) % 4]);
    acc[(h / 2 + 1) % 4] = __ffma2_rn(r1, make_float2(wv.z, wv.w), acc[(h / 2 + 1) % 4]);
  }
  const float p0 = acc[0].x + acc[0].y;
  const float p1 = acc[1].x + acc[1].y;
  const float p2 = acc[2].x + acc[2].y;
  const float p3 = acc[3].x + acc[3].y;
  return ((p0 + p1) + (p2 + p3)) * 0.5f;
}

// Candidate lists of one token's chunks (global memory, written by other CTAs of this launch,
// so read through L2 with ld.global.cg).  Chunk c's list is in ascending key order and chunk
// ranges ascend with c.
struct ListSrc {
  const uint32_t* u;
  const int32_t* i;
  const int32_t* n;
  int nchunks;
  int topk;
  __device__ __forceinline__ int segments() const { return nchunks; }
  __device__ __forceinline__ int seg_len(int c) const { return min(max(__ldcg(n + c), 0), topk); }
  __device__ __forceinline__ uint32_t key(int c, int j) const {
    return __ldcg(u + static_cast<int64_t>(c) * topk + j);
  }
  __device__ __forceinline__ int32_t index(int c, int j) const {
    return __ldcg(i + static_cast<int64_t>(c) * topk + j);
  }
};

// Accumulator-stage geometry of an item with ntok tokens: MMA width, key tiles per 256-column
// stage (kps), columns per tile slot, and epilogue groups per tile (gpt = 4 / kps).
struct StageGeom {
  int n_mma;
  int kps;
  int slot_cols;
  int gpt;
};

__host__ __device__ __forceinline__ StageGeom stage_geom(int ntok, int H) {
  StageGeom g;
  g.n_mma = ((ntok * H + 15) / 16) * 16;
  if (g.n_mma > kMaxCols) g.n_mma = kMaxCols;
  g.kps = g.n_mma <= 64 ? 4 : (g.n_mma <= 128 ? 2 : 1);
  g.slot_cols = kMaxCols / g.kps;
  g.gpt = kEpiGroups / g.kps;
  return g;
}

// Exact top-k of one token's row (fused mode) by a team of NT threads; writes the final indices
// or, for a chunk of a split row, the chunk's candidate list, and merges the lists when this is
// the row's last chunk to finish.
template <int NT>
__device__ __forceinline__ void select_token(const IndexParams& p, const ItemInfo& it, int t, int2 wn,
                                             uint32_t* row, int row_stride, uint32_t* hist, uint32_t* bm, int ttid,
                                             SelectScratch* sc, int bar_id) {
  const int n = max(0, wn.y - wn.x);
  const RowKeys src{row, wn.x - it.k_lo, n, wn.x};
  const int tok = it.tok0 + t;
  if (it.nchunks == 1) {
    int32_t* out = p.idx + static_cast<int64_t>(tok) * p.topk;
    const int cnt = row_topk<NT>(src, p.topk, hist, 24, 0u, bm, ttid, sc, bar_id, [&](int q, int j) { out[q] = wn.x + j; });
    for (int q = cnt + ttid; q < p.topk; q += NT) out[q] = -1;
    return;
  }
  const int slot0 = it.slot_base + t * it.nchunks;
  const int64_t slot = slot0 + it.chunk;
  uint32_t* lu = p.list_u + slot * p.topk;
  int32_t* li = p.list_i + slot * p.topk;
  const int cnt = row_topk<NT>(src, p.topk, hist, 24, 0u, bm, ttid, sc, bar_id, [&](int q, int j) {
    lu[q] = src.key(0, j);
    li[q] = wn.x + j;
  });
  if (ttid == 0) p.list_n[slot] = cnt;
  __threadfence();
  group_sync<NT>(bar_id);
  if (ttid == 0) {
    const unsigned old = atomicAdd(p.counters + slot0, 1u);
    sc->bcast[4] = (old == static_cast<unsigned>(it.nchunks - 1)) ? 1 : 0;
  }
  group_sync<NT>(bar_id);
  const int last = sc->bcast[4];
  group_sync<NT>(bar_id);
  if (!last) return;
  // This team finished the token's last chunk: merge every chunk's candidates.  The lists are in
  // ascending key order chunk after chunk, so their concatenation is too.
  __threadfence();
  const ListSrc ls{p.list_u + static_cast<int64_t>(slot0) * p.topk, p.list_i + static_cast<int64_t>(slot0) * p.topk,
                   p.list_n + slot0, it.nchunks, p.topk};
  const int lane = ttid & 31;
  const int nch = it.nchunks;
  // List lengths and their exclusive prefix, 32 chunks per step in every warp (all list-length
  // loads of a step in flight together); the team's first warp keeps the offsets of the first
  // kCandCap chunks in the scratch's candidate array for the staged merge below.
  uint32_t* seg_off = sc->cand_u;
  uint32_t* seg_len = reinterpret_cast<uint32_t*>(sc->cand_i);
  int total = 0;
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int cc = c0 + lane;
    const int len = cc < nch ? ls.seg_len(cc) : 0;
    int incl = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (ttid < 32 && cc < min(nch, kCandCap)) {
      seg_off[cc] = static_cast<uint32_t>(total + incl - len);
      seg_len[cc] = static_cast<uint32_t>(len);
    }
    total += __shfl_sync(0xffffffffu, incl, 31);
  }
  int32_t* out = p.idx + static_cast<int64_t>(tok) * p.topk;
  int mc;
  const int cap = row_stride / 2;  // (key, index) pairs that fit the token's row buffer
  if (total <= cap && nch <= kCandCap) {
    // fast merge: stage the lists in shared memory, then row_topk.  The lists are walked as one
    // padded [nch][topk] array, 4 loads (4-wide when topk % 4 == 0) per thread per pass, every
    // global load of a pass issued before its shared stores.  Every candidate is some chunk's
    // top-k, so the keys are close and share their top bits: the first digit of the select is
    // taken just below the prefix common to the smallest and largest staged key.
    uint32_t* keys = row;
    int32_t* idxs = reinterpret_cast<int32_t*>(row + cap);
    uint32_t* kmin = reinterpret_cast<uint32_t*>(&sc->bcast[5]);
    uint32_t* kmax = reinterpret_cast<uint32_t*>(&sc->bcast[6]);
    for (int b = ttid; b < 256; b += NT) hist[b] = 0u;
    if (ttid == 0) {
      *kmin = 0xFFFFFFFFu;
      *kmax = 0u;
    }
    uint32_t lo_key = 0xFFFFFFFFu, hi_key = 0u;
    group_sync<NT>(bar_id);  // offsets written, histogram and key range cleared
    const int padded = nch * p.topk;
    if ((p.topk & 3) == 0) {
      for (int g0 = 0; g0 < padded; g0 += 4 * 4 * NT) {
        uint4 ku[4], ki[4];
        int base[4], cnt[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int g = g0 + 4 * (v * NT + ttid);
          const int cc = g / p.topk;
          const int j = g - cc * p.topk;
          cnt[v] = 0;
          base[v] = 0;
          if (g < padded) {
            const int len = static_cast<int>(seg_len[cc]);
            cnt[v] = min(4, max(0, len - j));
            base[v] = static_cast<int>(seg_off[cc]) + j;
          }
          if (cnt[v] > 0) {
            ku[v] = __ldcg(reinterpret_cast<const uint4*>(ls.u + g));
            ki[v] = __ldcg(reinterpret_cast<const uint4*>(ls.i + g));
          } else {
            ku[v] = make_uint4(0u, 0u, 0u, 0u);
            ki[v] = ku[v];
          }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t uu[4] = {ku[v].x, ku[v].y, ku[v].z, ku[v].w};
          const uint32_t ii[4] = {ki[v].x, ki[v].y, ki[v].z, ki[v].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (e < cnt[v]) {
              keys[base[v] + e] = uu[e];
              idxs[base[v] + e] = static_cast<int32_t>(ii[e]);
              lo_key = min(lo_key, uu[e]);
              hi_key = max(hi_key, uu[e]);
            }
          }
        }
      }
    } else {
      for (int g0 = 0; g0 < padded; g0 += 4 * NT) {
        uint32_t ku[4];
        int32_t ki[4];
        int dst[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int g = g0 + v * NT + ttid;
          const int cc = g / p.topk;
          const int j = g - cc * p.topk;
          dst[v] = -1;
          ku[v] = 0u;
          ki[v] = 0;
          if (g < padded && j < static_cast<int>(seg_len[cc])) {
            dst[v] = static_cast<int>(seg_off[cc]) + j;
            ku[v] = __ldcg(ls.u + g);
            ki[v] = __ldcg(ls.i + g);
          }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          if (dst[v] >= 0) {
            keys[dst[v]] = ku[v];
            idxs[dst[v]] = ki[v];
            lo_key = min(lo_key, ku[v]);
            hi_key = max(hi_key, ku[v]);
          }
        }
      }
    }
    lo_key = __reduce_min_sync(0xffffffffu, lo_key);
    hi_key = __reduce_max_sync(0xffffffffu, hi_key);
    if (lane == 0) {
      atomicMin(kmin, lo_key);
      atomicMax(kmax, hi_key);
    }
    group_sync<NT>(bar_id);
    const uint32_t diff = *kmin ^ *kmax;
    const int top = diff == 0u ? 0 : 31 - __clz(diff);  // highest bit in which staged keys differ
    const int shift0 = top > 7 ? top - 7 : 0;
    const uint32_t prefix0 = shift0 + 8 < 32 ? (*kmax >> (shift0 + 8)) : 0u;
    for (int j0 = 0; j0 < total; j0 += 4 * NT) {
      const int j = j0 + 4 * ttid;
      if (j < total) {
        const uint4 v = *reinterpret_cast<const uint4*>(keys + j);
        const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (j + q < total) atomicAdd(&hist[(e[q] >> shift0) & 0xFFu], 1u);
      }
    }
    group_sync<NT>(bar_id);
    const RowKeys merged{keys, 0, total, 0};
    mc = row_topk<NT>(merged, p.topk, hist, shift0, prefix0, bm, ttid, sc, bar_id,
                      [&](int q, int j) { out[q] = idxs[j]; });
  } else {
    const SelectResult mr = group_select<NT>(ls, total, p.topk, ttid, sc, bar_id, nullptr);
    mc = group_emit_segments<NT, 4>(ls, mr, ttid, sc, bar_id, [&](int q, int s, int j) {
      if (q < p.topk) out[q] = ls.index(s, j);  // never past the row
    });
    mc = min(mc, p.topk);
  }
  for (int q = mc + ttid; q < p.topk; q += NT) out[q] = -1;
  if (ttid == 0) p.counters[slot0] = 0u;  // every chunk has arrived: re-arm for the next run
}

template <int H, int D, bool FUSED>
__global__ void __launch_bounds__(kIndexThreads, 1)
    index_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                 const IndexParams p) {
  static_assert(H == 4 || H == 8 || H == 16 || H == 32 || H == 64, "H");
  static_assert(kAccStages == 2, "the MMA issuer toggles between two accumulator stages");
  static_assert(D == 64 || D == 128, "D");
  constexpr int kTileBytes = kKeysPerTile * D;
  constexpr int kColsPerGroup = kMaxCols / kEpiGroups;  // 64
  constexpr int TPG = kColsPerGroup / H;                // tokens per 64-column group slot
  constexpr int kEpiThreads = kEpiGroups * kGroupThreads;
  constexpr int kEpiBar = 1 + kEpiGroups;  // named barrier of all epilogue threads

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base for the swizzled TMA / MMA tiles.  The pad is computed from the
  // shared-window address and applied to the shared array itself, so every pointer below stays
  // visibly in shared memory (plain shared loads, stores and atomics, not generic ones).
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem + p.off_ring;
  uint8_t* qbuf = smem + p.off_q;
  uint32_t* rows = reinterpret_cast<uint32_t*>(smem + p.off_rows);
  float* w_s = reinterpret_cast<float*>(smem + p.off_w);
  int2* win_s = reinterpret_cast<int2*>(smem + p.off_win);
  SelectScratch* scratch = reinterpret_cast<SelectScratch*>(smem + p.off_sc);
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + p.off_hist);
  uint32_t* bitmap_s = reinterpret_cast<uint32_t*>(smem + p.off_bitmap);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  const int S = p.stages;
  uint64_t* k_full = bars;
  uint64_t* k_empty = bars + S;
  uint64_t* acc_full = bars + 2 * S;
  uint64_t* acc_empty = acc_full + kAccStages;
  uint64_t* q_full = acc_empty + kAccStages;
  uint64_t* q_empty = q_full + 2;
  uint64_t* drain = q_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* item_full = drain + 2;
  uint64_t* item_empty = item_full + kItemRing;
  volatile int* item_ring = reinterpret_cast<volatile int*>(item_empty + kItemRing);  // + 2 broadcast slots

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int a = 0; a < kAccStages; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiGroups * 4);  // one arrival per epilogue warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
    }
    mbar_init(drain, 1);
    for (int b = 0; b < kItemRing; ++b) {
      mbar_init(&item_full[b], 1);
      mbar_init(&item_empty[b], 1 + kProducers);  // the other producers, the MMA issuer, the epilogue
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&qmap);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // Launched as a programmatic dependent of the planner, the prologue above overlaps the
  // planner's tail; the plan is read only after the planner grid has completed.  (A no-op when
  // the launch has no such dependency.)
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int n_items = FUSED ? p.plan->n_items : p.nblocks * p.nsplit;
  const int G = gridDim.x;
  const int c = blockIdx.x;

  if (warp == 0 || warp == 2 || warp == 3) {
    // ------------------------------------------------------------------ TMA producers
    // Three producer threads (lane 0 of warps 0, 2 and 3) share the K ring: producer pr issues
    // the tiles that land in stages st with st % kProducers == pr.  One thread issuing every
    // tile load caps the ring's fill rate (each thread's bulk-tensor copies proceed one after
    // another, whatever their size); three in parallel keep the tensor core fed.
    // Producer 0 also decides which items this CTA runs and passes each one (then -1) to the
    // other producers, the MMA issuer and the epilogue through item_ring, and loads the Q block
    // of each item.  Fused: CTA c starts with item c and then claims the next unclaimed item
    // from the plan's counter as soon as it has issued its loads of the current one; the planner
    // orders items longest first, so this is a longest-processing-time greedy schedule.  Each
    // CTA that had an item makes exactly one failing claim, hence n_items claims in all, and the
    // one that draws n_items - 1 (the last) re-arms the counter for the next run of the same
    // plan.  Score mode: a fixed snake order over the CTAs.
    const int pr = warp == 0 ? 0 : warp - 1;
    if (lane == 0) {
      uint32_t kt = 0;  // tiles of this CTA before the current item (all producers count alike)
      int qi = 0;
      int seq = 0;
      int r = 0;
      bool ok = true;
      auto next_item = [&]() -> int {
        if constexpr (FUSED) {
          const int v = atomicAdd(p.queue, 1);
          if (v == n_items - 1) atomicExch(p.queue, 0);
          return G + v < n_items ? G + v : -1;
        } else {
          for (; r * G < n_items; ++r) {
            const int ps = item_pos(r, G, c);
            if (ps < n_items) {
              ++r;
              return ps;
            }
          }
          return -1;
        }
      };
      // this producer's share of an item's K tiles
      auto load_tiles = [&](const ItemInfo& it) {
        for (int i = 0; i < it.ntiles; ++i) {
          const uint32_t t = kt + static_cast<uint32_t>(i);
          const int st = static_cast<int>(t % S);
          if (st % kProducers != pr) continue;
          const uint32_t ph = (t / S) & 1u;
          if (!mbar_wait(&k_empty[st], ph ^ 1u, abort_flag, p.err, 2)) return false;
          mbar_arrive_expect_tx(&k_full[st], static_cast<uint32_t>(kTileBytes));
          tma_load_2d(ring + st * kTileBytes, &kmap, &k_full[st], 0, it.k_lo + i * kKeysPerTile);
        }
        return true;
      };
      if (pr == 0) {
        int pos = FUSED ? (c < n_items ? c : -1) : next_item();
        while (true) {
          const ItemInfo it = pos >= 0 ? item_info<FUSED>(p, pos, 0, 1) : ItemInfo{};
          if (pos >= 0 && it.ntiles == 0) {  // nothing to compute: not handed on
            pos = next_item();
            continue;
          }
          const int sl = seq % kItemRing;
          if (!mbar_wait(&item_empty[sl], (static_cast<uint32_t>(seq / kItemRing) & 1u) ^ 1u, abort_flag, p.err,
                         7)) {
            ok = false;
            break;
          }
          item_ring[sl] = pos;
          mbar_arrive(&item_full[sl]);
          ++seq;
          if (pos < 0) break;
          const int qb = qi % p.qbufs;
          const uint32_t qph = static_cast<uint32_t>(qi / p.qbufs) & 1u;
          if (!mbar_wait(&q_empty[qb], qph ^ 1u, abort_flag, p.err, 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&q_full[qb], static_cast<uint32_t>(p.n_mma_max * D));
          tma_load_2d(qbuf + qb * p.n_mma_max * D, &qmap, &q_full[qb], 0, it.tok0 * H);
          ++qi;
          if (!load_tiles(it)) {
            ok = false;
            break;
          }
          kt += static_cast<uint32_t>(it.ntiles);
          pos = next_item();
        }
      } else {
        for (;; ++seq) {
          const int sl = seq % kItemRing;
          if (!mbar_wait(&item_full[sl], static_cast<uint32_t>(seq / kItemRing) & 1u, abort_flag, p.err, 10)) {
            ok = false;
            break;
          }
          const int pos = item_ring[sl];
          mbar_arrive(&item_empty[sl]);
          if (pos < 0) break;
          const ItemInfo it = item_info<FUSED>(p, pos, 0, 1);
          if (!load_tiles(it)) {
            ok = false;
            break;
          }
          kt += static_cast<uint32_t>(it.ntiles);
        }
      }
      if (!ok) {
        // let the copies this producer issued land before the CTA can exit
        for (uint32_t back = 0; back < static_cast<uint32_t>(S) && back < kt; ++back) {
          const uint32_t t = kt - 1 - back;
          if (static_cast<int>(t % S) % kProducers == pr) mbar_wait_drain(&k_full[t % S], (t / S) & 1u);
        }
        if (pr == 0 && qi > 0)
          mbar_wait_drain(&q_full[(qi - 1) % p.qbufs], static_cast<uint32_t>((qi - 1) / p.qbufs) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Ring slot, accumulator stage and their mbarrier phases advance as counters (no division
    // per tile), and the operand descriptors are formed once and advanced by address offsets:
    // this thread shares its scheduler with four epilogue warps, so every instruction it saves
    // is an MMA issued sooner.
    if (lane == 0) {
      int qi = 0;
      bool ok = true;
      int kst = 0;         // ring slot of the next key tile
      uint32_t kph = 0;    // phase of that slot's k_full
      int as = 0;          // accumulator stage being filled
      uint32_t aph = 0;    // phase of that stage
      const uint64_t a_desc0 = smem_desc_kmajor<D>(smem_addr(ring));
      for (int seq = 0;; ++seq) {
        const int sl = seq % kItemRing;
        if (!mbar_wait(&item_full[sl], static_cast<uint32_t>(seq / kItemRing) & 1u, abort_flag, p.err, 8)) break;
        const int pos = item_ring[sl];
        mbar_arrive(&item_empty[sl]);
        if (pos < 0) break;
        const ItemInfo it = item_info<FUSED>(p, pos, 0, 1);
        const StageGeom sg = stage_geom(it.ntok, H);
        const uint32_t idesc = idesc_f8_e4m3(kKeysPerTile, sg.n_mma);
        const int qb = qi % p.qbufs;
        if (!mbar_wait(&q_full[qb], static_cast<uint32_t>(qi / p.qbufs) & 1u, abort_flag, p.err, 3)) {
          ok = false;
          break;
        }
        const uint64_t b_desc = smem_desc_kmajor<D>(smem_addr(qbuf + qb * p.n_mma_max * D));
        // tile i of the item goes to tile slot ts = i % kps of an accumulator stage; a stage is
        // committed to the epilogue after its last tile
        int ts = 0;
        for (int i = 0; i < it.ntiles; ++i) {
          if (ts == 0 && !mbar_wait(&acc_empty[as], aph ^ 1u, abort_flag, p.err, 5)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&k_full[kst], kph, abort_flag, p.err, 4)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t a_desc = a_desc0 + static_cast<uint64_t>((kst * kTileBytes) >> 4);
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(as * kMaxCols + ts * sg.slot_cols);
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)  // K steps of 32 bytes: descriptor address + 2 (16-byte units)
            mma_f8(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, kk > 0 ? 1u : 0u);
          mma_commit(&k_empty[kst]);
          if (++kst == S) {
            kst = 0;
            kph ^= 1u;
          }
          if (++ts == sg.kps || i == it.ntiles - 1) {
            mma_commit(&acc_full[as]);
            ts = 0;
            as ^= 1;
            if (as == 0) aph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&q_empty[qb]);
        ++qi;
      }
      // every MMA issued by this thread has completed once `drain` flips
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    // After an expired wait (abort) the epilogue finishes the item in hand (every later wait
    // returns at once; the item's loops have plan-determined ends, so every thread still reaches
    // every barrier) and then stops: thread 0 broadcasts -1 when its wait for the next item
    // fails.  The output is then garbage and the error word says so.
    const int g = (warp - 4) >> 2;  // group: accumulator columns [64g, 64g + 64) of a stage
    const int gtid = threadIdx.x - 128 - g * kGroupThreads;
    const int etid = threadIdx.x - 128;
    const int quarter = warp & 3;  // tensor-memory lane quarter = key rows quarter*32 .. +31
    if constexpr (FUSED) {
      // tokens with an empty window: all -1 rows (spread over the CTAs)
      const int n_empty = p.plan->n_empty;
      for (int e = blockIdx.x; e < n_empty; e += gridDim.x) {
        int32_t* out = p.idx + static_cast<int64_t>(p.empty[e]) * p.topk;
        for (int q = etid; q < p.topk; q += kEpiThreads) out[q] = -1;
      }
    }
    uint32_t at = 0;
    for (int seq = 0;; ++seq) {
      // Thread 0 takes the next item from the ring and broadcasts it (two alternating slots: a
      // slot is rewritten only after every thread has passed the barrier that follows its next
      // read).  The barrier also means the previous item is finished by every group before the
      // shared per-item state (weights, windows, histograms, row buffer) is rewritten.
      if (etid == 0) {
        const int sl = seq % kItemRing;
        int ps = -1;
        if (mbar_wait(&item_full[sl], static_cast<uint32_t>(seq / kItemRing) & 1u, abort_flag, p.err, 9)) {
          ps = item_ring[sl];
          mbar_arrive(&item_empty[sl]);
        }
        item_ring[kItemRing + (seq & 1)] = ps;
      }
      named_bar_sync(kEpiBar, kEpiThreads);
      const int pos = item_ring[kItemRing + (seq & 1)];
      if (pos < 0) break;
      const ItemInfo it = item_info<FUSED>(p, pos, lane, 32);
      const StageGeom sg = stage_geom(it.ntok, H);
      const int ts = g / sg.gpt;          // key tile of the stage this group reads
      const int cs = g % sg.gpt;          // 64-column slot within that tile
      const int t0 = cs * TPG;            // first token of this group
      const int tn = max(0, min(TPG, it.ntok - t0));
      const int row_stride = FUSED ? row_stride_keys(p.row_keys, it.ntok) : 0;
      for (int e = etid; e < it.ntok * H; e += kEpiThreads)
        w_s[e] = __ldg(p.w + static_cast<int64_t>(it.tok0) * H + e);
      for (int t = etid; t < it.ntok; t += kEpiThreads) {
        const int a = clamp_key(p.ks[it.tok0 + t], p.N);
        const int e = clamp_key(p.ke[it.tok0 + t], p.N);
        win_s[t] = make_int2(max(a, it.k_lo), min(e, it.k_hi));
      }
      if constexpr (FUSED) {
        for (int e = etid; e < it.ntok * 256; e += kEpiThreads) hist_s[e] = 0u;
      }
      named_bar_sync(kEpiBar, kEpiThreads);

      const int nst = ceil_div(it.ntiles, sg.kps);
      // H = 64: the group's one token and its window, fixed for the item
      const int2 wn64 = (H == 64 && tn > 0) ? win_s[t0] : make_int2(0, 0);
      // k_scale of this lane's key, loaded one stage ahead so its latency hides behind a stage
      float ksc_next = 0.f;
      {
        const int j = it.k_lo + ts * kKeysPerTile + quarter * 32 + lane;
        if (ts < it.ntiles && j < p.N) ksc_next = __ldg(p.k_scale + j);
      }
      for (int sidx = 0; sidx < nst; ++sidx, ++at) {
        const int i = sidx * sg.kps + ts;  // this group's key tile
        const int j0 = it.k_lo + i * kKeysPerTile;
        const int wj = j0 + quarter * 32;
        const int my_j = wj + lane;
        const float ksc = ksc_next;
        {
          const int jn = my_j + sg.kps * kKeysPerTile;
          if (i + sg.kps < it.ntiles && jn < p.N) ksc_next = __ldg(p.k_scale + jn);
        }
        const int as = static_cast<int>(at % kAccStages);
        // score of (token t of the item, key my_j): logits store, or row buffer + first-digit histogram
        auto emit_score = [&](int t, int2 wn, float score) {
          const bool in = my_j >= wn.x && my_j < wn.y;
          if constexpr (FUSED) {
            const uint32_t u = score_key(score);
            if (in) rows[t * row_stride + (my_j - it.k_lo)] = u;
            if (in) atomicAdd(&hist_s[t * 256 + (u >> 24)], 1u);
          } else {
            if (in) p.logits[static_cast<int64_t>(it.tok0 + t) * p.N + my_j] = score;
          }
        };
        mbar_wait(&acc_full[as], (at / kAccStages) & 1u, abort_flag, p.err, 6);
        tc_fence_after_sync();
        bool any = false;
        if (i < it.ntiles) {
          if constexpr (H == 64) {
            any = tn > 0 && !(wj >= wn64.y || wj + 32 <= wn64.x);
          } else {
#pragma unroll
            for (int tt = 0; tt < TPG; ++tt) {
              if (tt < tn) {
                const int2 wn = win_s[t0 + tt];
                any |= !(wj >= wn.y || wj + 32 <= wn.x);
              }
            }
          }
        }
        if (any) {  // warp-uniform
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 static_cast<uint32_t>(as * kMaxCols + ts * sg.slot_cols + cs * kColsPerGroup);
          // H = 64: one token's 64 heads, summed into 4 packed partial sums (heads 2p, 2p + 1 go
          // to sum p % 4) and then in head_sum's tree, in both modes.  H <= 32: the 64 columns
          // are read in two halves of 32 (every token lies inside one half) and summed by
          // head_sum<H>.
          float2 acc64[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) acc64[q4] = make_float2(0.f, 0.f);
          // relu, weight and accumulate heads hh .. hh + 3 (accumulator columns v[0..3])
          auto heads4 = [&](const float* v, const float4 wq, int hh) {
            const float2 r0 = make_float2(relu2x(v[0]), relu2x(v[1]));
            const float2 r1 = make_float2(relu2x(v[2]), relu2x(v[3]));
            acc64[(hh / 2) % 4] = __ffma2_rn(r0, make_float2(wq.x, wq.y), acc64[(hh / 2) % 4]);
            acc64[(hh / 2 + 1) % 4] = __ffma2_rn(r1, make_float2(wq.z, wq.w), acc64[(hh / 2 + 1) % 4]);
          };
          if constexpr (H == 64) {
            // Quarters of 16 columns: the next quarter's tensor-memory load is in flight while
            // this one is summed.
            const float* wt = w_s + t0 * H;
            float sa[16], sb[16];
            tmem_ld_x16(taddr, sa);
            tmem_wait_ld_regs16(sa);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              float* cur = (qq & 1) ? sb : sa;
              float* nxt = (qq & 1) ? sa : sb;
              if (qq < 3) tmem_ld_x16(taddr + 16 * (qq + 1), nxt);
              float4 wv[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) wv[q] = *reinterpret_cast<const float4*>(wt + 16 * qq + 4 * q);
#pragma unroll
              for (int h = 0; h < 16; h += 4) heads4(cur + h, wv[h / 4], 16 * qq + h);
              if (qq < 3) tmem_wait_ld_regs16(nxt);
            }
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float s[32];
            if constexpr (H == 64) {
              // done above
            } else if (half * (32 / H) < tn) {  // (a half without tokens of this item is not read)
              constexpr int TPH = 32 / H;  // tokens per half
              // columns of this half that hold the item's tokens
              const int cols = (min(tn, (half + 1) * TPH) - half * TPH) * H;
              // 16-column loads, each waited for (a 32-column load waits far longer when the
              // lane quarter's four epilogue warps all load at once)
              tmem_ld_x16(taddr + 32 * half, s);
              tmem_wait_ld_regs16(s);
              if (cols > 16) {
                tmem_ld_x16(taddr + 32 * half + 16, s + 16);
                tmem_wait_ld_regs16(s + 16);
              }
#pragma unroll
              for (int tl = 0; tl < TPH; ++tl) {
                const int tt = half * TPH + tl;
                if (tt < tn) {
                  const int t = t0 + tt;
                  const int2 wn = win_s[t];
                  if (!(wj >= wn.y || wj + 32 <= wn.x)) {  // warp-uniform
                    const float score = head_sum<H>(s + tl * H, w_s + t * H) * ksc;
                    emit_score(t, wn, score);
                  }
                }
              }
            }
          }
          if constexpr (H == 64) {  // (any: the token's window meets this warp's keys)
            const float p0 = acc64[0].x + acc64[0].y;
            const float p1 = acc64[1].x + acc64[1].y;
            const float p2 = acc64[2].x + acc64[2].y;
            const float p3 = acc64[3].x + acc64[3].y;
            emit_score(t0, wn64, ((p0 + p1) + (p2 + p3)) * (0.5f * ksc));  // (the doubled sum, halved)
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[as]);
      }

      if constexpr (FUSED) {
        // ---------------------------------------------------------------- selection
        // Teams: as many as there are tokens, up to one per group (more, smaller teams select
        // more rows at once); team `team` takes tokens team, team + nteams, ...
        // Every row-buffer and histogram write of the tokens a team selects is visible after this
        // barrier.  With 64 heads and four tokens, group g scored exactly token g, which team g
        // selects: the group's own barrier suffices (no wait for the slowest group).
        if (H == 64 && it.ntok == kEpiGroups) {
          named_bar_sync(1 + g, kGroupThreads);
        } else {
          named_bar_sync(kEpiBar, kEpiThreads);
        }
        const int nteams = it.ntok >= kEpiGroups ? kEpiGroups : (it.ntok >= 2 ? 2 : 1);
        const int team = g % nteams;
        const int ttid = (g / nteams) * kGroupThreads + gtid;
        SelectScratch* sc = scratch + team;
        const int bar_id = 1 + team;
        for (int t = team; t < it.ntok; t += nteams) {
          uint32_t* row = rows + t * row_stride;
          uint32_t* bm = bitmap_s + t * (row_stride / 32);
          uint32_t* hist = hist_s + t * 256;
          if (nteams == 1) {
            select_token<4 * kGroupThreads>(p, it, t, win_s[t], row, row_stride, hist, bm, ttid, sc, bar_id);
          } else if (nteams == 2) {
            select_token<2 * kGroupThreads>(p, it, t, win_s[t], row, row_stride, hist, bm, ttid, sc, bar_id);
          } else {
            select_token<kGroupThreads>(p, it, t, win_s[t], row, row_stride, hist, bm, ttid, sc, bar_id);
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace dsa
