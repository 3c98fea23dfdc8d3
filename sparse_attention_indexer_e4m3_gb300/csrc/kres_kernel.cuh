// K-resident / Q-streaming variant of the FP8 indexer scorer (logits output, like
// dsa_index_score).  The layout is the one the Modular page "sparse_index_fp8_sm100_prefill"
// describes as the shipped scorer: a key tile stays in shared memory while query-token blocks
// stream past it.  Here it is a persistent tcgen05 kernel with the same roles as index_kernel:
//   warps 0, 2, 3  TMA producers: warp 0 claims work items (key tile, run of token blocks) from
//                  a counter, lists the blocks whose windows meet the tile, loads the tile into
//                  one of two K buffers and hands the item on; the three lane-0 threads then
//                  stream the item's Q blocks ([ntok * H, D] e4m3 boxes) through an S-slot ring,
//                  slot st filled by producer st % 3;
//   warp 1         MMA issuer and tensor-memory owner: per Q block one accumulator stage
//                  S^T = K . Q^T = [128 keys, ntok * H = 256 columns] (D / 32 tcgen05.mma of
//                  kind::f8f6f4, A = the resident tile, B = the streamed block);
//   warps 4..19    epilogue: four groups of four warps (one per 32-lane tensor-memory quarter);
//                  group g reads columns [64g, 64g + 64), i.e. 64 / H tokens, and writes
//                  logits[t, key] for in-window pairs with exactly the arithmetic of the
//                  Q-resident kernel (so both variants give the same bits).
// Which operand stays resident only changes what is re-read from L2: a 256-column Q block
// (32 KB at D = 128) per 128 keys here, a 16 KB key tile per 256 columns there.
#pragma once

#include <climits>
#include <cstdint>

#include "common.cuh"
#include "index_kernel.cuh"
#include "ptx.cuh"
#include "types.cuh"

namespace dsa {

// Clamped window of every token and the union of each block's windows; zeroes the item counter.
static __global__ void __launch_bounds__(256) kres_windows_kernel(const int32_t* ks, const int32_t* ke, int T, int N,
                                                           int ntok, int nblocks, int2* blk_win, int2* tok_win,
                                                           int* queue) {
  // the scorer may be scheduled now; it waits for this grid before reading what it writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0) *queue = 0;
  if (b >= nblocks) return;
  int lo = INT_MAX, hi = INT_MIN;
  const int t1 = min(T, (b + 1) * ntok);
  for (int t = b * ntok; t < t1; ++t) {
    const int a = clamp_key(ks[t], N), e = clamp_key(ke[t], N);
    tok_win[t] = make_int2(a, e);
    if (e > a) {
      lo = min(lo, a);
      hi = max(hi, e);
    }
  }
  blk_win[b] = hi > lo ? make_int2(lo, hi) : make_int2(0, 0);
}

template <int H, int D>
__global__ void __launch_bounds__(kIndexThreads, 1)
    kres_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                const KresParams p) {
  static_assert(H == 4 || H == 8 || H == 16 || H == 32 || H == 64, "H");
  static_assert(D == 64 || D == 128, "D");
  constexpr int kTileBytes = kKeysPerTile * D;
  constexpr int kQBytes = kMaxCols * D;
  constexpr int TPG = 64 / H;  // tokens per epilogue group
  constexpr int kEpiThreads = kEpiGroups * kGroupThreads;
  extern __shared__ __align__(1024) uint8_t kres_smem_raw[];
  uint8_t* smem = kres_smem_raw + ((1024u - (smem_addr(kres_smem_raw) & 1023u)) & 1023u);
  uint8_t* kbuf = smem;  // two key tiles
  uint8_t* qring = smem + p.off_q;
  const int S = p.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + S;
  uint64_t* k_full = bars + 2 * S;
  uint64_t* k_empty = k_full + 2;
  uint64_t* acc_full = k_empty + 2;
  uint64_t* acc_empty = acc_full + kAccStages;
  uint64_t* item_full = acc_empty + kAccStages;
  uint64_t* item_empty = item_full + kItemRing;
  uint64_t* drain = item_empty + kItemRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 2);  // 2 epilogue broadcast slots
  int* items = reinterpret_cast<int*>(smem + p.off_items);              // kItemRing x kKresItemInts

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&k_full[b], 1);
      mbar_init(&k_empty[b], 1);
    }
    for (int a = 0; a < kAccStages; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiGroups * 4);  // one arrival per epilogue warp
    }
    for (int b = 0; b < kItemRing; ++b) {
      mbar_init(&item_full[b], 1);
      mbar_init(&item_empty[b], (kKresProducers - 1) + 2);  // helper producers, MMA issuer, epilogue
    }
    mbar_init(drain, 1);
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
  // launched as a programmatic dependent of the window pass: wait for its results
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n_items = p.ntiles * p.nchunks;

  if (warp == 0 || warp == 2 || warp == 3) {
    // ------------------------------------------------------------------ TMA producers
    const int pr = warp == 0 ? 0 : warp - 1;
    uint32_t bt = 0;  // Q blocks of this CTA before the current item (all producers count alike)
    int kb_i = 0;     // key tiles loaded so far
    bool ok = true;
    // this producer's share of an item's Q blocks
    auto load_blocks = [&](const int* slot) {
      const int cnt = slot[1];
      for (int i = 0; i < cnt; ++i) {
        const uint32_t t = bt + static_cast<uint32_t>(i);
        const int st = static_cast<int>(t % static_cast<uint32_t>(S));
        if (st % kKresProducers != pr) continue;
        if (!mbar_wait(&q_empty[st], ((t / S) & 1u) ^ 1u, abort_flag, p.err, 0x71)) return false;
        mbar_arrive_expect_tx(&q_full[st], static_cast<uint32_t>(kQBytes));
        tma_load_2d(qring + st * kQBytes, &qmap, &q_full[st], 0, slot[2 + i] * p.ntok * H);
      }
      return true;
    };
    if (warp == 0) {
      // the whole warp claims items and lists their blocks; lane 0 issues the copies
      for (int seq = 0;; ++seq) {
        const int sl = seq % kItemRing;
        int* slot = items + sl * kKresItemInts;
        int ok_w = 1;
        if (lane == 0)
          ok_w = mbar_wait(&item_empty[sl], (static_cast<uint32_t>(seq / kItemRing) & 1u) ^ 1u, abort_flag, p.err,
                           0x72)
                     ? 1
                     : 0;
        ok_w = __shfl_sync(0xffffffffu, ok_w, 0);
        if (!ok_w) {
          ok = false;
          break;
        }
        int tile = -1, cnt = 0;
        while (true) {
          int id = 0;
          if (lane == 0) id = atomicAdd(p.queue, 1);
          id = __shfl_sync(0xffffffffu, id, 0);
          if (id >= n_items) {
            tile = -1;
            break;
          }
          tile = id / p.nchunks;
          const int b0 = (id - tile * p.nchunks) * p.chunk;
          const int b1 = min(p.nblocks, b0 + p.chunk);
          const int k0 = tile * kKeysPerTile, k1 = min(p.N, k0 + kKeysPerTile);
          cnt = 0;
          for (int bb = b0; bb < b1; bb += 32) {
            const int b = bb + lane;
            bool meets = false;
            if (b < b1) {
              const int2 wb = p.blk_win[b];
              meets = wb.x < wb.y && wb.x < k1 && wb.y > k0;
            }
            const unsigned m = __ballot_sync(0xffffffffu, meets);
            if (meets) slot[2 + cnt + __popc(m & ((1u << lane) - 1u))] = b;
            cnt += __popc(m);
          }
          if (cnt > 0) break;  // (an item no block's windows meet is skipped)
        }
        if (lane == 0) {
          slot[0] = tile;
          slot[1] = cnt;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_full[sl]);
        if (tile < 0) break;
        if (lane == 0) {
          const int kb = kb_i & 1;
          if (!mbar_wait(&k_empty[kb], (static_cast<uint32_t>(kb_i >> 1) & 1u) ^ 1u, abort_flag, p.err, 0x73)) {
            ok = false;
          } else {
            mbar_arrive_expect_tx(&k_full[kb], static_cast<uint32_t>(kTileBytes));
            tma_load_2d(kbuf + kb * kTileBytes, &kmap, &k_full[kb], 0, tile * kKeysPerTile);
            ++kb_i;
            ok = load_blocks(slot);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        bt += static_cast<uint32_t>(cnt);
      }
    } else if (lane == 0) {
      for (int seq = 0;; ++seq) {
        const int sl = seq % kItemRing;
        if (!mbar_wait(&item_full[sl], static_cast<uint32_t>(seq / kItemRing) & 1u, abort_flag, p.err, 0x74)) {
          ok = false;
          break;
        }
        const int* slot = items + sl * kKresItemInts;
        const int tile = slot[0], cnt = slot[1];
        if (tile < 0) {
          mbar_arrive(&item_empty[sl]);
          break;
        }
        ok = load_blocks(slot);
        mbar_arrive(&item_empty[sl]);  // (the block list was read while loading)
        if (!ok) break;
        bt += static_cast<uint32_t>(cnt);
      }
    }
    if (!ok && lane == 0) {
      // let the copies this producer issued land before the CTA can exit
      for (uint32_t back = 0; back < static_cast<uint32_t>(S) && back < bt; ++back) {
        const uint32_t t = bt - 1 - back;
        if (static_cast<int>(t % S) % kKresProducers == pr) mbar_wait_drain(&q_full[t % S], (t / S) & 1u);
      }
      if (warp == 0 && kb_i > 0) mbar_wait_drain(&k_full[(kb_i - 1) & 1], ((kb_i - 1) >> 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f8_e4m3(kKeysPerTile, kMaxCols);
      uint32_t bt = 0;
      int kb_i = 0;
      int as = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        const int sl = seq % kItemRing;
        if (!mbar_wait(&item_full[sl], static_cast<uint32_t>(seq / kItemRing) & 1u, abort_flag, p.err, 0x75)) break;
        const int tile = items[sl * kKresItemInts];
        const int cnt = items[sl * kKresItemInts + 1];
        mbar_arrive(&item_empty[sl]);
        if (tile < 0) break;
        const int kb = kb_i & 1;
        if (!mbar_wait(&k_full[kb], static_cast<uint32_t>(kb_i >> 1) & 1u, abort_flag, p.err, 0x76)) break;
        tc_fence_after_sync();
        const uint64_t a_desc = smem_desc_kmajor<D>(smem_addr(kbuf + kb * kTileBytes));
        for (int i = 0; i < cnt; ++i) {
          const uint32_t t = bt + static_cast<uint32_t>(i);
          const int st = static_cast<int>(t % static_cast<uint32_t>(S));
          if (!mbar_wait(&acc_empty[as], aph ^ 1u, abort_flag, p.err, 0x77) ||
              !mbar_wait(&q_full[st], (t / S) & 1u, abort_flag, p.err, 0x78)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t b_desc = smem_desc_kmajor<D>(smem_addr(qring + st * kQBytes));
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(as * kMaxCols);
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)  // K steps of 32 bytes: descriptor address + 2 (16-byte units)
            mma_f8(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, kk > 0 ? 1u : 0u);
          mma_commit(&q_empty[st]);
          mma_commit(&acc_full[as]);
          as ^= 1;
          if (as == 0) aph ^= 1u;
        }
        if (!ok) break;
        mma_commit(&k_empty[kb]);
        ++kb_i;
        bt += static_cast<uint32_t>(cnt);
      }
      // every MMA issued by this thread has completed once `drain` flips
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    // After an expired wait the epilogue finishes the item in hand (later waits return at once)
    // and stops: thread 0 broadcasts -1 when its wait for the next item fails.
    const int g = (warp - 4) >> 2;
    const int etid = threadIdx.x - 128;
    const int quarter = warp & 3;
    uint32_t at = 0;  // accumulator stages consumed
    for (int seq = 0;; ++seq) {
      const int sl = seq % kItemRing;
      if (etid == 0) {
        int tl = -1;
        if (mbar_wait(&item_full[sl], static_cast<uint32_t>(seq / kItemRing) & 1u, abort_flag, p.err, 0x79))
          tl = items[sl * kKresItemInts];
        bcast[seq & 1] = tl;
      }
      named_bar_sync(kKresEpiBar, kEpiThreads);
      const int tile = bcast[seq & 1];
      if (tile < 0) {
        if (etid == 0) mbar_arrive(&item_empty[sl]);
        break;
      }
      const int* slot = items + sl * kKresItemInts;
      const int cnt = slot[1];
      const int wj = tile * kKeysPerTile + quarter * 32;  // this warp's first key
      const int my_j = wj + lane;
      const float ksc = my_j < p.N ? __ldg(p.k_scale + my_j) : 0.f;
      for (int i = 0; i < cnt; ++i, ++at) {
        const int as = static_cast<int>(at % kAccStages);
        const int t0 = slot[2 + i] * p.ntok + g * TPG;  // this group's first token
        const int tn = max(0, min(TPG, p.T - t0));
        mbar_wait(&acc_full[as], (at / kAccStages) & 1u, abort_flag, p.err, 0x7A);
        tc_fence_after_sync();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(as * kMaxCols + g * 64);
        if constexpr (H == 64) {
          // one token: its 64 heads in quarters of 16 columns, summed exactly as the Q-resident
          // kernel sums them
          const int2 wn = tn > 0 ? __ldg(p.tok_win + t0) : make_int2(0, 0);
          if (tn > 0 && !(wj >= wn.y || wj + 32 <= wn.x)) {  // warp-uniform
            const float* wt = p.w + static_cast<int64_t>(t0) * H;
            float2 acc64[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) acc64[q4] = make_float2(0.f, 0.f);
            auto heads4 = [&](const float* v, const float4 wq, int hh) {
              const float2 r0 = make_float2(relu2x(v[0]), relu2x(v[1]));
              const float2 r1 = make_float2(relu2x(v[2]), relu2x(v[3]));
              acc64[(hh / 2) % 4] = __ffma2_rn(r0, make_float2(wq.x, wq.y), acc64[(hh / 2) % 4]);
              acc64[(hh / 2 + 1) % 4] = __ffma2_rn(r1, make_float2(wq.z, wq.w), acc64[(hh / 2 + 1) % 4]);
            };
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
              for (int q = 0; q < 4; ++q) wv[q] = __ldg(reinterpret_cast<const float4*>(wt + 16 * qq + 4 * q));
#pragma unroll
              for (int h = 0; h < 16; h += 4) heads4(cur + h, wv[h / 4], 16 * qq + h);
              if (qq < 3) tmem_wait_ld_regs16(nxt);
            }
            const float p0 = acc64[0].x + acc64[0].y;
            const float p1 = acc64[1].x + acc64[1].y;
            const float p2 = acc64[2].x + acc64[2].y;
            const float p3 = acc64[3].x + acc64[3].y;
            const float score = ((p0 + p1) + (p2 + p3)) * (0.5f * ksc);  // (the doubled sum, halved)
            if (my_j >= wn.x && my_j < wn.y) p.logits[static_cast<int64_t>(t0) * p.N + my_j] = score;
          }
        } else {
          // 64 / H tokens: two halves of 32 columns (every token lies inside one half)
          constexpr int TPH = 32 / H;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (half * TPH < tn) {  // (warp-uniform)
              // the window of each of the half's tokens, read by one lane each
              int2 wl = make_int2(0, 0);
              if (lane < TPH && half * TPH + lane < tn) wl = __ldg(p.tok_win + t0 + half * TPH + lane);
              bool any = false;
#pragma unroll
              for (int tl = 0; tl < TPH; ++tl) {
                const int wx = __shfl_sync(0xffffffffu, wl.x, tl), wy = __shfl_sync(0xffffffffu, wl.y, tl);
                any |= half * TPH + tl < tn && !(wj >= wy || wj + 32 <= wx);
              }
              if (!any) continue;
              const int cols = (min(tn, (half + 1) * TPH) - half * TPH) * H;
              float s[32];
              tmem_ld_x16(taddr + 32 * half, s);
              tmem_wait_ld_regs16(s);
              if (cols > 16) {
                tmem_ld_x16(taddr + 32 * half + 16, s + 16);
                tmem_wait_ld_regs16(s + 16);
              }
#pragma unroll
              for (int tl = 0; tl < TPH; ++tl) {
                const int wx = __shfl_sync(0xffffffffu, wl.x, tl), wy = __shfl_sync(0xffffffffu, wl.y, tl);
                const int t = t0 + half * TPH + tl;
                if (half * TPH + tl < tn && !(wj >= wy || wj + 32 <= wx)) {  // warp-uniform
                  const float score = head_sum<H>(s + tl * H, p.w + static_cast<int64_t>(t) * H) * ksc;
                  if (my_j >= wx && my_j < wy) p.logits[static_cast<int64_t>(t) * p.N + my_j] = score;
                }
              }
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[as]);
      }
      named_bar_sync(kKresEpiBar, kEpiThreads);  // every thread is done with the item's block list
      if (etid == 0) mbar_arrive(&item_empty[sl]);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace dsa
