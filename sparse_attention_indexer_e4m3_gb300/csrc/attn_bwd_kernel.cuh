// Gradients of the sparse attention on the tensor cores (TileLang README, "Sparse MLA Backward":
// delta = the row-wise product of the output and its gradient, dS = P (dP - delta), dQ = dS KV,
// dKV = dS^T Q + P^T dO accumulated atomically at the listed positions).  For query row t and
// head h, with p_j = e^{s_j - lse[t,h]} over the listed entries j (s_j = scale q[t,h,:].kv[j,:]):
//     dP_j = do[t,h,:] . kv[j,:],   delta = do[t,h,:] . o[t,h,:],   ds_j = scale p_j (dP_j - delta)
//     dq[t,h,:] = sum_j ds_j kv[j,:]
//     dkv[j,:] += ds_j q[t,h,:] + p_j do[t,h,:]
//     dsink[h] += -e^{sink[h] - lse[t,h]} delta
// (the scale is folded into ds once, so both products that use ds carry it).
//
// The structure follows the forward kernel: one CTA per query row at a time, all H <= 64 heads in
// one MMA column block, the row's list in blocks of 128 entries.  Per block:
//   gather (warps 12-15)  the block's kv rows into shared memory (cp.async, 128-byte swizzled
//                         chunks of [128 keys x 64 dims]); at a row's start also q and do (as
//                         [64 heads x 64 dims] chunks) and, per head, delta and lse (log2 units);
//   MMA (warp 0)          S^T and dP^T together: KV.[Q ; dO]^T (M = 128 keys, N = 2 x 64 heads,
//                         K = D);
//                         after the gradient warps: dQ^T += KV^T.dS^T (M = 128 dims per tile,
//                         N = 64 heads, K = 128 keys) and the block's
//                         dKV = dS.Q + P.dO (M = 128 keys, N = D, K = 64 heads);
//   gradient (warps 4-11) thread = (key, 32 heads): p and ds from S and dP in tensor memory,
//                         written as bf16 rows P[key][head], dS[key][head]; at a row's end dQ^T
//                         read out as fp32;
//   dKV (warps 12-15)     once the block's dKV is in tensor memory, thread = key row: its D
//                         columns added to dkv[j, :] with 16-byte atomic adds (masked entries
//                         skipped), overlapping the next block's gradient work.
// P and dS are stored once and read both as K-major A operands (dKV) and as MN-major B operands
// (dQ), exactly as the forward's weights are read in its second product.
//
// Tensor memory: S^T [0, 64), dP^T [64, 128), dQ^T tile m [128 + 64 m, 192 + 64 m),
// the block's dKV [256, 256 + D).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_kernel.cuh"
#include "attn_tc_kernel.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {

template <int D>
struct TcBwdLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kTiles = D / 128;
  static constexpr int kChunkBytes = kTcAttnKeys * 128;
  static constexpr int kQChunkBytes = kTcAttnHeads * 128;
  static constexpr int kKv = 0;
  static constexpr int kQ = kKv + kChunks * kChunkBytes;
  // q and do chunk c side by side: [q (64 heads) ; do (64 heads)] x 64 dims, 16 KB, so that one
  // N = 128 product computes S^T and dP^T together
  static constexpr int kQdChunkBytes = 2 * kQChunkBytes;
  static constexpr int kP = kQ + kChunks * kQdChunkBytes;   // bf16 [128 keys][64 heads]
  static constexpr int kDs = kP + kTcAttnKeys * 128;        // bf16 [128 keys][64 heads]
  static constexpr int kStage = kDs + kTcAttnKeys * 128;    // fp32 [128 keys][64 + 4] dKV columns
  static constexpr int kStagePitch = 64 * 4 + 16;           // bytes per staged row (padded)
  static constexpr int kIdx = kStage + kTcAttnKeys * kStagePitch;  // int32 [2][128] block entries
  static constexpr int kStat = kIdx + 2 * kTcAttnKeys * 4;  // float [2 rows][delta 64, lse 64]
  static constexpr int kMisc = kStat + 2 * 2 * kTcAttnHeads * 4;
  static constexpr int kBar = kMisc + 64;
  static constexpr int kNumBars = 12 + 2 * kTiles;
  static constexpr int kSmem = kBar + kNumBars * 8 + 1024;
};

__device__ __forceinline__ void red_add_f32x4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

template <int D>
__global__ void __launch_bounds__(kTcAttnThreads, 1) sparse_attn_bwd_tc_kernel(const AttnBwdParams p, unsigned* err) {
  static_assert(D == 128 || D == 256, "D: 128 or 256");
  using L = TcBwdLayout<D>;
  constexpr int kCh = L::kChunks;
  constexpr int kTi = L::kTiles;
  extern __shared__ __align__(1024) uint8_t tc_bwd_smem[];
  uint8_t* smem = tc_bwd_smem + ((1024u - (smem_addr(tc_bwd_smem) & 1023u)) & 1023u);
  uint8_t* kv_s = smem + L::kKv;
  uint8_t* q_s = smem + L::kQ;                        // q of chunk c at c * 16 KB
  uint8_t* do_s = smem + L::kQ + L::kQChunkBytes;     // do of chunk c at c * 16 KB + 8 KB
  uint8_t* p_s = smem + L::kP;
  uint8_t* ds_s = smem + L::kDs;
  uint8_t* stage_s = smem + L::kStage;
  int32_t* idx_s = reinterpret_cast<int32_t*>(smem + L::kIdx);
  float* stat_s = reinterpret_cast<float*>(smem + L::kStat);
  // [0] blocks of the row in flight, [1] its copy for the gradient warps, [2] for the gather
  // warps, [8..11] the gather warps' partial results
  volatile int* misc = reinterpret_cast<volatile int*>(smem + L::kMisc);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars + 0;      // q, do and the row's statistics staged (gather, 128)
  uint64_t* q_empty = bars + 1;     // the row's products are done with q and do (MMA)
  uint64_t* s_full = bars + 2;      // S^T, dP^T in tensor memory (MMA)
  uint64_t* p_full = bars + 3;      // P, dS written, S^T, dP^T read (gradient, 256)
  uint64_t* dkv_full = bars + 4;    // the block's dKV in tensor memory; P, dS read (MMA)
  uint64_t* dkv_empty = bars + 5;   // the block's dKV added to dkv (gather, 128)
  uint64_t* dq_done = bars + 6;     // the row's dQ^T complete (MMA)
  uint64_t* dq_empty = bars + 7;    // dQ^T read (gradient, 256)
  uint64_t* tok_full = bars + 8;
  uint64_t* tok_empty = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* kv_full = bars + 11;
  uint64_t* kv_empty = kv_full + kTi;
  uint64_t* drain = kv_empty + kTi;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = p.H;
  constexpr float kLog2e = 1.4426950408889634f;
  const float scale_log2 = p.scale * kLog2e;

  // q / do chunks: rows past H stay zero for the whole kernel
  for (int i = threadIdx.x; i < 2 * kCh * L::kQChunkBytes / 16; i += kTcAttnThreads)
    reinterpret_cast<uint4*>(q_s)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    mbar_init(q_full, kTcGatherThreads);
    mbar_init(q_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, kTcSoftThreads);
    mbar_init(dkv_full, 1);
    mbar_init(dkv_empty, kTcGatherThreads);
    mbar_init(dq_done, 1);
    mbar_init(dq_empty, kTcSoftThreads);
    mbar_init(tok_full, 1);
    mbar_init(tok_empty, 2);  // the MMA issuer and the gradient warps
    for (int m = 0; m < kTi; ++m) {
      mbar_init(&kv_full[m], kTcGatherThreads);
      mbar_init(&kv_empty[m], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  fence_proxy_async_shared();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  const uint32_t s_tmem = tbase;
  const uint32_t dp_tmem = tbase + 64;
  const uint32_t dq_tmem = tbase + 128;
  const uint32_t dkv_tmem = tbase + 256;

  if (warp >= 12) {
    // ------------------------------------------------------------------ gather and dKV
    // The gather warps also add each block's dKV (in tensor memory after the block's products)
    // to dkv: thread = key row gtid of the block (lane quarter gw), all D columns, 16-byte
    // atomic adds; this runs while the gradient warps work on the next block.  A row's
    // statistics (delta, lse) are computed one row ahead, during the previous row's gathers.
    const int gtid = threadIdx.x - 384;
    const int gw = warp - 12;
    const uint32_t lane_off = static_cast<uint32_t>(gw * 32) << 16;
    uint32_t gb = 0;
    int n = 0;
    // delta[h] = do . o and lse[h] in log2 units for row t into buffer `slot`, 16 heads per warp
    // (rows past H: delta 0, lse +inf, so their weights are 0); all loads of 4 heads in flight
    auto row_stats = [&](int t, int slot) {
      float* st = stat_s + slot * 2 * kTcAttnHeads;
      for (int h0 = 0; h0 < kTcAttnHeads / 4; h0 += 4) {
        uint32_t ov[4][D / 64], dv[4][D / 64];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int h = gw * (kTcAttnHeads / 4) + h0 + u;
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            ov[u][c] = dv[u][c] = 0u;
            if (h < H) {
              const int64_t off = (static_cast<int64_t>(t) * p.hs + h) * D / 2 + lane + 32 * c;
              ov[u][c] = __ldg(reinterpret_cast<const uint32_t*>(p.o) + off);
              dv[u][c] = __ldg(reinterpret_cast<const uint32_t*>(p.dout) + off);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int h = gw * (kTcAttnHeads / 4) + h0 + u;
          float acc = 0.f;
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            acc = fmaf(bf16_to_float(ov[u][c] & 0xFFFFu), bf16_to_float(dv[u][c] & 0xFFFFu), acc);
            acc = fmaf(bf16_to_float(ov[u][c] >> 16), bf16_to_float(dv[u][c] >> 16), acc);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
          if (lane == 0) {
            st[h] = acc;
            st[kTcAttnHeads + h] = h < H ? __ldg(p.lse + static_cast<int64_t>(t) * p.hs + h) * kLog2e : INFINITY;
          }
        }
      }
    };
    // adds block gbk's dKV to dkv (its entries are in idx_s slot gbk & 1), 64 columns at a time:
    // thread = key row reads them from tensor memory into a shared staging tile, then each warp
    // adds 2 rows x 256 bytes per instruction (16-byte atomic adds, whole cache lines per row)
    auto flush = [&](uint32_t gbk) {
      mbar_wait(dkv_full, gbk & 1u, abort_flag, err, 0x83);
      tc_fence_after_sync();
      const int32_t* ents = idx_s + (gbk & 1u) * kTcAttnKeys;
      for (int c0 = 0; c0 < D; c0 += 64) {
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          float v[16];
          tmem_ld_x16(dkv_tmem + lane_off + c0 + c, v);
          tmem_wait_ld_regs16(v);
          float4* dst = reinterpret_cast<float4*>(stage_s + gtid * L::kStagePitch + c * 4);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        }
        named_bar_sync(kTcGatherBar, kTcGatherThreads);
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          const int row = gw * 32 + 2 * i + (lane >> 4);
          const int ent = ents[row];
          if (ent >= 0) {
            const float4 x = *reinterpret_cast<const float4*>(stage_s + row * L::kStagePitch + (lane & 15) * 16);
            red_add_f32x4(p.dkv + static_cast<int64_t>(ent) * D + c0 + (lane & 15) * 4, x.x, x.y, x.z, x.w);
          }
        }
        named_bar_sync(kTcGatherBar, kTcGatherThreads);  // the staging tile is rewritten next
      }
      tc_fence_before_sync();
      mbar_arrive(dkv_empty);
    };
    if (static_cast<int>(blockIdx.x) < p.T) row_stats(blockIdx.x, 0);
    for (int t = blockIdx.x; t < p.T; t += gridDim.x, ++n) {
      const int32_t* list = p.idx + static_cast<int64_t>(t) * p.K;
      int last = -1;
      for (int j = gtid; j < p.K; j += kTcGatherThreads) {
        const int v = __ldg(list + j);
        if (v >= 0 && v < p.N) last = j;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      if (lane == 0) misc[8 + gw] = last;
      named_bar_sync(kTcGatherBar, kTcGatherThreads);
      if (gtid == 0) {
        int l4 = -1;
        for (int w = 0; w < 4; ++w) l4 = max(l4, misc[8 + w]);
        const int nb = (l4 + kTcAttnKeys) / kTcAttnKeys;
        mbar_wait(tok_empty, (static_cast<uint32_t>(n) & 1u) ^ 1u, abort_flag, err, 0x80);
        misc[0] = nb;
        mbar_arrive(tok_full);
        misc[2] = nb;
      }
      named_bar_sync(kTcGatherBar, kTcGatherThreads);
      const int nb = misc[2];
      // q and do of the row once the previous row's products are done with them
      if (n > 0) mbar_wait(q_empty, static_cast<uint32_t>(n - 1) & 1u, abort_flag, err, 0x81);
      for (int i = gtid; i < H * (D / 8); i += kTcGatherThreads) {
        const int h = i / (D / 8), pc = i % (D / 8);
        const uint32_t off = (pc / 8) * L::kQdChunkBytes + swz128(h, (pc % 8) * 16);
        const int64_t src = (static_cast<int64_t>(t) * p.hs + h) * D + pc * 8;
        cp_async16(smem_addr(q_s + off), p.q + src);
        cp_async16(smem_addr(do_s + off), p.dout + src);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_shared();
      mbar_arrive(q_full);
      const int rsub = gtid >> 4;
      const int cpiece = gtid & 15;
      const uint32_t dst0 = smem_addr(kv_s) + static_cast<uint32_t>((cpiece >> 3) * L::kChunkBytes + rsub * 128 +
                                                                      (((cpiece & 7) ^ (rsub & 7)) << 4));
      for (int b = 0; b < nb; ++b, ++gb) {
        // this block's entries: slot gb & 1 was last used by block gb - 2, already added to dkv
        int32_t* ent = idx_s + (gb & 1u) * kTcAttnKeys;
        {
          const int j = b * kTcAttnKeys + gtid;
          const int v = j < p.K ? __ldg(list + j) : -1;
          ent[gtid] = (v >= 0 && v < p.N) ? v : -1;
        }
        named_bar_sync(kTcGatherBar, kTcGatherThreads);
        const uint16_t* src[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) src[k] = p.kv + static_cast<int64_t>(max(ent[rsub + 8 * k], 0)) * D + cpiece * 8;
        for (int m = 0; m < kTi; ++m) {
          if (gb > 0) mbar_wait(&kv_empty[m], (gb - 1) & 1u, abort_flag, err, 0x82);
          const uint32_t dst = dst0 + static_cast<uint32_t>(2 * m * L::kChunkBytes);
#pragma unroll
          for (int k = 0; k < 16; ++k) cp_async16(dst + k * 1024, src[k] + 128 * m);
          cp_async_commit();
          if (m > 0) {
            cp_async_wait<1>();
            fence_proxy_async_shared();
            mbar_arrive(&kv_full[m - 1]);
          }
        }
        cp_async_wait<0>();
        fence_proxy_async_shared();
        mbar_arrive(&kv_full[kTi - 1]);
        if (b > 0) flush(gb - 1);  // the previous block's dKV, while the next products run
      }
      // this row's last dKV, then the next row's statistics (their buffer was last read by row
      // n - 1, whose products ended before this row's q and do were staged)
      if (nb > 0) flush(gb - 1);
      if (t + static_cast<int>(gridDim.x) < p.T) row_stats(t + gridDim.x, (n + 1) & 1);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_sdp = idesc_bf16(kTcAttnKeys, 2 * kTcAttnHeads, false, false);  // K-major x K-major
      const uint32_t id_dq = idesc_bf16(128, kTcAttnHeads, true, true);           // MN-major x MN-major
      const uint32_t id_dkv = idesc_bf16(kTcAttnKeys, D, false, true);            // K-major x MN-major
      const uint64_t kv_k = desc_sw128(smem_addr(kv_s), 16, 1024);          // keys x dims, K-major
      const uint64_t qd_k = desc_sw128(smem_addr(q_s), 16, 1024);   // [q ; do] 128 rows x dims, K-major
      const uint64_t kv_mn = desc_sw128(smem_addr(kv_s), L::kChunkBytes, 1024);   // dims x keys, MN-major
      const uint64_t ds_mn = desc_sw128(smem_addr(ds_s), 16384, 1024);            // heads x keys, MN-major
      const uint64_t ds_k = desc_sw128(smem_addr(ds_s), 16, 1024);                // keys x heads, K-major
      const uint64_t p_k = desc_sw128(smem_addr(p_s), 16, 1024);
      const uint64_t q_mn = desc_sw128(smem_addr(q_s), L::kQdChunkBytes, 1024);   // dims x heads, MN-major
      const uint64_t do_mn = desc_sw128(smem_addr(do_s), L::kQdChunkBytes, 1024);
      uint32_t gb = 0;
      int n = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.T; t += gridDim.x, ++n) {
        if (!mbar_wait(tok_full, static_cast<uint32_t>(n) & 1u, abort_flag, err, 0x90)) break;
        const int nb = misc[0];
        mbar_arrive(tok_empty);
        if (!mbar_wait(q_full, static_cast<uint32_t>(n) & 1u, abort_flag, err, 0x91)) break;
        for (int b = 0; b < nb; ++b, ++gb) {
          // S^T and dP^T = KV . [Q ; dO]^T over D / 16 steps (chunk c: dims [64c, 64c + 64))
          for (int c = 0; c < kCh; ++c) {
            if ((c & 1) == 0) {
              if (!mbar_wait(&kv_full[c / 2], gb & 1u, abort_flag, err, 0x92)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = kv_k + ((c * L::kChunkBytes + kk * 32) >> 4);
              // columns [0, 64): S^T, [64, 128): dP^T
              mma_bf16(s_tmem, a, qd_k + ((c * L::kQdChunkBytes + kk * 32) >> 4), id_sdp, (c | kk) ? 1u : 0u);
            }
          }
          if (!ok) break;
          mma_commit(s_full);
          if (!mbar_wait(p_full, gb & 1u, abort_flag, err, 0x93)) {
            ok = false;
            break;
          }
          // the row's first dQ product overwrites dQ^T: the previous row's must have been read
          if (b == 0 && n > 0 && !mbar_wait(dq_empty, static_cast<uint32_t>(n - 1) & 1u, abort_flag, err, 0x94)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // dQ^T += KV^T . dS^T: tile m = dims [128m, 128m + 128), K = 128 keys
          for (int m = 0; m < kTi; ++m) {
#pragma unroll
            for (int ks = 0; ks < kTcAttnKeys / 16; ++ks)
              mma_bf16(dq_tmem + 64 * m, kv_mn + ((2 * m * L::kChunkBytes + ks * 16 * 128) >> 4),
                       ds_mn + ((ks * 16 * 128) >> 4), id_dq, (b > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&kv_empty[m]);
          }
          // the block's dKV = dS . Q + P . dO (K = 64 heads in steps of 16), once the previous
          // block's has been read
          if (gb > 0 && !mbar_wait(dkv_empty, (gb - 1) & 1u, abort_flag, err, 0x95)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int hs = 0; hs < kTcAttnHeads / 16; ++hs)
            mma_bf16(dkv_tmem, ds_k + ((hs * 32) >> 4), q_mn + ((hs * 16 * 128) >> 4), id_dkv, hs > 0 ? 1u : 0u);
#pragma unroll
          for (int hs = 0; hs < kTcAttnHeads / 16; ++hs)
            mma_bf16(dkv_tmem, p_k + ((hs * 32) >> 4), do_mn + ((hs * 16 * 128) >> 4), id_dkv, 1u);
          mma_commit(dkv_full);
        }
        if (!ok) break;
        mma_commit(dq_done);
        mma_commit(q_empty);
      }
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ gradients
    const int etid = threadIdx.x - 128;
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    const int hb = half * kTcHalfHeads;  // heads [hb, hb + 32)
    const int r = quarter * 32 + lane;   // key of the block / dim of a dQ tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t gb = 0;
    int n = 0;
    for (int t = blockIdx.x; t < p.T; t += gridDim.x, ++n) {
      const int32_t* list = p.idx + static_cast<int64_t>(t) * p.K;
      if (etid == 0) {
        mbar_wait(tok_full, static_cast<uint32_t>(n) & 1u, abort_flag, err, 0xA0);
        misc[1] = misc[0];
        mbar_arrive(tok_empty);
      }
      named_bar_sync(kTcEpiBar, kTcSoftThreads);
      const int nb = misc[1];
      mbar_wait(q_full, static_cast<uint32_t>(n) & 1u, abort_flag, err, 0xA1);
      const float* st = stat_s + (n & 1) * 2 * kTcAttnHeads;
      // the sink's gradient: -e^{sink - lse} delta per head
      if (p.dsink != nullptr && p.sink != nullptr && etid < H)
        atomicAdd(p.dsink + etid, -exp2_approx(__ldg(p.sink + etid) * kLog2e - st[kTcAttnHeads + etid]) * st[etid]);
      int ent_next = (nb > 0 && r < p.K) ? __ldg(list + r) : -1;
      for (int b = 0; b < nb; ++b, ++gb) {
        const int ent = ent_next;
        {
          const int j = (b + 1) * kTcAttnKeys + r;
          ent_next = (b + 1 < nb && j < p.K) ? __ldg(list + j) : -1;
        }
        const bool valid = ent >= 0 && ent < p.N;
        mbar_wait(s_full, gb & 1u, abort_flag, err, 0xA2);
        tc_fence_after_sync();
        float x[kTcHalfHeads], y[kTcHalfHeads];
        tmem_ld_x16(s_tmem + lane_off + hb, x);
        tmem_ld_x16(s_tmem + lane_off + hb + 16, x + 16);
        tmem_ld_x16(dp_tmem + lane_off + hb, y);
        tmem_ld_x16(dp_tmem + lane_off + hb + 16, y + 16);
        tmem_wait_ld();
        // P and dS rows (bf16) of key r, heads [hb, hb + 32), once the previous block's products
        // have read both buffers
        if (gb > 0) mbar_wait(dkv_full, (gb - 1) & 1u, abort_flag, err, 0xA3);
#pragma unroll
        for (int h0 = 0; h0 < kTcHalfHeads; h0 += 8) {
          uint32_t pk[4], dk[4];
#pragma unroll
          for (int u = 0; u < 8; u += 2) {
            float pp[2], dd[2];
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              const int h = h0 + u + v;
              const float pr = valid ? exp2_approx(x[h] * scale_log2 - st[kTcAttnHeads + hb + h]) : 0.f;
              pp[v] = pr;
              dd[v] = p.scale * pr * (y[h] - st[hb + h]);
            }
            const __nv_bfloat162 a = __floats2bfloat162_rn(pp[0], pp[1]);
            const __nv_bfloat162 c = __floats2bfloat162_rn(dd[0], dd[1]);
            pk[u / 2] = *reinterpret_cast<const uint32_t*>(&a);
            dk[u / 2] = *reinterpret_cast<const uint32_t*>(&c);
          }
          const uint32_t off = swz128(r, 2 * (hb + h0));
          *reinterpret_cast<uint4*>(p_s + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(ds_s + off) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
        }
        fence_proxy_async_shared();
        tc_fence_before_sync();
        mbar_arrive(p_full);
      }
      // end of the row: dQ^T (lane = dim of tile m, columns = heads) as fp32 dq[t, h, d]
      mbar_wait(dq_done, static_cast<uint32_t>(n) & 1u, abort_flag, err, 0xA4);
      tc_fence_after_sync();
      float* dq = p.dq + static_cast<int64_t>(t) * p.hs * D;
      for (int m = 0; m < kTi; ++m) {
        const int d = 128 * m + r;
#pragma unroll
        for (int c = 0; c < kTcHalfHeads; c += 16) {
          float v[16];
          if (nb > 0) {
            tmem_ld_x16(dq_tmem + lane_off + 64 * m + hb + c, v);
            tmem_wait_ld_regs16(v);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int h = hb + c + e;
            if (h < H) dq[static_cast<int64_t>(h) * D + d] = v[e];
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(dq_empty);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

}  // namespace dsa
