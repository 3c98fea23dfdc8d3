// Sparse attention over the selected keys on the tensor cores: the step that consumes the top-k
// indices (DeepSeek V4.1 sparse_attn_kernel page; TileLang README, "Sparse MLA Forward").  For
// query row t and head h, over the entries j of idx[t, :] that name a key:
//     s_j = scale * q[t,h,:] . kv[j,:]
//     o[t,h,:] = sum_j e^{s_j - m} kv[j,:] / ( sum_j e^{s_j - m} + e^{sink[h] - m} )
// (every kv row is both key and value, the sink joins the denominator only, a row without keys
// writes zeros).  The weights e^{s_j - m} enter the weighted sum as bf16, as the V4.1 kernel
// casts them before its second product; the denominator sums them in fp32.
//
// One CTA per query row at a time (persistent over rows), all H <= 64 heads together, so each
// listed kv row is gathered once per query row.  The row's index list is walked in blocks of 128
// entries; per block:
//   gather   (warps 12-15) the block's kv rows into shared memory with cp.async, as D / 64
//                          chunks of [128 keys x 128 bytes] in the 128-byte swizzled layout;
//   score    (warp 0)      S^T = KV . Q^T: M = 128 keys, N = 64 heads, K = D in 16-element
//                          steps (tcgen05.mma kind::f16, bf16 x bf16 -> fp32 in tensor memory);
//   softmax  (warps 4-11)  thread = (key, half of the heads): its 32 scores from tensor memory, masked, scaled to
//                          log2 units; the running per-head maximum is raised only when a score
//                          exceeds it by more than 2^8 (then the partial sums and the output
//                          accumulators are rescaled); weights 2^(x - m) written as bf16 rows
//                          P[key][head] into shared memory; per-thread partial sums;
//   weighted (warp 0)      O^T += KV^T . P^T: M = 128 output dims (D / 128 tiles), N = 64
//                          heads, K = 128 keys, reading the same kv chunks as an MN-major
//                          operand and P as an MN-major operand.
// The gather of the next block's chunk pair m starts as soon as the weighted sum of tile m has
// read it.  At the end of a row: the partial sums are reduced across the 128 keys, the sink
// added, and O^T divided and written as bf16.
//
// Tensor memory: S^T in columns [0, 64), O^T tile m in columns [128 + 64 m, 192 + 64 m).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_kernel.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {

constexpr int kTcAttnKeys = 128;      // listed keys per block (M of the score product)
constexpr int kTcAttnHeads = 64;      // heads per row (N of both products); H <= 64
constexpr int kTcAttnThreads = 512;   // warp 0: MMA + tensor memory; 4-11: softmax / output; 12-15: gather
constexpr int kTcGatherThreads = 128;
constexpr int kTcSoftThreads = 256;   // 8 warps: lane quarter q = warp % 4, heads [32 half, 32 half + 32)
constexpr int kTcHalfHeads = 32;
constexpr int kTcEpiBar = 1;          // named barrier of the softmax warps
constexpr int kTcGatherBar = 2;       // named barrier of the gather warps
constexpr float kTcLazyLog2 = 8.f;    // the running maximum moves only when exceeded by 2^8

template <int D>
struct TcAttnLayout {
  static constexpr int kChunks = D / 64;                     // 128-byte chunks of a row
  static constexpr int kTiles = D / 128;                     // output tiles = chunk pairs
  static constexpr int kChunkBytes = kTcAttnKeys * 128;      // one chunk of the kv block
  static constexpr int kQChunkBytes = kTcAttnHeads * 128;    // one chunk of q
  static constexpr int kKv = 0;
  static constexpr int kQ = kKv + kChunks * kChunkBytes;
  static constexpr int kP = kQ + kChunks * kQChunkBytes;     // bf16 [128 keys][64 heads]
  static constexpr int kIdx = kP + kTcAttnKeys * 128;        // int32 [2][128] block entries
  static constexpr int kRed = kIdx + 2 * kTcAttnKeys * 4;    // float [4][64] cross-warp scratch
  static constexpr int kMax = kRed + 4 * kTcAttnHeads * 4;   // float [64] running maximum (log2 units)
  static constexpr int kAlpha = kMax + kTcAttnHeads * 4;     // float [64] rescale factors / 1 / l
  static constexpr int kMisc = kAlpha + kTcAttnHeads * 4;    // int [16]
  static constexpr int kBar = kMisc + 64;
  static constexpr int kNumBars = 10 + 2 * kTiles;
  static constexpr int kSmem = kBar + kNumBars * 8 + 1024;   // + alignment slack
};

// Byte offset of (row, byte) in a 128-byte swizzled [rows x 128 B] chunk.
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t byte) {
  return row * 128u + ((((byte >> 4) ^ (row & 7u)) << 4) | (byte & 15u));
}

// tcgen05 shared-memory descriptor, 128-byte swizzle: leading / stride byte offsets as given.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16 with bf16 operands and an fp32 accumulator; a_mn / b_mn:
// the operand is MN-major (transposed) rather than K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn ? 1u << 15 : 0u) | (b_mn ? 1u << 16 : 0u) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const float* v) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// OR of a predicate over the `n` threads of named barrier `id` (a barrier too).
__device__ __forceinline__ bool bar_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Reduces 64 values per lane across the warp's 32 lanes, one value of each of 64 heads per lane,
// by recursive halving: each step a lane keeps one half of its values and receives the other
// half from its partner.  Afterwards v[0], v[1] hold the reduction of heads 2 lane, 2 lane + 1.
template <class Op>
__device__ __forceinline__ void xpose_reduce64(float (&v)[64], int lane, Op op) {
  // partner offsets 16, 8, 4, 2, 1 over 64, 32, 16, 8, 4 values
#define DSA_XR_STEP(OFF, HALF)                                        \
  {                                                                   \
    const bool up = (lane & (OFF)) != 0;                              \
    _Pragma("unroll") for (int i = 0; i < (HALF); ++i) {              \
      const float send = up ? v[i] : v[i + (HALF)];                   \
      const float keep = up ? v[i + (HALF)] : v[i];                   \
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, (OFF)));     \
    }                                                                 \
  }
  DSA_XR_STEP(16, 32)
  DSA_XR_STEP(8, 16)
  DSA_XR_STEP(4, 8)
  DSA_XR_STEP(2, 4)
  DSA_XR_STEP(1, 2)
#undef DSA_XR_STEP
}

// The same over 32 values per lane (one of each of 32 heads): afterwards v[0] holds head `lane`.
template <class Op>
__device__ __forceinline__ void xpose_reduce32(float (&v)[32], int lane, Op op) {
#define DSA_XR_STEP(OFF, HALF)                                        \
  {                                                                   \
    const bool up = (lane & (OFF)) != 0;                              \
    _Pragma("unroll") for (int i = 0; i < (HALF); ++i) {              \
      const float send = up ? v[i] : v[i + (HALF)];                   \
      const float keep = up ? v[i + (HALF)] : v[i];                   \
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, (OFF)));     \
    }                                                                 \
  }
  DSA_XR_STEP(16, 16)
  DSA_XR_STEP(8, 8)
  DSA_XR_STEP(4, 4)
  DSA_XR_STEP(2, 2)
  DSA_XR_STEP(1, 1)
#undef DSA_XR_STEP
}

// 2^x for x <= 2^8 (the hardware approximation; 2^-inf = 0).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(kTcAttnThreads, 1) sparse_attn_tc_kernel(const AttnParams p, unsigned* err) {
  static_assert(D == 128 || D == 256 || D == 512, "D: 128, 256 or 512");
  using L = TcAttnLayout<D>;
  constexpr int kCh = L::kChunks;
  constexpr int kTi = L::kTiles;
  extern __shared__ __align__(1024) uint8_t tc_attn_smem[];
  uint8_t* smem = tc_attn_smem + ((1024u - (smem_addr(tc_attn_smem) & 1023u)) & 1023u);
  uint8_t* kv_s = smem + L::kKv;
  uint8_t* q_s = smem + L::kQ;
  uint8_t* p_s = smem + L::kP;
  int32_t* idx_s = reinterpret_cast<int32_t*>(smem + L::kIdx);
  float* red_s = reinterpret_cast<float*>(smem + L::kRed);
  float* max_s = reinterpret_cast<float*>(smem + L::kMax);
  float* alpha_s = reinterpret_cast<float*>(smem + L::kAlpha);
  // [0] blocks of the row in flight, [1] its copy for the softmax warps, [2] for the gather warps,
  // [8..11] the gather warps' partial results
  volatile int* misc = reinterpret_cast<volatile int*>(smem + L::kMisc);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* s_full = bars + 2;
  uint64_t* p_full = bars + 3;
  uint64_t* pv_done = bars + 4;
  uint64_t* o_empty = bars + 5;
  uint64_t* tok_full = bars + 6;   // [1]: one row in flight between the gather and the rest
  uint64_t* tok_empty = bars + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* kv_full = bars + 9;
  uint64_t* kv_empty = kv_full + kTi;
  uint64_t* drain = kv_empty + kTi;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = p.H;
  const float scale_log2 = p.scale * 1.4426950408889634f;

  // q chunks: rows past H stay zero for the whole kernel
  for (int i = threadIdx.x; i < kCh * L::kQChunkBytes / 16; i += kTcAttnThreads)
    reinterpret_cast<uint4*>(q_s)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    mbar_init(q_full, kTcGatherThreads);
    mbar_init(q_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, kTcSoftThreads);
    mbar_init(pv_done, 1);
    mbar_init(o_empty, kTcSoftThreads);
    mbar_init(tok_full, 1);
    mbar_init(tok_empty, 2);  // the MMA issuer and the softmax warps
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
  const uint32_t o_tmem = tbase + 128;

  if (warp >= 12) {
    // ------------------------------------------------------------------ gather
    const int gtid = threadIdx.x - 384;
    uint32_t gb = 0;  // blocks of this CTA so far
    int n = 0;        // rows of this CTA so far
    for (int t = blockIdx.x; t < p.T; t += gridDim.x, ++n) {
      const int32_t* list = p.idx + static_cast<int64_t>(t) * p.K;
      // blocks to walk: up to the last entry that names a key
      int last = -1;
      for (int j = gtid; j < p.K; j += kTcGatherThreads) {
        const int v = __ldg(list + j);
        if (v >= 0 && v < p.N) last = j;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      if (lane == 0) misc[8 + (warp - 12)] = last;
      named_bar_sync(kTcGatherBar, kTcGatherThreads);
      if (gtid == 0) {
        int l4 = -1;
        for (int w = 0; w < 4; ++w) l4 = max(l4, misc[8 + w]);
        const int nb = (l4 + kTcAttnKeys) / kTcAttnKeys;  // ceil((l4 + 1) / 128)
        mbar_wait(tok_empty, (static_cast<uint32_t>(n) & 1u) ^ 1u, abort_flag, err, 0x40);
        misc[0] = nb;
        mbar_arrive(tok_full);
        misc[2] = nb;  // for the gather warps
      }
      named_bar_sync(kTcGatherBar, kTcGatherThreads);
      const int nb = misc[2];
      // q of the row (H rows of D bf16) once the previous row's score products are done
      if (n > 0) mbar_wait(q_empty, static_cast<uint32_t>(n - 1) & 1u, abort_flag, err, 0x41);
      for (int i = gtid; i < H * (D / 8); i += kTcGatherThreads) {
        const int h = i / (D / 8), pc = i % (D / 8);
        cp_async16(smem_addr(q_s + (pc / 8) * L::kQChunkBytes + swz128(h, (pc % 8) * 16)),
                   p.q + (static_cast<int64_t>(t) * p.hs + h) * D + pc * 8);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_shared();
      mbar_arrive(q_full);
      // Thread gtid copies, for every chunk pair, the 16-byte piece (gtid & 15) of rows
      // gtid / 16 + 8k (k < 16): the row's low 3 bits, hence its swizzle, are fixed per thread.
      const int rsub = gtid >> 4;
      const int cpiece = gtid & 15;
      const uint32_t dst0 = smem_addr(kv_s) + static_cast<uint32_t>((cpiece >> 3) * L::kChunkBytes + rsub * 128 +
                                                                      (((cpiece & 7) ^ (rsub & 7)) << 4));
      for (int b = 0; b < nb; ++b, ++gb) {
        // this block's entries (a free slot: the softmax of block gb - 2 is finished, since the
        // weighted sum of block gb - 1, awaited below for the previous block, followed it)
        int32_t* ent = idx_s + (gb & 1u) * kTcAttnKeys;
        {
          const int j = b * kTcAttnKeys + gtid;
          const int v = j < p.K ? __ldg(list + j) : -1;
          ent[gtid] = (v >= 0 && v < p.N) ? v : -1;
        }
        named_bar_sync(kTcGatherBar, kTcGatherThreads);
        const uint16_t* src[16];  // piece cpiece of the thread's 16 rows (a masked entry reads row 0)
#pragma unroll
        for (int k = 0; k < 16; ++k) src[k] = p.kv + static_cast<int64_t>(max(ent[rsub + 8 * k], 0)) * D + cpiece * 8;
        for (int m = 0; m < kTi; ++m) {
          if (gb > 0) mbar_wait(&kv_empty[m], (gb - 1) & 1u, abort_flag, err, 0x42);
          // chunks 2m, 2m + 1 of the 128 rows
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
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16(kTcAttnKeys, kTcAttnHeads, false, false);
      const uint32_t id_pv = idesc_bf16(128, kTcAttnHeads, true, true);
      const uint64_t kv_k = desc_sw128(smem_addr(kv_s), 16, 1024);         // K-major: keys x dims
      const uint64_t q_k = desc_sw128(smem_addr(q_s), 16, 1024);           // K-major: heads x dims
      const uint64_t kv_mn = desc_sw128(smem_addr(kv_s), L::kChunkBytes, 1024);  // MN-major: dims x keys
      const uint64_t p_mn = desc_sw128(smem_addr(p_s), 16384, 1024);       // MN-major: heads x keys
      uint32_t gb = 0;
      int n = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.T; t += gridDim.x, ++n) {
        if (!mbar_wait(tok_full, static_cast<uint32_t>(n) & 1u, abort_flag, err, 0x50)) break;
        const int nb = misc[0];
        mbar_arrive(tok_empty);
        if (!mbar_wait(q_full, static_cast<uint32_t>(n) & 1u, abort_flag, err, 0x51)) break;
        for (int b = 0; b < nb; ++b, ++gb) {
          // S^T = KV . Q^T over D / 16 steps; chunk c holds dims [64c, 64c + 64)
          for (int c = 0; c < kCh; ++c) {
            if ((c & 1) == 0) {
              if (!mbar_wait(&kv_full[c / 2], gb & 1u, abort_flag, err, 0x53)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(s_tmem, kv_k + ((c * L::kChunkBytes + kk * 32) >> 4), q_k + ((c * L::kQChunkBytes + kk * 32) >> 4),
                       id_qk, (c | kk) ? 1u : 0u);
          }
          if (!ok) break;
          mma_commit(s_full);
          // O^T += KV^T . P^T: tile m = dims [128m, 128m + 128) = chunks 2m, 2m + 1; K = 128 keys
          if (!mbar_wait(p_full, gb & 1u, abort_flag, err, 0x54)) {
            ok = false;
            break;
          }
          // the row's first weighted sum overwrites O: the previous row's output must be read
          if (b == 0 && n > 0 && !mbar_wait(o_empty, static_cast<uint32_t>(n - 1) & 1u, abort_flag, err, 0x52)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          for (int m = 0; m < kTi; ++m) {
#pragma unroll
            for (int ks = 0; ks < kTcAttnKeys / 16; ++ks)
              mma_bf16(o_tmem + 64 * m, kv_mn + ((2 * m * L::kChunkBytes + ks * 16 * 128) >> 4),
                       p_mn + ((ks * 16 * 128) >> 4), id_pv, (b > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&kv_empty[m]);
          }
          mma_commit(pv_done);
        }
        if (!ok) break;
        mma_commit(q_empty);
      }
      // every MMA issued by this thread has completed once `drain` flips
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax and output
    const int etid = threadIdx.x - 128;
    const int quarter = warp & 3;                 // tensor-memory lane quarter
    const int hb = ((warp - 4) >> 2) * kTcHalfHeads;  // this thread's heads [hb, hb + 32)
    const int r = quarter * 32 + lane;            // key of the block (score rows) / dim of a tile (output rows)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t gb = 0;
    int n = 0;
    float lsum[kTcHalfHeads];
    for (int t = blockIdx.x; t < p.T; t += gridDim.x, ++n) {
      const int32_t* list = p.idx + static_cast<int64_t>(t) * p.K;
      if (etid == 0) {
        mbar_wait(tok_full, static_cast<uint32_t>(n) & 1u, abort_flag, err, 0x60);
        misc[1] = misc[0];
        mbar_arrive(tok_empty);
      }
      if (etid < kTcAttnHeads) max_s[etid] = -INFINITY;
#pragma unroll
      for (int h = 0; h < kTcHalfHeads; ++h) lsum[h] = 0.f;
      named_bar_sync(kTcEpiBar, kTcSoftThreads);
      const int nb = misc[1];
      int ent_next = (nb > 0 && r < p.K) ? __ldg(list + r) : -1;  // this key's list entry, one block ahead
      for (int b = 0; b < nb; ++b, ++gb) {
        const int ent = ent_next;
        {
          const int j = (b + 1) * kTcAttnKeys + r;
          ent_next = (b + 1 < nb && j < p.K) ? __ldg(list + j) : -1;
        }
        const bool valid = ent >= 0 && ent < p.N;
        mbar_wait(s_full, gb & 1u, abort_flag, err, 0x61);
        tc_fence_after_sync();
        float x[kTcHalfHeads];
        tmem_ld_x16(s_tmem + lane_off + hb, x);
        tmem_ld_x16(s_tmem + lane_off + hb + 16, x + 16);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < kTcHalfHeads; ++h) x[h] = valid ? x[h] * scale_log2 : -INFINITY;
        // does a score exceed its head's running maximum by more than 2^8 (or is it the first)?
        bool exceed = false;
#pragma unroll
        for (int h = 0; h < kTcHalfHeads; h += 4) {
          const float4 mv = *reinterpret_cast<const float4*>(max_s + hb + h);
          exceed |= (x[h] > mv.x + kTcLazyLog2) | (x[h + 1] > mv.y + kTcLazyLog2) | (x[h + 2] > mv.z + kTcLazyLog2) |
                    (x[h + 3] > mv.w + kTcLazyLog2);
        }
        const bool raise = bar_or(kTcEpiBar, kTcSoftThreads, exceed);
        if (raise) {
          // (the reduction consumes x; the scores are read again from tensor memory below)
          xpose_reduce32(x, lane, [](float a, float c) { return fmaxf(a, c); });
          red_s[quarter * kTcAttnHeads + hb + lane] = x[0];
          named_bar_sync(kTcEpiBar, kTcSoftThreads);
          if (etid < kTcAttnHeads) {
            const float bm = fmaxf(fmaxf(red_s[etid], red_s[kTcAttnHeads + etid]),
                                   fmaxf(red_s[2 * kTcAttnHeads + etid], red_s[3 * kTcAttnHeads + etid]));
            const float mo = max_s[etid];
            const float mn = (bm > mo + kTcLazyLog2) ? bm : mo;
            alpha_s[etid] = (mo == -INFINITY || mn == mo) ? 1.f : exp2f(mo - mn);
            max_s[etid] = mn;
          }
          named_bar_sync(kTcEpiBar, kTcSoftThreads);
          bool rescale = false;
#pragma unroll
          for (int h = 0; h < kTcHalfHeads; ++h) {
            const float a = alpha_s[hb + h];
            lsum[h] *= a;
            rescale |= a != 1.f;
          }
          // the output accumulators of earlier blocks follow the new maximum (this thread: its
          // dim row r of every tile, its 32 head columns)
          rescale = bar_or(kTcEpiBar, kTcSoftThreads, rescale);
          if (b > 0 && rescale) {
            mbar_wait(pv_done, (gb - 1) & 1u, abort_flag, err, 0x62);
            tc_fence_after_sync();
            for (int m = 0; m < kTi; ++m) {
#pragma unroll
              for (int c = 0; c < kTcHalfHeads; c += 16) {
                float o[16];
                tmem_ld_x16(o_tmem + lane_off + 64 * m + hb + c, o);
                tmem_wait_ld_regs16(o);
#pragma unroll
                for (int j = 0; j < 16; ++j) o[j] *= alpha_s[hb + c + j];
                tmem_st_x16(o_tmem + lane_off + 64 * m + hb + c, o);
              }
            }
            tmem_wait_st();
          }
          tmem_ld_x16(s_tmem + lane_off + hb, x);
          tmem_ld_x16(s_tmem + lane_off + hb + 16, x + 16);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < kTcHalfHeads; ++h) x[h] = valid ? x[h] * scale_log2 : -INFINITY;
        }
        // weights 2^(x - m) (the maximum of a head without keys yet counts as 0), written into
        // the bf16 row P[key r] (this thread: heads [hb, hb + 32)) once the previous block's
        // weighted sum has read P
        if (gb > 0) mbar_wait(pv_done, (gb - 1) & 1u, abort_flag, err, 0x63);
#pragma unroll
        for (int h0 = 0; h0 < kTcHalfHeads; h0 += 8) {
          uint32_t pk[4];
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const float4 mv = *reinterpret_cast<const float4*>(max_s + hb + h0 + 4 * q2);
            const float mu[4] = {mv.x, mv.y, mv.z, mv.w};
            float e[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int h = h0 + 4 * q2 + u;
              e[u] = exp2_approx(x[h] - (mu[u] == -INFINITY ? 0.f : mu[u]));
              lsum[h] += e[u];
            }
            const __nv_bfloat162 a = __floats2bfloat162_rn(e[0], e[1]);
            const __nv_bfloat162 c = __floats2bfloat162_rn(e[2], e[3]);
            pk[2 * q2] = *reinterpret_cast<const uint32_t*>(&a);
            pk[2 * q2 + 1] = *reinterpret_cast<const uint32_t*>(&c);
          }
          *reinterpret_cast<uint4*>(p_s + swz128(r, 2 * (hb + h0))) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async_shared();
        tc_fence_before_sync();
        mbar_arrive(p_full);
      }
      // end of the row: denominators (partial sums across the 128 keys, plus the sink)
      xpose_reduce32(lsum, lane, [](float a, float c) { return a + c; });
      red_s[quarter * kTcAttnHeads + hb + lane] = lsum[0];
      named_bar_sync(kTcEpiBar, kTcSoftThreads);
      if (etid < kTcAttnHeads) {
        float l = (red_s[etid] + red_s[kTcAttnHeads + etid]) + (red_s[2 * kTcAttnHeads + etid] + red_s[3 * kTcAttnHeads + etid]);
        const float m = max_s[etid] == -INFINITY ? 0.f : max_s[etid];
        if (p.sink != nullptr && etid < H) l += exp2f(__ldg(p.sink + etid) * 1.4426950408889634f - m);
        alpha_s[etid] = l > 0.f ? 1.f / l : 0.f;
        // ln of the denominator: the weights were 2^(x - m) in log2 units
        if (p.lse != nullptr && etid < H)
          p.lse[static_cast<int64_t>(t) * p.hs + etid] = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
      named_bar_sync(kTcEpiBar, kTcSoftThreads);
      uint16_t* out = p.out + static_cast<int64_t>(t) * p.hs * D;
      if (nb > 0) {
        mbar_wait(pv_done, (gb - 1) & 1u, abort_flag, err, 0x64);
        tc_fence_after_sync();
        for (int m = 0; m < kTi; ++m) {
          const int d = 128 * m + r;
#pragma unroll
          for (int c = 0; c < kTcHalfHeads; c += 16) {
            float o[16];
            tmem_ld_x16(o_tmem + lane_off + 64 * m + hb + c, o);
            tmem_wait_ld_regs16(o);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int h = hb + c + j;
              if (h < H) {
                const __nv_bfloat16 ob = __float2bfloat16_rn(o[j] * alpha_s[h]);
                out[static_cast<int64_t>(h) * D + d] = *reinterpret_cast<const uint16_t*>(&ob);
              }
            }
          }
        }
      } else {
        for (int m = 0; m < kTi; ++m)
          for (int h = hb; h < min(H, hb + kTcHalfHeads); ++h) out[static_cast<int64_t>(h) * D + 128 * m + r] = 0;
      }
      tc_fence_before_sync();
      mbar_arrive(o_empty);
      named_bar_sync(kTcEpiBar, kTcSoftThreads);  // alpha_s / max_s / misc[1] are rewritten by the next row
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

}  // namespace dsa
