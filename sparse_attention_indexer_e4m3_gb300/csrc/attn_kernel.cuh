// Sparse attention over the selected keys: the step that consumes the top-k indices (DeepSeek
// V4.1 sparse_attn_kernel page; TileLang README, "Sparse MLA Forward").  For query row t and
// head h, over the entries j of idx[t, :] that are not -1:
//     s_j = scale * q[t,h,:] . kv[j,:]
//     o[t,h,:] = sum_j e^{s_j - m} kv[j,:] / ( sum_j e^{s_j - m} + e^{sink[h] - m} )
// with a running maximum m (online softmax) and the optional per-head sink in the denominator
// only; every kv row is both key and value.  A row without keys writes zeros.
//
// First version, on the CUDA cores: a CTA takes one query row and kAttnHeads heads (two per
// warp), stages those heads' q in shared memory as fp32, and walks the index list in blocks of
// kAttnKeys entries: the block's kv rows are gathered into shared memory (rows padded by one
// word so that lane j reading row j is free of bank conflicts), lane j scores key j for the
// warp's two heads, the warp updates its running maximum and sum, and every lane accumulates
// D / 32 output columns per head.  bf16 in, fp32 arithmetic, bf16 out.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace dsa {

constexpr int kAttnThreads = 256;
constexpr int kAttnHeads = 2 * (kAttnThreads / 32);  // heads per CTA: two per warp
constexpr int kAttnKeys = 32;                        // index-list entries per block (one per lane)

struct AttnParams {
  const uint16_t* q;     // bf16 [T, hs, D] (heads [0, H) used)
  const uint16_t* kv;    // bf16 [N, D]
  const float* sink;     // [H] or null
  const int32_t* idx;    // [T, K]
  uint16_t* out;         // bf16 [T, hs, D]
  float* lse;            // [T, hs] or null: ln of each softmax denominator (the sink included)
  int T, N, H, K;
  float scale;
  int hs;  // heads per token in q / out / lse (row stride in heads, >= H)
};

// Arguments of the backward (gradient) kernel.
struct AttnBwdParams {
  const uint16_t* q;     // bf16 [T, hs, D] (heads [0, H) used)
  const uint16_t* kv;    // bf16 [N, D]
  const float* sink;     // [H] or null
  const int32_t* idx;    // [T, K]
  const uint16_t* o;     // bf16 [T, hs, D], the forward's output
  const float* lse;      // [T, hs], the forward's ln denominators
  const uint16_t* dout;  // bf16 [T, hs, D]
  float* dq;             // [T, hs, D]
  float* dkv;            // [N, D], zeroed before the launch
  float* dsink;          // [H] or null, zeroed before the launch
  int T, N, H, K;
  float scale;
  int hs;  // heads per token in q / o / lse / dout / dq (row stride in heads, >= H)
};

__host__ __device__ constexpr size_t attn_smem_bytes(int D) {
  return static_cast<size_t>(kAttnHeads) * D * 4 + static_cast<size_t>(kAttnKeys) * (D + 1) * 4 + kAttnKeys * 4;
}

__device__ __forceinline__ float bf16_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

template <int D>
__global__ void __launch_bounds__(kAttnThreads) sparse_attn_kernel(const AttnParams p) {
  static_assert(D % 32 == 0 && D <= 512, "D: a multiple of 32, at most 512");
  constexpr int C = D / 32;  // output columns per lane and head
  constexpr int KVS = D + 1;  // padded kv row stride (words)
  extern __shared__ __align__(16) uint8_t smem_raw[];
  float* q_s = reinterpret_cast<float*>(smem_raw);            // [kAttnHeads][D]
  float* kv_s = q_s + kAttnHeads * D;                          // [kAttnKeys][D + 1]
  int32_t* idx_s = reinterpret_cast<int32_t*>(kv_s + kAttnKeys * KVS);  // [kAttnKeys]

  const int t = blockIdx.x;
  const int h0 = blockIdx.y * kAttnHeads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // this CTA's heads of q[t] (rows past H are zeros and never stored)
  for (int e = tid; e < kAttnHeads * D; e += kAttnThreads) {
    const int hh = e / D, d = e % D;
    const int h = h0 + hh;
    q_s[e] = h < p.H ? bf16_to_float(p.q[(static_cast<int64_t>(t) * p.hs + h) * D + d]) : 0.f;
  }

  // per warp: heads hA = h0 + 2 warp, hB = hA + 1
  const float* qa = q_s + (2 * warp) * D;
  const float* qb = qa + D;
  float m[2] = {-1e30f, -1e30f};  // running maxima (finite: an all-masked block leaves them unchanged)
  float l[2] = {0.f, 0.f};        // running sums of e^{s - m}
  float acc[2][C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[0][c] = acc[1][c] = 0.f;

  const int32_t* row_idx = p.idx + static_cast<int64_t>(t) * p.K;
  for (int b0 = 0; b0 < p.K; b0 += kAttnKeys) {
    __syncthreads();  // the previous block's kv rows are no longer read (and q_s is written)
    if (tid < kAttnKeys) {
      int j = b0 + tid < p.K ? row_idx[b0 + tid] : -1;
      if (j < 0 || j >= p.N) j = -1;  // (an entry outside [0, N) is skipped like -1)
      idx_s[tid] = j;
    }
    __syncthreads();
    // gather: the block's kv rows as bf16 pairs (consecutive lanes, consecutive words), zeros
    // for skipped entries
    constexpr int PAIRS = D / 2;
    for (int c = tid; c < kAttnKeys * PAIRS; c += kAttnThreads) {
      const int r = c / PAIRS, pw = c % PAIRS;
      const int j = idx_s[r];
      const uint32_t w = j >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(p.kv + static_cast<int64_t>(j) * D) + pw) : 0u;
      float* dst = kv_s + r * KVS + 2 * pw;
      dst[0] = bf16_to_float(w & 0xFFFFu);
      dst[1] = bf16_to_float(w >> 16);
    }
    __syncthreads();

    // scores of key `lane` for the warp's two heads
    const bool valid = idx_s[lane] >= 0;
    const float* kr = kv_s + lane * KVS;
    float sa = 0.f, sb = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; d += 4) {
      const float4 a4 = *reinterpret_cast<const float4*>(qa + d);
      const float4 b4 = *reinterpret_cast<const float4*>(qb + d);
      const float k0 = kr[d], k1 = kr[d + 1], k2 = kr[d + 2], k3 = kr[d + 3];
      sa = fmaf(a4.x, k0, sa);
      sa = fmaf(a4.y, k1, sa);
      sa = fmaf(a4.z, k2, sa);
      sa = fmaf(a4.w, k3, sa);
      sb = fmaf(b4.x, k0, sb);
      sb = fmaf(b4.y, k1, sb);
      sb = fmaf(b4.z, k2, sb);
      sb = fmaf(b4.w, k3, sb);
    }
    const float ninf = __int_as_float(0xff800000);  // -inf: e^{-inf - m} = 0
    float s[2] = {valid ? sa * p.scale : ninf, valid ? sb * p.scale : ninf};

    // online softmax update per head, then the block's weighted kv rows
    float pr[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float mb = s[hh];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
      const float mn = fmaxf(m[hh], mb);
      const float alpha = expf(m[hh] - mn);
      pr[hh] = expf(s[hh] - mn);  // 0 for a skipped entry
      float sum = pr[hh];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l[hh] = l[hh] * alpha + sum;
      m[hh] = mn;
#pragma unroll
      for (int c = 0; c < C; ++c) acc[hh][c] *= alpha;
    }
    for (int r = 0; r < kAttnKeys; ++r) {
      const float pa = __shfl_sync(0xffffffffu, pr[0], r);
      const float pb = __shfl_sync(0xffffffffu, pr[1], r);
      const float* vr = kv_s + r * KVS + lane;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const float v = vr[32 * c];
        acc[0][c] = fmaf(pa, v, acc[0][c]);
        acc[1][c] = fmaf(pb, v, acc[1][c]);
      }
    }
  }

  // normalise: the sink joins the maximum, then the denominator
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = h0 + 2 * warp + hh;
    if (h >= p.H) continue;
    float mf = m[hh], lf = l[hh], f = 1.f;
    float den = lf;
    if (p.sink) {
      const float sk = p.sink[h];
      mf = fmaxf(m[hh], sk);
      f = expf(m[hh] - mf);
      den = lf * f + expf(sk - mf);
    }
    const float inv = den > 0.f ? f / den : 0.f;  // no key and no sink: zeros
    if (p.lse) p.lse[static_cast<int64_t>(t) * p.hs + h] = den > 0.f ? mf + logf(den) : -INFINITY;
    uint16_t* o = p.out + (static_cast<int64_t>(t) * p.hs + h) * D + lane;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const __nv_bfloat16 v = __float2bfloat16_rn(acc[hh][c] * inv);
      o[32 * c] = *reinterpret_cast<const uint16_t*>(&v);
    }
  }
}

}  // namespace dsa
