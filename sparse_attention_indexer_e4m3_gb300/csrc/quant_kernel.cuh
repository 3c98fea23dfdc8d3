// e4m3 quantise-on-write of index key rows: the step that produces the fp8 index keys the scorer
// reads (TileLang deepseek_v32 README, "Lightning Indexer": the index vectors are FP8-quantized;
// 448 is the largest e4m3 value, as the FlashInfer MLA-decode discussion notes).
//
// Per row of D bf16 values x:  s = max_j |x_j| / 448 (fp32 division);  code_j = x_j / s (fp32
// division) rounded to the nearest e4m3 value, ties to even, saturating at +-448 (the hardware
// conversion cvt.rn.satfinite).  A row of zeros gets s = 0 and all codes 0.  Inputs must be
// finite.
//
// HBM-bound (2D bytes read, D + 4 written per row).  A warp takes kRowsPerWarp consecutive rows
// per step with all their loads issued first, so that enough bytes are in flight per SM; the
// step's codes and scales are written as contiguous runs.
#pragma once

#include <cstdint>
#include <type_traits>

namespace dsa {

constexpr int kQuantThreads = 256;
constexpr int kRowsPerWarp = 8;

// Two floats to two e4m3 codes (nearest, ties to even, saturating); lo lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int D>
__global__ void __launch_bounds__(kQuantThreads) quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t N,
                                                                      uint8_t* __restrict__ codes,
                                                                      float* __restrict__ scale) {
  static_assert(D == 64 || D == 128, "D");
  constexpr int V = D / 32;  // bf16 values per lane: 2 or 4
  using Raw = typename std::conditional<V == 4, uint2, uint32_t>::type;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * (kQuantThreads / 32) + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kQuantThreads / 32);
  for (int64_t r0 = warp0 * kRowsPerWarp; r0 < N; r0 += nwarps * kRowsPerWarp) {
    Raw raw[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int64_t r = r0 + i;
      if (r < N) raw[i] = __ldcs(reinterpret_cast<const Raw*>(x + r * D) + lane);
    }
    float my_s = 0.0f;  // lane i keeps row r0 + i's scale: one 32-byte store per step
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int64_t r = r0 + i;
      if (r >= N) break;  // warp-uniform
      float v[V];
      if constexpr (V == 4) {
        v[0] = __uint_as_float(raw[i].x << 16);
        v[1] = __uint_as_float(raw[i].x & 0xFFFF0000u);
        v[2] = __uint_as_float(raw[i].y << 16);
        v[3] = __uint_as_float(raw[i].y & 0xFFFF0000u);
      } else {
        v[0] = __uint_as_float(raw[i] << 16);
        v[1] = __uint_as_float(raw[i] & 0xFFFF0000u);
      }
      uint32_t amax = 0u;  // largest magnitude, compared as bits (finite inputs)
#pragma unroll
      for (int j = 0; j < V; ++j) amax = max(amax, __float_as_uint(v[j]) & 0x7FFFFFFFu);
      amax = __reduce_max_sync(0xffffffffu, amax);
      const float m = __uint_as_float(amax);
      const float s = m / 448.0f;
      uint32_t c = 0u;
      if (m != 0.0f) {
#pragma unroll
        for (int j = 0; j < V; j += 2) c |= cvt_e4m3x2(v[j] / s, v[j + 1] / s) << (8 * j);
      }
      if constexpr (V == 4) {
        reinterpret_cast<uint32_t*>(codes + r * D)[lane] = c;
      } else {
        reinterpret_cast<uint16_t*>(codes + r * D)[lane] = static_cast<uint16_t>(c);
      }
      my_s = lane == i ? s : my_s;
    }
    if (lane < kRowsPerWarp && r0 + lane < N) scale[r0 + lane] = my_s;
  }
}

}  // namespace dsa
