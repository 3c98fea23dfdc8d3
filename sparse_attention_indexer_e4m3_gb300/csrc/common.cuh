// Shared device-side definitions of the indexer library: the device error word, the
// order-preserving float -> uint32 key map, and small helpers.
#pragma once

#include <cstdint>

namespace dsa {

// Wall-time limit of any single device-side wait (1 s).  A correct run never waits longer than a
// few milliseconds; the limit exists so that a broken pipeline returns instead of hanging.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// Wall-time limit of a wait issued while tearing down after an abort (10 ms).
constexpr uint64_t kDrainLimitNs = 10000000ull;

// Device error word bits.
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrPlan = 2u;  // the planner could not fit a plan into the workspace

// The device error word lives in the C-ABI translation unit; kernels receive its address.
// An expired wait records kErrTimeout and its site in bits [8, 16).
// Wait sites 0xF0 and 0xF1 belong to the bounded-wait self-check.
constexpr int kSiteWaitCheck = 0xF0;

__device__ __forceinline__ void record_timeout(unsigned* err, int site) {
  atomicOr(err, kErrTimeout | (static_cast<unsigned>(site & 0xFF) << 8));
}

__device__ __forceinline__ void record_error(unsigned* err, unsigned bits) { atomicOr(err, bits); }

// Order-preserving image of an fp32 score as an unsigned integer (TileLang README, "Top-k
// Selector": floats processed as unsigned integers such that a larger float maps to a larger
// integer).  A non-negative float gets its sign bit set; a negative float, sign | magnitude,
// maps to 2^31 - magnitude (its two's-complement negation), below every non-negative key and
// decreasing with the magnitude.  -0 so lands on the key of +0: the two zeros, which compare
// equal as floats, share one key.  NaN inputs are not supported.
__device__ __forceinline__ uint32_t score_key(float x) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t m = static_cast<uint32_t>(static_cast<int32_t>(b) >> 31);  // all ones if negative
  return (b ^ (m | 0x80000000u)) - m;
}

__host__ __device__ __forceinline__ int64_t clamp_i64(int64_t x, int64_t lo, int64_t hi) {
  return x < lo ? lo : (x > hi ? hi : x);
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace dsa
