// The C ABI of the FP8 lightning indexer and top-k selector (declared in include/dsa.h).
//
// Host side only: argument checks, the choice of tile configuration and shared-memory carve-up,
// tensor-memory-accelerator descriptors, the fused path's workspace layout, and the launches.
// Every step of the computation runs in the kernels of this library; there is no host or
// fallback compute path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/dsa.h"
#include "attn_kernel.cuh"
#include "common.cuh"
#include "launch.h"
#include "types.cuh"

// The device error word of this library (one per device context).
__device__ unsigned int g_dsa_error_word;

namespace dsa {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxRingStages = 8;
constexpr int kPrefillRowBytes = 128 * 1024;  // fused prefill: row buffer of all tokens of an item
constexpr int kDecodeRowBytes = 128 * 1024;   // fused decode (one token per item)
constexpr int kChunkMinKeys = 4096;           // shortest chunk when rows are split for parallelism
// Tokens of a fused prefill item: each needs its own first-digit histogram (1 KB) and its window
// in the row buffer, so items hold at most 8 tokens even when few heads would let the MMA take
// more (256 / H); the planner halves items whose windows do not fit.
constexpr int kFusedTokensMax = 8;

struct DeviceInfo {
  bool init = false;
  int sms = 0;
  int max_smem = 0;
  unsigned* err = nullptr;
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// Device facts of the current device (cached).  Returns nullptr on a CUDA error.
const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return nullptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dsa_error_word) != cudaSuccess) return nullptr;
    d.err = static_cast<unsigned*>(p);
    d.init = true;
  }
  return &d;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 2-D map over a row-major [rows, D] e4m3 matrix, box = [box_rows, D], swizzle matching D.
bool make_row_map(CUtensorMap* map, const void* base, int64_t rows, int D, int box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool supported_h(int H) { return H == 4 || H == 8 || H == 16 || H == 32 || H == 64; }
bool supported_d(int D) { return D == 64 || D == 128; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ----------------------------------------------------------------------------- index kernel config

struct IndexConfig {
  int ntok_max;
  int n_mma_max;
  int row_keys;  // fused only: requested on input, granted on output
  int stages;
  int qbufs;
  int off_ring, off_q, off_rows, off_w, off_win, off_sc, off_hist, off_bitmap, off_bar;
  int smem;  // dynamic shared memory to request (includes 1 KB alignment slack)
};

constexpr int kMinFusedStages = 3;

// Shared-memory carve-up.  The fused mode first reserves kMinFusedStages ring stages and shrinks
// the row buffer (a multiple of 1024 keys) to what is left; the remaining space then becomes
// ring stages (up to kMaxRingStages) and, if at least 4 stages remain, a second Q buffer.
bool layout_index(IndexConfig& c, int H, int D, bool fused, int max_smem) {
  const int tile = 128 * D;
  const int q_bytes = c.n_mma_max * D;
  const int w_bytes = static_cast<int>(round_up(static_cast<size_t>(c.ntok_max) * H * 4, 16));
  const int win_bytes = static_cast<int>(round_up(static_cast<size_t>(c.ntok_max) * 8, 16));
  const int sc_bytes = static_cast<int>(round_up(kEpiGroups * sizeof(SelectScratch), 16));
  const int hist_bytes = fused ? c.ntok_max * 256 * 4 : 0;
  const int bar_max = (2 * kMaxRingStages + 2 * kAccStages + kMiscBarWords) * 8 + 64;
  const int misc = 1024 + w_bytes + win_bytes + sc_bytes + hist_bytes + bar_max;
  int rows = 0, bitmap = 0;
  if (fused) {
    // row buffer (4 bytes per key) + selection bitmap (1 bit per key)
    const int avail = max_smem - misc - q_bytes - kMinFusedStages * tile;
    int keys = std::min(c.row_keys, avail * 8 / 33) / 1024 * 1024;
    if (keys < 1024) return false;
    c.row_keys = keys;
    rows = keys * 4;
    bitmap = keys / 8;
  }
  for (int qbufs = 2; qbufs >= 1; --qbufs) {
    const int fixed = misc + qbufs * q_bytes + rows + bitmap;
    int stages = (max_smem - fixed) / tile;
    if (stages > kMaxRingStages) stages = kMaxRingStages;
    if (qbufs == 2 && stages < 4) continue;
    if (stages < 2) return false;
    c.stages = stages;
    c.qbufs = qbufs;
    int off = 0;
    c.off_ring = off;
    off += stages * tile;
    c.off_q = off;
    off += qbufs * q_bytes;
    c.off_rows = off;
    off += rows;
    c.off_w = off;
    off += w_bytes;
    c.off_win = off;
    off += win_bytes;
    c.off_sc = off;
    off += sc_bytes;
    c.off_hist = off;
    off += hist_bytes;
    c.off_bitmap = off;
    off += bitmap;
    c.off_bar = off;
    off += (2 * stages + 2 * kAccStages + kMiscBarWords) * 8 + 64;
    c.smem = off + 1024;
    return c.smem <= max_smem;
  }
  return false;
}

void fill_params(IndexParams& p, const IndexConfig& c) {
  p.ntok_max = c.ntok_max;
  p.n_mma_max = c.n_mma_max;
  p.stages = c.stages;
  p.qbufs = c.qbufs;
  p.off_ring = c.off_ring;
  p.off_q = c.off_q;
  p.off_rows = c.off_rows;
  p.off_w = c.off_w;
  p.off_win = c.off_win;
  p.off_sc = c.off_sc;
  p.off_hist = c.off_hist;
  p.off_bitmap = c.off_bitmap;
  p.off_bar = c.off_bar;
}

int round16(int x) { return (x + 15) / 16 * 16; }

cudaError_t launch_index(int D, int H, bool fused, int grid, size_t smem, cudaStream_t st, const CUtensorMap& km,
                         const CUtensorMap& qm, const IndexParams& p) {
  return D == 128 ? launch_index_d128(H, fused, grid, smem, st, km, qm, p)
                  : launch_index_d64(H, fused, grid, smem, st, km, qm, p);
}

// ----------------------------------------------------------------------------- fused config + workspace

// A launch is treated as decode-like when keys vastly outnumber queries (packed requests, one
// window each): one token per item.  Otherwise tokens are blocked (the planner still falls back
// to one unit per token for blocks whose windows do not overlap).
bool decode_like(int T, int N) { return static_cast<int64_t>(N) >= 16 * static_cast<int64_t>(T); }

struct FusedPlan {
  IndexConfig cfg;
  int target;
  int max_units, max_items, max_slots, groups;
  size_t off_hdr, off_units, off_items, off_empty, off_cnt, off_ln, off_lu, off_li, total;
};

bool fused_plan(FusedPlan& f, int T, int N, int H, int D, int topk, int sms, int max_smem) {
  IndexConfig& c = f.cfg;
  const bool dec = decode_like(T, N);
  c.ntok_max = dec ? 1 : std::min(256 / H, kFusedTokensMax);
  c.n_mma_max = round16(c.ntok_max * H);
  c.row_keys = (dec ? kDecodeRowBytes : kPrefillRowBytes) / 4;
  if (!layout_index(c, H, D, true, max_smem)) return false;
  f.target = sms;
  f.groups = (T + c.ntok_max - 1) / c.ntok_max;
  f.max_units = std::max(T, 1);
  int64_t slots = 0;
  if (N > c.row_keys) slots += static_cast<int64_t>(T) * ((static_cast<int64_t>(N) + c.row_keys - 1) / c.row_keys);
  if (f.groups < f.target) slots += 2 * static_cast<int64_t>(f.target) * c.ntok_max;
  if (slots > INT_MAX / 2) return false;
  f.max_slots = static_cast<int>(slots);
  const int64_t items = static_cast<int64_t>(T) + slots + 1;
  if (items > INT_MAX / 2) return false;
  f.max_items = static_cast<int>(items);
  size_t off = 0;
  f.off_hdr = off;
  off += 256;
  f.off_units = off;
  off = round_up(off + static_cast<size_t>(f.max_units) * sizeof(PlanUnit), 256);
  f.off_items = off;
  off = round_up(off + static_cast<size_t>(f.max_items) * sizeof(PlanItem), 256);
  f.off_empty = off;
  off = round_up(off + static_cast<size_t>(std::max(T, 1)) * 4, 256);
  f.off_cnt = off;
  off = round_up(off + static_cast<size_t>(f.max_slots) * 4, 256);
  f.off_ln = off;
  off = round_up(off + static_cast<size_t>(f.max_slots) * 4, 256);
  f.off_lu = off;
  off = round_up(off + static_cast<size_t>(f.max_slots) * topk * 4, 256);
  f.off_li = off;
  off = round_up(off + static_cast<size_t>(f.max_slots) * topk * 4, 256);
  f.total = off;
  return true;
}

dsa_status check_common(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale, const int32_t* ks,
                        const int32_t* ke, int T, int N, int H, int D) {
  if (T < 0 || N < 0) return DSA_ERR_INVALID_ARG;
  if (!supported_h(H) || !supported_d(D)) return DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * H > INT_MAX) return DSA_ERR_UNSUPPORTED;
  if (T > 0 && (!q || !w || !ks || !ke)) return DSA_ERR_INVALID_ARG;
  if (N > 0 && (!k || !k_scale)) return DSA_ERR_INVALID_ARG;
  if ((q && !aligned(q, 16)) || (k && !aligned(k, 16))) return DSA_ERR_INVALID_ARG;
  if ((w && !aligned(w, 4)) || (k_scale && !aligned(k_scale, 4)) || (ks && !aligned(ks, 4)) ||
      (ke && !aligned(ke, 4)))
    return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// Few heads on long windows: a fused unit then holds only one or two tokens (each needs its
// whole window in the row buffer), the MMA is narrow and the selection runs in large teams, so
// the call is routed through the unfused scorer and selector instead, a slab of rows at a
// time (the slab's logits live in the workspace; measured faster for 16 heads and fewer on
// 8192-token causal prefill).
bool route_unfused(int T, int N, int H, const FusedPlan& f) {
  return H <= 16 && !decode_like(T, N) && N > f.cfg.row_keys / f.cfg.ntok_max;
}

constexpr size_t kRouteLogitsBytes = size_t(256) << 20;  // logits slab of the routed call

size_t route_workspace(int T, int N) {
  const size_t row = static_cast<size_t>(N) * 4;
  const size_t rows = std::max<size_t>(1, std::min<size_t>(static_cast<size_t>(T), kRouteLogitsBytes / row));
  return rows * row;
}

// The routed call: dsa_index_score + dsa_topk over slabs of the rows that fit the workspace.
dsa_status run_routed(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale, const int32_t* ks,
                      const int32_t* ke, int T, int N, int H, int D, int topk, int32_t* idx, void* workspace,
                      size_t workspace_bytes, void* stream) {
  const size_t row = static_cast<size_t>(N) * 4;
  const int64_t slab = static_cast<int64_t>(std::min<size_t>(static_cast<size_t>(T), workspace_bytes / row));
  if (slab < 1) return DSA_ERR_WORKSPACE;
  float* logits = static_cast<float*>(workspace);
  for (int64_t r0 = 0; r0 < T; r0 += slab) {
    const int rows = static_cast<int>(std::min<int64_t>(slab, T - r0));
    dsa_status st = dsa_index_score(q + r0 * H * D, w + r0 * H, k, k_scale, ks + r0, ke + r0, rows, N, H, D, logits,
                                    stream);
    if (st != DSA_OK) return st;
    st = dsa_topk(logits, ks + r0, ke + r0, rows, N, topk, idx + r0 * topk, nullptr, 0, stream);
    if (st != DSA_OK) return st;
  }
  return DSA_OK;
}

// ----------------------------------------------------------------------------- K-resident scorer

struct KresConfig {
  KresParams p;  // the shape fields and shared-memory offsets
  int smem;
  size_t off_blk, off_tok, total;  // workspace: item counter at 0, block windows, token windows
};

bool kres_config(KresConfig& c, int T, int N, int H, int D, int sms, int max_smem) {
  KresParams& p = c.p;
  p.T = T;
  p.N = N;
  p.ntok = kMaxCols / H;
  p.nblocks = (T + p.ntok - 1) / p.ntok;
  p.ntiles = (N + kKeysPerTile - 1) / kKeysPerTile;
  // runs of token blocks per work item: about four items per SM over the (tile, block) grid
  const int64_t work = static_cast<int64_t>(p.nblocks) * p.ntiles;
  int64_t chunk = (work + 4LL * sms - 1) / (4LL * sms);
  chunk = std::max<int64_t>(1, std::min<int64_t>(chunk, std::min(kKresMaxChunk, std::max(p.nblocks, 1))));
  p.chunk = static_cast<int>(chunk);
  p.nchunks = (p.nblocks + p.chunk - 1) / p.chunk;
  if (static_cast<int64_t>(p.ntiles) * p.nchunks > INT_MAX / 2) return false;
  const int tile = kKeysPerTile * D, qblk = kMaxCols * D;
  const int items_bytes = kItemRing * kKresItemInts * 4;
  p.off_q = 2 * tile;
  int stages = (max_smem - 1024 - p.off_q - items_bytes - kres_barrier_bytes(kMaxRingStages)) / qblk;
  stages = std::min(stages, kMaxRingStages);
  if (stages < 2) return false;
  p.stages = stages;
  p.off_bar = p.off_q + stages * qblk;
  p.off_items = p.off_bar + static_cast<int>(round_up(static_cast<size_t>(kres_barrier_bytes(stages)), 16));
  c.smem = p.off_items + items_bytes + 1024;
  if (c.smem > max_smem) return false;
  c.off_blk = 256;
  c.off_tok = round_up(c.off_blk + static_cast<size_t>(std::max(p.nblocks, 1)) * 8, 256);
  c.total = round_up(c.off_tok + static_cast<size_t>(std::max(T, 1)) * 8, 256);
  return true;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_version(void) { return 10000; }

const char* dsa_status_string(dsa_status s) {
  switch (s) {
    case DSA_OK:
      return "DSA_OK";
    case DSA_ERR_INVALID_ARG:
      return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED:
      return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_WORKSPACE:
      return "DSA_ERR_WORKSPACE";
    case DSA_ERR_CUDA:
      return "DSA_ERR_CUDA";
    case DSA_ERR_TIMEOUT:
      return "DSA_ERR_TIMEOUT";
  }
  return "DSA_ERR_UNKNOWN";
}

dsa_status dsa_index_score(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale,
                           const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, float* logits,
                           void* stream) {
  dsa_status st = check_common(q, w, k, k_scale, ks, ke, T, N, H, D);
  if (st != DSA_OK) return st;
  if (T > 0 && N > 0 && (!logits || !aligned(logits, 4))) return DSA_ERR_INVALID_ARG;
  if (T == 0 || N == 0) return DSA_OK;  // no window holds a key: nothing to write
  const DeviceInfo* dev = device_info();
  if (!dev) return DSA_ERR_CUDA;
  IndexConfig c{};
  c.ntok_max = 256 / H;
  c.n_mma_max = round16(c.ntok_max * H);
  c.row_keys = 0;
  if (!layout_index(c, H, D, false, dev->max_smem)) return DSA_ERR_UNSUPPORTED;
  CUtensorMap kmap, qmap;
  if (!make_row_map(&kmap, k, N, D, 128)) return DSA_ERR_CUDA;
  if (!make_row_map(&qmap, q, static_cast<int64_t>(T) * H, D, c.n_mma_max)) return DSA_ERR_CUDA;
  IndexParams p{};
  fill_params(p, c);
  p.w = w;
  p.k_scale = k_scale;
  p.ks = ks;
  p.ke = ke;
  p.err = dev->err;
  p.T = T;
  p.N = N;
  p.logits = logits;
  p.nblocks = (T + c.ntok_max - 1) / c.ntok_max;
  const int target = 2 * dev->sms;
  int nsplit = (target + p.nblocks - 1) / p.nblocks;
  const int max_split = std::max(1, (N + 1023) / 1024);  // at least ~1024 keys per split
  nsplit = std::max(1, std::min(nsplit, max_split));
  p.nsplit = nsplit;
  const int64_t n_items = static_cast<int64_t>(p.nblocks) * nsplit;
  const int grid = static_cast<int>(std::min<int64_t>(n_items, dev->sms));
  cudaError_t e = launch_index(D, H, false, grid, c.smem, static_cast<cudaStream_t>(stream), kmap, qmap, p);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

size_t dsa_index_score_kres_workspace_size(int T, int N, int H, int D) {
  if (T < 0 || N < 0 || !supported_h(H) || !supported_d(D)) return 0;
  KresConfig c{};
  // the workspace depends only on T and H (the SM count and shared memory do not enter it)
  if (!kres_config(c, T, std::max(N, 1), H, D, 1, INT_MAX)) return 0;
  return c.total;
}

dsa_status dsa_index_score_kres(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale,
                                const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, float* logits,
                                void* workspace, size_t workspace_bytes, void* stream) {
  dsa_status st = check_common(q, w, k, k_scale, ks, ke, T, N, H, D);
  if (st != DSA_OK) return st;
  if (T > 0 && N > 0 && (!logits || !aligned(logits, 4) || !aligned(w, 16))) return DSA_ERR_INVALID_ARG;
  if (T == 0 || N == 0) return DSA_OK;  // no window holds a key: nothing to write
  const DeviceInfo* dev = device_info();
  if (!dev) return DSA_ERR_CUDA;
  KresConfig c{};
  if (!kres_config(c, T, N, H, D, dev->sms, dev->max_smem)) return DSA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < c.total || !aligned(workspace, 256)) return DSA_ERR_WORKSPACE;
  CUtensorMap kmap, qmap;
  if (!make_row_map(&kmap, k, N, D, kKeysPerTile)) return DSA_ERR_CUDA;
  if (!make_row_map(&qmap, q, static_cast<int64_t>(T) * H, D, kMaxCols)) return DSA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  KresParams p = c.p;
  p.w = w;
  p.k_scale = k_scale;
  p.logits = logits;
  p.err = dev->err;
  p.queue = reinterpret_cast<int*>(ws);
  p.blk_win = reinterpret_cast<const int2*>(ws + c.off_blk);
  p.tok_win = reinterpret_cast<const int2*>(ws + c.off_tok);
  const int64_t n_items = static_cast<int64_t>(p.ntiles) * p.nchunks;
  const int grid = static_cast<int>(std::min<int64_t>(n_items, dev->sms));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = D == 128 ? launch_kres_d128(H, grid, c.smem, s, kmap, qmap, p, ks, ke)
                           : launch_kres_d64(H, grid, c.smem, s, kmap, qmap, p, ks, ke);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

size_t dsa_topk_workspace_size(int T, int N, int topk) {
  (void)T;
  (void)N;
  (void)topk;
  return 0;
}

dsa_status dsa_topk(const float* logits, const int32_t* ks, const int32_t* ke, int T, int N, int topk, int32_t* idx,
                    void* workspace, size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (T < 0 || N < 0) return DSA_ERR_INVALID_ARG;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!ks || !ke || !idx || (N > 0 && !logits)) return DSA_ERR_INVALID_ARG;
  if (!aligned(ks, 4) || !aligned(ke, 4) || !aligned(idx, 4) || (logits && !aligned(logits, 4)))
    return DSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = device_info();
  if (!dev) return DSA_ERR_CUDA;
  TopkParams p{};
  p.logits = logits;
  p.ks = ks;
  p.ke = ke;
  p.idx = idx;
  p.T = T;
  p.N = N;
  p.topk = topk;
  p.err = dev->err;
  const size_t head = round_up(sizeof(SelectScratch), 16);
  if (N <= kTopkStreamMaxKeys && aligned(logits, 16)) {
    // every row fits a streaming CTA's row buffer: one buffer per CTA, several CTAs per SM
    p.cache_keys = (N + 31) / 32 * 32;
    const size_t smem = head + static_cast<size_t>(p.cache_keys + 8) * 4 +
                        static_cast<size_t>(((p.cache_keys + 31) / 32 + 3) & ~3) * 4 + 32;
    cudaError_t e = launch_topk_stream(T, smem, static_cast<cudaStream_t>(stream), p);
    return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  // key cache (4 bytes per key) + selection bitmap (1 bit per key)
  const int cap = static_cast<int>((static_cast<size_t>(dev->max_smem) - head - 256) * 8 / 33) / 32 * 32;
  p.cache_keys = std::max(0, std::min(N, cap));
  const size_t smem = head + static_cast<size_t>((p.cache_keys + 3) & ~3) * 4 + (p.cache_keys + 31) / 32 * 4 + 16;
  const int grid = std::min(T, 8 * dev->sms);
  cudaError_t e = launch_topk_rows(grid, smem, static_cast<cudaStream_t>(stream), p);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

size_t dsa_index_topk_workspace_size(int T, int N, int H, int D, int topk) {
  if (T < 0 || N < 0 || !supported_h(H) || !supported_d(D) || topk < 1 || topk > DSA_MAX_TOPK) return 0;
  const DeviceInfo* dev = device_info();
  if (!dev) return 0;
  FusedPlan f{};
  if (!fused_plan(f, T, N, H, D, topk, dev->sms, dev->max_smem)) return 0;
  if (route_unfused(T, N, H, f)) return route_workspace(T, N);
  return f.total;
}

// Checks shared by the fused entry points; fills the plan geometry.
static dsa_status fused_prologue(const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, int topk,
                                 void* workspace, size_t workspace_bytes, const DeviceInfo** dev_out,
                                 FusedPlan* f) {
  if (T < 0 || N < 0) return DSA_ERR_INVALID_ARG;
  if (!supported_h(H) || !supported_d(D)) return DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(T) * H > INT_MAX) return DSA_ERR_UNSUPPORTED;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (T > 0 && (!ks || !ke || !aligned(ks, 4) || !aligned(ke, 4))) return DSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = device_info();
  if (!dev) return DSA_ERR_CUDA;
  if (!fused_plan(*f, T, N, H, D, topk, dev->sms, dev->max_smem)) return DSA_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256)) return DSA_ERR_INVALID_ARG;
  if (workspace_bytes < (route_unfused(T, N, H, *f) ? route_workspace(T, N) : f->total)) return DSA_ERR_WORKSPACE;
  *dev_out = dev;
  return DSA_OK;
}

dsa_status dsa_index_topk_plan(const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, int topk,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (T == 0 && N >= 0 && supported_h(H) && supported_d(D) && topk >= 1 && topk <= DSA_MAX_TOPK) return DSA_OK;
  const DeviceInfo* dev = nullptr;
  FusedPlan f{};
  dsa_status st = fused_prologue(ks, ke, T, N, H, D, topk, workspace, workspace_bytes, &dev, &f);
  if (st != DSA_OK) return st;
  if (route_unfused(T, N, H, f)) return DSA_OK;  // the routed run needs no plan
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PlanArgs a{};
  a.ks = ks;
  a.ke = ke;
  a.T = T;
  a.N = N;
  a.topk = topk;
  a.ntok_max = f.cfg.ntok_max;
  a.row_keys = f.cfg.row_keys;
  a.target_items = f.target;
  a.cl_min = kChunkMinKeys;
  a.max_units = f.max_units;
  a.max_items = f.max_items;
  a.max_slots = f.max_slots;
  a.hdr = reinterpret_cast<PlanHeader*>(ws + f.off_hdr);
  a.units = reinterpret_cast<PlanUnit*>(ws + f.off_units);
  a.items = reinterpret_cast<PlanItem*>(ws + f.off_items);
  a.counters = reinterpret_cast<uint32_t*>(ws + f.off_cnt);
  a.empty = reinterpret_cast<int32_t*>(ws + f.off_empty);
  a.err = dev->err;
  a.stage_windows = static_cast<int64_t>(T) * 8 + 1024 <= dev->max_smem ? 1 : 0;
  return launch_plan(static_cast<cudaStream_t>(stream), a) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status dsa_index_topk_run(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale,
                              const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, int topk,
                              int32_t* idx, void* workspace, size_t workspace_bytes, void* stream) {
  dsa_status st = check_common(q, w, k, k_scale, ks, ke, T, N, H, D);
  if (st != DSA_OK) return st;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!idx || !aligned(idx, 4)) return DSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  FusedPlan f{};
  st = fused_prologue(ks, ke, T, N, H, D, topk, workspace, workspace_bytes, &dev, &f);
  if (st != DSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    // no keys: every window is empty, every row is -1 (all-ones bytes)
    return cudaMemsetAsync(idx, 0xFF, static_cast<size_t>(T) * topk * sizeof(int32_t), s) == cudaSuccess
               ? DSA_OK
               : DSA_ERR_CUDA;
  }
  if (route_unfused(T, N, H, f))
    return run_routed(q, w, k, k_scale, ks, ke, T, N, H, D, topk, idx, workspace, workspace_bytes, stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  CUtensorMap kmap, qmap;
  if (!make_row_map(&kmap, k, N, D, 128)) return DSA_ERR_CUDA;
  if (!make_row_map(&qmap, q, static_cast<int64_t>(T) * H, D, f.cfg.n_mma_max)) return DSA_ERR_CUDA;
  IndexParams p{};
  fill_params(p, f.cfg);
  p.w = w;
  p.k_scale = k_scale;
  p.ks = ks;
  p.ke = ke;
  p.err = dev->err;
  p.T = T;
  p.N = N;
  p.topk = topk;
  p.row_keys = f.cfg.row_keys;
  p.plan = reinterpret_cast<const PlanHeader*>(ws + f.off_hdr);
  p.queue = &reinterpret_cast<PlanHeader*>(ws + f.off_hdr)->next_item;
  p.units = reinterpret_cast<const PlanUnit*>(ws + f.off_units);
  p.items = reinterpret_cast<const PlanItem*>(ws + f.off_items);
  p.idx = idx;
  p.list_u = reinterpret_cast<uint32_t*>(ws + f.off_lu);
  p.list_i = reinterpret_cast<int32_t*>(ws + f.off_li);
  p.list_n = reinterpret_cast<int32_t*>(ws + f.off_ln);
  p.counters = reinterpret_cast<uint32_t*>(ws + f.off_cnt);
  p.empty = reinterpret_cast<const int32_t*>(ws + f.off_empty);
  cudaError_t e = launch_index(D, H, true, dev->sms, f.cfg.smem, s, kmap, qmap, p);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status dsa_index_topk(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale,
                          const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, int topk, int32_t* idx,
                          void* workspace, size_t workspace_bytes, void* stream) {
  dsa_status st = check_common(q, w, k, k_scale, ks, ke, T, N, H, D);
  if (st != DSA_OK) return st;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!idx || !aligned(idx, 4)) return DSA_ERR_INVALID_ARG;
  st = dsa_index_topk_plan(ks, ke, T, N, H, D, topk, workspace, workspace_bytes, stream);
  if (st != DSA_OK) return st;
  return dsa_index_topk_run(q, w, k, k_scale, ks, ke, T, N, H, D, topk, idx, workspace, workspace_bytes, stream);
}

// ----------------------------------------------------------------------------- allocation-free variant
//
// Some callers cannot allocate device memory at the point where they need the top-k indices:
// code running inside a memory pool or arena that owns every byte of the device, code on a
// path where a cudaMalloc would synchronise the device or fail under a hard memory cap, or
// runtimes that forbid allocation after start-up.  For them, dsa_index_topk_noalloc keeps the
// fused path's scratch (the work plan) in a fixed array of this library, defined below.  Every
// device that loads the library holds the array until the process exits.

// Scratch of dsa_index_topk_noalloc: 32 MiB per device.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mutex;

// Device address of g_noalloc_scratch on the current device (looked up once per device).
void* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}
}  // namespace

dsa_status dsa_index_topk_noalloc(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale,
                                  const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, int topk,
                                  int32_t* idx, void* stream) {
  dsa_status st = check_common(q, w, k, k_scale, ks, ke, T, N, H, D);
  if (st != DSA_OK) return st;
  if (topk < 1 || topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!idx || !aligned(idx, 4)) return DSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = device_info();
  if (!dev) return DSA_ERR_CUDA;
  FusedPlan f{};
  if (!fused_plan(f, T, N, H, D, topk, dev->sms, dev->max_smem)) return DSA_ERR_UNSUPPORTED;
  if (route_unfused(T, N, H, f)) {
    // routed: the scratch holds as many rows' logits as fit (at least one)
    if (static_cast<size_t>(N) * 4 > kNoAllocScratchBytes) return DSA_ERR_WORKSPACE;
    void* scratch = noalloc_scratch();
    if (!scratch) return DSA_ERR_CUDA;
    return run_routed(q, w, k, k_scale, ks, ke, T, N, H, D, topk, idx, scratch, kNoAllocScratchBytes, stream);
  }
  const size_t need = f.total;
  if (need > kNoAllocScratchBytes) return DSA_ERR_WORKSPACE;  // the fixed scratch is too small
  void* scratch = noalloc_scratch();
  if (!scratch) return DSA_ERR_CUDA;
  // The plan kernel writes every scratch word the run reads, so nothing left by an earlier call
  // needs clearing.
  return dsa_index_topk(q, w, k, k_scale, ks, ke, T, N, H, D, topk, idx, scratch, kNoAllocScratchBytes, stream);
}

dsa_status dsa_get_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DSA_ERR_CUDA;
  const DeviceInfo* dev = device_info();
  if (!dev) return DSA_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, dev->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return DSA_ERR_CUDA;
  if (word == 0) return DSA_OK;
  if (cudaMemset(dev->err, 0, sizeof(unsigned)) != cudaSuccess) return DSA_ERR_CUDA;
  if (word & kErrTimeout) return DSA_ERR_TIMEOUT;
  return DSA_ERR_WORKSPACE;
}

dsa_status dsa_quantize_k(const uint16_t* k, int N, int D, uint8_t* k_e4m3, float* k_scale, void* stream) {
  if (N < 0) return DSA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return DSA_ERR_UNSUPPORTED;
  if (N == 0) return DSA_OK;
  if (!k || !k_e4m3 || !k_scale || !aligned(k, 8) || !aligned(k_e4m3, 4) || !aligned(k_scale, 4))
    return DSA_ERR_INVALID_ARG;
  const cudaError_t e = launch_quantize(D, k, N, k_e4m3, k_scale, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status dsa_sparse_attn(const uint16_t* q, const uint16_t* kv, const float* attn_sink, const int32_t* idx,
                           int T, int N, int H, int D, int K, float scale, uint16_t* out, float* lse, void* stream) {
  if (T < 0 || N < 0 || H < 1 || K < 0) return DSA_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256 && D != 512) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!q || !out || !aligned(q, 2) || !aligned(out, 2)) return DSA_ERR_INVALID_ARG;
  if (K > 0 && (!idx || !aligned(idx, 4))) return DSA_ERR_INVALID_ARG;
  if (N > 0 && (!kv || !aligned(kv, 4))) return DSA_ERR_INVALID_ARG;
  if (attn_sink && !aligned(attn_sink, 4)) return DSA_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return DSA_ERR_INVALID_ARG;
  if (H > 65535 * kAttnHeads) return DSA_ERR_UNSUPPORTED;  // (head groups on the grid's y axis)
  AttnParams p{q, kv, attn_sink, idx, out, lse, T, N, H, K, scale, H};
  // Tensor cores for D in {128, 256, 512} and 16-byte aligned q and kv (copied in 16-byte
  // pieces): all heads of a row in one MMA column block, so up to 64 heads per launch, and a
  // layer with more heads as groups of 64 (the softmax and its sink are per head), one launch
  // per group over the same lists.  The CUDA-core kernel otherwise.
  const DeviceInfo* dev = device_info();
  if (!dev) return DSA_ERR_CUDA;
  const int tc_smem = sparse_attn_tc_smem(D);
  if (tc_smem > 0 && tc_smem <= dev->max_smem && K > 0 && N > 0 && aligned(q, 16) && aligned(kv, 16)) {
    const int grid = std::min(T, dev->sms);
    for (int h0 = 0; h0 < H; h0 += kTcMaxHeads) {
      AttnParams g = p;
      g.H = std::min(kTcMaxHeads, H - h0);
      g.q = q + static_cast<size_t>(h0) * D;
      g.out = out + static_cast<size_t>(h0) * D;
      g.sink = attn_sink ? attn_sink + h0 : nullptr;
      g.lse = lse ? lse + h0 : nullptr;
      if (launch_sparse_attn_tc(D, grid, g, dev->err, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
  }
  const cudaError_t e = launch_sparse_attn(D, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status dsa_sparse_attn_bwd(const uint16_t* q, const uint16_t* kv, const float* attn_sink, const int32_t* idx,
                               const uint16_t* out, const float* lse, const uint16_t* dout, int T, int N, int H, int D,
                               int K, float scale, float* dq, float* dkv, float* dsink, void* stream) {
  if (T < 0 || N < 0 || H < 1 || K < 0) return DSA_ERR_INVALID_ARG;
  if (D != 128 && D != 256) return DSA_ERR_UNSUPPORTED;
  if (N > 0 && (!kv || !aligned(kv, 16) || !dkv || !aligned(dkv, 16))) return DSA_ERR_INVALID_ARG;
  if (attn_sink && !aligned(attn_sink, 4)) return DSA_ERR_INVALID_ARG;
  if (dsink && !aligned(dsink, 4)) return DSA_ERR_INVALID_ARG;
  if (T > 0 && (!q || !aligned(q, 16) || !out || !aligned(out, 4) || !lse || !aligned(lse, 4) || !dout ||
                !aligned(dout, 16) || !dq || !aligned(dq, 4)))
    return DSA_ERR_INVALID_ARG;
  if (T > 0 && K > 0 && (!idx || !aligned(idx, 4))) return DSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = device_info();
  if (!dev) return DSA_ERR_CUDA;
  const int smem = sparse_attn_bwd_tc_smem(D);
  if (smem <= 0 || smem > dev->max_smem) return DSA_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (N > 0 && cudaMemsetAsync(dkv, 0, static_cast<size_t>(N) * D * sizeof(float), st) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (dsink && cudaMemsetAsync(dsink, 0, static_cast<size_t>(H) * sizeof(float), st) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (T == 0) return DSA_OK;
  AttnBwdParams p{q, kv, attn_sink, K > 0 ? idx : nullptr, out, lse, dout, dq, dkv, attn_sink ? dsink : nullptr,
                  T, N, H, K, scale, H};
  // up to 64 heads per launch; a layer with more heads as groups of 64, one launch per group
  // over the same lists, every group adding into the one dkv
  const int grid = std::min(T, dev->sms);
  for (int h0 = 0; h0 < H; h0 += kTcMaxHeads) {
    AttnBwdParams g = p;
    g.H = std::min(kTcMaxHeads, H - h0);
    g.q = q + static_cast<size_t>(h0) * D;
    g.o = out + static_cast<size_t>(h0) * D;
    g.dout = dout + static_cast<size_t>(h0) * D;
    g.dq = dq + static_cast<size_t>(h0) * D;
    g.lse = lse + h0;
    g.sink = attn_sink ? attn_sink + h0 : nullptr;
    g.dsink = p.dsink ? p.dsink + h0 : nullptr;
    if (launch_sparse_attn_bwd_tc(D, grid, g, dev->err, st) != cudaSuccess) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

// Device times of the two waits of the bounded-wait self-check (written by its kernel).
static __device__ unsigned long long g_wait_check_ns[2];

dsa_status dsa_check_bounded_wait(uint64_t* wait_ns, void* stream) {
  const DeviceInfo* dev = device_info();
  if (!dev) return DSA_ERR_CUDA;
  void* took = nullptr;
  if (cudaGetSymbolAddress(&took, g_wait_check_ns) != cudaSuccess) return DSA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_wait_check(st, dev->err, static_cast<unsigned long long*>(took)) != cudaSuccess) return DSA_ERR_CUDA;
  unsigned long long h[2] = {0ull, 0ull};
  if (cudaMemcpyAsync(h, took, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DSA_ERR_CUDA;
  if (wait_ns) {
    wait_ns[0] = h[0];
    wait_ns[1] = h[1];
  }
  return DSA_OK;
}

}  // extern "C"

namespace dsa {
int max_dynamic_smem() {
  const DeviceInfo* d = device_info();
  return d ? d->max_smem : 0;
}
}  // namespace dsa
