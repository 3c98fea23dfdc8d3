// Types and constants shared by the kernels and the host side of the library (no kernels
// here, so the C-ABI translation unit can include it without compiling any kernel).
#pragma once

#include <cstdint>

namespace dsa {

constexpr int kTopkThreads = 512;
constexpr int kPlanThreads = 1024;

constexpr int kKeysPerTile = 128;  // MMA M
constexpr int kMaxCols = 256;      // largest MMA N = tokens * heads of an item
constexpr int kAccStages = 2;
// Items handed from the TMA producer (which claims them) to the MMA issuer and the epilogue.
constexpr int kItemRing = 4;
// 8-byte shared words after the K-ring and accumulator barriers: q_full[2], q_empty[2], drain,
// TMEM-address + abort word, item_full[kItemRing], item_empty[kItemRing], then kItemRing item
// slots and two epilogue broadcast slots (ints).
constexpr int kMiscBarWords = 4 + 1 + 1 + 2 * kItemRing + (kItemRing + 2 + 1) / 2;
constexpr int kTmemCols = 512;
constexpr int kEpiGroups = 4;       // epilogue groups; group g owns accumulator columns [64g, 64g + 64)
constexpr int kGroupThreads = 128;  // 4 warps, one per 32-lane tensor-memory quarter
constexpr int kIndexThreads = 128 + kEpiGroups * kGroupThreads;
constexpr int kProducers = 3;  // TMA producer threads of the index kernel (lane 0 of warps 0, 2, 3)

// ---------------------------------------------------------------------------- plan (fused mode)

struct PlanHeader {
  int n_items;
  int n_units;
  int n_slots;
  int status;
  int n_empty;     // tokens whose clamped window is empty (their rows are all -1)
  int next_item;   // run kernel's item counter: 0 between runs (the planner zeroes it, the run re-arms it)
  int pad[2];
};

// A unit: `ntok` consecutive tokens scored together over key range [lo, hi), cut into
// `nchunks` chunks of `chunk_len` keys.  A unit with nchunks > 1 writes per-chunk candidate
// lists to slots [slot_base, slot_base + ntok * nchunks) and the last chunk merges them.
// 16-byte aligned, so that a record is stored and loaded as two 16-byte vectors.
struct alignas(16) PlanUnit {
  int tok0;
  int ntok;
  int lo;
  int hi;
  int chunk_len;
  int nchunks;
  int slot_base;
  int pad;
};

struct alignas(8) PlanItem {
  int unit;
  int chunk;
};

struct IndexParams {
  const float* w;
  const float* k_scale;
  const int32_t* ks;
  const int32_t* ke;
  unsigned* err;
  int T;
  int N;
  int ntok_max;   // tokens per item (upper bound)
  int n_mma_max;  // rows of the Q box = MMA N of a full item (multiple of 16, <= 256)
  int stages;     // K ring depth
  int qbufs;      // Q buffers (1 or 2)
  // shared-memory carve-up, byte offsets from the 1024-aligned base
  int off_ring;
  int off_q;
  int off_rows;
  int off_w;
  int off_win;
  int off_sc;
  int off_hist;    // fused: per-token most-significant-digit histograms [ntok_max][256]
  int off_bitmap;  // fused: selection bitmaps, one bit per row-buffer key [row_keys / 32]
  int off_bar;
  int* queue;  // FUSED: &plan->next_item, items gridDim.x, gridDim.x + 1, ... are claimed from it
  // SCORE mode: items are (token block, key split), decoded arithmetically
  float* logits;
  int nblocks;
  int nsplit;
  // FUSED mode: items come from the planner
  int topk;
  int row_keys;  // row-buffer capacity in keys (all tokens of an item together)
  const PlanHeader* plan;
  const PlanUnit* units;
  const PlanItem* items;
  int32_t* idx;
  uint32_t* list_u;
  int32_t* list_i;
  int32_t* list_n;
  uint32_t* counters;
  const int32_t* empty;  // [plan->n_empty] tokens with an empty window
};

// ---------------------------------------------------------------------------- K-resident scorer

constexpr int kKresMaxChunk = 64;                  // token blocks per work item (at most)
constexpr int kKresItemInts = 2 + kKresMaxChunk;   // tile, block count, block list
constexpr int kKresProducers = 3;
constexpr int kKresEpiBar = 1;                     // named barrier of the 512 epilogue threads

struct KresParams {
  const float* w;         // [T, H], 16-byte aligned
  const float* k_scale;   // [N]
  float* logits;          // [T, N]
  unsigned* err;
  const int2* blk_win;    // [nblocks] union of the block's clamped windows (empty: x >= y)
  const int2* tok_win;    // [T] clamped windows
  int* queue;             // work-item counter (zeroed by the window pass before each launch)
  int T;
  int N;
  int ntok;               // tokens per Q block (256 / H)
  int nblocks;            // ceil(T / ntok)
  int ntiles;             // ceil(N / 128)
  int chunk;              // token blocks per work item, <= kKresMaxChunk
  int nchunks;            // ceil(nblocks / chunk)
  int stages;             // Q ring depth
  int off_q;              // byte offsets from the 1024-aligned base (the two K buffers are at 0)
  int off_bar;
  int off_items;
};

// Bytes of the K-resident kernel's barrier block: the Q-ring, key-buffer, accumulator and item
// barriers and `drain`, then the tensor-memory address, the abort flag and two broadcast words.
__host__ __device__ constexpr int kres_barrier_bytes(int stages) {
  return (2 * stages + 4 + 2 * kAccStages + 2 * kItemRing + 1) * 8 + 16;
}

// ---------------------------------------------------------------------------- selection

struct SelectResult {
  uint32_t prefix;
  int shift;    // 0, 8, 16 or 24
  int take_eq;  // how many keys with (u >> shift) == prefix to take, lowest index first
  int all;      // nonzero: every key is selected (n <= k)
};

// Shared scratch a group needs: 256 histogram bins, 32 scan slots, 4 broadcast words.
constexpr int kCandCap = 64;  // threshold-bin candidates ranked exactly by the fast select

struct SelectScratch {
  uint32_t hist[256];  // general radix passes
  uint32_t warp_tot[32];
  uint32_t warp_eq[32];
  uint32_t cand_u[kCandCap];
  int32_t cand_i[kCandCap];
  int cand_n;
  int bcast[7];
};

// ---------------------------------------------------------------------------- top-k kernel

struct TopkParams {
  const float* logits;
  const int32_t* ks;
  const int32_t* ke;
  int32_t* idx;
  int T;
  int N;
  int topk;
  int cache_keys;  // shared-memory key cache capacity (per row buffer)
  unsigned* err;   // device error word (bounded waits)
};

// Streaming top-k kernel: threads per CTA, and the longest row it stages in shared memory.
constexpr int kTopkStreamThreads = 128;
constexpr int kTopkStreamMaxKeys = 8192;

// ---------------------------------------------------------------------------- planner

struct PlanArgs {
  const int32_t* ks;
  const int32_t* ke;
  int T;
  int N;
  int topk;
  int ntok_max;
  int row_keys;
  int target_items;
  int cl_min;
  int max_units;
  int max_items;
  int max_slots;
  PlanHeader* hdr;
  PlanUnit* units;
  PlanItem* items;
  uint32_t* counters;
  int32_t* empty;    // [T] tokens with an empty window
  int stage_windows; // nonzero: the launch has T * 8 bytes of dynamic shared memory for the windows
  unsigned* err;
};

}  // namespace dsa
