// Host-side launchers of the library's kernels (one translation unit per head dimension and
// one for the selection kernels, so they compile in parallel).  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace dsa {

struct IndexParams;
struct TopkParams;
struct PlanArgs;
struct AttnParams;
struct AttnBwdParams;
struct KresParams;

// Index kernel for head dimension 128 / 64; `fused` selects the fused index + top-k mode.
cudaError_t launch_index_d128(int H, bool fused, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                              const CUtensorMap& qmap, const IndexParams& p);
cudaError_t launch_index_d64(int H, bool fused, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                             const CUtensorMap& qmap, const IndexParams& p);

// K-resident scorer (window pass, then the scorer) for head dimension 128 / 64.
cudaError_t launch_kres_d128(int H, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                             const CUtensorMap& qmap, const KresParams& p, const int32_t* ks, const int32_t* ke);
cudaError_t launch_kres_d64(int H, int grid, size_t smem, cudaStream_t stream, const CUtensorMap& kmap,
                            const CUtensorMap& qmap, const KresParams& p, const int32_t* ks, const int32_t* ke);

cudaError_t launch_topk_rows(int grid, size_t smem, cudaStream_t stream, const TopkParams& p);
// Streaming top-k for rows of at most kTopkStreamMaxKeys keys; as many CTAs as fit, <= max_grid.
cudaError_t launch_topk_stream(int max_grid, size_t smem, cudaStream_t stream, const TopkParams& p);
cudaError_t launch_plan(cudaStream_t stream, const PlanArgs& a);
// e4m3 quantise-on-write of N rows of D (64 or 128) bf16 values.
cudaError_t launch_quantize(int D, const uint16_t* x, int64_t N, uint8_t* codes, float* scale, cudaStream_t stream);
// One CTA exercising the bounded wait on barriers that never complete (about kWaitLimitNs).
cudaError_t launch_wait_check(cudaStream_t stream, unsigned* err, unsigned long long* took_ns);

// Sparse attention over the selected keys, head dimension D (64, 128, 256 or 512): CUDA cores.
cudaError_t launch_sparse_attn(int D, const AttnParams& p, cudaStream_t stream);
// Heads one tensor-core attention launch takes (the N of its products); a layer with more heads
// runs as groups of at most this many, each a launch over the same lists (p.hs = the layer's heads).
constexpr int kTcMaxHeads = 64;
// The same on the tensor cores (D in {128, 256, 512}, H <= kTcMaxHeads, q and kv 16-byte
// aligned): `grid` persistent CTAs over the query rows; its bounded waits record into *err.
// Dynamic shared memory it needs (0 for an unsupported D).
cudaError_t launch_sparse_attn_tc(int D, int grid, const AttnParams& p, unsigned* err, cudaStream_t stream);
int sparse_attn_tc_smem(int D);
// Gradients of the sparse attention on the tensor cores (D in {128, 256}, H <= kTcMaxHeads): `grid`
// persistent CTAs over the query rows; dkv and dsink must be zeroed first.
cudaError_t launch_sparse_attn_bwd_tc(int D, int grid, const AttnBwdParams& p, unsigned* err, cudaStream_t stream);
int sparse_attn_bwd_tc_smem(int D);

// Largest dynamic shared memory a CTA of this device may use (bytes).
int max_dynamic_smem();

}  // namespace dsa
