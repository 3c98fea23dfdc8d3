/*
 * dsa.h -- C ABI of the GB300 (sm_103a) FP8 lightning indexer and exact top-k selector.
 *
 * The operation (Modular docs, "sparse_index_fp8_sm100_prefill", the per-(token, key) logit
 * formula; TileLang examples/deepseek_v32 README, "Lightning Indexer" and "Top-k Selector"):
 *
 *     score[t, j] = k_scale[j] * sum_{h < H} relu( sum_{d < D} q[t, h, d] * k[j, d] ) * w[t, h]
 *
 * for every query token t and key j inside the token's window [ks[t], ke[t]) (both clamped to
 * [0, N], as the README clamps its per-token CuSeqLenKS / CuSeqLenKE bounds to the key count),
 * followed by the selection of the topk keys of largest score in each token's window.  Two
 * neighbouring steps are provided too: dsa_quantize_k writes the e4m3 keys and their scales
 * (upstream), and dsa_sparse_attn evaluates attention over the selected keys (downstream).
 *
 * Common conventions
 *   - q, k are OCP E4M3FN fp8 codes (one byte each, NaN codes 0x7F / 0xFF must not occur).
 *     w is the per-(token, head) fp32 weight with any q dequantisation scale folded in;
 *     k_scale is the per-key fp32 scale.  Scores accumulate in fp32.
 *   - All arrays are row-major and contiguous, in DEVICE memory owned by the caller.  The
 *     library never allocates, frees, or keeps a pointer past the call.  q and k must be
 *     16-byte aligned (they are read by the tensor-memory accelerator).
 *   - There is no batch dimension: several requests are packed along T (queries) and N (keys),
 *     each token's window selecting its own request's keys.
 *   - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t, 0 = the legacy
 *     default stream) on the current CUDA device.  Argument checks are synchronous: any status
 *     other than DSA_OK means nothing was launched.  DSA_ERR_CUDA reports a launch failure.
 *   - Every device-side wait is bounded.  A wait that expires sets a device error word and the
 *     kernel returns early; dsa_get_device_error() reports it as DSA_ERR_TIMEOUT.  The outputs of
 *     such a call are unspecified.
 *   - Limits of the indexer calls: H in {4, 8, 16, 32, 64}; D in {64, 128}; 1 <= topk <= 2048;
 *     0 <= T, N < 2^31.  Other values return DSA_ERR_UNSUPPORTED (not an undefined result).
 *     dsa_quantize_k and dsa_sparse_attn state their own limits.
 *
 * Output conventions (TileLang README, "Top-k Selector"; DeepSeek V4.1 model page,
 * sparse_attn_kernel, where an index of -1 marks "no key"):
 *   - idx[t, :] holds absolute key positions in ASCENDING order, followed by -1 padding when the
 *     window holds fewer than topk keys.  An empty window (ke <= ks after clamping) gives an
 *     all -1 row.
 *   - Ties: a larger score wins; among equal scores the lower key index wins.  -0 and +0 are
 *     equal.  The result is deterministic (independent of scheduling).
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

/* Every entry point is exported from the shared library; everything else in it is hidden. */
#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, negative size, bad workspace pointer */
  DSA_ERR_UNSUPPORTED = 2, /* H, D or topk outside the supported set */
  DSA_ERR_WORKSPACE = 3,   /* workspace_bytes smaller than the *_workspace_size() query */
  DSA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  DSA_ERR_TIMEOUT = 5      /* a bounded device-side wait expired (see dsa_get_device_error) */
} dsa_status;

#define DSA_MAX_TOPK 2048

/*
 * dsa_index_score -- the lightning-indexer scorer (TileLang README, "Lightning Indexer":
 * the key-tile x (token, head) GEMM, relu, weight, key scale, head sum, and the per-token key
 * window with the block key-range skip; Modular "sparse_index_fp8_sm100_prefill": the same
 * logit formula, computed as S^T = K . Q^T with Q resident and K streamed).
 *
 *   q        uint8 e4m3 [T, H, D]   query index vectors
 *   w        float      [T, H]      per-(token, head) weights
 *   k        uint8 e4m3 [N, D]      key index vectors
 *   k_scale  float      [N]         per-key scales
 *   ks, ke   int32      [T]         window [ks[t], ke[t]) per token
 *   logits   float      [T, N]      OUTPUT.  Only in-window entries are written; entries
 *                                   outside a token's window are left as they were.
 *
 * The scores are bit-identical to those dsa_index_topk ranks (same arithmetic, same order).
 */
DSA_API dsa_status dsa_index_score(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale,
                                   const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, float* logits,
                                   void* stream);

/*
 * dsa_index_score_kres_workspace_size / dsa_index_score_kres -- the same scorer with the other
 * operand resident (Modular "sparse_index_fp8_sm100_prefill": the shipped scorer it describes
 * is K-resident / Q-streaming -- a key tile stays on chip while the query tokens stream past it;
 * the logit formula is the one above).  Each work item keeps one 128-key tile in shared memory
 * and streams a run of query-token blocks (256 / H tokens each) whose windows meet the tile.
 * Arguments and output as in dsa_index_score, and the scores are bit-identical to its scores.
 *
 *   w          must be 16-byte aligned here (DSA_ERR_INVALID_ARG otherwise)
 *   workspace  device scratch of at least dsa_index_score_kres_workspace_size(T, N, H, D)
 *              bytes (a work counter and the clamped windows), 256-byte aligned; its contents
 *              on entry do not matter; two calls running at the same time must not share it.
 *              DSA_ERR_WORKSPACE if it is missing, short or misaligned.
 * The workspace size depends only on T and H (0 for an unsupported H or D, or T < 0).
 */
DSA_API size_t dsa_index_score_kres_workspace_size(int T, int N, int H, int D);
DSA_API dsa_status dsa_index_score_kres(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale,
                                        const int32_t* ks, const int32_t* ke, int T, int N, int H, int D,
                                        float* logits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_topk_workspace_size / dsa_topk -- the exact top-k selector over a logits buffer
 * (TileLang README, "Top-k Selector": radix selection on an order-preserving unsigned
 * integer image of the float logits, an 8-bit histogram pass followed by refinement passes on
 * the threshold bin; here 4 passes of 8 bits resolve the full 32-bit key, and the tie rule and
 * ascending output make the result deterministic).
 *
 *   logits   float [T, N]   scores; only entries inside each token's window are read.  4-byte
 *                           alignment suffices; with N <= 8192 and a 16-byte aligned pointer the
 *                           rows are staged by bulk copies (same result, faster)
 *   ks, ke   int32 [T]      windows, clamped to [0, N]
 *   idx      int32 [T, topk] OUTPUT
 *   workspace / workspace_bytes: device scratch of at least dsa_topk_workspace_size(T, N, topk)
 *            bytes (may be NULL when that size is 0).  Its contents on entry do not matter.
 */
DSA_API size_t dsa_topk_workspace_size(int T, int N, int topk);
DSA_API dsa_status dsa_topk(const float* logits, const int32_t* ks, const int32_t* ke, int T, int N, int topk,
                            int32_t* idx, void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_index_topk_workspace_size / dsa_index_topk -- scorer and selector fused, so that the
 * [T, N] logits buffer is never written (Modular "sparse_index_fp8_sm100_prefill": a CTA that
 * keeps its query-token block resident sees every key of that block, which is what a fused
 * score + top-k select needs).  Arguments as in dsa_index_score and dsa_topk.  The result equals
 * dsa_topk applied to the output of dsa_index_score, bit for bit.  With 16 heads or fewer on
 * windows too long for a block of tokens to share the on-chip row buffer, the call runs exactly
 * that pair instead, over slabs of rows whose logits fit the workspace (faster there), so the
 * workspace then holds a logits slab (up to 256 MiB).
 *
 *   workspace: device scratch of at least dsa_index_topk_workspace_size(T, N, H, D, topk)
 *   bytes, 256-byte aligned.  Its contents on entry do not matter.  Two calls that run at the
 *   same time must not share a workspace.
 */
DSA_API size_t dsa_index_topk_workspace_size(int T, int N, int H, int D, int topk);
DSA_API dsa_status dsa_index_topk(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale,
                                  const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, int topk,
                                  int32_t* idx, void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_index_topk_plan / dsa_index_topk_run -- the two halves of dsa_index_topk, which is
 * exactly plan followed by run.  The plan (the split of the tokens into work items, written into
 * the workspace by one small kernel) depends only on (ks, ke, T, N, H, D, topk), so a caller
 * whose layers share the same windows plans once and runs once per layer.
 *
 *   dsa_index_topk_plan: reads ks / ke, writes the plan into the workspace.
 *   dsa_index_topk_run:  requires a workspace holding a plan made on the same stream (or
 *                        otherwise ordered before it) with the same ks, ke, T, N, H, D and topk,
 *                        not modified since; every run leaves the plan valid for the next run.
 *                        Runs that share a workspace must not execute concurrently.
 * Errors as for dsa_index_topk.
 */
DSA_API dsa_status dsa_index_topk_plan(const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, int topk,
                                       void* workspace, size_t workspace_bytes, void* stream);
DSA_API dsa_status dsa_index_topk_run(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale,
                                      const int32_t* ks, const int32_t* ke, int T, int N, int H, int D, int topk,
                                      int32_t* idx, void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_index_topk_noalloc -- dsa_index_topk for callers that cannot allocate device memory when
 * they need the indices: code that runs inside a memory pool or arena owning every byte of the
 * device, code on a path where an allocation would synchronise the device or fail under a hard
 * memory cap, and runtimes that forbid allocation after start-up.  It takes the same inputs and
 * output as dsa_index_topk but no workspace: its scratch is a fixed 32 MiB array inside this
 * library (every device that loads the library keeps it until the process exits).  The pages
 * this library follows have no counterpart of this entry point.
 *
 *   Limits (nothing is launched when a problem is refused; use dsa_index_topk for it):
 *   - problems that dsa_index_topk runs fused are refused with DSA_ERR_WORKSPACE when
 *     dsa_index_topk_workspace_size(T, N, H, D, topk) exceeds 32 MiB;
 *   - problems that dsa_index_topk routes through the scorer and the selector (16 heads or
 *     fewer on long windows) are refused only when one row of logits, 4 * N bytes, exceeds
 *     32 MiB; otherwise they run in slabs of floor(32 MiB / (4 * N)) rows.  Their
 *     dsa_index_topk_workspace_size may therefore exceed 32 MiB.
 *   Allocation: none.  No cudaMalloc, cudaFree or other allocating call is made.
 *   Set-up: the first call on a device looks up the device address of the scratch array on
 *   that device; make that first call before any stream capture.
 *   Concurrency: all calls on a device share the one scratch array, so calls that may overlap
 *   on the GPU (different streams without ordering between them) race and must be avoided.
 *   Earlier calls' scratch contents are never read: every call rebuilds what it uses.
 */
DSA_API dsa_status dsa_index_topk_noalloc(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale,
                                          const int32_t* ks, const int32_t* ke, int T, int N, int H, int D,
                                          int topk, int32_t* idx, void* stream);

/*
 * Device state kept between calls: the library caches, per device ordinal, the device addresses
 * of its error word and of the dsa_index_topk_noalloc scratch array in the device's primary
 * context.  They stay valid as long as that context is not reset (cudaDeviceReset) while the
 * library is loaded; calls made under another (non-primary) context are not supported.
 */

/*
 * dsa_get_device_error -- synchronises `stream`, then reads and clears the current device's
 * error word.  Returns DSA_ERR_TIMEOUT if a bounded wait in any kernel of this library expired
 * since the last call, DSA_ERR_CUDA if synchronisation itself failed, DSA_OK otherwise.
 */
DSA_API dsa_status dsa_get_device_error(void* stream);

/*
 * dsa_quantize_k -- e4m3 quantise-on-write of index key rows: the step that writes the fp8 keys
 * the scorer reads (TileLang README, "Lightning Indexer": the index vectors are FP8-quantized;
 * 448 is the largest e4m3 value, FlashInfer MLA-decode discussion).  Per row of D values x:
 *     k_scale = max_j |x_j| / 448                       (fp32 division)
 *     k_e4m3[j] = x_j / k_scale rounded to the nearest e4m3 value, ties to even, magnitudes
 *                 beyond 448 saturating to 448           (fp32 division)
 * so that x_j ~= e4m3(k_e4m3[j]) * k_scale; a row of zeros gets k_scale = 0 and codes 0.
 *
 *   k        bf16 (uint16 bits) [N, D]  input rows, finite values; 8-byte aligned
 *   k_e4m3   uint8 [N, D]   OUTPUT codes (the dsa_index_* k argument); 4-byte aligned
 *   k_scale  float [N]      OUTPUT per-row scales (the dsa_index_* k_scale argument)
 *   D in {64, 128}.  Device memory owned by the caller; asynchronous on `stream`.  Returns
 *   DSA_ERR_UNSUPPORTED for another D and DSA_ERR_INVALID_ARG for a null / misaligned pointer
 *   or N < 0 (nothing launched).
 */
DSA_API dsa_status dsa_quantize_k(const uint16_t* k, int N, int D, uint8_t* k_e4m3, float* k_scale, void* stream);

/*
 * dsa_sparse_attn -- attention of each query row over its selected keys, the step that consumes
 * the top-k indices (DeepSeek V4.1 sparse_attn_kernel page; TileLang README, "Sparse MLA
 * Forward").  For token t and head h, over the entries j of idx[t, :] other than -1 (a key
 * listed twice counts twice):
 *     s_j = scale * sum_d q[t,h,d] kv[j,d]
 *     out[t,h,:] = sum_j e^{s_j} kv[j,:] / ( sum_j e^{s_j} + e^{attn_sink[h]} )
 * Each kv row is both key and value; without attn_sink the denominator is sum_j e^{s_j}.  A row
 * whose list holds no key gets zeros.  fp32 arithmetic, bf16 output.
 *
 *   q          bf16 (uint16 bits) [T, H, D]   queries
 *   kv         bf16 (uint16 bits) [N, D]      keys = values; 4-byte aligned
 *   attn_sink  float [H] or NULL              per-head sink logit
 *   idx        int32 [T, K]                   key indices, -1 = none (dsa_index_topk's output);
 *                                             an entry outside [0, N) is skipped like -1
 *   scale      softmax scale (1 / sqrt(D) in the page's default)
 *   out        bf16 (uint16 bits) [T, H, D]   OUTPUT
 *   lse        float [T, H] or NULL           OUTPUT: ln( sum_j e^{s_j} + e^{attn_sink[h]} ), the
 *                                             natural log of each denominator (-inf for a row
 *                                             with neither keys nor sink); dsa_sparse_attn_bwd
 *                                             takes it
 *   D in {64, 128, 256, 512}, H >= 1, K >= 0.  Device memory owned by the caller; asynchronous
 *   on `stream`.  Returns DSA_ERR_UNSUPPORTED for another D and DSA_ERR_INVALID_ARG for a null /
 *   misaligned pointer or a negative size (nothing launched).  Tensor cores for D >= 128 with
 *   16-byte aligned q and kv: up to 64 heads per kernel launch, more heads as consecutive groups
 *   of 64 (one launch each, every group reading the listed kv rows again); CUDA cores otherwise.
 */
DSA_API dsa_status dsa_sparse_attn(const uint16_t* q, const uint16_t* kv, const float* attn_sink, const int32_t* idx,
                                   int T, int N, int H, int D, int K, float scale, uint16_t* out, float* lse,
                                   void* stream);

/*
 * dsa_sparse_attn_bwd -- gradients of dsa_sparse_attn (TileLang README, "Sparse MLA Backward":
 * delta = the row-wise product of the output and its gradient; dS = P (dP - delta); dQ from dS
 * and the listed rows; dKV from dS and q plus P and dO, accumulated atomically at the listed
 * positions).  For the loss sum_{t,h,d} do[t,h,d] out[t,h,d], per token t and head h, with
 * p_j = e^{s_j - lse[t,h]} over the listed entries:
 *     dP_j = do[t,h,:] . kv[j,:],   delta = do[t,h,:] . out[t,h,:]
 *     ds_j = p_j (dP_j - delta)
 *     dq[t,h,:] = scale sum_j ds_j kv[j,:]
 *     dkv[j,:] += scale ds_j q[t,h,:] + p_j do[t,h,:]   (every listed occurrence)
 *     dsink[h] += -e^{attn_sink[h] - lse[t,h]} delta
 * P and dS enter the three products as bf16 (as the forward's weights do); products accumulate
 * in fp32.
 *
 *   q, kv, attn_sink, idx, scale   as passed to dsa_sparse_attn (q and kv 16-byte aligned)
 *   out        bf16 [T, H, D]   the forward's output
 *   lse        float [T, H]     the forward's lse output
 *   dout       bf16 [T, H, D]   gradient of the loss with respect to out
 *   dq         float [T, H, D]  OUTPUT (overwritten)
 *   dkv        float [N, D]     OUTPUT (overwritten; 16-byte aligned)
 *   dsink      float [H] or NULL  OUTPUT (overwritten) when attn_sink is given
 *   D in {128, 256}, H >= 1 (up to 64 heads per kernel launch; more heads as consecutive groups
 *   of 64, one launch each, all adding into dkv).  Returns DSA_ERR_UNSUPPORTED for another D and
 *   DSA_ERR_INVALID_ARG for a null / misaligned pointer or a negative size (nothing launched).
 *   dkv is summed with atomic adds, so its last bits may differ from run to run.
 */
DSA_API dsa_status dsa_sparse_attn_bwd(const uint16_t* q, const uint16_t* kv, const float* attn_sink,
                                       const int32_t* idx, const uint16_t* out, const float* lse,
                                       const uint16_t* dout, int T, int N, int H, int D, int K, float scale,
                                       float* dq, float* dkv, float* dsink, void* stream);

/*
 * dsa_check_bounded_wait -- failure-detection self-check (no counterpart in the method's
 * description: it tests the library's own guarantee that no device-side wait is unbounded).
 * Runs one CTA on `stream` in which one warp waits, through the same bounded wait as every
 * pipeline wait of the library, on a barrier that nothing ever completes, and a second warp
 * waits on another such barrier once the first has given up.  The first wait expires after the
 * library's limit (about one second), records a timeout in the device error word and raises the
 * CTA's abort flag; the second then returns at once without recording anything.  Synchronises
 * `stream`.  If wait_ns (HOST memory, 2 entries) is not null it receives the device time each
 * wait took in nanoseconds (0 / UINT64_MAX: the wait completed, which must not happen).
 * Returns DSA_OK when the kernel ran, DSA_ERR_CUDA otherwise; the timeout it recorded is then
 * reported, and cleared, by the next dsa_get_device_error().  The CUDA context stays usable.
 */
DSA_API dsa_status dsa_check_bounded_wait(uint64_t* wait_ns, void* stream);

/* dsa_status_string -- a static, human-readable name for a status code. */
DSA_API const char* dsa_status_string(dsa_status status);

/* dsa_version -- the ABI version (major * 10000 + minor * 100 + patch). */
DSA_API int dsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
