/*
 * sfc.h — fused sample · filter · support capture for one LLM decode step.
 *
 * C ABI of libsfc.so (GB300 / sm_103a). Plain pointers and sizes only.
 *
 * What one call computes, per row r of a [B, V] logits matrix:
 *   z = l / T; p = softmax(z) over every finite logit;
 *   K = {l >= k-th largest logit}          (ties at the cut all kept, so |K| may exceed k)
 *   P = {mass of strictly larger logits <= top_p}   (measured on the full, un-renormalised p)
 *   M = {z - z_max >= ln(min_p)}
 *   S = K ∩ P ∩ M   (the post-filter support, S = {i | w[i] > 0})
 *   token = argmax_{i in S} (z_i - ln E_i),  E_i = -ln u_i,  u_i from Philox4x32-10
 *   logprob_i = z_i - z_max - ln sum_{j in S} exp(z_j - z_max)   (renormalised over S)
 * Sources, by page title and section:
 *   - prhub summary of SGLang PR #36630 ("sampler 原生捕获支持集…"), sections 实现拆解 2-4 and
 *     关键源码片段 (joint top-k/top-p keep-sets intersected, ties at a threshold kept, min-p after,
 *     support = positive weights, selected logprob = log(w[y] / sum w) from the same capture);
 *   - "[Sampling] Stream sampling masks as per-request arrays" (SGLang PR #40986), sections
 *     Contract, Checks removed item 1 and Correctness (per-row packed ids, logprobs, length,
 *     OK/OVERFLOW status against the packed width; selected logprob equals the token's entry;
 *     no opt-in, no cost);
 *   - "vLLM Sampling Mask（Distribution Replay）深入解析", sections 前置要求与参数约束 and
 *     工作原理 Step 1-2 (temperature > 0; survivors are the finite processed logits);
 *   - "topk-subset-sampler" (Gaudi cookbook), section The fix (exponential race; one top-k
 *     candidate subset instead of a full-vocabulary sort).
 *
 * Conventions shared by every entry point:
 *   - Every array argument is a DEVICE pointer, allocated and owned by the caller. The library
 *     allocates nothing and keeps no state between calls other than per-device launch settings
 *     (and what a call leaves in the caller's workspace: see sfc_workspace_size).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream): a
 *     return of SFC_OK means the work was enqueued. The caller synchronises before reading outputs.
 *   - Results are deterministic: identical inputs give bitwise identical outputs.
 */
#ifndef SFC_H_
#define SFC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Logit element types. */
#define SFC_BF16 0 /* bfloat16, stored as 16-bit patterns */
#define SFC_F32 1  /* IEEE float32 */

/* Host return codes. */
#define SFC_OK 0
#define SFC_EINVAL (-1)     /* a required pointer is NULL, a size or the dtype is out of range */
#define SFC_EWORKSPACE (-2) /* workspace_bytes < sfc_workspace_size(...) */
#define SFC_ECUDA (-3)      /* a CUDA launch or attribute call failed; see cudaGetLastError */

/* Per-row device status, written to row_status[r]. */
#define SFC_ROW_OK 0
#define SFC_ROW_OVERFLOW 1   /* capturing row with |S| > packed_width: the first packed_width
                                entries of S (canonical order) were written, lengths[r] = |S| */
#define SFC_ROW_BADPARAM (-1) /* T not finite or <= 0, top_p NaN or < 0, min_p outside [0, 1],
                                 a NaN or +inf logit, or no finite logit in the row */
#define SFC_ROW_TIMEOUT (-2)  /* a bounded wait of the kernel for its own copies gave up (not
                                 expected to happen); the row's other outputs are undefined */
#define SFC_ROW_OUTSIDE 2     /* replay only: the token is not in the row's support */

/* Flags of sfc_sample_filter_capture_ex. */
#define SFC_FLAG_GREEDY_T0 1u /* a row whose temperature is exactly 0 is a greedy row: the token is the
                                 lowest id among the largest logits, a capturing row's support is that
                                 token alone (length 1, log-probability 0); without the flag such a row
                                 is BADPARAM */
#define SFC_FLAG_POSITIONAL 2u /* top-k and top-p truncate the canonical order by position, as the
                                  PyTorch producer does (prhub summary of SGLang PR #36630,
                                  实现拆解 item 5): top-k keeps the first k positions and top-p the positions
                                  whose own exclusive cumulative probability is <= top_p, so the last tie
                                  group can be cut to its lowest ids; min-p stays a threshold on the value */
#define SFC_FLAG_MIN_P_FIRST 4u /* the vLLM sampler's order ("vLLM Sampling Mask（Distribution Replay）
                                   深入解析", 工作原理 Step 1): min-p first drops its tokens (writes
                                   -inf), then top-k / top-p run as one joint step on what is left, so
                                   top-p measures masses renormalised over the min-p survivors; rows
                                   without both min-p and top-p are unaffected */
#define SFC_FLAG_TEST_STALL 8u /* for tests of the failure path only: each CTA never issues the copy of
                                  its first ring stage, so its bounded waits for it give up (after a few
                                  polls instead of seconds); every row that streams reports
                                  SFC_ROW_TIMEOUT, with tokens -1 and lengths 0 (other outputs undefined),
                                  and the copies that were issued are awaited before the kernel ends */

/* Largest packed_width accepted. */
#define SFC_MAX_PACKED_WIDTH 16384

/*
 * Bytes of device workspace that sfc_sample_filter_capture needs for these sizes (0: none; workspace
 * may then be NULL). Short batches of long rows split each row into several independent CTAs
 * ("slices", up to 8) so that some rows stream from HBM while others finish; each slice publishes its
 * candidates, its sample threshold and its softmax statistics in the workspace, and the slice that
 * arrives last (an atomic ticket per row) merges them and finishes the row. The count depends only on
 * B, V, packed_width and dtype. Contract of a non-empty workspace:
 *   - 16-byte aligned, at least this many bytes;
 *   - ZERO-FILLED before its first use (e.g. cudaMemsetAsync once after allocating it); every call
 *     returns each byte it wrote to zero before it completes, so the workspace is reused as is, by
 *     calls of any size (one sized for the largest call serves all);
 *   - used by one call at a time: calls that may overlap on the GPU (other streams) need their own.
 * Returns 0 for arguments out of range.
 */
size_t sfc_workspace_size(int64_t B, int64_t V, int32_t packed_width, int dtype);

/*
 * The same for sfc_sample_filter_capture_ex with a `slices` argument (0: the library's choice, as
 * sfc_workspace_size; 1: no split, 0 bytes; 2..8: that many slices per row, fewer on rows of fewer
 * 16-byte vectors; packed widths above 2048 are never split).
 */
size_t sfc_workspace_size_ex(int64_t B, int64_t V, int32_t packed_width, int dtype, int32_t slices);

/*
 * One decode step: filter, draw and (for opted-in rows) capture the support.
 *
 * logits          [B, row_stride] elements of `dtype`, row-major; only the first V of each row
 *                 are read. Must be aligned to the element size. NaN / +inf make a row BADPARAM;
 *                 -inf tokens are never in the support.
 * dtype           SFC_BF16 or SFC_F32.
 * B, V            rows and vocabulary size: 1 <= B <= 2^31-1, 1 <= V <= 2^31-1.
 * row_stride      elements between row starts, >= V.
 * temperature     [B] float32, finite and > 0.
 * top_k           [B] int32; <= 0 or >= V disables top-k.
 * top_p           [B] float32 in [0, 1]; >= 1 disables top-p.
 * min_p           [B] float32 in [0, 1]; 0 disables min-p.
 * seed, step      race noise: u_i = Philox4x32-10 with key (seed lo, seed hi) and counter
 *                 (token id, row, step lo, step hi), word 0 w, u = (2 (w >> 9) + 1) 2^-24.
 * capture_rows    [B] uint8, nonzero = the row opts in to support capture; NULL = no row does.
 * packed_width    W, 1 <= W <= SFC_MAX_PACKED_WIDTH: columns of the packed outputs.
 * tokens          [B] int32 out: the drawn token, -1 on BADPARAM rows.
 * support_ids     [B, W] int32 out: for capturing rows, the first min(|S|, W) ids of S in
 *                 canonical order (logit descending, id ascending); other entries untouched.
 *                 May be NULL only when capture_rows is NULL.
 * support_logprobs[B, W] float32 out, aligned with support_ids; NULL = "selected" mode (the
 *                 support ids and the selected logprob only). The chosen mode changes no
 *                 other output bit.
 * lengths         [B] int32 out: |S| for capturing rows (not clamped to W), 0 for the others.
 *                 May be NULL only when capture_rows is NULL.
 * selected_logprob[B] float32 out: for capturing rows, the drawn token's logprob over S, bitwise
 *                 equal to its support_logprobs entry; NaN on capturing BADPARAM rows; other
 *                 rows untouched. May be NULL only when capture_rows is NULL.
 * row_status      [B] int32 out: SFC_ROW_OK / SFC_ROW_OVERFLOW / SFC_ROW_BADPARAM /
 *                 SFC_ROW_TIMEOUT.
 * workspace       device scratch of workspace_bytes bytes, with the contract of sfc_workspace_size
 *                 (may be NULL when that returns 0).
 * stream          cudaStream_t to enqueue on.
 *
 * Returns SFC_OK or a negative code (SFC_EWORKSPACE: the rows are split and the workspace is NULL or
 * smaller than sfc_workspace_size; SFC_EINVAL also for a workspace not 16-byte aligned); on error
 * nothing is enqueued.
 */
int sfc_sample_filter_capture(const void* logits, int dtype, int64_t B, int64_t V, int64_t row_stride,
                              const float* temperature, const int32_t* top_k, const float* top_p,
                              const float* min_p, uint64_t seed, uint64_t step, const uint8_t* capture_rows,
                              int32_t packed_width, int32_t* tokens, int32_t* support_ids,
                              float* support_logprobs, int32_t* lengths, float* selected_logprob,
                              int32_t* row_status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * sfc_sample_filter_capture plus the exact support of overflowing rows as a bitmask (the fallback
 * encoding that "vLLM Sampling Mask（Distribution Replay）深入解析" describes in 工作原理 Step 2 for
 * rows whose support is wider than the compact id buffer) and mode flags.
 *
 * support_mask    [B, ceil(V / 32)] uint32 out, or NULL (then this call is sfc_sample_filter_capture).
 *                 For each capturing row with |S| > W (status SFC_ROW_OVERFLOW): bit i % 32 of word
 *                 i / 32 is 1 iff token i is in S (little-endian: bit i % 8 of byte i / 8). Other
 *                 rows are untouched. Needs capture_rows != NULL. Rows whose support is held on
 *                 chip set their bits from it; rows on the multi-pass path read the row once more.
 * flags           0 or an OR of SFC_FLAG_GREEDY_T0 (greedy rows, the width-1 supports of the greedy
 *                 producer that the same page names in Checks removed item 1) and SFC_FLAG_POSITIONAL
 *                 (positional truncation) and SFC_FLAG_MIN_P_FIRST (min-p before top-p) and
 *                 SFC_FLAG_TEST_STALL (failure-path tests); other bits: SFC_EINVAL.
 * max_top_k       the largest top_k among the rows if the caller knows it (as the Gaudi cookbook page
 *                 "topk-subset-sampler", section The fix, reads it from a host copy), else 0. With
 *                 1 <= max_top_k <= 256 and slices = 0, a short batch that the GPU's CTA slots hold
 *                 at once is split into thread-block clusters: each row is streamed by 2, 4 or 8 CTAs
 *                 that exchange their candidates through distributed shared memory (no workspace).
 *                 A row whose top-k exceeds the value is still exact (it falls back to the
 *                 multi-pass path).
 * row_offset      added to each row's index b in the race's Philox counter (row word = row_offset + b;
 *                 0 in sfc_sample_filter_capture). A batch sharded over several calls or GPUs, each
 *                 passing the global index of its first row, draws what one call over the whole batch
 *                 draws: tokens, support ids, lengths and statuses are identical. Support and selected
 *                 logprobs are identical when the shards split their rows as the whole call does, and
 *                 otherwise agree within float32 rounding of the softmax sums (the slice count, which
 *                 depends on B, fixes the order in which partial sums merge). Negative, or
 *                 row_offset + B > 2^32: SFC_EINVAL.
 * slices          0: the library chooses (as sfc_sample_filter_capture); 1: one CTA per row (or a
 *                 cluster, see max_top_k); 2..8: that many slices per row (fewer on rows of fewer
 *                 16-byte vectors; never for packed widths above 2048); other values: SFC_EINVAL.
 *                 The workspace must then hold sfc_workspace_size_ex(B, V, packed_width, dtype, slices)
 *                 bytes. Only the speed and the order of floating-point merges depend on max_top_k and
 *                 slices: identical inputs with the same values give identical outputs.
 * All other arguments, outputs and return codes are those of sfc_sample_filter_capture.
 */
int sfc_sample_filter_capture_ex(const void* logits, int dtype, int64_t B, int64_t V, int64_t row_stride,
                                 const float* temperature, const int32_t* top_k, const float* top_p,
                                 const float* min_p, uint64_t seed, uint64_t step, const uint8_t* capture_rows,
                                 int32_t packed_width, int32_t* tokens, int32_t* support_ids,
                                 float* support_logprobs, int32_t* lengths, float* selected_logprob,
                                 int32_t* row_status, uint32_t* support_mask, uint32_t flags, int32_t max_top_k,
                                 int64_t row_offset, int32_t slices, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * Training-side replay of a captured support: the sampled token's log-probability under (another
 * policy's) logits renormalised over the support S, as the page "vLLM Sampling Mask（Distribution
 * Replay）深入解析" describes in section RL 训练侧使用 (tokens outside S masked to -inf, log-softmax,
 * read at the sampled token). Per row r, with n = lengths[r] and S = support_ids[r, 0:n]:
 *   z = l / T,  token_logprob[r] = z_tok - max_S z - ln sum_{i in S} exp(z_i - max_S z).
 *
 * logits          [B, row_stride] elements of `dtype` (the policy being trained), row-major;
 *                 aligned to the element size.
 * temperature     [B] float32, finite and > 0 (1 replays raw logits).
 * support_ids     [B, W] int32: row r's support in its first lengths[r] entries (as a capture writes
 *                 them); the ids must be distinct — repeated ids give unspecified results.
 * lengths         [B] int32: |S|.
 * packed_width    W, 1 <= W <= SFC_MAX_PACKED_WIDTH.
 * tokens          [B] int32: the sampled tokens.
 * token_logprob   [B] float32 out: the token's log-probability over S; -inf when the token is not
 *                 in S (status SFC_ROW_OUTSIDE); NaN on OVERFLOW and BADPARAM rows.
 * support_logprobs[B, W] float32 out, or NULL: entry j < lengths[r] is support_ids[r, j]'s
 *                 log-probability over S (written on OK and OUTSIDE rows); other entries untouched.
 * row_status      [B] int32 out: SFC_ROW_OK; SFC_ROW_OUTSIDE; SFC_ROW_OVERFLOW when lengths[r] > W
 *                 (the ids are incomplete); SFC_ROW_BADPARAM when T is not finite or <= 0,
 *                 lengths[r] < 1, an id lies outside [0, V), a support logit is NaN or +inf, or no
 *                 support logit is finite.
 * stream          cudaStream_t to enqueue on.
 * Every array is a device pointer owned by the caller; nothing is allocated. Returns SFC_OK or a
 * negative code (nothing enqueued).
 */
int sfc_replay_logprob(const void* logits, int dtype, int64_t B, int64_t V, int64_t row_stride,
                       const float* temperature, const int32_t* support_ids, const int32_t* lengths,
                       int32_t packed_width, const int32_t* tokens, float* token_logprob,
                       float* support_logprobs, int32_t* row_status, void* stream);

/*
 * Realized-size packing of captured supports ("[Sampling] Stream sampling masks as per-request
 * arrays", section Limitations: a capacity-sized [B, W] copy moves far more than was captured).
 * With n_r = min(max(lengths[r], 0), W):
 *   offsets[0] = 0, offsets[r + 1] = offsets[r] + n_r                     (B + 1 int64)
 *   ids_out[offsets[r] + j] = support_ids[r, j],  lps_out[...] = support_logprobs[r, j],  j < n_r
 * Entries whose packed index is >= capacity are not written (offsets[B] still tells the total).
 *
 * lengths, support_ids, support_logprobs: [B], [B, W], [B, W] device arrays as a capture wrote them
 *                 (rows that do not capture have length 0); support_logprobs and lps_out are both
 *                 NULL or both set.
 * offsets, ids_out, lps_out: device memory, or host memory that the device can address (pinned,
 *                 e.g. cudaHostAlloc): then this call is the device-to-host move itself, sized by
 *                 what was captured.
 * Two kernels on `stream`; returns SFC_OK or SFC_EINVAL / SFC_ECUDA (nothing enqueued on EINVAL).
 */
int sfc_pack_supports(const int32_t* lengths, const int32_t* support_ids, const float* support_logprobs,
                      int64_t B, int32_t packed_width, int64_t* offsets, int32_t* ids_out, float* lps_out,
                      int64_t capacity, void* stream);

/*
 * sfc_sample_filter_capture for callers that cannot allocate device memory. The pages describe no such
 * call; it exists for callers whose device memory is owned by a planner that forbids allocations it
 * did not make (an inference engine that pre-plans every buffer, a plugin limited to its host
 * framework's allocator), or that cannot take cudaMalloc's implicit synchronisation on their hot path.
 * They still pass inputs and outputs, but no workspace: rows that the call splits into slices use a
 * scratch array of SFC_STATIC_SCRATCH_BYTES inside the library instead. Every GPU that loads the
 * library holds that array until the process exits.
 *
 * Arguments, outputs and results are those of sfc_sample_filter_capture; `slices` is that of
 * sfc_sample_filter_capture_ex (0: the library's choice, which always fits the array).
 * - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine is called.
 * - The first call on a device (with it current) looks up the array's device address and, if the
 *   library's code is not yet loaded on that device, loads it; make that first call before any stream
 *   capture.
 * - Every call uses the same array on a device, which keeps the last call's contents: each call clears
 *   the per-row tickets it relies on (a cudaMemsetAsync of 4 B bytes on `stream`) before its kernel.
 *   Calls that may overlap on the GPU (other streams, other threads) race on the array: serialise them.
 * - SFC_EWORKSPACE when the requested split needs more than SFC_STATIC_SCRATCH_BYTES; SFC_ECUDA when the
 *   array's address or the clear fails; otherwise the codes of sfc_sample_filter_capture_ex. The clear
 *   is enqueued before that call checks its other arguments, so an argument error may still leave that
 *   clear of the library's own array enqueued (nothing of the caller's is touched).
 */
#define SFC_STATIC_SCRATCH_BYTES (5u * 1024u * 1024u)
int sfc_sample_filter_capture_noalloc(const void* logits, int dtype, int64_t B, int64_t V, int64_t row_stride,
                                      const float* temperature, const int32_t* top_k, const float* top_p,
                                      const float* min_p, uint64_t seed, uint64_t step, const uint8_t* capture_rows,
                                      int32_t packed_width, int32_t* tokens, int32_t* support_ids,
                                      float* support_logprobs, int32_t* lengths, float* selected_logprob,
                                      int32_t* row_status, int32_t slices, void* stream);

/* Static, NUL-terminated text for a return code. */
const char* sfc_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* SFC_H_ */
