// C ABI of libsfc.so: argument checks, kernel-class choice, launch.
//
// The declarations and their contracts live in include/sfc.h.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "../../include/sfc.h"
#include "sfc_launch.cuh"

extern "C" size_t sfc_workspace_size(int64_t, int64_t, int32_t, int) { return 0; }

namespace {
// CTAs per row for a short batch (class A only): the largest C in {8, 4, 2} such that B C rows fit
// the GPU's CTA slots at once and each slice keeps at least two ring stages of 16-byte vectors
// (shorter slices measured slower than one CTA per row); only when every row's top-k is known to be
// small (each slice keeps its own top-k candidates on chip).
constexpr int kSplitMaxK = 256;
int sm_count() {
  static int cached[64] = {0};
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}
int choose_split(int64_t B, int64_t V, int elt, int32_t max_top_k) {
  if (max_top_k < 1 || max_top_k > kSplitMaxK) return 1;
  const int64_t slots = static_cast<int64_t>(sfc::ClassA::kCtasPerSm) * sm_count();
  const int64_t vectors = V * elt / 16;
  constexpr int64_t kStageVectors = sfc::ClassA::kStageBytes / 16;
  for (int c = 8; c >= 2; c /= 2)
    if (B * c <= slots && vectors / c >= 2 * kStageVectors) return c;
  return 1;
}
}  // namespace

extern "C" const char* sfc_strerror(int code) {
  switch (code) {
    case SFC_OK: return "success";
    case SFC_EINVAL: return "invalid argument (null pointer, size or dtype out of range, misaligned logits)";
    case SFC_EWORKSPACE: return "workspace too small";
    case SFC_ECUDA: return "CUDA launch failed";
    default: return "unknown sfc error code";
  }
}

extern "C" int sfc_sample_filter_capture_ex(const void* logits, int dtype, int64_t B, int64_t V,
                                            int64_t row_stride, const float* temperature, const int32_t* top_k,
                                            const float* top_p, const float* min_p, uint64_t seed, uint64_t step,
                                            const uint8_t* capture_rows, int32_t packed_width, int32_t* tokens,
                                            int32_t* support_ids, float* support_logprobs, int32_t* lengths,
                                            float* selected_logprob, int32_t* row_status, uint32_t* support_mask,
                                            uint32_t flags, int32_t max_top_k, int64_t row_offset,
                                            void* workspace, size_t workspace_bytes, void* stream) {
  (void)workspace;
  if (support_mask && !capture_rows) return SFC_EINVAL;
  if (flags & ~static_cast<uint32_t>(SFC_FLAG_GREEDY_T0 | SFC_FLAG_POSITIONAL | SFC_FLAG_MIN_P_FIRST)) return SFC_EINVAL;
  if (!logits || !temperature || !top_k || !top_p || !min_p || !tokens || !row_status) return SFC_EINVAL;
  if (dtype != SFC_BF16 && dtype != SFC_F32) return SFC_EINVAL;
  if (B < 1 || B > INT32_MAX || V < 1 || V > INT32_MAX || row_stride < V) return SFC_EINVAL;
  if (row_offset < 0 || row_offset + B > (int64_t{1} << 32)) return SFC_EINVAL;  // the counter's row word
  if (packed_width < 1 || packed_width > SFC_MAX_PACKED_WIDTH) return SFC_EINVAL;
  if (capture_rows && (!support_ids || !lengths || !selected_logprob)) return SFC_EINVAL;
  const int elt = dtype == SFC_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % elt) return SFC_EINVAL;
  if (workspace_bytes < sfc_workspace_size(B, V, packed_width, dtype)) return SFC_EWORKSPACE;

  const int cls = packed_width <= sfc::ClassA::kMaxW ? 0 : 1;
  const int split = (cls == 0) ? choose_split(B, V, elt, max_top_k) : 1;

  sfc::Params p;
  p.logits = logits;
  p.row_stride = row_stride;
  p.V = V;
  p.B = static_cast<int32_t>(B);
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p;
  p.min_p = min_p;
  p.seed = seed;
  p.step = step;
  p.capture_rows = capture_rows;
  p.W = packed_width;
  p.tokens = tokens;
  p.support_ids = support_ids;
  p.support_logprobs = support_logprobs;
  p.lengths = lengths;
  p.selected_logprob = selected_logprob;
  p.row_status = row_status;
  p.support_mask = support_mask;
  p.flags = flags;
  p.split = split;
  p.row_offset = row_offset;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t err = dtype == SFC_BF16 ? sfc::launch_bf16(p, cls, st) : sfc::launch_f32(p, cls, st);
  if (err != cudaSuccess) {
    (void)cudaGetLastError();  // clear the launch error so later, unrelated calls do not see it
    return SFC_ECUDA;
  }
  return SFC_OK;
}

extern "C" int sfc_sample_filter_capture(const void* logits, int dtype, int64_t B, int64_t V, int64_t row_stride,
                                         const float* temperature, const int32_t* top_k, const float* top_p,
                                         const float* min_p, uint64_t seed, uint64_t step,
                                         const uint8_t* capture_rows, int32_t packed_width, int32_t* tokens,
                                         int32_t* support_ids, float* support_logprobs, int32_t* lengths,
                                         float* selected_logprob, int32_t* row_status, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  return sfc_sample_filter_capture_ex(logits, dtype, B, V, row_stride, temperature, top_k, top_p, min_p, seed, step,
                                      capture_rows, packed_width, tokens, support_ids, support_logprobs, lengths,
                                      selected_logprob, row_status, nullptr, 0u, 0, 0, workspace,
                                      workspace_bytes, stream);
}
