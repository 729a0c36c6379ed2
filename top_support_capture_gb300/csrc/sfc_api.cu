// C ABI of libsfc.so: argument checks, kernel-class choice, launch.
//
// The declarations and their contracts live in include/sfc.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>

#include "../../include/sfc.h"
#include "sfc_launch.cuh"

namespace {
// ---- rows split into independent slices (class A) ----
// A row of a short batch is split into S ordinary CTAs that stream its slices in parallel. The split
// pays only while every slice of every row runs at once: each slice CTA and each row's merge carry a
// fixed cost of several microseconds (the first copy's latency, the candidate gather and publish, the
// ticket, the merge), which extra waves of CTAs would add rather than hide. S is the largest count
// with B S <= kSliceSlots (the CTA slots of a GB300: 2 per SM x 152 SMs) and at least two ring
// stages per slice, at most kMaxSlices. It depends on B, V, the dtype and the packed width only (not
// on the device), so identical inputs split the same way everywhere.
constexpr int64_t kSliceSlots = 304;
constexpr int kMaxSlices = 8;
constexpr int kSliceCap = 2048;  // candidates one slice may publish (16 KB of workspace)

int64_t body_vectors(int64_t V, int elt) { return V * elt / 16; }

// Slices per row; `requested` 0 lets the library choose, 1..kMaxSlices asks for that many (fewer if
// the row has fewer 16-byte vectors).
int resolve_slices(int64_t B, int64_t V, int elt, int32_t W, int32_t requested) {
  if (W > sfc::ClassA::kMaxW) return 1;  // the wide class keeps one CTA per row
  const int64_t vectors = body_vectors(V, elt);
  if (requested >= 1) return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(requested, vectors)));
  constexpr int64_t kMinVectors = 2 * (sfc::ClassA::kStageBytes / 16);  // two ring stages
  const int64_t smax = std::min<int64_t>({kMaxSlices, vectors / kMinVectors, kSliceSlots / B});
  return static_cast<int>(std::max<int64_t>(1, smax));
}

// Workspace of S > 1 slices per row: [B] tickets (padded to 256 bytes), [B S] records of 16 bytes
// (padded to 256), [B S kSliceCap] candidates of 8 bytes.
struct SliceLayout {
  size_t tickets, rec, pool, total;
};
SliceLayout slice_layout(int64_t B, int S) {
  auto pad = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  SliceLayout l{};
  if (S <= 1) return l;
  const size_t b = static_cast<size_t>(B), s = static_cast<size_t>(S);
  l.tickets = 0;
  l.rec = pad(b * 4);
  l.pool = l.rec + pad(b * s * 16);
  l.total = l.pool + b * s * static_cast<size_t>(kSliceCap) * 8;
  return l;
}

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

extern "C" size_t sfc_workspace_size_ex(int64_t B, int64_t V, int32_t packed_width, int dtype, int32_t slices) {
  if (B < 1 || V < 1 || (dtype != SFC_BF16 && dtype != SFC_F32) || slices < 0 || slices > kMaxSlices) return 0;
  const int elt = dtype == SFC_BF16 ? 2 : 4;
  return slice_layout(B, resolve_slices(B, V, elt, packed_width, slices)).total;
}

extern "C" size_t sfc_workspace_size(int64_t B, int64_t V, int32_t packed_width, int dtype) {
  return sfc_workspace_size_ex(B, V, packed_width, dtype, 0);
}

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
                                            int32_t slices, void* workspace, size_t workspace_bytes,
                                            void* stream) {
  if (support_mask && !capture_rows) return SFC_EINVAL;
  if (slices < 0 || slices > kMaxSlices) return SFC_EINVAL;
  if (flags & ~static_cast<uint32_t>(SFC_FLAG_GREEDY_T0 | SFC_FLAG_POSITIONAL | SFC_FLAG_MIN_P_FIRST | SFC_FLAG_TEST_STALL))
    return SFC_EINVAL;
  if (!logits || !temperature || !top_k || !top_p || !min_p || !tokens || !row_status) return SFC_EINVAL;
  if (dtype != SFC_BF16 && dtype != SFC_F32) return SFC_EINVAL;
  if (B < 1 || B > INT32_MAX || V < 1 || V > INT32_MAX || row_stride < V) return SFC_EINVAL;
  if (row_offset < 0 || row_offset + B > (int64_t{1} << 32)) return SFC_EINVAL;  // the counter's row word
  if (packed_width < 1 || packed_width > SFC_MAX_PACKED_WIDTH) return SFC_EINVAL;
  if (capture_rows && (!support_ids || !lengths || !selected_logprob)) return SFC_EINVAL;
  const int elt = dtype == SFC_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % elt) return SFC_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) % 16) return SFC_EINVAL;

  const int cls = packed_width <= sfc::ClassA::kMaxW ? 0 : 1;
  // A cluster split only when the caller bounds top_k and asks for no slice count; else slices.
  const int split = (cls == 0 && slices == 0) ? choose_split(B, V, elt, max_top_k) : 1;
  const int nslices = split > 1 ? 1 : resolve_slices(B, V, elt, packed_width, slices);
  if (B * nslices > INT32_MAX) return SFC_EINVAL;  // the grid
  const SliceLayout lay = slice_layout(B, nslices);
  if (nslices > 1 && (workspace == nullptr || workspace_bytes < lay.total)) return SFC_EWORKSPACE;

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
  p.slices = nslices;
  p.slice_cap = kSliceCap;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.tickets = nslices > 1 ? reinterpret_cast<uint32_t*>(ws + lay.tickets) : nullptr;
  p.slice_rec = nslices > 1 ? reinterpret_cast<uint4*>(ws + lay.rec) : nullptr;
  p.slice_pool = nslices > 1 ? reinterpret_cast<uint64_t*>(ws + lay.pool) : nullptr;

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
                                      selected_logprob, row_status, nullptr, 0u, 0, 0, 0, workspace,
                                      workspace_bytes, stream);
}
