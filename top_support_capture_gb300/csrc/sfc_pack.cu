// Realized-size packing of captured supports ("[Sampling] Stream sampling masks as per-request
// arrays", section Limitations: the capacity-sized [B, W] device-to-host copy moves far more than the
// supports captured). Two launches on the caller's stream: one CTA scans min(|S_r|, W) into CSR
// offsets; then one warp per row copies its entries to their packed place. The outputs may be device
// memory or host memory the device can address (pinned), which makes this the device-to-host move
// itself, sized by what was captured.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/sfc.h"
#include "sfc_device.cuh"

namespace sfc {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kPackRowsPerCta = 8;

__global__ void __launch_bounds__(kScanThreads) pack_scan_kernel(const int32_t* lengths, int64_t B, int32_t W,
                                                                 int64_t* offsets) {
  __shared__ int64_t warp_tot[kScanThreads / 32];
  __shared__ int64_t carry;
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  if (tid == 0) {
    carry = 0;
    offsets[0] = 0;
  }
  __syncthreads();
  for (int64_t r0 = 0; r0 < B; r0 += kScanThreads) {  // uniform
    const int64_t r = r0 + tid;
    const int n = r < B ? min(max(lengths[r], 0), W) : 0;
    const int incl = warp_incl_scan(n);
    if (lane == 31) warp_tot[wp] = incl;
    __syncthreads();
    int64_t before = carry;
    for (int v = 0; v < wp; ++v) before += warp_tot[v];
    if (r < B) offsets[r + 1] = before + incl;
    __syncthreads();  // every thread has read carry and warp_tot
    if (tid == kScanThreads - 1) carry = before + incl;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(32 * kPackRowsPerCta)
    pack_copy_kernel(const int32_t* lengths, const int32_t* ids, const float* lps, int64_t B, int32_t W,
                     const int64_t* offsets, int32_t* ids_out, float* lps_out, int64_t capacity) {
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * kPackRowsPerCta + (threadIdx.x >> 5);
  if (r >= B) return;
  const int n = min(max(lengths[r], 0), W);
  const int64_t base = offsets[r];
  const int32_t* src = ids + r * W;
  const float* srcl = lps ? lps + r * W : nullptr;
  for (int j = lane; j < n; j += 32) {
    const int64_t d = base + j;
    if (d >= capacity) break;
    ids_out[d] = src[j];
    if (srcl) lps_out[d] = srcl[j];
  }
}

}  // namespace
}  // namespace sfc

extern "C" int sfc_pack_supports(const int32_t* lengths, const int32_t* support_ids, const float* support_logprobs,
                                 int64_t B, int32_t packed_width, int64_t* offsets, int32_t* ids_out, float* lps_out,
                                 int64_t capacity, void* stream) {
  if (!lengths || !support_ids || !offsets || !ids_out) return SFC_EINVAL;
  if ((support_logprobs == nullptr) != (lps_out == nullptr)) return SFC_EINVAL;
  if (B < 1 || B > INT32_MAX * static_cast<int64_t>(sfc::kPackRowsPerCta)) return SFC_EINVAL;
  if (packed_width < 1 || packed_width > SFC_MAX_PACKED_WIDTH || capacity < 0) return SFC_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  sfc::pack_scan_kernel<<<1, sfc::kScanThreads, 0, st>>>(lengths, B, packed_width, offsets);
  if (cudaGetLastError() != cudaSuccess) return SFC_ECUDA;
  const unsigned grid = static_cast<unsigned>((B + sfc::kPackRowsPerCta - 1) / sfc::kPackRowsPerCta);
  sfc::pack_copy_kernel<<<grid, 32 * sfc::kPackRowsPerCta, 0, st>>>(lengths, support_ids, support_logprobs, B,
                                                                     packed_width, offsets, ids_out, lps_out,
                                                                     capacity);
  if (cudaGetLastError() != cudaSuccess) return SFC_ECUDA;
  return SFC_OK;
}
