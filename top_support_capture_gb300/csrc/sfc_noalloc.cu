// sfc_sample_filter_capture_noalloc: the decode-step call for callers that cannot allocate device
// memory. Its scratch (the workspace of rows split into slices) is a fixed array inside the library.
//
// Who needs it: a caller whose device memory is owned by a planner that forbids allocations it did
// not make (inference engines that pre-plan every buffer, plugins that may only use the host
// framework's allocator), or a caller on a latency-critical path that cannot take cudaMalloc's
// implicit device synchronisation. Such a caller can still pass its own inputs and outputs, but
// cannot hand the library a workspace of its own.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/sfc.h"

namespace {

// The scratch: 5 MiB, enough for every split the library chooses by itself (at most 304 slices of
// 16 KB of candidates each, plus their tickets and records). Every GPU that loads the library keeps
// it for the life of the process.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SFC_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};
std::atomic<bool> g_scratch_ready[kMaxDevices] = {};

// The scratch's device address on the current device. In host code g_noalloc_scratch names a
// host-side stand-in, not device memory, so the address comes from the runtime, once per device
// (the first call on a device; it loads the library's module there if it is not loaded yet).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return SFC_ECUDA;
  }
  if (!g_scratch_ready[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ready[dev].load(std::memory_order_relaxed)) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return SFC_ECUDA;
      }
      g_scratch_addr[dev] = p;
      g_scratch_ready[dev].store(true, std::memory_order_release);
    }
  }
  *out = g_scratch_addr[dev];
  return SFC_OK;
}

}  // namespace

extern "C" int sfc_sample_filter_capture_noalloc(const void* logits, int dtype, int64_t B, int64_t V,
                                                 int64_t row_stride, const float* temperature,
                                                 const int32_t* top_k, const float* top_p, const float* min_p,
                                                 uint64_t seed, uint64_t step, const uint8_t* capture_rows,
                                                 int32_t packed_width, int32_t* tokens, int32_t* support_ids,
                                                 float* support_logprobs, int32_t* lengths,
                                                 float* selected_logprob, int32_t* row_status, int32_t slices,
                                                 void* stream) {
  const size_t need = sfc_workspace_size_ex(B, V, packed_width, dtype, slices);
  if (need > SFC_STATIC_SCRATCH_BYTES) return SFC_EWORKSPACE;  // the split needs more than the array holds
  void* ws = nullptr;
  if (need > 0) {
    const int rc = scratch_address(&ws);
    if (rc != SFC_OK) return rc;
    // The array keeps whatever the previous call left in it, and a call with another batch size lays
    // its per-row tickets over bytes that call used for other things: clear the tickets (the first
    // 4 B bytes) on the caller's stream before the kernel counts on them being zero.
    const size_t tickets = static_cast<size_t>(B) * 4;
    if (cudaMemsetAsync(ws, 0, tickets, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
      (void)cudaGetLastError();
      return SFC_ECUDA;
    }
  }
  return sfc_sample_filter_capture_ex(logits, dtype, B, V, row_stride, temperature, top_k, top_p, min_p, seed, step,
                                      capture_rows, packed_width, tokens, support_ids, support_logprobs, lengths,
                                      selected_logprob, row_status, nullptr, 0u, 0, 0, slices, ws, need, stream);
}
