// Launch of one instantiation of the fused kernel on the caller's stream: one CTA per row, p.slices
// independent CTAs per row (meeting through the workspace), or one thread-block cluster of p.split
// CTAs per row.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "sfc_kernel.cuh"

namespace sfc {

// Kernel classes: the CTA size, the ring of bulk-copy stages (its space also holds the candidate
// pool after the pass, and so bounds the widest packed output sorted on chip), the candidate bitmap
// (one bit per 16-byte vector of the row) and the stages sampled for the threshold. Class A: 256
// threads, 2 x 32 KB stages, two CTAs per SM (each bulk copy carries a fixed cost, so fewer, larger
// copies stream a row faster: 4 x 16 KB measured 4-15 % slower; a third stage measured no faster and
// costs registers). Class B: 512 threads, 10 x 16 KB stages, one CTA per SM, for wide packed outputs
// (its ring also holds their large candidate pools).
struct ClassA {
  static constexpr int kThreads = 256;
  static constexpr int kStages = 2;
  static constexpr int kStageBytes = 32768;
  static constexpr int kBitmapWords = 4096;
  static constexpr int kMaxW = 2048;
  static constexpr int kCtasPerSm = 2;
  static constexpr int kSampleStages = 2;
};
struct ClassB {
  static constexpr int kThreads = 512;
  static constexpr int kStages = 10;
  static constexpr int kStageBytes = 16384;
  static constexpr int kBitmapWords = 8192;
  static constexpr int kMaxW = 16384;
  static constexpr int kCtasPerSm = 1;
  static constexpr int kSampleStages = 10;
};

template <int DT, class Cls>
cudaError_t launch_fused(const Params& p, cudaStream_t stream) {
  auto kern = fused_kernel<DT, Cls::kThreads, Cls::kStages, Cls::kStageBytes, Cls::kBitmapWords, Cls::kCtasPerSm,
                           Cls::kSampleStages>;
  const size_t smem = static_cast<size_t>(Cls::kStages) * Cls::kStageBytes + static_cast<size_t>(Cls::kBitmapWords) * 4;
  static std::atomic<uint64_t> configured{0};  // one bit per device ordinal < 64
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const uint64_t bit = (dev < 64) ? (1ull << dev) : 0ull;
  if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  if (p.split <= 1) {  // one CTA per row, or p.slices ordinary CTAs per row
    kern<<<static_cast<unsigned>(p.B) * static_cast<unsigned>(p.slices), Cls::kThreads, smem, stream>>>(p);
    return cudaGetLastError();
  }
  // p.split CTAs per row as one thread-block cluster (distributed shared memory between them)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B) * static_cast<unsigned>(p.split), 1, 1);
  cfg.blockDim = dim3(Cls::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_bf16(const Params& p, int cls, cudaStream_t stream);
cudaError_t launch_f32(const Params& p, int cls, cudaStream_t stream);

}  // namespace sfc
