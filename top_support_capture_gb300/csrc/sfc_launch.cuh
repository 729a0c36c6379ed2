// Launch of one instantiation of the fused kernel (cluster launch on the caller's stream).
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "sfc_kernel.cuh"

namespace sfc {

// Kernel classes: the candidate buffer (and thus the widest packed output that can be sorted on
// chip) and the CTA size. Class A: 4 Ki candidates, 256 threads, several CTAs per SM. Class B:
// 24 Ki candidates, 512 threads, one CTA per SM, for wide packed outputs and large top-k.
struct ClassA {
  static constexpr int kThreads = 256;
  static constexpr int kBuf = 4096;
  static constexpr int kMaxW = 2048;
  static constexpr int kCtasPerSm = 4;
};
struct ClassB {
  static constexpr int kThreads = 512;
  static constexpr int kBuf = 24576;
  static constexpr int kMaxW = 16384;
  static constexpr int kCtasPerSm = 1;
};

template <int DT, class Cls>
cudaError_t launch_fused(const Params& p, int split, cudaStream_t stream) {
  constexpr int U = 4;  // 16-byte vectors per thread per tile
  auto kern = fused_kernel<DT, Cls::kThreads, Cls::kBuf, U, Cls::kCtasPerSm>;
  const size_t smem = static_cast<size_t>(Cls::kBuf) * sizeof(uint64_t);
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B) * static_cast<unsigned>(split), 1, 1);
  cfg.blockDim = dim3(Cls::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_bf16(const Params& p, int cls, int split, cudaStream_t stream);
cudaError_t launch_f32(const Params& p, int cls, int split, cudaStream_t stream);

}  // namespace sfc
