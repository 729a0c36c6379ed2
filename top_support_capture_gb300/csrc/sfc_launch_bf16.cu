// bf16 instantiations of the fused kernel.
#include "sfc_launch.cuh"

namespace sfc {
cudaError_t launch_bf16(const Params& p, int cls, cudaStream_t stream) {
  return cls == 0 ? launch_fused<0, ClassA>(p, stream) : launch_fused<0, ClassB>(p, stream);
}
}  // namespace sfc
