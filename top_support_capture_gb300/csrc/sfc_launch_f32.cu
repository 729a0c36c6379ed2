// float32 instantiations of the fused kernel.
#include "sfc_launch.cuh"

namespace sfc {
cudaError_t launch_f32(const Params& p, int cls, cudaStream_t stream) {
  return cls == 0 ? launch_fused<1, ClassA>(p, stream) : launch_fused<1, ClassB>(p, stream);
}
}  // namespace sfc
