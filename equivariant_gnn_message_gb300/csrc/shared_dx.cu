// Gradient of x for shared weights: the fused shared-weight kernel run over
// the sender view (transposed walk), fp32 storage.
#include "launch_shared.cuh"

namespace eqmp {
eqmp_status launch_shared_dx_f32(const LayerArgs& a, int C, const CUtensorMap& map, cudaStream_t st,
                                 const DeviceInfo& dev) {
  return launch_shared_c<float, true, true>(a, C, map, st, dev);
}
}  // namespace eqmp
