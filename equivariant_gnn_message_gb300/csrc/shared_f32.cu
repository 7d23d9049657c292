// Shared-weight fused / tp_scatter kernels, fp32 storage.
#include "launch_shared.cuh"

namespace eqmp {
eqmp_status launch_shared_f32(const LayerArgs& a, int C, bool from_vec, const CUtensorMap& map,
                              cudaStream_t st, const DeviceInfo& dev) {
  return from_vec ? launch_shared_c<float, true>(a, C, map, st, dev)
                  : launch_shared_c<float, false>(a, C, map, st, dev);
}
}  // namespace eqmp
