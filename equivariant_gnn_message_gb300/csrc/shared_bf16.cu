// Shared-weight fused / tp_scatter kernels, bf16 storage of x and out.
#include "launch_shared.cuh"

namespace eqmp {
eqmp_status launch_shared_bf16(const LayerArgs& a, int C, bool from_vec, const CUtensorMap& map,
                               cudaStream_t st, const DeviceInfo& dev) {
  return from_vec ? launch_shared_c<__nv_bfloat16, true>(a, C, map, st, dev)
                  : launch_shared_c<__nv_bfloat16, false>(a, C, map, st, dev);
}
}  // namespace eqmp
