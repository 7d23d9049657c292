// Radial-weight fused / tp_scatter kernels (fp32 and bf16 storage).
#include "k_radial.cuh"
#include "launch.h"

namespace eqmp {

template <int C, typename XT, bool FV>
static eqmp_status launch_radial_t(const LayerArgs& a, cudaStream_t st, const DeviceInfo& dev) {
  constexpr int NT = C > kRadialThreads ? C : kRadialThreads;
  constexpr int GROUPS = NT / C;
  const long long want = (a.N + GROUPS - 1) / GROUPS;
  const long long cap = (long long)dev.sms * 16;
  const int grid = (int)(want < cap ? want : cap);
  if (grid <= 0) return EQMP_OK;
  k_radial<C, XT, FV><<<grid, NT, 0, st>>>(a);
  return cuda_status(cudaGetLastError());
}

template <typename XT, bool FV>
static eqmp_status launch_radial_c(const LayerArgs& a, int C, cudaStream_t st, const DeviceInfo& dev) {
  switch (C) {
    case 8: return launch_radial_t<8, XT, FV>(a, st, dev);
    case 16: return launch_radial_t<16, XT, FV>(a, st, dev);
    case 32: return launch_radial_t<32, XT, FV>(a, st, dev);
    case 64: return launch_radial_t<64, XT, FV>(a, st, dev);
    case 128: return launch_radial_t<128, XT, FV>(a, st, dev);
    default: return EQMP_ERR_UNSUPPORTED;
  }
}

eqmp_status launch_radial_f32(const LayerArgs& a, int C, bool from_vec, cudaStream_t st,
                              const DeviceInfo& dev) {
  return from_vec ? launch_radial_c<float, true>(a, C, st, dev)
                  : launch_radial_c<float, false>(a, C, st, dev);
}

eqmp_status launch_radial_bf16(const LayerArgs& a, int C, bool from_vec, cudaStream_t st,
                               const DeviceInfo& dev) {
  return from_vec ? launch_radial_c<__nv_bfloat16, true>(a, C, st, dev)
                  : launch_radial_c<__nv_bfloat16, false>(a, C, st, dev);
}

}  // namespace eqmp
