// Launch of the shared-weight kernel for one (C, KQ, storage, SH source).
#pragma once

#include "k_shared.cuh"
#include "launch.h"

namespace eqmp {

template <int C, int KQ, typename XT, bool FV>
eqmp_status launch_shared_t(const LayerArgs& a, const CUtensorMap& map, cudaStream_t st,
                            const DeviceInfo& dev) {
  using K = SharedCfg<C, KQ, XT, FV>;
  auto kern = k_shared<C, KQ, XT, FV>;
  static unsigned long long attr_done = 0;
  static int occ_cache[64] = {0};
  cudaError_t err = ensure_smem_attr(kern, K::SMEM_BYTES, &attr_done);
  if (err != cudaSuccess) return EQMP_ERR_CUDA;
  int d = 0;
  cudaGetDevice(&d);
  int occ = __atomic_load_n(&occ_cache[d & 63], __ATOMIC_RELAXED);
  if (occ == 0) {
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, K::NTHREADS, K::SMEM_BYTES);
    if (err != cudaSuccess || occ < 1) return EQMP_ERR_CUDA;
    __atomic_store_n(&occ_cache[d & 63], occ, __ATOMIC_RELAXED);
  }
  const long long slots = (long long)dev.sms * occ;
  const int grid = (int)(a.N < slots ? a.N : slots);
  if (grid <= 0) return EQMP_OK;
  kern<<<grid, K::NTHREADS, K::SMEM_BYTES, st>>>(map, a);
  return cuda_status(cudaGetLastError());
}

// KQ per channel count and storage: 4 k1 per thread (64 accumulators) for
// fp32 up to C = 64; 8 (128 accumulators) for bf16 from C = 32 (keeps the
// swizzled reads conflict-free) and for fp32 at C = 128.
template <typename XT, bool FV>
eqmp_status launch_shared_c(const LayerArgs& a, int C, const CUtensorMap& map, cudaStream_t st,
                            const DeviceInfo& dev) {
  constexpr bool B = sizeof(XT) == 2;
  switch (C) {
    case 8: return launch_shared_t<8, 4, XT, FV>(a, map, st, dev);
    case 16: return launch_shared_t<16, 4, XT, FV>(a, map, st, dev);
    case 32: return launch_shared_t<32, B ? 8 : 4, XT, FV>(a, map, st, dev);
    case 64: return launch_shared_t<64, B ? 8 : 4, XT, FV>(a, map, st, dev);
    case 128: return launch_shared_t<128, 8, XT, FV>(a, map, st, dev);
    default: return EQMP_ERR_UNSUPPORTED;
  }
}

}  // namespace eqmp
