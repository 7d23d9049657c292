// Launch of the shared-weight kernel for one (C, KQ, storage, SH source).
#pragma once

#include "k_shared.cuh"
#include "launch.h"

namespace eqmp {

template <int C, int KQ, typename XT, bool FV, bool TRANS = false>
eqmp_status launch_shared_t(const LayerArgs& a, const CUtensorMap& map, cudaStream_t st,
                            const DeviceInfo& dev) {
  using K = SharedCfg<C, KQ, XT, FV>;
  auto kern = k_shared<C, KQ, XT, FV, TRANS>;
  static unsigned long long attr_done = 0;
  static int occ_cache[64] = {0};
  cudaError_t err = ensure_smem_attr(kern, K::SMEM_BYTES, &attr_done);
  if (err != cudaSuccess) return EQMP_ERR_CUDA;
  int d = 0;
  cudaGetDevice(&d);
  int occ = __atomic_load_n(&occ_cache[d & 63], __ATOMIC_RELAXED);
  if (occ == 0) {
    // setmaxnreg.inc waits until the CTA's register pool can cover the
    // request, with no time limit: launch only if the compiled register
    // count gives a pool at least as large as the split needs.
    if constexpr (K::WS) {
      cudaFuncAttributes fa;
      err = cudaFuncGetAttributes(&fa, kern);
      if (err != cudaSuccess) return EQMP_ERR_CUDA;
      if ((long long)fa.numRegs * K::NTHREADS < (long long)K::RP * 128 + (long long)K::RC * K::NCONS)
        return EQMP_ERR_UNSUPPORTED;
    }
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

// KQ per channel count and storage comes from SharedTune (k_shared.cuh).
template <typename XT, bool FV, bool TRANS = false>
eqmp_status launch_shared_c(const LayerArgs& a, int C, const CUtensorMap& map, cudaStream_t st,
                            const DeviceInfo& dev) {
  switch (C) {
    case 8: return launch_shared_t<8, SharedTune<8, XT>::KQ, XT, FV, TRANS>(a, map, st, dev);
    case 16: return launch_shared_t<16, SharedTune<16, XT>::KQ, XT, FV, TRANS>(a, map, st, dev);
    case 32: return launch_shared_t<32, SharedTune<32, XT>::KQ, XT, FV, TRANS>(a, map, st, dev);
    case 64: return launch_shared_t<64, SharedTune<64, XT>::KQ, XT, FV, TRANS>(a, map, st, dev);
    case 128: return launch_shared_t<128, SharedTune<128, XT>::KQ, XT, FV, TRANS>(a, map, st, dev);
    default: return EQMP_ERR_UNSUPPORTED;
  }
}

}  // namespace eqmp
