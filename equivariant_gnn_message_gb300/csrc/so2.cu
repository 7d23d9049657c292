// eqmp_fused_so2: the fused layer in the aligned (SO(2)) frame.
#include "k_so2.cuh"
#include "launch.h"

namespace eqmp {

template <int C, typename XT, bool RADIAL>
static eqmp_status launch_so2_t(const LayerArgs& a, const CUtensorMap& map, cudaStream_t st,
                                const DeviceInfo& dev) {
  using K = So2Cfg<C, XT, RADIAL>;
  auto kern = k_so2<C, XT, RADIAL>;
  static unsigned long long attr_done = 0;
  static int clusters_cache[64] = {0};
  if (ensure_smem_attr(kern, K::SMEM_BYTES, &attr_done) != cudaSuccess) return EQMP_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = K::Q;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(K::NTHREADS);
  cfg.dynamicSmemBytes = K::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int d = 0;
  cudaGetDevice(&d);
  // Clusters resident at once on the whole device: the persistent grid.
  int nc = __atomic_load_n(&clusters_cache[d & 63], __ATOMIC_RELAXED);
  if (nc == 0) {
    cfg.gridDim = dim3(K::Q * dev.sms);
    if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess || nc < 1) return EQMP_ERR_CUDA;
    __atomic_store_n(&clusters_cache[d & 63], nc, __ATOMIC_RELAXED);
  }
  const long long need = ((long long)a.N + K::Q - 1) / K::Q;  // at least one receiver per cluster
  const int clusters = (int)(need < nc ? need : nc);
  if (clusters <= 0) return EQMP_OK;
  cfg.gridDim = dim3(clusters * K::Q);
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, map, a));
}

template <typename XT, bool RADIAL>
static eqmp_status launch_so2_c(const LayerArgs& a, int C, const CUtensorMap& map, cudaStream_t st,
                                const DeviceInfo& dev) {
  switch (C) {
    case 8: return launch_so2_t<8, XT, RADIAL>(a, map, st, dev);
    case 16: return launch_so2_t<16, XT, RADIAL>(a, map, st, dev);
    case 32: return launch_so2_t<32, XT, RADIAL>(a, map, st, dev);
    case 64: return launch_so2_t<64, XT, RADIAL>(a, map, st, dev);
    case 128: return launch_so2_t<128, XT, RADIAL>(a, map, st, dev);
  }
  return EQMP_ERR_UNSUPPORTED;
}

static bool al(const void* p, unsigned n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

}  // namespace eqmp

using namespace eqmp;

extern "C" eqmp_status eqmp_fused_so2(const float* vec, const void* x, int64_t N_src, eqmp_dtype x_dtype,
                                      const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E,
                                      int32_t C, eqmp_weights wt, void* out, eqmp_dtype out_dtype,
                                      eqmp_stream_t stream) {
  if (N < 0 || E < 0 || N_src < 0) return EQMP_ERR_INVALID_ARG;
  if (N > INT32_MAX - 1 || E > INT32_MAX || N_src > INT32_MAX) return EQMP_ERR_INVALID_ARG;
  if ((x_dtype != EQMP_F32 && x_dtype != EQMP_BF16) || out_dtype != x_dtype) return EQMP_ERR_INVALID_ARG;
  const bool shared = wt.w != nullptr;
  if (shared) {
    if (wt.R || wt.M || wt.K != 0) return EQMP_ERR_INVALID_ARG;
  } else {
    if (wt.K != 8) return EQMP_ERR_UNSUPPORTED;
    if (E > 0 && (!wt.R || !wt.M)) return EQMP_ERR_INVALID_ARG;
    if (!al(wt.R, 16) || !al(wt.M, 4)) return EQMP_ERR_INVALID_ARG;
  }
  if (C != 8 && C != 16 && C != 32 && C != 64 && C != 128) return EQMP_ERR_UNSUPPORTED;
  if (N == 0) return EQMP_OK;
  if (!row_offsets || !out || !al(out, 16)) return EQMP_ERR_INVALID_ARG;
  if (E > 0 && (!vec || !src || !x || N_src < 1 || !al(x, 16) || !al(vec, 4) || !al(src, 4)))
    return EQMP_ERR_INVALID_ARG;
  DeviceInfo dev;
  eqmp_status s = device_info(&dev);
  if (s != EQMP_OK) return s;
  LayerArgs a{};
  a.vec = vec; a.x = x; a.off = row_offsets; a.src = src; a.w = wt.w; a.R = wt.R; a.M = wt.M;
  a.out = out; a.watchdog = dev.watchdog; a.N = (int)N; a.E = (int)E; a.N_src = (int)N_src;
  const bool bf16 = x_dtype == EQMP_BF16;
  CUtensorMap map;
  if (E > 0) {
    s = encode_x_map(x, N_src, C, bf16, &map);
    if (s != EQMP_OK) return s;
  } else {
    memset(&map, 0, sizeof(map));
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (bf16) return shared ? launch_so2_c<__nv_bfloat16, false>(a, C, map, st, dev)
                          : launch_so2_c<__nv_bfloat16, true>(a, C, map, st, dev);
  return shared ? launch_so2_c<float, false>(a, C, map, st, dev) : launch_so2_c<float, true>(a, C, map, st, dev);
}
