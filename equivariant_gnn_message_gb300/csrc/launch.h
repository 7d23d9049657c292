// Host-side launcher declarations shared by the translation units of libeqmp.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "eqmp.h"
#include "layer_args.cuh"

namespace eqmp {

struct DeviceInfo {
  int sms = 0;          // multiprocessors
  int* watchdog = nullptr;  // device address of the watchdog word
};

// Per-device facts, initialised once per device (thread-safe).
eqmp_status device_info(DeviceInfo* out);

// TMA descriptor for x viewed as [N_src * C*16*elem/128 rows][128 bytes],
// box = one node row, 128-byte swizzle, zero fill out of bounds.
eqmp_status encode_x_map(const void* x, long long n_src, int C, bool bf16, CUtensorMap* map);

// Fused / tp_scatter layer launchers (one per storage type and weight mode).
eqmp_status launch_shared_f32(const LayerArgs& a, int C, bool from_vec, const CUtensorMap& map,
                              cudaStream_t st, const DeviceInfo& dev);
eqmp_status launch_shared_bf16(const LayerArgs& a, int C, bool from_vec, const CUtensorMap& map,
                               cudaStream_t st, const DeviceInfo& dev);
// Gradient of x, shared weights: LayerArgs of the transposed walk (rows =
// senders through perm/dst, x = upstream gradient, map over its rows).
eqmp_status launch_shared_dx_f32(const LayerArgs& a, int C, const CUtensorMap& map, cudaStream_t st,
                                 const DeviceInfo& dev);
eqmp_status launch_radial_f32(const LayerArgs& a, int C, bool from_vec, cudaStream_t st,
                              const DeviceInfo& dev);
eqmp_status launch_radial_bf16(const LayerArgs& a, int C, bool from_vec, cudaStream_t st,
                               const DeviceInfo& dev);

inline eqmp_status cuda_status(cudaError_t e) { return e == cudaSuccess ? EQMP_OK : EQMP_ERR_CUDA; }

// Sets the dynamic shared memory limit of `kernel` once per device.
template <typename Kernel>
cudaError_t ensure_smem_attr(Kernel kernel, int bytes, unsigned long long* done_mask) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const unsigned long long bit = 1ull << (dev & 63);
  if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) __atomic_fetch_or(done_mask, bit, __ATOMIC_RELEASE);
  return err;
}

}  // namespace eqmp
