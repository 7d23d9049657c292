// Backward entry points: eqmp_fused_backward and its workspace size query.
#include <mutex>

#include "k_bwd.cuh"
#include "k_bwd_sw.cuh"
#include "launch.h"

namespace eqmp {

constexpr int kBwdGridPerSm = 8;

// dw and dvec with shared weights in the forward kernel's schedule
// (k_bwd_sw.cuh); C = 32 and 64.  One workspace row of [34][C] partial dw
// per CTA (at most max_rows CTAs), summed in order by k_bwd_reduce_w.
template <int C, int KQ = 4, bool DW = true, bool DV = true>
static eqmp_status launch_bwd_sw(const BwdArgs& a, float* gw, long long max_rows, cudaStream_t st,
                                 const DeviceInfo& dev) {
  using K = BwdSwCfg<C, KQ, DW, DV>;
  auto kern = k_bwd_sw<C, KQ, DW, DV>;
  static unsigned long long attr_done = 0;
  static int occ_cache[64] = {0};
  if (ensure_smem_attr(kern, K::SMEM_BYTES, &attr_done) != cudaSuccess) return EQMP_ERR_CUDA;
  int d = 0;
  cudaGetDevice(&d);
  int occ = __atomic_load_n(&occ_cache[d & 63], __ATOMIC_RELAXED);
  if (occ == 0) {
    // setmaxnreg.inc waits, without a limit, for the registers it asks for:
    // launch only if the compiled count gives a pool that covers the split
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return EQMP_ERR_CUDA;
    if ((long long)fa.numRegs * K::NTHREADS < (long long)K::RP * 128 + (long long)K::RC * K::NCONS)
      return EQMP_ERR_UNSUPPORTED;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, K::NTHREADS, K::SMEM_BYTES) != cudaSuccess ||
        occ < 1)
      return EQMP_ERR_CUDA;
    __atomic_store_n(&occ_cache[d & 63], occ, __ATOMIC_RELAXED);
  }
  long long grid = (long long)dev.sms * occ;
  if (grid > a.N) grid = a.N;
  if (grid > max_rows) grid = max_rows;
  if (grid <= 0) return EQMP_OK;
  CUtensorMap map;
  if (a.E > 0) {
    const eqmp_status s = encode_x_map(a.x, a.N_src, C, false, &map);
    if (s != EQMP_OK) return s;
  } else {
    memset(&map, 0, sizeof(map));  // never dereferenced: no edge, no load
  }
  kern<<<(int)grid, K::NTHREADS, K::SMEM_BYTES, st>>>(map, a, dev.watchdog);
  if (cudaGetLastError() != cudaSuccess) return EQMP_ERR_CUDA;
  if (DW && gw) {
    k_bwd_reduce_w<<<(34 * C + kRedX - 1) / kRedX, dim3(kRedX, kRedY), 0, st>>>(a.ws, (int)grid, 34 * C, gw);
    if (cudaGetLastError() != cudaSuccess) return EQMP_ERR_CUDA;
  }
  return EQMP_OK;
}

template <int C>
static long long bwd_slots(long long N, int sms) {
  using K = BwdCfg<C, false>;
  const long long want = (N + K::GROUPS - 1) / K::GROUPS;
  const long long cap = (long long)sms * kBwdGridPerSm;
  return (want < cap ? want : cap) * K::GROUPS;
}

// Blocks of k_bwd_wv with radial weights (no per-block workspace rows).
template <int C>
static long long radial_wv_grid(long long N, int sms) {
  using K = BwdCfg<C, true>;
  const long long want = (N + K::NODES - 1) / K::NODES;
  const long long cap = (long long)sms * kBwdGridPerSm;
  return want < cap ? want : cap;
}

static long long slots_for(int C, long long N, int sms) {
  switch (C) {
    case 8: return bwd_slots<8>(N, sms);
    case 16: return bwd_slots<16>(N, sms);
    case 32: return bwd_slots<32>(N, sms);
    case 64: return bwd_slots<64>(N, sms);
    case 128: return bwd_slots<128>(N, sms);
  }
  return -1;
}

// dw and dvec with shared weights.  C = 32: one kernel forms both (KQ = 4,
// A and H in registers together).  C = 64: dw by the forward's schedule
// (KQ = 8, A contracted with g per receiver) and dvec by a second pass
// (KQ = 8, H only), each with half the threads of the fused kernel; the
// fused form at KQ = 4 spent most of its issue slots on the per-edge dY
// reduction over its 256 threads.
template <int C>
static eqmp_status run_dw_dvec(const BwdArgs& a, float* gw, long long max_rows, cudaStream_t st,
                               const DeviceInfo& dev) {
  if constexpr (C == 64) {
    if (gw) {
      const eqmp_status s = launch_bwd_sw<C, 8, true, false>(a, gw, max_rows, st, dev);
      if (s != EQMP_OK) return s;
    }
    if (a.gvec) return launch_bwd_sw<C, 8, false, true>(a, nullptr, max_rows, st, dev);
    return EQMP_OK;
  } else {
    return launch_bwd_sw<C>(a, gw, max_rows, st, dev);
  }
}

// Gradient of x with shared weights:
//   gx[j,c,k1] = sum_p w[p,c] sum_{k3,k2} C_p[k3,k1,k2] B[j,c,k3,k2],
//   B[j,c,k3,k2] = sum_{e: src_e = j} g[dst_e,c,k3] Y_e[k2],
// which is the forward layer's schedule (accumulate outer products, then
// contract once per row) over the sender view, gathering rows of g, with the
// CG tables transposed.  The fused shared-weight kernel runs it.
static eqmp_status run_dx_shared(const BwdArgs& b, int C, cudaStream_t st, const DeviceInfo& dev) {
  if (b.N_src == 0) return EQMP_OK;
  if (b.N == 0) return cuda_status(cudaMemsetAsync(b.gx, 0, (size_t)b.N_src * C * 16 * 4, st));
  LayerArgs a{};
  a.vec = b.vec;
  a.x = b.g;
  a.off = b.send_off;
  a.w = b.w;
  a.out = b.gx;
  a.watchdog = dev.watchdog;
  a.N = b.N_src;
  a.E = b.n_send;
  a.N_src = b.N;
  a.perm = b.send_edges;
  a.dst = b.dst;
  a.E_edges = b.E;
  CUtensorMap map;
  if (b.n_send > 0) {
    const eqmp_status s = encode_x_map(b.g, b.N, C, false, &map);
    if (s != EQMP_OK) return s;
  } else {
    memset(&map, 0, sizeof(map));  // never dereferenced: no edge, no load
  }
  return launch_shared_dx_f32(a, C, map, st, dev);
}

// dL/dM from the per-edge path sums S (a.ws, [E][34C]): chunk partials
// after S in the workspace, then their fixed-order sum.
static eqmp_status reduce_M(const BwdArgs& a, int C, float* gM, cudaStream_t st) {
  const int cols = 34 * C;
  float* part = a.ws + (size_t)a.E * cols;
  k_bwd_partial_M<<<dim3((cols + kRedX - 1) / kRedX, kRmChunks), dim3(kRedX, kRedY), 0, st>>>(
      a.R, a.ws, a.off, a.N, a.E, cols, part);
  if (cudaGetLastError() != cudaSuccess) return EQMP_ERR_CUDA;
  k_bwd_reduce_w<<<(8 * cols + kRedX - 1) / kRedX, dim3(kRedX, kRedY), 0, st>>>(part, kRmChunks, 8 * cols, gM);
  return cuda_status(cudaGetLastError());
}

// Radial workspace: S rows for every edge, then the chunk partials of dL/dM.
static long long radial_ws_floats(long long E, int C) { return (E + 8ll * kRmChunks) * 34 * C; }

template <int C, bool RADIAL>
static eqmp_status run_bwd(const BwdArgs& a, bool want_x, bool want_wv, float* gw, float* gM,
                           cudaStream_t st, const DeviceInfo& dev) {
  using K = BwdCfg<C, RADIAL>;
  if (!RADIAL && want_x) {
    const eqmp_status s = run_dx_shared(a, C, st, dev);
    if (s != EQMP_OK) return s;
  } else if (want_x && a.N_src > 0) {
    if constexpr (RADIAL) {  // per-edge weights: one group of lanes (or a block) per sender
      const long long want = (a.N_src + K::NODES - 1) / K::NODES;
      const long long cap = (long long)dev.sms * 16;
      k_bwd_x<C, RADIAL><<<(int)(want < cap ? want : cap), K::NT, 0, st>>>(a);
      if (cudaGetLastError() != cudaSuccess) return EQMP_ERR_CUDA;
    }
  }
  if constexpr (!RADIAL && (C == 32 || C == 64)) {
    if (want_wv && a.N > 0) return run_dw_dvec<C>(a, gw, 1ll << 40, st, dev);
    return EQMP_OK;
  }
  if (want_wv && a.N > 0) {
    const int grid = (int)(RADIAL ? radial_wv_grid<C>(a.N, dev.sms) : bwd_slots<C>(a.N, dev.sms) / K::GROUPS);
    const int smem = RADIAL ? 0 : K::GROUPS * 34 * C * 4;
    static unsigned long long attr_done = 0;
    if (ensure_smem_attr(k_bwd_wv<C, RADIAL>, smem > 0 ? smem : 1, &attr_done) != cudaSuccess)
      return EQMP_ERR_CUDA;
    k_bwd_wv<C, RADIAL><<<grid, K::NT, smem, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return EQMP_ERR_CUDA;
    if (!RADIAL && gw) {
      k_bwd_reduce_w<<<(34 * C + kRedX - 1) / kRedX, dim3(kRedX, kRedY), 0, st>>>(a.ws, grid * K::GROUPS, 34 * C, gw);
      if (cudaGetLastError() != cudaSuccess) return EQMP_ERR_CUDA;
    }
    if (RADIAL && gM) return reduce_M(a, C, gM, st);
  }
  return EQMP_OK;
}

template <bool RADIAL>
static eqmp_status dispatch_bwd(int C, const BwdArgs& a, bool want_x, bool want_wv, float* gw, float* gM,
                                cudaStream_t st, const DeviceInfo& dev) {
  switch (C) {
    case 8: return run_bwd<8, RADIAL>(a, want_x, want_wv, gw, gM, st, dev);
    case 16: return run_bwd<16, RADIAL>(a, want_x, want_wv, gw, gM, st, dev);
    case 32: return run_bwd<32, RADIAL>(a, want_x, want_wv, gw, gM, st, dev);
    case 64: return run_bwd<64, RADIAL>(a, want_x, want_wv, gw, gM, st, dev);
    case 128: return run_bwd<128, RADIAL>(a, want_x, want_wv, gw, gM, st, dev);
  }
  return EQMP_ERR_UNSUPPORTED;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace eqmp

using namespace eqmp;

extern "C" {

int64_t eqmp_fused_backward_workspace_size(int64_t N, int64_t E, int32_t C, int32_t radial) {
  if (N < 0 || E < 0) return -1;
  if (radial) return radial_ws_floats(E, C) * 4;
  DeviceInfo dev;
  if (device_info(&dev) != EQMP_OK) return -1;
  const long long slots = slots_for(C, N, dev.sms);
  return slots < 0 ? -1 : slots * 34 * (int64_t)C * 4;
}

eqmp_status eqmp_fused_backward(const float* vec, const float* x, int64_t N_src, const int32_t* row_offsets,
                                const int32_t* src, const int32_t* dst, const int32_t* send_offsets,
                                const int32_t* send_edges, int64_t E_send, int64_t N, int64_t E, int32_t C,
                                eqmp_weights weights, const float* grad_out, float* grad_x, float* grad_w,
                                float* grad_R, float* grad_M, float* grad_vec, void* workspace,
                                int64_t workspace_bytes, eqmp_stream_t stream) {
  if (N < 0 || E < 0 || N_src < 0 || E_send < 0) return EQMP_ERR_INVALID_ARG;
  if (N > INT32_MAX - 1 || E > INT32_MAX || N_src > INT32_MAX - 1 || E_send > INT32_MAX)
    return EQMP_ERR_INVALID_ARG;
  if (C != 8 && C != 16 && C != 32 && C != 64 && C != 128) return EQMP_ERR_UNSUPPORTED;
  const bool radial = weights.w == nullptr;
  if (!radial && (weights.R || weights.M || weights.K != 0)) return EQMP_ERR_INVALID_ARG;
  if (radial && weights.K != 8) return EQMP_ERR_UNSUPPORTED;
  if (radial && E > 0 && (!weights.R || !weights.M)) return EQMP_ERR_INVALID_ARG;
  if (!radial && (grad_R || grad_M)) return EQMP_ERR_INVALID_ARG;
  if (radial && grad_w) return EQMP_ERR_INVALID_ARG;
  const bool want_x = grad_x != nullptr;
  const bool want_wv = grad_vec || grad_w || grad_R || grad_M;
  if (want_x && (!send_offsets || (E_send > 0 && (!send_edges || !dst)) || !aligned16(grad_x)))
    return EQMP_ERR_INVALID_ARG;
  if ((want_x || want_wv) && N > 0 && (!row_offsets || !grad_out || !aligned16(grad_out)))
    return EQMP_ERR_INVALID_ARG;
  if (E > 0 && (want_x || want_wv) && (!vec || !src || !x || !aligned16(x) || N_src < 1))
    return EQMP_ERR_INVALID_ARG;
  if (radial && E > 0 && (!aligned16(weights.R) || (grad_R && !aligned16(grad_R)))) return EQMP_ERR_INVALID_ARG;
  DeviceInfo dev;
  eqmp_status s = device_info(&dev);
  if (s != EQMP_OK) return s;
  const int64_t need = want_wv ? eqmp_fused_backward_workspace_size(N, E, C, radial ? 1 : 0) : 0;
  if (need < 0) return EQMP_ERR_CUDA;
  if (want_wv && need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return EQMP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  BwdArgs a{};
  a.vec = vec; a.x = x; a.off = row_offsets; a.src = src; a.dst = dst;
  a.send_off = send_offsets; a.send_edges = send_edges;
  a.w = weights.w; a.R = weights.R; a.M = weights.M; a.g = grad_out;
  a.gx = grad_x; a.gvec = grad_vec; a.gR = grad_R; a.ws = static_cast<float*>(workspace);
  a.N = (int)N; a.E = (int)E; a.N_src = (int)N_src; a.n_send = (int)E_send;
  if (radial && grad_M && N == 0) {  // no receiver, no edge: dL/dM = 0
    if (cudaMemsetAsync(grad_M, 0, (size_t)8 * 34 * C * 4, st) != cudaSuccess) return EQMP_ERR_CUDA;
    grad_M = nullptr;
  }
  if (!radial && grad_w && N == 0) {
    if (cudaMemsetAsync(grad_w, 0, (size_t)34 * C * 4, st) != cudaSuccess) return EQMP_ERR_CUDA;
  }
  return radial ? dispatch_bwd<true>(C, a, want_x, want_wv, nullptr, grad_M, st, dev)
                : dispatch_bwd<false>(C, a, want_x, want_wv, grad_w, nullptr, st, dev);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// eqmp_fused_backward_noalloc: the same backward with its scratch in a
// static device array instead of a caller-supplied workspace.
//
// Some callers cannot hand the library extra device memory: code running as
// a plugin inside a host framework that owns the whole device memory pool,
// or a tight simulation loop that must not pay for an allocation every
// step.  This entry point needs nothing beyond its inputs and outputs.  Its
// scratch is the array below, of kNoAllocBytes (8 MiB); every GPU that loads
// the library holds it until the process exits.  All calls share the array
// and it keeps the previous call's contents; the kernels overwrite every
// part they later read, so nothing has to start at zero.  Two calls that
// overlap on the GPU (other streams, other threads) race on the array.
namespace eqmp {

constexpr size_t kNoAllocBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch for the current device, looked up once
// per device.  Host code must not pass the symbol itself to a kernel: on the
// host it is only a stand-in, not a device address.
static eqmp_status noalloc_scratch(float** out) {
  static std::once_flag once[64];
  static void* addr[64];
  static cudaError_t err[64];
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return EQMP_ERR_CUDA;
  std::call_once(once[d], [d]() { err[d] = cudaGetSymbolAddress(&addr[d], g_noalloc_scratch); });
  if (err[d] != cudaSuccess || addr[d] == nullptr) return EQMP_ERR_CUDA;
  *out = static_cast<float*>(addr[d]);
  return EQMP_OK;
}

template <int C, bool RADIAL>
static eqmp_status run_bwd_noalloc(const BwdArgs& a, bool want_x, bool want_wv, float* gw, float* gM,
                                   cudaStream_t st, const DeviceInfo& dev) {
  using K = BwdCfg<C, RADIAL>;
  if (!RADIAL && want_x) {
    const eqmp_status s = run_dx_shared(a, C, st, dev);
    if (s != EQMP_OK) return s;
  } else if (want_x && a.N_src > 0) {
    if constexpr (RADIAL) {  // per-edge weights: one group of lanes (or a block) per sender
      const long long want = (a.N_src + K::NODES - 1) / K::NODES;
      const long long cap = (long long)dev.sms * 16;
      k_bwd_x<C, RADIAL><<<(int)(want < cap ? want : cap), K::NT, 0, st>>>(a);
      if (cudaGetLastError() != cudaSuccess) return EQMP_ERR_CUDA;
    }
  }
  if constexpr (!RADIAL && (C == 32 || C == 64)) {
    if (want_wv && a.N > 0)
      return run_dw_dvec<C>(a, gw, (long long)(kNoAllocBytes / ((size_t)34 * C * 4)), st, dev);
    return EQMP_OK;
  }
  if (want_wv && a.N > 0) {
    // as many receiver groups as the static scratch holds partial rows for
    const long long fit = (long long)(kNoAllocBytes / ((size_t)34 * C * 4)) / K::GROUPS;
    long long grid = RADIAL ? radial_wv_grid<C>(a.N, dev.sms) : bwd_slots<C>(a.N, dev.sms) / K::GROUPS;
    if (!RADIAL && grid > fit) grid = fit;
    const int smem = RADIAL ? 0 : K::GROUPS * 34 * C * 4;
    static unsigned long long attr_done = 0;
    if (ensure_smem_attr(k_bwd_wv<C, RADIAL>, smem > 0 ? smem : 1, &attr_done) != cudaSuccess)
      return EQMP_ERR_CUDA;
    k_bwd_wv<C, RADIAL><<<(int)grid, K::NT, smem, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return EQMP_ERR_CUDA;
    if (!RADIAL && gw) {
      k_bwd_reduce_w<<<(34 * C + kRedX - 1) / kRedX, dim3(kRedX, kRedY), 0, st>>>(a.ws, (int)grid * K::GROUPS, 34 * C, gw);
      if (cudaGetLastError() != cudaSuccess) return EQMP_ERR_CUDA;
    }
    if (RADIAL && gM) return reduce_M(a, C, gM, st);
  }
  return EQMP_OK;
}

template <bool RADIAL>
static eqmp_status dispatch_bwd_noalloc(int C, const BwdArgs& a, bool want_x, bool want_wv, float* gw, float* gM,
                                        cudaStream_t st, const DeviceInfo& dev) {
  switch (C) {
    case 8: return run_bwd_noalloc<8, RADIAL>(a, want_x, want_wv, gw, gM, st, dev);
    case 16: return run_bwd_noalloc<16, RADIAL>(a, want_x, want_wv, gw, gM, st, dev);
    case 32: return run_bwd_noalloc<32, RADIAL>(a, want_x, want_wv, gw, gM, st, dev);
    case 64: return run_bwd_noalloc<64, RADIAL>(a, want_x, want_wv, gw, gM, st, dev);
    case 128: return run_bwd_noalloc<128, RADIAL>(a, want_x, want_wv, gw, gM, st, dev);
  }
  return EQMP_ERR_UNSUPPORTED;
}

}  // namespace eqmp

extern "C" {

int64_t eqmp_fused_backward_noalloc_max_bytes(void) { return (int64_t)eqmp::kNoAllocBytes; }

eqmp_status eqmp_fused_backward_noalloc(const float* vec, const float* x, int64_t N_src,
                                        const int32_t* row_offsets, const int32_t* src, const int32_t* dst,
                                        const int32_t* send_offsets, const int32_t* send_edges, int64_t E_send,
                                        int64_t N, int64_t E, int32_t C, eqmp_weights weights,
                                        const float* grad_out, float* grad_x, float* grad_w, float* grad_R,
                                        float* grad_M, float* grad_vec, eqmp_stream_t stream) {
  if (N < 0 || E < 0 || N_src < 0 || E_send < 0) return EQMP_ERR_INVALID_ARG;
  if (N > INT32_MAX - 1 || E > INT32_MAX || N_src > INT32_MAX - 1 || E_send > INT32_MAX)
    return EQMP_ERR_INVALID_ARG;
  if (C != 8 && C != 16 && C != 32 && C != 64 && C != 128) return EQMP_ERR_UNSUPPORTED;
  const bool radial = weights.w == nullptr;
  if (!radial && (weights.R || weights.M || weights.K != 0)) return EQMP_ERR_INVALID_ARG;
  if (radial && weights.K != 8) return EQMP_ERR_UNSUPPORTED;
  if (radial && E > 0 && (!weights.R || !weights.M)) return EQMP_ERR_INVALID_ARG;
  if (!radial && (grad_R || grad_M)) return EQMP_ERR_INVALID_ARG;
  if (radial && grad_w) return EQMP_ERR_INVALID_ARG;
  const bool want_x = grad_x != nullptr;
  const bool want_wv = grad_vec || grad_w || grad_R || grad_M;
  if (want_x && (!send_offsets || (E_send > 0 && (!send_edges || !dst)) || !aligned16(grad_x)))
    return EQMP_ERR_INVALID_ARG;
  if ((want_x || want_wv) && N > 0 && (!row_offsets || !grad_out || !aligned16(grad_out)))
    return EQMP_ERR_INVALID_ARG;
  if (E > 0 && (want_x || want_wv) && (!vec || !src || !x || !aligned16(x) || N_src < 1))
    return EQMP_ERR_INVALID_ARG;
  if (radial && E > 0 && (!aligned16(weights.R) || (grad_R && !aligned16(grad_R)))) return EQMP_ERR_INVALID_ARG;
  // Radial weights keep one scratch row of 34*C floats per edge (and the
  // dL/dM chunk partials): beyond the static array this entry point cannot
  // run (use eqmp_fused_backward).
  if (radial && want_wv && (size_t)radial_ws_floats(E, C) * 4 > kNoAllocBytes) return EQMP_ERR_UNSUPPORTED;
  DeviceInfo dev;
  eqmp_status s = device_info(&dev);
  if (s != EQMP_OK) return s;
  float* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != EQMP_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  BwdArgs a{};
  a.vec = vec; a.x = x; a.off = row_offsets; a.src = src; a.dst = dst;
  a.send_off = send_offsets; a.send_edges = send_edges;
  a.w = weights.w; a.R = weights.R; a.M = weights.M; a.g = grad_out;
  a.gx = grad_x; a.gvec = grad_vec; a.gR = grad_R; a.ws = scratch;
  a.N = (int)N; a.E = (int)E; a.N_src = (int)N_src; a.n_send = (int)E_send;
  if (radial && grad_M && N == 0) {
    if (cudaMemsetAsync(grad_M, 0, (size_t)8 * 34 * C * 4, st) != cudaSuccess) return EQMP_ERR_CUDA;
    grad_M = nullptr;
  }
  if (!radial && grad_w && N == 0) {
    if (cudaMemsetAsync(grad_w, 0, (size_t)34 * C * 4, st) != cudaSuccess) return EQMP_ERR_CUDA;
  }
  return radial ? dispatch_bwd_noalloc<true>(C, a, want_x, want_wv, nullptr, grad_M, st, dev)
                : dispatch_bwd_noalloc<false>(C, a, want_x, want_wv, grad_w, nullptr, st, dev);
}

}  // extern "C"
