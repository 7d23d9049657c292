// C ABI of libeqmp.so: argument checks, dispatch, the standalone SH kernel,
// graph validation and the device watchdog.  Declarations and contracts are
// in include/eqmp.h.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace eqmp {

// Watchdog word, one per device (module globals are per context).
__device__ int g_watchdog_word = 0;
// Result word of eqmp_validate_graph.
__device__ int g_validate_word = 0;

// ------------------------------------------------------------ SH kernel
// One thread per edge; the 16 values go through shared memory so the block
// writes its [256][16] tile of Y with contiguous 16-byte stores.
constexpr int kShThreads = 256;

__global__ void __launch_bounds__(kShThreads) k_sh(const float* __restrict__ vec, int E,
                                                   float* __restrict__ Y) {
  __shared__ float4 tile[kShThreads * 4 + kShThreads / 8];  // padded rows
  const int base = blockIdx.x * kShThreads;
  const int e = base + threadIdx.x;
  float y[16];
  if (e < E) {
    real_sh16(__ldg(vec + 3 * (size_t)e), __ldg(vec + 3 * (size_t)e + 1),
              __ldg(vec + 3 * (size_t)e + 2), y);
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) y[k] = 0.0f;
  }
  // row t occupies float4 slots 4t..4t+3, shifted by t/8 to spread banks
  const int rowp = 4 * threadIdx.x + threadIdx.x / 8;
#pragma unroll
  for (int h = 0; h < 4; ++h) tile[rowp + h] = make_float4(y[4 * h], y[4 * h + 1], y[4 * h + 2], y[4 * h + 3]);
  __syncthreads();
  const int n_valid = min(kShThreads, E - base);
  float4* dst = reinterpret_cast<float4*>(Y) + 4 * (size_t)base;
  for (int i = threadIdx.x; i < 4 * n_valid; i += kShThreads) {
    const int t = i >> 2, h = i & 3;
    dst[i] = tile[4 * t + t / 8 + h];
  }
}

// ------------------------------------------------------------ validation
__global__ void k_validate(const int32_t* __restrict__ off, const int32_t* __restrict__ src, int N,
                           int N_src, int E, int* flag) {
  const int stride = gridDim.x * blockDim.x;
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int o0 = off[0], oN = off[N];
  if (tid == 0 && (o0 < 0 || oN > E || o0 > oN)) atomicOr(flag, 1);
  for (int i = tid; i < N; i += stride)
    if (off[i] > off[i + 1]) atomicOr(flag, 2);
  const int lo = min(max(o0, 0), E), hi = min(max(oN, 0), E);
  for (int e = lo + tid; e < hi; e += stride) {
    const int s = src[e];
    if (s < 0 || s >= N_src) atomicOr(flag, 4);
  }
}

// ------------------------------------------------------------ watchdog self-test
// One thread waits on an mbarrier that nothing will ever complete, with a
// limit of limit_ns; when the wait gives up it records code 5 in the
// watchdog word and the kernel ends.  Shows on a live GPU that an expired
// wait is reported to the host and leaves the context usable, without any
// fault or hang.
__global__ void k_wait_selftest(unsigned long long limit_ns, int* watchdog) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  const unsigned long long t0 = global_ns();
  while (!mbar_test_wait(b, 0)) {
    if (global_ns() - t0 > limit_ns) {
      watchdog_trip(watchdog, 5);
      break;
    }
  }
}

// Eight independent paired-FMA chains per thread: enough independent work
// to keep the FMA pipe busy from any resident warp.
__global__ void __launch_bounds__(256) k_fp32_peak(int iters, float* out) {
  const float t = (float)threadIdx.x * 1e-7f;
  float2 v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = make_float2(t + (float)k * 1e-3f, t - (float)k * 1e-3f);
  const float2 m = make_float2(0.999999f, 1.000001f), c = make_float2(1e-7f, -1e-7f);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __ffma2_rn(v[k], m, c);
  }
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) s += v[k].x + v[k].y;
  if (s == 1234567.0f) *out = s;
}

// ------------------------------------------------------------ device state
eqmp_status device_info(DeviceInfo* out) {
  static std::once_flag once[64];
  static DeviceInfo info[64];
  static cudaError_t init_err[64];
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return EQMP_ERR_CUDA;
  std::call_once(once[d], [d]() {
    DeviceInfo v;
    cudaError_t e = cudaDeviceGetAttribute(&v.sms, cudaDevAttrMultiProcessorCount, d);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&v.watchdog), g_watchdog_word);
    init_err[d] = e;
    info[d] = v;
  });
  if (init_err[d] != cudaSuccess) return EQMP_ERR_CUDA;
  *out = info[d];
  return EQMP_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

eqmp_status encode_x_map(const void* x, long long n_src, int C, bool bf16, CUtensorMap* map) {
  auto fn = encode_fn();
  if (!fn) return EQMP_ERR_CUDA;
  const int elem = bf16 ? 2 : 4;
  const int row_bytes = C * 16 * elem;
  const cuuint64_t inner = 128 / elem;
  const cuuint64_t rows = (cuuint64_t)n_src * (row_bytes / 128);
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {(cuuint32_t)inner, (cuuint32_t)(row_bytes / 128)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                  const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? EQMP_OK : EQMP_ERR_CUDA;
}

static bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static eqmp_status run_layer(bool from_vec, const float* vec_or_Y, const void* x, int64_t N_src,
                             eqmp_dtype x_dtype, const int32_t* off, const int32_t* src, int64_t N,
                             int64_t E, int32_t C, eqmp_weights wt, void* out, eqmp_dtype out_dtype,
                             cudaStream_t st) {
  if (N < 0 || E < 0 || N_src < 0) return EQMP_ERR_INVALID_ARG;
  if (N > INT32_MAX - 1 || E > INT32_MAX || N_src > INT32_MAX) return EQMP_ERR_INVALID_ARG;
  if ((x_dtype != EQMP_F32 && x_dtype != EQMP_BF16) || out_dtype != x_dtype) return EQMP_ERR_INVALID_ARG;
  const bool shared = wt.w != nullptr;
  if (shared) {
    if (wt.R || wt.M || wt.K != 0) return EQMP_ERR_INVALID_ARG;
  } else {
    if (wt.K != 8) return EQMP_ERR_UNSUPPORTED;
    if (E > 0 && (!wt.R || !wt.M)) return EQMP_ERR_INVALID_ARG;  // nothing is read when E == 0
    if (!aligned(wt.R, 16) || !aligned(wt.M, 4)) return EQMP_ERR_INVALID_ARG;
  }
  if (C != 8 && C != 16 && C != 32 && C != 64 && C != 128) return EQMP_ERR_UNSUPPORTED;
  if (N == 0) return EQMP_OK;
  if (!off || !out || !aligned(out, 16)) return EQMP_ERR_INVALID_ARG;
  if (E > 0) {
    if (!vec_or_Y || !src || !x || N_src < 1) return EQMP_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(vec_or_Y, from_vec ? 4 : 16) || !aligned(src, 4))
      return EQMP_ERR_INVALID_ARG;
  }
  DeviceInfo dev;
  eqmp_status s = device_info(&dev);
  if (s != EQMP_OK) return s;
  LayerArgs a{};
  a.vec = from_vec ? vec_or_Y : nullptr;
  a.Y = from_vec ? nullptr : vec_or_Y;
  a.x = x;
  a.off = off;
  a.src = src;
  a.w = wt.w;
  a.R = wt.R;
  a.M = wt.M;
  a.out = out;
  a.watchdog = dev.watchdog;
  a.N = (int)N;
  a.E = (int)E;
  a.N_src = (int)N_src;
  const bool bf16 = x_dtype == EQMP_BF16;
  if (!shared) {
    // Per-edge weights: the fused layer takes the aligned-frame schedule
    // (k_so2: same result, about half the FMAs and twice as fast here);
    // with the harmonics read from memory only the dense kernel applies.
    if (from_vec)
      return eqmp_fused_so2(vec_or_Y, x, N_src, x_dtype, off, src, N, E, C, wt, out, out_dtype,
                            reinterpret_cast<eqmp_stream_t>(st));
    return bf16 ? launch_radial_bf16(a, C, from_vec, st, dev) : launch_radial_f32(a, C, from_vec, st, dev);
  }
  CUtensorMap map;
  if (E > 0) {
    s = encode_x_map(x, N_src, C, bf16, &map);
    if (s != EQMP_OK) return s;
  } else {
    memset(&map, 0, sizeof(map));  // never dereferenced: no edge, no load
  }
  return bf16 ? launch_shared_bf16(a, C, from_vec, map, st, dev)
              : launch_shared_f32(a, C, from_vec, map, st, dev);
}

}  // namespace eqmp

using namespace eqmp;

extern "C" {

int32_t eqmp_num_paths(void) { return tables::kNumPaths; }

eqmp_status eqmp_path_table(int32_t* l1l2l3) {
  if (!l1l2l3) return EQMP_ERR_INVALID_ARG;
  for (int p = 0; p < tables::kNumPaths; ++p) {
    l1l2l3[3 * p + 0] = tables::kPaths[p].l1;
    l1l2l3[3 * p + 1] = tables::kPaths[p].l2;
    l1l2l3[3 * p + 2] = tables::kPaths[p].l3;
  }
  return EQMP_OK;
}

const char* eqmp_status_string(eqmp_status s) {
  switch (s) {
    case EQMP_OK: return "ok";
    case EQMP_ERR_INVALID_ARG: return "invalid argument";
    case EQMP_ERR_UNSUPPORTED: return "unsupported configuration";
    case EQMP_ERR_CUDA: return "CUDA error";
    case EQMP_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case EQMP_ERR_GRAPH: return "graph precondition violated";
  }
  return "unknown status";
}

eqmp_status eqmp_sh(const float* vec, int64_t E, float* Y, eqmp_stream_t stream) {
  if (E < 0 || E > INT32_MAX) return EQMP_ERR_INVALID_ARG;
  if (E == 0) return EQMP_OK;
  if (!vec || !Y || !aligned(vec, 4) || !aligned(Y, 16)) return EQMP_ERR_INVALID_ARG;
  const int grid = (int)((E + kShThreads - 1) / kShThreads);
  k_sh<<<grid, kShThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(vec, (int)E, Y);
  return cuda_status(cudaGetLastError());
}

eqmp_status eqmp_tp_scatter(const float* Y, const void* x, int64_t N_src, eqmp_dtype x_dtype,
                            const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E,
                            int32_t C, eqmp_weights weights, void* out, eqmp_dtype out_dtype,
                            eqmp_stream_t stream) {
  return run_layer(false, Y, x, N_src, x_dtype, row_offsets, src, N, E, C, weights, out, out_dtype,
                   reinterpret_cast<cudaStream_t>(stream));
}

eqmp_status eqmp_fused(const float* vec, const void* x, int64_t N_src, eqmp_dtype x_dtype,
                       const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E,
                       int32_t C, eqmp_weights weights, void* out, eqmp_dtype out_dtype,
                       eqmp_stream_t stream) {
  return run_layer(true, vec, x, N_src, x_dtype, row_offsets, src, N, E, C, weights, out, out_dtype,
                   reinterpret_cast<cudaStream_t>(stream));
}

eqmp_status eqmp_fused_staged(const void* h_in, void* d_in, size_t in_bytes, const float* vec,
                              const void* x, int64_t N_src, eqmp_dtype x_dtype,
                              const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E,
                              int32_t C, eqmp_weights weights, void* out, eqmp_dtype out_dtype,
                              void* h_out, size_t out_bytes, eqmp_stream_t stream) {
  if ((in_bytes > 0 && (!h_in || !d_in)) || (out_bytes > 0 && (!h_out || !out))) return EQMP_ERR_INVALID_ARG;
  if (N < 0 || C <= 0 || (out_dtype != EQMP_F32 && out_dtype != EQMP_BF16)) return EQMP_ERR_INVALID_ARG;
  const size_t out_size = (size_t)N * (size_t)C * 16 * (out_dtype == EQMP_BF16 ? 2 : 4);
  if (out_bytes > out_size) return EQMP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (in_bytes > 0 && cudaMemcpyAsync(d_in, h_in, in_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return EQMP_ERR_CUDA;
  const eqmp_status s = run_layer(true, vec, x, N_src, x_dtype, row_offsets, src, N, E, C, weights, out,
                                  out_dtype, st);
  if (s != EQMP_OK) return s;
  if (out_bytes > 0 && cudaMemcpyAsync(h_out, out, out_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return EQMP_ERR_CUDA;
  return EQMP_OK;
}

struct eqmp_plan_st {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

eqmp_status eqmp_plan_staged(const void* h_in, void* d_in, size_t in_bytes, const float* vec, const void* x,
                             int64_t N_src, eqmp_dtype x_dtype, const int32_t* row_offsets, const int32_t* src,
                             int64_t N, int64_t E, int32_t C, eqmp_weights weights, void* out,
                             eqmp_dtype out_dtype, void* h_out, size_t out_bytes, eqmp_plan* plan) {
  if (!plan) return EQMP_ERR_INVALID_ARG;
  *plan = nullptr;
  // per-device state first: nothing below may allocate while capturing
  DeviceInfo dev;
  eqmp_status s = device_info(&dev);
  if (s != EQMP_OK) return s;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return EQMP_ERR_CUDA;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return EQMP_ERR_CUDA;
  }
  s = eqmp_fused_staged(h_in, d_in, in_bytes, vec, x, N_src, x_dtype, row_offsets, src, N, E, C, weights, out,
                        out_dtype, h_out, out_bytes, reinterpret_cast<eqmp_stream_t>(cs));
  cudaGraph_t g = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(cs, &g);  // ends the capture whatever happened inside
  cudaStreamDestroy(cs);
  if (s != EQMP_OK || ce != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();  // clear the error a failed capture reports, so the next call does not see it
    return s != EQMP_OK ? s : EQMP_ERR_CUDA;
  }
  cudaGraphExec_t ex = nullptr;
  if (cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return EQMP_ERR_CUDA;
  }
  *plan = new eqmp_plan_st{g, ex};
  return EQMP_OK;
}

eqmp_status eqmp_plan_launch(eqmp_plan plan, eqmp_stream_t stream) {
  if (!plan) return EQMP_ERR_INVALID_ARG;
  return cuda_status(cudaGraphLaunch(plan->exec, reinterpret_cast<cudaStream_t>(stream)));
}

eqmp_status eqmp_plan_destroy(eqmp_plan plan) {
  if (!plan) return EQMP_OK;
  const cudaError_t a = cudaGraphExecDestroy(plan->exec);
  const cudaError_t b = cudaGraphDestroy(plan->graph);
  delete plan;
  return a == cudaSuccess && b == cudaSuccess ? EQMP_OK : EQMP_ERR_CUDA;
}

eqmp_status eqmp_validate_graph(const int32_t* row_offsets, const int32_t* src, int64_t N,
                                int64_t N_src, int64_t E, eqmp_stream_t stream) {
  if (N < 0 || N_src < 0 || E < 0 || N > INT32_MAX - 1 || N_src > INT32_MAX || E > INT32_MAX)
    return EQMP_ERR_INVALID_ARG;
  if (!row_offsets || (E > 0 && !src)) return EQMP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* flag = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&flag), g_validate_word) != cudaSuccess)
    return EQMP_ERR_CUDA;
  if (cudaMemsetAsync(flag, 0, sizeof(int), st) != cudaSuccess) return EQMP_ERR_CUDA;
  k_validate<<<64, 256, 0, st>>>(row_offsets, src, (int)N, (int)N_src, (int)E, flag);
  if (cudaGetLastError() != cudaSuccess) return EQMP_ERR_CUDA;
  int h = 0;
  if (cudaMemcpyAsync(&h, flag, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return EQMP_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return EQMP_ERR_CUDA;
  return h ? EQMP_ERR_GRAPH : EQMP_OK;
}

eqmp_status eqmp_watchdog_selftest(int32_t wait_ms, eqmp_stream_t stream) {
  if (wait_ms < 1 || wait_ms > 1000) return EQMP_ERR_INVALID_ARG;
  DeviceInfo dev;
  eqmp_status s = device_info(&dev);
  if (s != EQMP_OK) return s;
  k_wait_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      (unsigned long long)wait_ms * 1000000ull, dev.watchdog);
  return cuda_status(cudaGetLastError());
}

eqmp_status eqmp_fp32_peak_probe(int32_t iters, int32_t blocks_per_sm, float* out, double* flops,
                                 eqmp_stream_t stream) {
  if (!out || !flops || iters < 1 || blocks_per_sm < 1 || blocks_per_sm > 8) return EQMP_ERR_INVALID_ARG;
  DeviceInfo dev;
  eqmp_status s = device_info(&dev);
  if (s != EQMP_OK) return s;
  const int grid = dev.sms * blocks_per_sm;
  *flops = (double)grid * 256.0 * 32.0 * (double)iters;
  k_fp32_peak<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(iters, out);
  return cuda_status(cudaGetLastError());
}

eqmp_status eqmp_device_error(int32_t* code) {
  if (!code) return EQMP_ERR_INVALID_ARG;
  DeviceInfo dev;
  eqmp_status s = device_info(&dev);
  if (s != EQMP_OK) return s;
  int h = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return EQMP_ERR_CUDA;
  if (cudaMemcpy(&h, dev.watchdog, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return EQMP_ERR_CUDA;
  if (h != 0 && cudaMemset(dev.watchdog, 0, sizeof(int)) != cudaSuccess) return EQMP_ERR_CUDA;
  *code = h;
  return h ? EQMP_ERR_DEVICE_TIMEOUT : EQMP_OK;
}

}  // extern "C"
