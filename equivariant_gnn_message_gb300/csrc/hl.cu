// The fused layer at degrees 4..6 (l_max = 4, 5, 6), aligned-frame schedule.
//
// The Batmobile blog stops at l <= 3 (section on limits and future work:
// higher degrees).  At degree L the dense CG product has O(L^6) terms; in the
// frame whose z axis is the edge the edge harmonics keep only m = 0
// (E2Former-V2, Lemma 4.1) and each output order takes one input order
// (Eq. 13), so the product becomes O(L^3) terms between two rotations:
//   x'_l = D_l^T x_l,   m'[k3] = sum_p W_p kappa_p x'[k1],   out_l += D_l m'_l,
// kappa_p[m3, m1] = C_p[m3, m1, 0] sqrt((2 l2 + 1) / 4 pi) (tables generated
// at build time from this library's real CG coefficients).
//
// Organisation: 128 threads per CTA in groups of C threads (thread =
// channel); a CTA owns one receiver at a time.  For each batch of its edges,
// one thread per edge builds the real Wigner-D blocks D_1..D_L of the edge
// frame in shared memory (frame by Duff et al. 2017; levels 2..L by the
// Ivanic-Ruedenberg recursion with compile-time coefficients, so the threads
// never diverge).  The groups then take the batch's edges: the sender row is
// staged in shared memory with coalesced loads, every thread rotates its
// channel in, applies the aligned terms with its path weights, and rotates
// back into its partial accumulators; the partials are added in group order
// at the end.  Deterministic (fixed order everywhere), no atomics.
// Zero-length edges (r^2 < 1e-30) take Y = (Y00, 0, ...): only the paths
// (l, 0, l) contribute, as W_p Y00 x_l.
#include <stdint.h>
#include <string.h>

#include <utility>

#include "common.cuh"
#include "eqmp_tables_hl.h"
#include "launch.h"

namespace eqmp {
namespace {

using tables_hl::Hl;

constexpr int kHlThreads = 128;
constexpr int kBatch = 16;  // edges whose Wigner blocks are built at once

struct HlArgs {
  const float* vec;
  const float* x;
  const int32_t* off;
  const int32_t* src;
  const float* w;
  const float* R;
  const float* M;
  float* out;
  int N, E, N_src, C;
};

template <int L>
struct HlCfg {
  static constexpr int NC = (L + 1) * (L + 1);
  static constexpr int P = Hl<L>::kNumPaths;
  // D_l rows padded to whole float4s
  static constexpr int stride(int l) { return (2 * l + 1 + 3) / 4 * 4; }
  static constexpr int off(int l) {
    int o = 0;
    for (int j = 1; j < l; ++j) o += (2 * j + 1) * stride(j);
    return o;
  }
  // Floats per edge slot (D_1..D_L): a multiple of 4 (rows are read as
  // float4s) that is 4 more than a multiple of 32, so the builders of a batch
  // (thread j writes slot j) spread over the banks (2-way, not 16-way).
  static constexpr int DS = (off(L + 1) + 31) / 32 * 32 + 4;
  static constexpr int XV = (NC + 3) / 4;                  // float4s of a staged row per thread
  // floats: a batch of kBatch edge slots (+ zero-length flags), the
  // accumulators of every thread [NC][128], the staged sender rows
  // [G][C][NC] (= [128][NC]), then the weights: shared [P][C], or the
  // current edge's radial weights of every thread [P][128]
  static constexpr int off_flag() { return kBatch * DS; }
  static constexpr int off_acc() { return off_flag() + kBatch; }
  static constexpr int off_x() { return off_acc() + NC * kHlThreads; }
  static constexpr int off_w() { return off_x() + NC * kHlThreads; }
  static constexpr int smem(int C, bool radial) { return (off_w() + (radial ? P * kHlThreads : P * C)) * 4; }
};

__device__ __forceinline__ void group_sync(int C, int g) {
  if (C <= 32) {
    const unsigned lane_base = (threadIdx.x & 31u) / (unsigned)C * (unsigned)C;
    const unsigned mask = C == 32 ? 0xffffffffu : (((1u << C) - 1u) << lane_base);
    __syncwarp(mask);
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(C) : "memory");
  }
}

// ---- Wigner-D of one edge, computed by one thread -----------------------
// Ivanic-Ruedenberg basis (real SH without the Condon-Shortley sign, l = 1
// block = the frame rotation in (y, z, x) order).  Level l entry (M, N) from
// level l-1 (Dp, padded rows) and R, with compile-time coefficients: no
// branches on the data, so the threads of a warp, each on its own edge,
// never diverge.
template <int L>
constexpr float hl_u(int l, int m, int n) { return tables_hl::kHlIrU[l - 2][m + 6][n + 6]; }
template <int L>
constexpr float hl_v(int l, int m, int n) { return tables_hl::kHlIrV[l - 2][m + 6][n + 6]; }
template <int L>
constexpr float hl_w(int l, int m, int n) { return tables_hl::kHlIrW[l - 2][m + 6][n + 6]; }

template <int LL, int l, int I, int A, int B>
__device__ __forceinline__ float hl_P(const float (&R)[3][3], const float* Dp) {
  constexpr int sp = HlCfg<LL>::stride(l - 1);
  auto dp = [&](int a, int b) { return Dp[(a + l - 1) * sp + (b + l - 1)]; };
  if constexpr (B == l) {
    return R[I + 1][2] * dp(A, l - 1) - R[I + 1][0] * dp(A, -l + 1);
  } else if constexpr (B == -l) {
    return R[I + 1][2] * dp(A, -l + 1) + R[I + 1][0] * dp(A, l - 1);
  } else {
    return R[I + 1][1] * dp(A, B);
  }
}

template <int LL, int l, int M, int N>
__device__ __forceinline__ float hl_entry(const float (&R)[3][3], const float* Dp) {
  constexpr float u = hl_u<LL>(l, M, N), v = hl_v<LL>(l, M, N), w = hl_w<LL>(l, M, N);
  float val = 0.0f;
  if constexpr (u != 0.0f) val = u * hl_P<LL, l, 0, M, N>(R, Dp);
  if constexpr (v != 0.0f) {
    float V;
    if constexpr (M == 0) {
      V = hl_P<LL, l, 1, 1, N>(R, Dp) + hl_P<LL, l, -1, -1, N>(R, Dp);
    } else if constexpr (M == 1) {
      V = hl_P<LL, l, 1, 0, N>(R, Dp) * 1.41421356237309515f;
    } else if constexpr (M > 1) {
      V = hl_P<LL, l, 1, M - 1, N>(R, Dp) - hl_P<LL, l, -1, -M + 1, N>(R, Dp);
    } else if constexpr (M == -1) {
      V = hl_P<LL, l, -1, 0, N>(R, Dp) * 1.41421356237309515f;
    } else {
      V = hl_P<LL, l, 1, M + 1, N>(R, Dp) + hl_P<LL, l, -1, -M - 1, N>(R, Dp);
    }
    val = fmaf(v, V, val);
  }
  if constexpr (w != 0.0f) {
    float Wt;
    if constexpr (M > 0)
      Wt = hl_P<LL, l, 1, M + 1, N>(R, Dp) + hl_P<LL, l, -1, -M - 1, N>(R, Dp);
    else
      Wt = hl_P<LL, l, 1, M - 1, N>(R, Dp) - hl_P<LL, l, -1, -M + 1, N>(R, Dp);
    val = fmaf(w, Wt, val);
  }
  return val;
}

template <int LL, int l, int... Is>
__device__ __forceinline__ void hl_level(const float (&R)[3][3], float* D, std::integer_sequence<int, Is...>) {
  constexpr int W = 2 * l + 1, st = HlCfg<LL>::stride(l), base = HlCfg<LL>::off(l), pbase = HlCfg<LL>::off(l - 1);
  ((D[base + (Is / W) * st + Is % W] = hl_entry<LL, l, Is / W - l, Is % W - l>(R, D + pbase)), ...);
}

template <int LL, int... ls>
__device__ __forceinline__ void hl_levels(const float (&R)[3][3], float* D, std::integer_sequence<int, ls...>) {
  (hl_level<LL, ls + 2>(R, D, std::make_integer_sequence<int, (2 * (ls + 2) + 1) * (2 * (ls + 2) + 1)>{}), ...);
}

// Frame of unit direction (x, y, z) and D_1..D_L into one edge slot.
template <int L>
__device__ __forceinline__ void hl_wigner(float x, float y, float z, float* D) {
  const float sg = z >= 0.0f ? 1.0f : -1.0f;
  const float ia = -1.0f / (sg + z);
  const float b = x * y * ia;
  const float Q[3][3] = {{fmaf(sg * x * x, ia, 1.0f), b, x}, {sg * b, fmaf(y * y, ia, sg), y}, {-sg * x, -y, z}};
  const float R[3][3] = {{Q[1][1], Q[1][2], Q[1][0]}, {Q[2][1], Q[2][2], Q[2][0]}, {Q[0][1], Q[0][2], Q[0][0]}};
#pragma unroll
  for (int i = 0; i < 3; ++i)
#pragma unroll
    for (int j = 0; j < 3; ++j) D[HlCfg<L>::off(1) + i * HlCfg<L>::stride(1) + j] = R[i][j];
  hl_levels<L>(R, D, std::make_integer_sequence<int, L - 1>{});
}

constexpr float sgn_m(int m) { return (m & 1) ? -1.0f : 1.0f; }  // (-1)^|m|

// x'_l[n] = sum_m D_l[m][n] x_l[m], this library's basis (signs s_m s_n on
// the recursion's entries); x_l read from global memory as needed.
// Row m of level l (padded to whole float4s) from shared memory.
template <int L, int l>
__device__ __forceinline__ void load_row(const float* D, int m, float (&row)[HlCfg<L>::stride(l)]) {
  constexpr int st = HlCfg<L>::stride(l), base = HlCfg<L>::off(l);
  const float4* p = reinterpret_cast<const float4*>(D + base + m * st);
#pragma unroll
  for (int h = 0; h < st / 4; ++h) {
    const float4 v = p[h];
    row[4 * h] = v.x; row[4 * h + 1] = v.y; row[4 * h + 2] = v.z; row[4 * h + 3] = v.w;
  }
}

template <int L, int l>
__device__ __forceinline__ void rotate_in(const float* D, const float* xrow, float (&xr)[HlCfg<L>::NC]) {
  constexpr int W = 2 * l + 1, o = l * l;
#pragma unroll
  for (int n = 0; n < W; ++n) xr[o + n] = 0.0f;
#pragma unroll
  for (int m = 0; m < W; ++m) {
    const float xm = xrow[o + m];
    float row[HlCfg<L>::stride(l)];
    load_row<L, l>(D, m, row);
#pragma unroll
    for (int n = 0; n < W; ++n) xr[o + n] = fmaf(sgn_m(m - l) * sgn_m(n - l) * row[n], xm, xr[o + n]);
  }
}

// acc_l3[m] += sum_n D_l3[m][n] m'_l3[n] for one output block (mp indexed
// from 0).  The receiver accumulators live in shared memory, component k of
// this thread at acc[k * C] (the group's C threads side by side).
template <int L, int l>
__device__ __forceinline__ void rotate_out(const float* D, const float (&mp)[2 * L + 1], float* acc, int C) {
  constexpr int W = 2 * l + 1, o = l * l;
#pragma unroll
  for (int m = 0; m < W; ++m) {
    float row[HlCfg<L>::stride(l)];
    load_row<L, l>(D, m, row);
    float s = acc[(o + m) * C];
#pragma unroll
    for (int n = 0; n < W; ++n) s = fmaf(sgn_m(m - l) * sgn_m(n - l) * row[n], mp[n], s);
    acc[(o + m) * C] = s;
  }
}

template <int L, int... ls>
__device__ __forceinline__ void rotate_in_all(const float* D, const float* xrow, float (&xr)[HlCfg<L>::NC],
                                              std::integer_sequence<int, ls...>) {
  (rotate_in<L, ls + 1>(D, xrow, xr), ...);
}
// Weight of path p for this thread's channel: shared weights staged in
// shared memory (ws[p * C + c]); radial weights of the current edge, formed
// per thread at the start of the edge (ws[p * 128 + thread]).
template <int L, bool RADIAL>
__device__ __forceinline__ float path_weight(const HlArgs& a, const float* ws, int p, int c, const float (&rad)[8]) {
  if constexpr (RADIAL) {
    return ws[p * kHlThreads + threadIdx.x];
  } else {
    return ws[p * a.C + c];
  }
}

// Terms of one path into the output block of its l3 (mp indexed from l3^2).
template <int L, int First, int O, int... Is>
__device__ __forceinline__ void path_terms(float wp, const float (&xr)[HlCfg<L>::NC], float (&mp)[2 * L + 1],
                                           std::integer_sequence<int, Is...>) {
  ((mp[Hl<L>::kTerms[First + Is].k3 - O] = fmaf(wp * Hl<L>::kTerms[First + Is].kappa,
                                                xr[Hl<L>::kTerms[First + Is].k1],
                                                mp[Hl<L>::kTerms[First + Is].k3 - O])),
   ...);
}

// Output block l3: the aligned terms of every path ending in l3, each with
// its weight, then the rotation back into the accumulators.  Working one
// output block at a time keeps only 2 l3 + 1 partial outputs live.
template <int L, bool RADIAL, int L3, int p>
__device__ __forceinline__ void block_path(const HlArgs& a, const float* ws, int c, const float (&rad)[8],
                                           const float (&xr)[HlCfg<L>::NC], float (&mp)[2 * L + 1]) {
  constexpr tables_hl::HlPath path = Hl<L>::kPaths[p];
  if constexpr (path.l3 == L3 && path.count > 0)
    path_terms<L, path.first, L3 * L3>(path_weight<L, RADIAL>(a, ws, p, c, rad), xr, mp,
                                       std::make_integer_sequence<int, path.count>{});
}

template <int L, bool RADIAL, int L3, int... Ps>
__device__ __forceinline__ void out_block(const HlArgs& a, const float* ws, int c, const float (&rad)[8],
                                          const float* D, const float (&xr)[HlCfg<L>::NC], float* acc,
                                          std::integer_sequence<int, Ps...>) {
  float mp[2 * L + 1];
#pragma unroll
  for (int k = 0; k < 2 * L + 1; ++k) mp[k] = 0.0f;
  (block_path<L, RADIAL, L3, Ps>(a, ws, c, rad, xr, mp), ...);
  if constexpr (L3 == 0) {
    acc[0] += mp[0];
  } else {
    rotate_out<L, L3>(D, mp, acc, a.C);
  }
}

template <int L, bool RADIAL, int... L3s>
__device__ __forceinline__ void all_blocks(const HlArgs& a, const float* ws, int c, const float (&rad)[8],
                                           const float* D, const float (&xr)[HlCfg<L>::NC], float* acc,
                                           std::integer_sequence<int, L3s...>) {
  (out_block<L, RADIAL, L3s>(a, ws, c, rad, D, xr, acc, std::make_integer_sequence<int, HlCfg<L>::P>{}), ...);
}

// Zero-length edge: out_l += W_(l,0,l) Y00 x_l.
template <int L, bool RADIAL, int p>
__device__ __forceinline__ void zero_len_path(const HlArgs& a, const float* ws, int c, const float (&rad)[8],
                                              const float* xrow, float* acc) {
  constexpr float y00 = 0.28209479177387814f;
  constexpr tables_hl::HlPath path = Hl<L>::kPaths[p];
  if constexpr (path.l2 == 0) {
    const float wy = path_weight<L, RADIAL>(a, ws, p, c, rad) * y00;
#pragma unroll
    for (int k = path.l1 * path.l1; k < (path.l1 + 1) * (path.l1 + 1); ++k)
      acc[k * a.C] = fmaf(wy, xrow[k], acc[k * a.C]);
  }
}

template <int L, bool RADIAL, int... Ps>
__device__ __forceinline__ void zero_len_terms(const HlArgs& a, const float* ws, int c, const float (&rad)[8],
                                               const float* xrow, float* acc, std::integer_sequence<int, Ps...>) {
  (zero_len_path<L, RADIAL, Ps>(a, ws, c, rad, xrow, acc), ...);
}

template <int L, bool RADIAL>
__global__ void __launch_bounds__(kHlThreads) k_hl(const HlArgs a) {
  using K = HlCfg<L>;
  constexpr int NC = K::NC;
  extern __shared__ float hsm[];
  const int C = a.C, G = kHlThreads / C;
  const int t = threadIdx.x, g = t / C, c = t % C;
  float* slots = hsm;                      // [kBatch][DS]
  float* flags = hsm + K::off_flag();      // [kBatch]: 1 for a zero-length edge
  float* accs = hsm + K::off_acc();        // partial accumulators [G][NC][C]
  float* acc = accs + (size_t)g * NC * C + c;
  float* xs = hsm + K::off_x() + (size_t)g * C * NC;  // the group's staged sender row [C][NC]
  float* ws = hsm + K::off_w();
  if constexpr (!RADIAL) {
    for (int i = t; i < K::P * C; i += kHlThreads) ws[i] = __ldg(a.w + i);
    __syncthreads();
  }
  // One receiver per CTA at a time.  Its edges go in batches of kBatch:
  // thread j builds the Wigner blocks of edge j of the batch (one edge per
  // thread, no divergence), then the G groups take the batch's edges
  // g, g + G, ... and add them into their partial sums, which are summed in
  // group order at the end: deterministic.
  for (long long r = blockIdx.x; r < a.N; r += gridDim.x) {
    const int e0 = min(max(__ldg(a.off + r), 0), a.E);
    const int e1 = max(e0, min(max(__ldg(a.off + r + 1), 0), a.E));
#pragma unroll
    for (int k = 0; k < NC; ++k) acc[k * C] = 0.0f;
    for (int b0 = e0; b0 < e1; b0 += kBatch) {
      const int nb = min(kBatch, e1 - b0);
      __syncthreads();  // the previous batch's slots are no longer read
      if (t < nb) {
        const int e = b0 + t;
        const float vx = __ldg(a.vec + 3 * (size_t)e), vy = __ldg(a.vec + 3 * (size_t)e + 1),
                    vz = __ldg(a.vec + 3 * (size_t)e + 2);
        const float r2 = fmaf(vx, vx, fmaf(vy, vy, vz * vz));
        if (r2 >= 1e-30f) {
          const float inv = rsqrtf(r2);
          hl_wigner<L>(vx * inv, vy * inv, vz * inv, slots + (size_t)t * K::DS);
          flags[t] = 0.0f;
        } else {
          flags[t] = 1.0f;  // zero length: Y = (Y00, 0, ...)
        }
      }
      __syncthreads();
      for (int j = g; j < nb; j += G) {
        const int e = b0 + j;
        const float* D = slots + (size_t)j * K::DS;
        const bool zero = flags[j] != 0.0f;
        float rad[8];
        if constexpr (RADIAL) {
          const float4* rp = reinterpret_cast<const float4*>(a.R) + 2 * (size_t)e;
          const float4 r0 = __ldg(rp), r1 = __ldg(rp + 1);
          rad[0] = r0.x; rad[1] = r0.y; rad[2] = r0.z; rad[3] = r0.w;
          rad[4] = r1.x; rad[5] = r1.y; rad[6] = r1.z; rad[7] = r1.w;
          // W[p] = sum_k R[e,k] M[k, p C + c] for every path, into this
          // thread's column (read only by this thread); eight paths at a time
          const float* mc = a.M + c;
          const size_t pc = (size_t)K::P * C;
#pragma unroll 1
          for (int p0 = 0; p0 < K::P; p0 += 8) {
            float m[8][8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
#pragma unroll
              for (int k = 0; k < 8; ++k)
                m[q][k] = p0 + q < K::P ? __ldg(mc + k * pc + (size_t)(p0 + q) * C) : 0.0f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float w = 0.0f;
#pragma unroll
              for (int k = 0; k < 8; ++k) w = fmaf(rad[k], m[q][k], w);
              if (p0 + q < K::P) ws[(p0 + q) * kHlThreads + t] = w;
            }
          }
        }
        const int s = __ldg(a.src + e);
        const bool in_range = (unsigned)s < (unsigned)a.N_src;  // an out-of-range sender adds nothing
        // stage the sender's row (C * NC floats, contiguous) with coalesced float4s
        {
          const float4* src4 = reinterpret_cast<const float4*>(a.x + (size_t)(in_range ? s : 0) * C * NC);
          float4* xs4 = reinterpret_cast<float4*>(xs);
          const int n4 = C * NC / 4;
#pragma unroll
          for (int v = 0; v < K::XV; ++v) {
            const int i = c + v * C;
            if (i < n4) xs4[i] = __ldg(src4 + i);
          }
        }
        group_sync(C, g);
        if (in_range) {
          const float* xrs = xs + c * NC;
          if (!zero) {
            float xr[NC];
            xr[0] = xrs[0];
            rotate_in_all<L>(D, xrs, xr, std::make_integer_sequence<int, L>{});
            all_blocks<L, RADIAL>(a, ws, c, rad, D, xr, acc, std::make_integer_sequence<int, L + 1>{});
          } else {
            zero_len_terms<L, RADIAL>(a, ws, c, rad, xrs, acc, std::make_integer_sequence<int, K::P>{});
          }
        }
        group_sync(C, g);  // the staged row (and radial weights) are rewritten next
      }
    }
    __syncthreads();
    // out[r][c][k] = sum over groups in order; thread (g, c) takes k = g, g + G, ...
    float* orow = a.out + ((size_t)r * C + c) * NC;
    for (int k = g; k < NC; k += G) {
      float v = 0.0f;
      for (int h = 0; h < G; ++h) v += accs[((size_t)h * NC + k) * C + c];
      orow[k] = v;
    }
    __syncthreads();  // the partials are zeroed for the next receiver
  }
}

template <int L, bool RADIAL>
eqmp_status launch_hl(const HlArgs& a, cudaStream_t st, const DeviceInfo& dev) {
  auto kern = k_hl<L, RADIAL>;
  const int smem = HlCfg<L>::smem(a.C, RADIAL);
  static unsigned long long attr_done = 0;
  if (ensure_smem_attr(kern, 227 * 1024, &attr_done) != cudaSuccess) return EQMP_ERR_CUDA;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kHlThreads, smem) != cudaSuccess || occ < 1)
    return EQMP_ERR_CUDA;
  const long long want = a.N;  // one receiver per CTA at a time
  const long long cap = (long long)dev.sms * occ;
  const int grid = (int)(want < cap ? want : cap);
  if (grid <= 0) return EQMP_OK;
  kern<<<grid, kHlThreads, smem, st>>>(a);
  return cuda_status(cudaGetLastError());
}

int num_paths(int l_max) {
  switch (l_max) {
    case 4: return Hl<4>::kNumPaths;
    case 5: return Hl<5>::kNumPaths;
    case 6: return Hl<6>::kNumPaths;
  }
  return -1;
}

}  // namespace
}  // namespace eqmp

using namespace eqmp;

extern "C" {

int32_t eqmp_num_paths_lmax(int32_t l_max) {
  if (l_max == 3) return eqmp_num_paths();
  return num_paths(l_max);
}

eqmp_status eqmp_fused_lmax(int32_t l_max, const float* vec, const float* x, int64_t N_src,
                            const int32_t* row_offsets, const int32_t* src, int64_t N, int64_t E, int32_t C,
                            eqmp_weights weights, float* out, eqmp_stream_t stream) {
  if (l_max < 4 || l_max > 6) return EQMP_ERR_UNSUPPORTED;
  if (N < 0 || E < 0 || N_src < 0 || N > INT32_MAX - 1 || E > INT32_MAX || N_src > INT32_MAX)
    return EQMP_ERR_INVALID_ARG;
  if (C != 8 && C != 16 && C != 32 && C != 64 && C != 128) return EQMP_ERR_UNSUPPORTED;
  const bool radial = weights.w == nullptr;
  if (!radial && (weights.R || weights.M || weights.K != 0)) return EQMP_ERR_INVALID_ARG;
  if (radial && weights.K != 8) return EQMP_ERR_UNSUPPORTED;
  if (radial && E > 0 && (!weights.R || !weights.M || (reinterpret_cast<uintptr_t>(weights.R) & 15)))
    return EQMP_ERR_INVALID_ARG;
  if (N == 0) return EQMP_OK;
  if (!row_offsets || !out) return EQMP_ERR_INVALID_ARG;
  if (E > 0 && (!vec || !src || !x || N_src < 1)) return EQMP_ERR_INVALID_ARG;
  DeviceInfo dev;
  eqmp_status s = device_info(&dev);
  if (s != EQMP_OK) return s;
  HlArgs a{};
  a.vec = vec; a.x = x; a.off = row_offsets; a.src = src;
  a.w = weights.w; a.R = weights.R; a.M = weights.M; a.out = out;
  a.N = (int)N; a.E = (int)E; a.N_src = (int)N_src; a.C = C;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  switch (l_max) {
    case 4: return radial ? launch_hl<4, true>(a, st, dev) : launch_hl<4, false>(a, st, dev);
    case 5: return radial ? launch_hl<5, true>(a, st, dev) : launch_hl<5, false>(a, st, dev);
    default: return radial ? launch_hl<6, true>(a, st, dev) : launch_hl<6, false>(a, st, dev);
  }
}

}  // extern "C"
