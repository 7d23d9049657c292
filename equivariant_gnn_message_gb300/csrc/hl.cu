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
// channel); a CTA owns one receiver at a time and deals its edges to its
// groups, whose partial sums it adds in group order at the end.  Per edge
// the group builds the real Wigner-D blocks D_1..D_L of the
// edge frame in shared memory (frame by Duff et al. 2017; levels 2..L by the
// Ivanic-Ruedenberg recursion, the entries of a level spread over the
// group's threads), then every thread rotates its channel in, applies the
// aligned terms with its path weights, and rotates back into its receiver
// accumulators.  D is double-buffered so one group barrier per level is the
// only synchronisation.  Deterministic (fixed order everywhere), no atomics.
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
  static constexpr int DS = (off(L + 1) + 31) / 32 * 32;  // floats per D set
  // D double buffers of every group + accumulators of every thread
  static constexpr int smem(int C) { return ((kHlThreads / C) * 2 * DS + NC * kHlThreads) * 4; }
  static constexpr int SMEM = smem(8);  // largest: 16 groups of 8
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

// One entry (m, n) of level l in the Ivanic-Ruedenberg basis (real SH
// without the Condon-Shortley sign, l = 1 block in (y, z, x) order).  R is
// the stored l = 1 block (row stride 4), Dp level l-1 with row stride sp.
__device__ __forceinline__ float ir_entry(int l, int m, int n, const float* R, const float* Dp, int sp) {
  const float* cf = &tables_hl::kHlIr[l - 2][m + 6][n + 6][0];
  const float u = __ldg(cf), v = __ldg(cf + 1), w = __ldg(cf + 2);
  auto dp = [&](int a, int b) { return Dp[(a + l - 1) * sp + (b + l - 1)]; };
  auto P = [&](const float* Ri, int a, int b) {  // Ri = row i + 1 of R
    if (b == l) return Ri[2] * dp(a, l - 1) - Ri[0] * dp(a, -l + 1);
    if (b == -l) return Ri[2] * dp(a, -l + 1) + Ri[0] * dp(a, l - 1);
    return Ri[1] * dp(a, b);
  };
  const float* Rm = R;
  const float* R0 = R + 4;
  const float* Rp = R + 8;
  float val = 0.0f;
  if (u != 0.0f) val = u * P(R0, m, n);
  if (v != 0.0f) {
    float V;
    if (m == 0) {
      V = P(Rp, 1, n) + P(Rm, -1, n);
    } else if (m > 0) {
      V = m == 1 ? P(Rp, 0, n) * 1.41421356237309515f : P(Rp, m - 1, n) - P(Rm, -m + 1, n);
    } else {
      V = m == -1 ? P(Rm, 0, n) * 1.41421356237309515f : P(Rp, m + 1, n) + P(Rm, -m - 1, n);
    }
    val = fmaf(v, V, val);
  }
  if (w != 0.0f) {
    const float Wt = m > 0 ? P(Rp, m + 1, n) + P(Rm, -m - 1, n) : P(Rp, m - 1, n) - P(Rm, -m + 1, n);
    val = fmaf(w, Wt, val);
  }
  return val;
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
    const float xm = __ldg(xrow + o + m);
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
// Weight of path p for channel c of edge e.
template <int L, bool RADIAL>
__device__ __forceinline__ float path_weight(const HlArgs& a, int p, int c, const float (&rad)[8]) {
  constexpr int P = HlCfg<L>::P;
  if constexpr (RADIAL) {
    // the eight loads of one path together; the empty asm keeps the
    // compiler from hoisting the loads of every path ahead at once
    const float* mp = a.M + (size_t)p * a.C + c;
    const size_t stride = (size_t)P * a.C;
    float m[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = __ldg(mp + k * stride);
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) s = fmaf(rad[k], m[k], s);
    asm volatile("" : "+f"(s));
    return s;
  } else {
    float wv = __ldg(a.w + (size_t)p * a.C + c);
    asm volatile("" : "+f"(wv));  // load as it is needed, not all paths ahead
    return wv;
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
__device__ __forceinline__ void block_path(const HlArgs& a, int c, const float (&rad)[8],
                                           const float (&xr)[HlCfg<L>::NC], float (&mp)[2 * L + 1]) {
  constexpr tables_hl::HlPath path = Hl<L>::kPaths[p];
  if constexpr (path.l3 == L3 && path.count > 0)
    path_terms<L, path.first, L3 * L3>(path_weight<L, RADIAL>(a, p, c, rad), xr, mp,
                                       std::make_integer_sequence<int, path.count>{});
}

template <int L, bool RADIAL, int L3, int... Ps>
__device__ __forceinline__ void out_block(const HlArgs& a, int c, const float (&rad)[8], const float* D,
                                          const float (&xr)[HlCfg<L>::NC], float* acc,
                                          std::integer_sequence<int, Ps...>) {
  float mp[2 * L + 1];
#pragma unroll
  for (int k = 0; k < 2 * L + 1; ++k) mp[k] = 0.0f;
  (block_path<L, RADIAL, L3, Ps>(a, c, rad, xr, mp), ...);
  if constexpr (L3 == 0) {
    acc[0] += mp[0];
  } else {
    rotate_out<L, L3>(D, mp, acc, a.C);
  }
}

template <int L, bool RADIAL, int... L3s>
__device__ __forceinline__ void all_blocks(const HlArgs& a, int c, const float (&rad)[8], const float* D,
                                           const float (&xr)[HlCfg<L>::NC], float* acc,
                                           std::integer_sequence<int, L3s...>) {
  (out_block<L, RADIAL, L3s>(a, c, rad, D, xr, acc, std::make_integer_sequence<int, HlCfg<L>::P>{}), ...);
}

// Zero-length edge: out_l += W_(l,0,l) Y00 x_l.
template <int L, bool RADIAL, int p>
__device__ __forceinline__ void zero_len_path(const HlArgs& a, int c, const float (&rad)[8], const float* xrow,
                                              float* acc) {
  constexpr float y00 = 0.28209479177387814f;
  constexpr tables_hl::HlPath path = Hl<L>::kPaths[p];
  if constexpr (path.l2 == 0) {
    const float wy = path_weight<L, RADIAL>(a, p, c, rad) * y00;
#pragma unroll
    for (int k = path.l1 * path.l1; k < (path.l1 + 1) * (path.l1 + 1); ++k)
      acc[k * a.C] = fmaf(wy, __ldg(xrow + k), acc[k * a.C]);
  }
}

template <int L, bool RADIAL, int... Ps>
__device__ __forceinline__ void zero_len_terms(const HlArgs& a, int c, const float (&rad)[8], const float* xrow,
                                               float* acc, std::integer_sequence<int, Ps...>) {
  (zero_len_path<L, RADIAL, Ps>(a, c, rad, xrow, acc), ...);
}

template <int L, bool RADIAL>
__global__ void __launch_bounds__(kHlThreads) k_hl(const HlArgs a) {
  using K = HlCfg<L>;
  constexpr int NC = K::NC;
  extern __shared__ float hsm[];
  const int C = a.C, G = kHlThreads / C;
  const int t = threadIdx.x, g = t / C, c = t % C;
  float* Dg = hsm + (size_t)g * 2 * K::DS;
  // partial accumulators of each group: [G][NC][C] after the D buffers
  float* accs = hsm + (size_t)G * 2 * K::DS;
  float* acc = accs + (size_t)g * NC * C + c;
  // D buffer of the group's step-th edge is step & 1, counted across
  // receivers, and every step passes at least one group barrier: a buffer is
  // rewritten only after every thread of the group has left the step that
  // last read it.
  unsigned step = 0;
  // One receiver per CTA at a time; its edges are dealt to the G groups
  // (group g takes e0 + g, e0 + g + G, ...), whose partial sums are added
  // in group order at the end: deterministic.
  for (long long r = blockIdx.x; r < a.N; r += gridDim.x) {
    const int e0 = min(max(__ldg(a.off + r), 0), a.E);
    const int e1 = max(e0, min(max(__ldg(a.off + r + 1), 0), a.E));
#pragma unroll
    for (int k = 0; k < NC; ++k) acc[k * C] = 0.0f;
    for (int e = e0 + g; e < e1; e += G, ++step) {
      float* D = Dg + (step & 1u) * K::DS;
      const float vx = __ldg(a.vec + 3 * (size_t)e), vy = __ldg(a.vec + 3 * (size_t)e + 1),
                  vz = __ldg(a.vec + 3 * (size_t)e + 2);
      const float r2 = fmaf(vx, vx, fmaf(vy, vy, vz * vz));
      const bool zero = !(r2 >= 1e-30f);  // group-uniform
      float rad[8];
      if constexpr (RADIAL) {
        const float4* rp = reinterpret_cast<const float4*>(a.R) + 2 * (size_t)e;
        const float4 r0 = __ldg(rp), r1 = __ldg(rp + 1);
        rad[0] = r0.x; rad[1] = r0.y; rad[2] = r0.z; rad[3] = r0.w;
        rad[4] = r1.x; rad[5] = r1.y; rad[6] = r1.z; rad[7] = r1.w;
      }
      const int s = __ldg(a.src + e);
      const bool in_range = (unsigned)s < (unsigned)a.N_src;  // an out-of-range sender adds nothing
      const float* xrow = a.x + ((size_t)(in_range ? s : 0) * C + c) * NC;
      if (!zero) {
        {
          // frame Q (columns t1, t2, n; Duff et al. 2017); level 1 is Q in
          // (y, z, x) order, entry (i, j) = 3 i + j written by thread
          // (3 i + j) mod C
          const float inv = rsqrtf(r2);
          const float x = vx * inv, y = vy * inv, z = vz * inv;
          const float sg = z >= 0.0f ? 1.0f : -1.0f;
          const float ia = -1.0f / (sg + z);
          const float b = x * y * ia;
          const float Q[3][3] = {{fmaf(sg * x * x, ia, 1.0f), b, x},
                                 {sg * b, fmaf(y * y, ia, sg), y},
                                 {-sg * x, -y, z}};
          for (int ij = c; ij < 9; ij += C) {
            const int i = ij / 3, j = ij % 3;
            const int qi = i == 0 ? 1 : i == 1 ? 2 : 0, qj = j == 0 ? 1 : j == 1 ? 2 : 0;
            float q = 0.0f;
#pragma unroll
            for (int u = 0; u < 3; ++u)
#pragma unroll
              for (int v = 0; v < 3; ++v) q = (u == qi && v == qj) ? Q[u][v] : q;
            D[K::off(1) + i * K::stride(1) + j] = q;
          }
        }
        group_sync(C, g);
#pragma unroll 1
        for (int l = 2; l <= L; ++l) {
          const int W = 2 * l + 1, n_ent = W * W;
          const int st = (W + 3) / 4 * 4, stp = (W - 2 + 3) / 4 * 4;
          int base = 0, basep = 0;
          for (int j = 1; j < l; ++j) {
            basep = base;
            base += (2 * j + 1) * ((2 * j + 1 + 3) / 4 * 4);
          }
          for (int i = c; i < n_ent; i += C) {
            const int m = i / W - l, n = i % W - l;
            D[base + (m + l) * st + (n + l)] = ir_entry(l, m, n, D + K::off(1), D + basep, stp);
          }
          group_sync(C, g);
        }
        if (in_range) {
          float xr[NC];
          xr[0] = __ldg(xrow);
          rotate_in_all<L>(D, xrow, xr, std::make_integer_sequence<int, L>{});
          all_blocks<L, RADIAL>(a, c, rad, D, xr, acc, std::make_integer_sequence<int, L + 1>{});
        }
      } else {
        group_sync(C, g);  // keeps one barrier per step (see above)
        if (in_range) zero_len_terms<L, RADIAL>(a, c, rad, xrow, acc, std::make_integer_sequence<int, K::P>{});
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
  const int smem = HlCfg<L>::smem(a.C);
  static unsigned long long attr_done = 0;
  if (ensure_smem_attr(kern, HlCfg<L>::SMEM, &attr_done) != cudaSuccess) return EQMP_ERR_CUDA;
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
