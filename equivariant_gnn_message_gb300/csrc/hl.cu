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
// Organisation (k_hl below): a producer warp builds the real Wigner-D
// blocks D_1..D_L of each edge's frame (frame by Duff et al. 2017; levels
// 2..L by the Ivanic-Ruedenberg recursion with compile-time coefficients, one
// edge per lane, so the lanes never diverge) into an edge ring and
// bulk-copies each sender row into a row ring; 128 consumer threads in
// groups of C (thread = channel) rotate their channel in, apply the aligned
// terms with their path weights, and rotate back into partial accumulators,
// added in group order at each receiver's end.  Deterministic (fixed order
// everywhere), no atomics.
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

constexpr int kHlThreads = 128;  // consumer threads per CTA (plus one producer warp)

struct HlArgs {
  const float* vec;
  const float* x;
  const int32_t* off;
  const int32_t* src;
  const float* w;
  const float* R;
  const float* M;
  float* out;
  int* watchdog;
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
  // float4s) that is 4 more than a multiple of 32, so the producer's lanes
  // (lane j writes slot j) spread their stores over the banks.
  static constexpr int DS = (off(L + 1) + 31) / 32 * 32 + 4;
};


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
// Weight of path p for this thread's channel.  RADIAL = 0: shared weights
// staged in shared memory (ws[p * C + c]).  RADIAL = 1: radial weights of
// the current edge, formed per thread at the start of the edge from M in
// global memory (ws[p * 128 + thread]).  RADIAL = 2: M staged in shared
// memory (ws[(k * P + p) * C + c]) and the weight formed here, 8 FMAs.
template <int L, int RADIAL>
__device__ __forceinline__ float path_weight(const HlArgs& a, const float* ws, int p, int c, const float (&rad)[8]) {
  if constexpr (RADIAL == 2) {
    constexpr int P = HlCfg<L>::P;
    float w = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) w = fmaf(rad[k], ws[(k * P + p) * a.C + c], w);
    return w;
  } else if constexpr (RADIAL == 1) {
    return ws[p * kHlThreads + threadIdx.x];
  } else {
    return ws[p * a.C + c];
  }
}

// Terms of one path into the output block of its l3 (mp indexed from l3^2).
// Terms of a path whose |kappa| is equal (the orders m and -m) share one
// product w |kappa| (about half as many multiplies as terms); the sign goes
// into the FMA.
template <int L>
constexpr float hl_akappa(int i) {
  return Hl<L>::kTerms[i].kappa < 0.0f ? -Hl<L>::kTerms[i].kappa : Hl<L>::kTerms[i].kappa;
}
template <int L, int First, int I>
constexpr int hl_kappa_slot() {
  for (int j = 0; j < I; ++j)
    if (hl_akappa<L>(First + j) == hl_akappa<L>(First + I)) return j;
  return I;
}
template <int L, int First, int O, int I, int NT>
__device__ __forceinline__ void path_term(float wp, float (&wk)[NT], const float (&xr)[HlCfg<L>::NC],
                                          float (&mp)[2 * L + 1]) {
  constexpr tables_hl::HlTerm t = Hl<L>::kTerms[First + I];
  constexpr int sl = hl_kappa_slot<L, First, I>();
  if constexpr (sl == I) wk[I] = wp * hl_akappa<L>(First + I);
  if constexpr (t.kappa < 0.0f) {
    mp[t.k3 - O] = fmaf(-wk[sl], xr[t.k1], mp[t.k3 - O]);
  } else {
    mp[t.k3 - O] = fmaf(wk[sl], xr[t.k1], mp[t.k3 - O]);
  }
}
template <int L, int First, int O, int... Is>
__device__ __forceinline__ void path_terms(float wp, const float (&xr)[HlCfg<L>::NC], float (&mp)[2 * L + 1],
                                           std::integer_sequence<int, Is...>) {
  float wk[sizeof...(Is) > 0 ? sizeof...(Is) : 1];
  (path_term<L, First, O, Is>(wp, wk, xr, mp), ...);
}

// Output block l3: the aligned terms of every path ending in l3, each with
// its weight, then the rotation back into the accumulators.  Working one
// output block at a time keeps only 2 l3 + 1 partial outputs live.
template <int L, int RADIAL, int L3, int p>
__device__ __forceinline__ void block_path(const HlArgs& a, const float* ws, int c, const float (&rad)[8],
                                           const float (&xr)[HlCfg<L>::NC], float (&mp)[2 * L + 1]) {
  constexpr tables_hl::HlPath path = Hl<L>::kPaths[p];
  if constexpr (path.l3 == L3 && path.count > 0)
    path_terms<L, path.first, L3 * L3>(path_weight<L, RADIAL>(a, ws, p, c, rad), xr, mp,
                                       std::make_integer_sequence<int, path.count>{});
}

template <int L, int RADIAL, int L3, int... Ps>
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

template <int L, int RADIAL, int... L3s>
__device__ __forceinline__ void all_blocks(const HlArgs& a, const float* ws, int c, const float (&rad)[8],
                                           const float* D, const float (&xr)[HlCfg<L>::NC], float* acc,
                                           std::integer_sequence<int, L3s...>) {
  (out_block<L, RADIAL, L3s>(a, ws, c, rad, D, xr, acc, std::make_integer_sequence<int, HlCfg<L>::P>{}), ...);
}

// Zero-length edge: out_l += W_(l,0,l) Y00 x_l.
template <int L, int RADIAL, int p>
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

template <int L, int RADIAL, int... Ps>
__device__ __forceinline__ void zero_len_terms(const HlArgs& a, const float* ws, int c, const float (&rad)[8],
                                               const float* xrow, float* acc, std::integer_sequence<int, Ps...>) {
  (zero_len_path<L, RADIAL, Ps>(a, ws, c, rad, xrow, acc), ...);
}

// Shared-memory plan of k_hl for one (L, C, weights): a producer batch of
// PB edges (their Wigner blocks built lane-parallel), an S-slot ring of
// gathered sender rows (S a multiple of the group count 128 / C), and an
// edge ring of YR = PB + S entries (the
// producer writes a batch's entries only after the rows S edges back have
// been released, so PB + S entries never collide).  Offsets in floats.
struct HlPlan {
  int PB, S, YR;
  int o_slot, o_flag, o_rad, o_acc, o_x, o_w, o_bar, bytes;
};

template <int L>
inline HlPlan hl_plan(int C, int radial, int pb, int S) {
  using K = HlCfg<L>;
  HlPlan q{};
  q.PB = pb;
  q.S = S;
  q.YR = pb + S;
  auto up4 = [](int v) { return (v + 3) / 4 * 4; };
  q.o_slot = 0;
  q.o_flag = up4(q.o_slot + q.YR * K::DS);
  q.o_rad = up4(q.o_flag + q.YR);
  q.o_acc = up4(q.o_rad + (radial ? 8 * q.YR : 0));
  q.o_x = up4(q.o_acc + K::NC * kHlThreads);
  q.o_w = up4(q.o_x + S * C * K::NC);
  const int wfloats = radial == 2 ? 8 * K::P * C : radial ? K::P * kHlThreads : K::P * C;
  q.o_bar = up4(q.o_w + wfloats);  // barriers, then the range (int4)
  q.bytes = q.o_bar * 4 + 2 * S * 8 + 16;
  return q;
}

// CTA: NCONS = 128 consumer threads in groups of C (thread = channel) and one
// producer warp.  The CTA owns a contiguous receiver range, balanced on edges
// (balanced_range_publish), and walks its edges in order across receivers.
// Producer, per batch of PB edges lane-parallel: the edge's unit vector, its
// frame and D_1..D_L into the edge ring (lane j builds edge j, no
// divergence), the zero-length flag and (radial) the 8 features; then one
// bulk copy of the sender row x[src] (C (L+1)^2 floats, contiguous) per edge
// into the row ring, completing on the slot's full barrier.  Group g takes
// the edges whose CTA ordinal is g mod G: it rotates its channel in, applies
// the aligned terms with its path weights, rotates back into its partial
// accumulators (shared memory), and releases the slot.  At each receiver's
// end the groups' partials are added in group order.
template <int L, int RADIAL>
__global__ void __launch_bounds__(kHlThreads + 32, 2) k_hl(const HlArgs a, const HlPlan q) {
  using K = HlCfg<L>;
  constexpr int NC = K::NC;
  extern __shared__ __align__(16) float hsm[];
  const int C = a.C, G = kHlThreads / C;
  const int t = threadIdx.x;
  const int S = q.S, YR = q.YR;
  float* slots = hsm + q.o_slot;  // [YR][DS]
  float* flags = hsm + q.o_flag;  // [YR]: 1 for a zero-length edge
  float* rads = hsm + q.o_rad;    // [YR][8] radial features
  float* accs = hsm + q.o_acc;    // partial accumulators [G][NC][C]
  float* xring = hsm + q.o_x;     // [S][C][NC]
  float* ws = hsm + q.o_w;
  const uint32_t full0 = smem_u32(hsm + q.o_bar);
  const uint32_t empty0 = full0 + 8 * S;
  int4* range_s = reinterpret_cast<int4*>(hsm + q.o_bar + 4 * S);
  balanced_range_publish(range_s, a.off, a.N, gridDim.x, blockIdx.x, 1);
  if (t < S) {
    mbar_init(full0 + 8 * t, 1);
    mbar_init(empty0 + 8 * t, C);  // the C threads of the owning group
    fence_mbar_init();
  }
  if constexpr (RADIAL == 0) {
    if (t < kHlThreads)
      for (int i = t; i < K::P * C; i += kHlThreads) ws[i] = __ldg(a.w + i);
  } else if constexpr (RADIAL == 2) {
    if (t < kHlThreads)  // M[k][p C + c], the same layout
      for (int i = t; i < 8 * K::P * C; i += kHlThreads) ws[i] = __ldg(a.M + i);
  }
  __syncthreads();
  const int4 rr = *range_s;
  const int r_begin = rr.x, r_end = rr.y;
  const int e_begin = min(max(rr.z, 0), a.E);
  const int e_end = max(e_begin, min(max(rr.w, 0), a.E));
  const int total = e_end - e_begin;
  const uint32_t row_bytes = (uint32_t)(C * NC * 4);

  if (t >= kHlThreads) {
    // ------------------------------------------------------------ producer
    const int lane = t & 31;
    bool ok = true;
    for (int base = 0; base < total && ok; base += q.PB) {
      const uint32_t n = (uint32_t)(base + lane);
      int node = 0;
      if (lane < q.PB && n < (uint32_t)total) {
        const int e = e_begin + (int)n;
        node = __ldg(a.src + e);
        const float vx = __ldg(a.vec + 3 * (size_t)e), vy = __ldg(a.vec + 3 * (size_t)e + 1),
                    vz = __ldg(a.vec + 3 * (size_t)e + 2);
        const int y = (int)(n % (uint32_t)YR);
        const float r2 = fmaf(vx, vx, fmaf(vy, vy, vz * vz));
        if (r2 >= 1e-30f) {
          const float inv = rsqrtf(r2);
          hl_wigner<L>(vx * inv, vy * inv, vz * inv, slots + (size_t)y * K::DS);
          flags[y] = 0.0f;
        } else {
          flags[y] = 1.0f;  // zero length: Y = (Y00, 0, ...)
        }
        if constexpr (RADIAL) {
          const float4* rp = reinterpret_cast<const float4*>(a.R) + 2 * (size_t)e;
          reinterpret_cast<float4*>(rads + 8 * y)[0] = __ldg(rp);
          reinterpret_cast<float4*>(rads + 8 * y)[1] = __ldg(rp + 1);
        }
      }
      const int cnt = min(q.PB, total - base);
      for (int j = 0; j < cnt; ++j) {
        int good = 1;
        if (lane == j) {
          const uint32_t s = n % (uint32_t)S, par = ((n / (uint32_t)S) & 1u) ^ 1u;
          if (mbar_try_wait(empty0 + 8 * s, par) || mbar_wait(empty0 + 8 * s, par, a.watchdog, 2)) {
            // an out-of-range sender copies row 0; its edge adds nothing
            const size_t row = (unsigned)node < (unsigned)a.N_src ? (size_t)node : 0;
            mbar_arrive_expect_tx(full0 + 8 * s, row_bytes);
            bulk_load(smem_u32(xring + (size_t)s * C * NC), a.x + row * C * NC, row_bytes, full0 + 8 * s);
          } else {
            good = 0;
          }
        }
        if (!__all_sync(0xffffffffu, good)) { ok = false; break; }
      }
    }
    // Drain: the last min(S, total) copies have landed before this warp leaves.
    if (lane == 0 && ok) {
      const uint32_t last = (uint32_t)total;
      const uint32_t first = last > (uint32_t)S ? last - S : 0;
      for (uint32_t i = first; i < last; ++i)
        if (!mbar_wait(full0 + 8 * (i % S), (i / S) & 1u, a.watchdog, 3)) break;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = t / C, c = t % C;
  float* acc = accs + (size_t)g * NC * C + c;
  bool failed = false;
  uint32_t n = 0;
  for (int r = r_begin; r < r_end; ++r) {
    const int a0 = min(max(__ldg(a.off + r), 0), a.E);
    const int a1 = min(max(__ldg(a.off + r + 1), 0), a.E);
    const int deg = min(max(a1 - a0, 0), total - (int)n);
#pragma unroll
    for (int k = 0; k < NC; ++k) acc[k * C] = 0.0f;
    // the group's edges of this receiver: ordinals n + j with j = j0, j0 + G, ...
    const int j0 = (int)(((uint32_t)g + (uint32_t)G - n % (uint32_t)G) % (uint32_t)G);
    for (int j = j0; j < deg; j += G) {
      const uint32_t m = n + j;
      const uint32_t s = m % (uint32_t)S, par = (m / (uint32_t)S) & 1u;
      if (!mbar_try_wait(full0 + 8 * s, par))
        if (!mbar_wait_slow(full0 + 8 * s, par, a.watchdog, 1, failed)) failed = true;
      const int y = (int)(m % (uint32_t)YR);
      const float* D = slots + (size_t)y * K::DS;
      const bool zero = flags[y] != 0.0f;
      const int e = e_begin + (int)m;
      const int snd = __ldg(a.src + e);
      float rad[8];
      if constexpr (RADIAL) {
#pragma unroll
        for (int k = 0; k < 8; ++k) rad[k] = rads[8 * y + k];
      }
      if constexpr (RADIAL == 1) {
        // W[p] = sum_k R[e,k] M[k, p C + c] for every path, into this
        // thread's column (read only by this thread); eight paths at a time,
        // two batches unrolled so one batch's loads are in flight while the
        // other's are summed
        const float* mc = a.M + c;
        const size_t pc = (size_t)K::P * C;
#pragma unroll 2
        for (int p0 = 0; p0 < K::P; p0 += 8) {
          float mm[8][8];
#pragma unroll
          for (int qq = 0; qq < 8; ++qq)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mm[qq][k] = p0 + qq < K::P ? __ldg(mc + k * pc + (size_t)(p0 + qq) * C) : 0.0f;
#pragma unroll
          for (int qq = 0; qq < 8; ++qq) {
            float w = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) w = fmaf(rad[k], mm[qq][k], w);
            if (p0 + qq < K::P) ws[(p0 + qq) * kHlThreads + t] = w;
          }
        }
      }
      if ((unsigned)snd < (unsigned)a.N_src) {  // an out-of-range sender adds nothing
        const float* xrs = xring + (size_t)s * C * NC + c * NC;
        if (!zero) {
          float xr[NC];
          xr[0] = xrs[0];
          rotate_in_all<L>(D, xrs, xr, std::make_integer_sequence<int, L>{});
          all_blocks<L, RADIAL>(a, ws, c, rad, D, xr, acc, std::make_integer_sequence<int, L + 1>{});
        } else {
          zero_len_terms<L, RADIAL>(a, ws, c, rad, xrs, acc, std::make_integer_sequence<int, K::P>{});
        }
      }
      // all reads of row slot s and of edge entry y are done
      mbar_arrive(empty0 + 8 * s);
    }
    n += deg;
    named_barrier(1, kHlThreads);
    // out[r][c][k] = sum over groups in order; thread (g, c) takes k = g, g + G, ...
    float* orow = a.out + ((size_t)r * C + c) * NC;
    for (int k = g; k < NC; k += G) {
      float v = 0.0f;
      for (int h = 0; h < G; ++h) v += accs[((size_t)h * NC + k) * C + c];
      orow[k] = v;
    }
    named_barrier(1, kHlThreads);  // the partials are zeroed for the next receiver
  }
}

// The plan for one weight mode: the ring's slot count is a multiple of the
// group count, so every slot is always used by the same group, which takes
// its edges in order (a group never waits on a slot more than one phase
// ahead of it; the parity wait could not tell that phase from an older
// one).  Plans that fit two CTAs per SM come first (a smaller producer batch
// if need be), then one CTA per SM.
template <int L, int RADIAL>
static bool hl_pick(int C, HlPlan& q) {
  const int G = kHlThreads / C;
  for (int cap : {113 * 1024 - 1024, 227 * 1024 - 1024})
    for (int pb : {32, 24, 16, 12, 8})
      for (int S : {8, 16, 4, 2}) {
        if (S % G != 0) continue;
        q = hl_plan<L>(C, RADIAL, pb, S);
        if (q.bytes <= cap) return true;
      }
  return false;
}

template <int L, int RADIAL>
static eqmp_status launch_hl_plan(const HlArgs& a, const HlPlan& q, cudaStream_t st, const DeviceInfo& dev) {
  auto kern = k_hl<L, RADIAL>;
  static unsigned long long attr_done = 0;
  if (ensure_smem_attr(kern, 227 * 1024, &attr_done) != cudaSuccess) return EQMP_ERR_CUDA;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kHlThreads + 32, q.bytes) != cudaSuccess ||
      occ < 1)
    return EQMP_ERR_CUDA;
  const long long cap = (long long)dev.sms * occ;
  const int grid = (int)(a.N < cap ? a.N : cap);
  if (grid <= 0) return EQMP_OK;
  kern<<<grid, kHlThreads + 32, q.bytes, st>>>(a, q);
  return cuda_status(cudaGetLastError());
}

// Radial weights keep M (8 P C floats) in shared memory when it fits beside
// the rings; otherwise every edge forms its weights from M in global memory.
template <int L>
eqmp_status launch_hl(const HlArgs& a, bool radial, cudaStream_t st, const DeviceInfo& dev) {
  HlPlan q{};
  if (!radial) return hl_pick<L, 0>(a.C, q) ? launch_hl_plan<L, 0>(a, q, st, dev) : EQMP_ERR_UNSUPPORTED;
  if (hl_pick<L, 2>(a.C, q)) return launch_hl_plan<L, 2>(a, q, st, dev);
  return hl_pick<L, 1>(a.C, q) ? launch_hl_plan<L, 1>(a, q, st, dev) : EQMP_ERR_UNSUPPORTED;
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
  if (E > 0 && (reinterpret_cast<uintptr_t>(x) & 15)) return EQMP_ERR_INVALID_ARG;  // rows are bulk-copied
  DeviceInfo dev;
  eqmp_status s = device_info(&dev);
  if (s != EQMP_OK) return s;
  HlArgs a{};
  a.vec = vec; a.x = x; a.off = row_offsets; a.src = src;
  a.w = weights.w; a.R = weights.R; a.M = weights.M; a.out = out; a.watchdog = dev.watchdog;
  a.N = (int)N; a.E = (int)E; a.N_src = (int)N_src; a.C = C;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  switch (l_max) {
    case 4: return launch_hl<4>(a, radial, st, dev);
    case 5: return launch_hl<5>(a, radial, st, dev);
    default: return launch_hl<6>(a, radial, st, dev);
  }
}

}  // extern "C"
