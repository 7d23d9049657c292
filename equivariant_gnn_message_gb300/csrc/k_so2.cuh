// Fused layer in the aligned (SO(2)) frame, E2Former-V2 section 2.1 (EAAS).
//
// Same result as k_shared / k_radial (the dense CG product), computed per
// edge in a frame whose z axis is the edge:
//   x'_l = D_l^T x_l                      (Wigner-D of the frame rotation Q, Q z = n)
//   m'[k3] = sum_p W_p kappa_p x'[k1]     (only m2 = 0 survives, Lemma 4.1; one m1
//                                          per output m3, Eq. 13: 111 terms)
//   out_l += D_l m'_l                     (back to the global frame, summed per receiver)
// About 2.5x fewer FMAs per edge and channel than the dense product, which
// pays off where the weights change per edge (radial weights).
//
// CTA: one producer warp + NCONS = 128 consumer threads split into EG = 128/C
// edge groups of C threads (thread = channel); group g takes the edges whose
// CTA ordinal is g mod EG.  Producer, per 32 edges lane-parallel: frame Q
// (branch-free orthonormal basis), D_1..D_3 by the Ivanic-Ruedenberg
// recursion (coefficients generated at build time), the 8 radial features,
// into a 64-entry edge ring; then one TMA row copy of x[src] per edge into an
// S-slot ring (128-byte swizzle), as in k_shared.  Receiver partials of the
// groups are summed through shared memory in group order (deterministic).
// CTAs run in clusters of Q; inside a cluster the edges are cut at edge
// granularity (cluster_cut_range), and the CTA after a cut hands its piece
// of the cut receiver to the CTA before it through distributed shared
// memory, which adds it to its own piece (deterministic: own piece first).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "k_shared.cuh"
#include "layer_args.cuh"

namespace eqmp {

constexpr float ir_u(int l, int m, int n) { return tables::kIrU[l - 2][m + 3][n + 3]; }
constexpr float ir_v(int l, int m, int n) { return tables::kIrV[l - 2][m + 3][n + 3]; }
constexpr float ir_w(int l, int m, int n) { return tables::kIrW[l - 2][m + 3][n + 3]; }
constexpr tables::AlignedTerm aligned_at(int i) { return tables::kAligned[i]; }

// Edge ring entry (floats), rows padded to whole 16-byte chunks: D_1 rows of
// 4 at 0 (3 x 4), D_2 rows of 8 at 12 (5 x 8), D_3 rows of 8 at 52 (7 x 8),
// radial features (8) at 108, zero-length flag at 116; 120 floats.
constexpr int kEntryFloats = 120;
constexpr int kD1 = 0, kD2 = 12, kD3 = 52, kRad = 108, kFlag = 116;
template <int L>
constexpr int d_off() { return L == 1 ? kD1 : L == 2 ? kD2 : kD3; }
template <int L>
constexpr int d_stride() { return L == 1 ? 4 : 8; }

// ---- Ivanic-Ruedenberg recursion (real SH without CS sign, (y,z,x) order) ---
// R[i+1][j+1], i,j in {-1,0,1}; Dp: level L-1, (2L-1)^2 row-major.
template <int L, int I, int A, int B>
__device__ __forceinline__ float ir_P(const float (&R)[3][3], const float* Dp) {
  constexpr int W = 2 * L - 1;
  auto dp = [&](int a, int b) { return Dp[(a + L - 1) * W + (b + L - 1)]; };
  if constexpr (B == L) {
    return R[I + 1][2] * dp(A, L - 1) - R[I + 1][0] * dp(A, -L + 1);
  } else if constexpr (B == -L) {
    return R[I + 1][2] * dp(A, -L + 1) + R[I + 1][0] * dp(A, L - 1);
  } else {
    return R[I + 1][1] * dp(A, B);
  }
}

template <int L, int M, int N>
__device__ __forceinline__ float ir_entry(const float (&R)[3][3], const float* Dp) {
  constexpr float u = ir_u(L, M, N), v = ir_v(L, M, N), w = ir_w(L, M, N);
  float val = 0.0f;
  if constexpr (u != 0.0f) val = u * ir_P<L, 0, M, N>(R, Dp);
  if constexpr (v != 0.0f) {
    float V;
    if constexpr (M == 0) {
      V = ir_P<L, 1, 1, N>(R, Dp) + ir_P<L, -1, -1, N>(R, Dp);
    } else if constexpr (M > 0) {
      constexpr float f1 = M == 1 ? 1.41421356237309515f : 1.0f;
      constexpr float f2 = M == 1 ? 0.0f : 1.0f;
      V = ir_P<L, 1, M - 1, N>(R, Dp) * f1;
      if constexpr (f2 != 0.0f) V -= ir_P<L, -1, -M + 1, N>(R, Dp);
    } else {
      constexpr float f1 = M == -1 ? 0.0f : 1.0f;
      constexpr float f2 = M == -1 ? 1.41421356237309515f : 1.0f;
      V = ir_P<L, -1, -M - 1, N>(R, Dp) * f2;
      if constexpr (f1 != 0.0f) V += ir_P<L, 1, M + 1, N>(R, Dp);
    }
    val = fmaf(v, V, val);
  }
  if constexpr (w != 0.0f) {
    float Wt;
    if constexpr (M > 0) {
      Wt = ir_P<L, 1, M + 1, N>(R, Dp) + ir_P<L, -1, -M - 1, N>(R, Dp);
    } else {
      Wt = ir_P<L, 1, M - 1, N>(R, Dp) - ir_P<L, -1, -M + 1, N>(R, Dp);
    }
    val = fmaf(w, Wt, val);
  }
  return val;
}

template <int L, int... Is>
__device__ __forceinline__ void ir_level(const float (&R)[3][3], const float* Dp, float* Dl,
                                         std::integer_sequence<int, Is...>) {
  constexpr int W = 2 * L + 1;
  ((Dl[Is] = ir_entry<L, Is / W - L, Is % W - L>(R, Dp)), ...);
}

constexpr float cs_sign_(int m) { return (m != 0 && (m & 1)) ? -1.0f : 1.0f; }

// Level L straight into the edge entry (this library's signs, padded rows),
// entry by entry, so the level is never held in registers.
template <int L, int... Is>
__device__ __forceinline__ void ir_level_store(const float (&R)[3][3], const float* Dp, float* out,
                                               std::integer_sequence<int, Is...>) {
  constexpr int W = 2 * L + 1, ST = L == 1 ? 4 : 8;
  ((out[(Is / W) * ST + Is % W] =
        cs_sign_(Is / W - L) * cs_sign_(Is % W - L) * ir_entry<L, Is / W - L, Is % W - L>(R, Dp)),
   ...);
}

constexpr float cs_sign(int m) { return (m != 0 && (m & 1)) ? -1.0f : 1.0f; }

// This library's basis: D[i][j] = s_i s_j D_IR[i][j], s = (-1)^|m|; rows
// stored with the padded stride of the edge ring.
template <int L, int... Is>
__device__ __forceinline__ void store_block(const float* Dir, float* out, std::integer_sequence<int, Is...>) {
  constexpr int W = 2 * L + 1, ST = d_stride<L>();
  ((out[(Is / W) * ST + Is % W] = cs_sign(Is / W - L) * cs_sign(Is % W - L) * Dir[Is]), ...);
}

// Frame and D_1..D_3 for unit direction (x, y, z) into entry e (83 floats).
__device__ __forceinline__ void wigner_blocks(float x, float y, float z, float* e) {
  const float s = z >= 0.0f ? 1.0f : -1.0f;
  const float a = -1.0f / (s + z);
  const float b = x * y * a;
  // Q columns: t1, t2, n
  const float Q[3][3] = {{fmaf(s * x * x, a, 1.0f), b, x},
                         {s * b, fmaf(y * y, a, s), y},
                         {-s * x, -y, z}};
  // (y, z, x) ordering
  const float R[3][3] = {{Q[1][1], Q[1][2], Q[1][0]},
                         {Q[2][1], Q[2][2], Q[2][0]},
                         {Q[0][1], Q[0][2], Q[0][0]}};
  float D2[25];
  ir_level<2>(R, &R[0][0], D2, std::make_integer_sequence<int, 25>{});
  store_block<1>(&R[0][0], e + kD1, std::make_integer_sequence<int, 9>{});
  store_block<2>(D2, e + kD2, std::make_integer_sequence<int, 25>{});
  ir_level_store<3>(R, D2, e + kD3, std::make_integer_sequence<int, 49>{});
}

template <int C, typename XT, bool RADIAL>
struct So2Cfg {
  static constexpr int NCONS = 128;
#ifdef EQMP_TUNE_SO2_Q
  static constexpr int Q = EQMP_TUNE_SO2_Q;            // cluster size (experiments)
#else
  static constexpr int Q = 2;                          // cluster size
#endif
  static constexpr int EG = NCONS / C;                 // edge groups
  static constexpr int NTHREADS = NCONS + 32;
  static constexpr int ROW_BYTES = C * 16 * (int)sizeof(XT);
  static constexpr int ROWS = ROW_BYTES / 128;
  static constexpr int SLOT = ROW_BYTES < 1024 ? 1024 : ROW_BYTES;
  static constexpr int YR = 64;
  // radial: M as [8][17][C] float2; shared: w as [34][C]
  static constexpr int M_BYTES = RADIAL ? 8 * 34 * C * 4 : 34 * C * 4;
  static constexpr int FIXED = YR * kEntryFloats * 4 + 2 * EG * 16 * C * 4 + M_BYTES + 16 * C * 4 + 2 * 16 * 8 + 16 +
                               32 + 2048;
  // two CTAs per SM when at least 4 slots fit in half the shared memory
  static constexpr int S_FIT2 = (113 * 1024 - FIXED) / SLOT;
  static constexpr int MINB = S_FIT2 >= 4 ? 2 : 1;
  static constexpr int S_FIT = MINB == 2 ? S_FIT2 : (227 * 1024 - FIXED) / SLOT;
  static constexpr int S = S_FIT >= 16 ? 16 : S_FIT >= 8 ? 8 : S_FIT >= 4 ? 4 : 2;
  static_assert(S % EG == 0 && S <= 32 && YR >= 32 + S && S_FIT >= 2, "ring layout");
  static constexpr int OFF_X = 0;
  static constexpr int OFF_E = OFF_X + S * SLOT;                       // edge ring
  static constexpr int OFF_RED = OFF_E + YR * kEntryFloats * 4;         // [2][EG][16][C]
  static constexpr int OFF_M = OFF_RED + 2 * EG * 16 * C * 4;          // radial: [8][17][C] float2
  static constexpr int OFF_EX = OFF_M + M_BYTES;                       // [16][C]: piece handed over
  static constexpr int OFF_BAR = OFF_EX + 16 * C * 4;                  // full[S], empty[S], xfull
  static constexpr int OFF_RANGE = OFF_BAR + 2 * S * 8 + 16;           // the CTA's CutRange
  static constexpr int SMEM_BYTES = OFF_RANGE + 32 + 1024;
};

// One padded D row (m) of level L from the edge entry into registers.
template <int L>
__device__ __forceinline__ void load_row(const float* ent, int m, float (&row)[8]) {
  const float4* p = reinterpret_cast<const float4*>(ent + d_off<L>() + m * d_stride<L>());
  const float4 a = p[0];
  row[0] = a.x; row[1] = a.y; row[2] = a.z; row[3] = a.w;
  if constexpr (d_stride<L>() == 8) {
    const float4 b = p[1];
    row[4] = b.x; row[5] = b.y; row[6] = b.z; row[7] = b.w;
  }
}
// x'_l[n] = sum_m D[m][n] x_l[m], rows of D streamed from shared memory
template <int L>
__device__ __forceinline__ void rotate_in(const float* ent, const float (&x)[16], float (&xr)[16]) {
  constexpr int W = 2 * L + 1, o = L * L;
#pragma unroll
  for (int n = 0; n < W; ++n) xr[o + n] = 0.0f;
#pragma unroll
  for (int m = 0; m < W; ++m) {
    float row[8];
    load_row<L>(ent, m, row);
#pragma unroll
    for (int n = 0; n < W; ++n) xr[o + n] = fmaf(row[n], x[o + m], xr[o + n]);
  }
}
// out_l[m] += sum_n D[m][n] m'_l[n]
template <int L>
__device__ __forceinline__ void rotate_out(const float* ent, const float (&mp)[16], float (&out)[16]) {
  constexpr int W = 2 * L + 1, o = L * L;
#pragma unroll
  for (int m = 0; m < W; ++m) {
    float row[8];
    load_row<L>(ent, m, row);
    float s = out[o + m];
#pragma unroll
    for (int n = 0; n < W; ++n) s = fmaf(row[n], mp[o + n], s);
    out[o + m] = s;
  }
}

// Aligned terms of one path (compile-time range of the table, sorted by path).
constexpr int aligned_first(int p) {
  for (int i = 0; i < tables::kNumAligned; ++i)
    if (tables::kAligned[i].p == p) return i;
  return tables::kNumAligned;
}
constexpr int aligned_count(int p) {
  int c = 0;
  for (int i = 0; i < tables::kNumAligned; ++i) c += tables::kAligned[i].p == p;
  return c;
}
template <int First, int... Is>
__device__ __forceinline__ void so2_path_terms(float wp, const float (&xr)[16], float (&mp)[16],
                                               std::integer_sequence<int, Is...>) {
  ((mp[aligned_at(First + Is).k3] =
        fmaf(wp, aligned_at(First + Is).kappa * xr[aligned_at(First + Is).k1], mp[aligned_at(First + Is).k3])),
   ...);
}
// Paths 2Q and 2Q+1: their weights (radial: one FFMA2 chain over k with M
// pairs from shared memory; shared: w[p][c] from shared memory), then their
// aligned terms.
template <int Q, int C, bool RADIAL>
__device__ __forceinline__ void so2_pair(const float2* Ms, int c, const float2 (&rr)[8],
                                         const float (&xr)[16], float (&mp)[16]) {
  constexpr int P0 = 2 * Q, P1 = 2 * Q + 1;
  float w0, w1;
  if constexpr (RADIAL) {
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc = __ffma2_rn(rr[k], Ms[(k * 17 + Q) * C + c], acc);
    w0 = acc.x;
    w1 = acc.y;
  } else {
    const float* ws = reinterpret_cast<const float*>(Ms);
    w0 = ws[P0 * C + c];
    w1 = ws[P1 * C + c];
  }
  so2_path_terms<aligned_first(P0)>(w0, xr, mp, std::make_integer_sequence<int, aligned_count(P0)>{});
  so2_path_terms<aligned_first(P1)>(w1, xr, mp, std::make_integer_sequence<int, aligned_count(P1)>{});
}
template <int C, bool RADIAL, int... Qs>
__device__ __forceinline__ void so2_all(const float2* Ms, int c, const float2 (&rr)[8], const float (&xr)[16],
                                        float (&mp)[16], std::integer_sequence<int, Qs...>) {
  (so2_pair<Qs, C, RADIAL>(Ms, c, rr, xr, mp), ...);
}

// The radial mixing matrix (or the shared weights) to shared memory by NT
// threads (t = 0 .. NT-1), while warp 0 searches the CTA's range; loads in
// batches of 8 per thread, each batch issued before its stores.
template <int C, bool RADIAL, int NT>
__device__ __forceinline__ void so2_stage_weights(const LayerArgs& a, float2* Ms, int t) {
  if constexpr (RADIAL) {
    // M[k][p*C + c] -> Ms[(k*17 + p/2)*C + c] = (M[k][p][c], M[k][p+1][c])
    if ((reinterpret_cast<uintptr_t>(a.M) & 15) == 0) {
      constexpr int Q4 = 8 * 17 * C / 4;  // (k, path pair, 4 channels)
      for (int base = 0; base < Q4; base += 8 * NT) {
        float4 va[8], vb[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = base + t + u * NT;
          if (i < Q4) {
            const int c4 = i % (C / 4), pp = (i / (C / 4)) % 17, k = i / (17 * (C / 4));
            const float* row = a.M + (size_t)k * 34 * C + (size_t)(2 * pp) * C + 4 * c4;
            va[u] = __ldg(reinterpret_cast<const float4*>(row));
            vb[u] = __ldg(reinterpret_cast<const float4*>(row + C));
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = base + t + u * NT;
          if (i < Q4) {
            const int c4 = i % (C / 4), pp = (i / (C / 4)) % 17, k = i / (17 * (C / 4));
            float4* d = reinterpret_cast<float4*>(Ms + (k * 17 + pp) * C + 4 * c4);
            d[0] = make_float4(va[u].x, vb[u].x, va[u].y, vb[u].y);
            d[1] = make_float4(va[u].z, vb[u].z, va[u].w, vb[u].w);
          }
        }
      }
    } else {
      for (int i = t; i < 8 * 17 * C; i += NT) {
        const int k = i / (17 * C), pp = (i / C) % 17, c = i % C;
        Ms[i] = make_float2(__ldg(a.M + (size_t)k * 34 * C + (2 * pp) * C + c),
                            __ldg(a.M + (size_t)k * 34 * C + (2 * pp + 1) * C + c));
      }
    }
  } else {
    float* ws = reinterpret_cast<float*>(Ms);
    for (int i = t; i < 34 * C; i += NT) ws[i] = __ldg(a.w + i);
  }
}

template <int C, typename XT, bool RADIAL>
__global__ void __launch_bounds__(So2Cfg<C, XT, RADIAL>::NTHREADS, So2Cfg<C, XT, RADIAL>::MINB)
    k_so2(const __grid_constant__ CUtensorMap tmap, const LayerArgs a) {
  using K = So2Cfg<C, XT, RADIAL>;
  constexpr int S = K::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align<1024>(smem_raw);
  float* ering = reinterpret_cast<float*>(smem + K::OFF_E);
  float* red = reinterpret_cast<float*>(smem + K::OFF_RED);
  float2* Ms = reinterpret_cast<float2*>(smem + K::OFF_M);
  float* ex = reinterpret_cast<float*>(smem + K::OFF_EX);
  const uint32_t full0 = smem_u32(smem + K::OFF_BAR);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t xfull = empty0 + 8 * S;  // the next CTA's piece is in its ex
  const int tid = threadIdx.x;
  // Edge range, balanced on edges (a receiver's group sum and store cost
  // about one edge here), cut at edge granularity inside the cluster.
  CutRange* range_s = reinterpret_cast<CutRange*>(smem + K::OFF_RANGE);
  if (tid < 32) {
    const CutRange cr = cluster_cut_range(a.off, a.N, gridDim.x, blockIdx.x, K::Q, 1);
    if (tid == 0) *range_s = cr;
  }
  if (tid >= 32 && tid < K::NCONS) so2_stage_weights<C, RADIAL, K::NCONS - 32>(a, Ms, tid - 32);
  if (tid < S) {
    mbar_init(full0 + 8 * tid, 1);
    mbar_init(empty0 + 8 * tid, C);  // the C threads of the owning edge group
    if (tid == 0) mbar_init(xfull, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Two cluster barriers: this one (arrive now, wait before any remote
  // access) publishes the initialised barriers; the one at the end keeps
  // every CTA's shared memory alive until the cluster's remote accesses are done.
  cluster_arrive();
  const CutRange cr = *range_s;
  const int r_begin = cr.r_begin, r_end = cr.r_end;
  const int e_begin = min(max(cr.e_begin, 0), a.E);
  const int e_end = max(e_begin, min(max(cr.e_end, 0), a.E));
  const int total = e_end - e_begin;

  if (tid >= K::NCONS) {
    // ------------------------------------------------------------ producer
    const int lane = tid & 31;
    if (lane == 0) prefetch_tmap(&tmap);
    bool ok = true;
    for (int base = 0; base < total && ok; base += 32) {
      const uint32_t n = (uint32_t)(base + lane);
      int node = 0;
      if (n < (uint32_t)total) {
        const int e = e_begin + (int)n;
        node = __ldg(a.src + e);
        const float* v = a.vec + 3 * (size_t)e;
        const float vx = __ldg(v), vy = __ldg(v + 1), vz = __ldg(v + 2);
        float* ent = ering + (size_t)(n % K::YR) * kEntryFloats;
        const float r2 = fmaf(vx, vx, fmaf(vy, vy, vz * vz));
        if (r2 >= 1e-30f) {
          const float inv = rsqrtf(r2);
          wigner_blocks(vx * inv, vy * inv, vz * inv, ent);
          ent[kFlag] = 0.0f;
        } else {
          ent[kFlag] = 1.0f;  // zero-length edge: only the l2 = 0 paths contribute
        }
        if constexpr (RADIAL) {
          const float4* rp = reinterpret_cast<const float4*>(a.R) + 2 * (size_t)e;
          reinterpret_cast<float4*>(ent + kRad)[0] = __ldg(rp);
          reinterpret_cast<float4*>(ent + kRad)[1] = __ldg(rp + 1);
        }
      }
      const int cnt = min(32, total - base);
      for (int j = 0; j < cnt; ++j) {
        int good = 1;
        if (lane == j) {
          const uint32_t s = n % S, par = ((n / S) & 1u) ^ 1u;
          if (mbar_try_wait(empty0 + 8 * s, par) || mbar_wait(empty0 + 8 * s, par, a.watchdog, 2)) {
            mbar_arrive_expect_tx(full0 + 8 * s, K::ROW_BYTES);
            tma_load_2d(smem_u32(smem + K::OFF_X + s * K::SLOT), &tmap, 0, node * K::ROWS, full0 + 8 * s);
          } else {
            good = 0;
          }
        }
        if (!__all_sync(0xffffffffu, good)) { ok = false; break; }
      }
    }
    // Drain: the last min(S, total) loads have landed before this warp leaves.
    if (lane == 0 && ok) {
      const uint32_t last = (uint32_t)total;
      const uint32_t first = last > (uint32_t)S ? last - S : 0;
      for (uint32_t i = first; i < last; ++i)
        if (!mbar_wait(full0 + 8 * (i % S), (i / S) & 1u, a.watchdog, 3)) break;
    }
    cluster_wait();
    cluster_arrive();
    cluster_wait();
    return;
  }

  // -------------------------------------------------------------- consumers
  cluster_wait();              // every CTA of the cluster has initialised its barriers
  const uint32_t rank = cluster_rank();

  const int c = tid % C, g = tid / C;
  const uint32_t xlog = (uint32_t)(c * 16 * (int)sizeof(XT));
  const uint32_t xo[2] = {swz128(xlog), swz128(xlog + 16)};
  bool failed = false;
  int buf = 0;
  uint32_t n = 0;
  for (int r = r_begin; r < r_end; ++r) {
    const int a0 = max(min(max(__ldg(a.off + r), 0), a.E), e_begin);
    const int a1 = min(min(max(__ldg(a.off + r + 1), 0), a.E), e_end);
    const int deg = min(max(a1 - a0, 0), total - (int)n);
    float out[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) out[k] = 0.0f;
    // the group's edges of this receiver: ordinals n + j with j = j0, j0 + EG, ...
    const int j0 = (int)(((uint32_t)g + (uint32_t)K::EG - n % (uint32_t)K::EG) % (uint32_t)K::EG);
    for (int j = j0; j < deg; j += K::EG) {
      const uint32_t m = n + j;
      const uint32_t s = m % S, par = (m / S) & 1u;
      if (!mbar_try_wait(full0 + 8 * s, par))
        if (!mbar_wait_slow(full0 + 8 * s, par, a.watchdog, 1, failed)) failed = true;
      const float* ent = ering + (size_t)(m % K::YR) * kEntryFloats;
      float x[16];
      {
        const uint8_t* slot = smem + K::OFF_X + s * K::SLOT;
        if constexpr (sizeof(XT) == 4) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float4 v = *reinterpret_cast<const float4*>(slot + swz128(xlog + 16 * h));
            x[4 * h] = v.x; x[4 * h + 1] = v.y; x[4 * h + 2] = v.z; x[4 * h + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 v = *reinterpret_cast<const uint4*>(slot + xo[h]);
            x[8 * h + 0] = bf16_lo(v.x); x[8 * h + 1] = bf16_hi(v.x);
            x[8 * h + 2] = bf16_lo(v.y); x[8 * h + 3] = bf16_hi(v.y);
            x[8 * h + 4] = bf16_lo(v.z); x[8 * h + 5] = bf16_hi(v.z);
            x[8 * h + 6] = bf16_lo(v.w); x[8 * h + 7] = bf16_hi(v.w);
          }
        }
      }
      float2 rr[8];
      if constexpr (RADIAL) {
#pragma unroll
        for (int k = 0; k < 8; ++k) rr[k] = make_float2(ent[kRad + k], ent[kRad + k]);
      }
      const bool zero_len = ent[kFlag] != 0.0f;
      if (!zero_len) {
        float xr[16], mp[16];
        xr[0] = x[0];
        rotate_in<1>(ent, x, xr);
        rotate_in<2>(ent, x, xr);
        rotate_in<3>(ent, x, xr);
#pragma unroll
        for (int k = 0; k < 16; ++k) mp[k] = 0.0f;
        so2_all<C, RADIAL>(Ms, c, rr, xr, mp, std::make_integer_sequence<int, 17>{});
        out[0] += mp[0];
        rotate_out<1>(ent, mp, out);
        rotate_out<2>(ent, mp, out);
        rotate_out<3>(ent, mp, out);
      } else {
        // n = 0: Y = (Y00, 0, ...): only the paths (l, 0, l), identity CG
        constexpr float y00 = 0.28209479177387814f;
        float w0, w4, w13, w24;
        if constexpr (RADIAL) {
          float2 a0 = make_float2(0.f, 0.f), a4 = a0, a12 = a0, a24 = a0;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            a0 = __ffma2_rn(rr[k], Ms[(k * 17 + 0) * C + c], a0);
            a4 = __ffma2_rn(rr[k], Ms[(k * 17 + 2) * C + c], a4);
            a12 = __ffma2_rn(rr[k], Ms[(k * 17 + 6) * C + c], a12);
            a24 = __ffma2_rn(rr[k], Ms[(k * 17 + 12) * C + c], a24);
          }
          w0 = a0.x; w4 = a4.x; w13 = a12.y; w24 = a24.x;
        } else {
          const float* ws = reinterpret_cast<const float*>(Ms);
          w0 = ws[0 * C + c]; w4 = ws[4 * C + c]; w13 = ws[13 * C + c]; w24 = ws[24 * C + c];
        }
        out[0] = fmaf(w0 * y00, x[0], out[0]);
#pragma unroll
        for (int k = 1; k < 4; ++k) out[k] = fmaf(w4 * y00, x[k], out[k]);
#pragma unroll
        for (int k = 4; k < 9; ++k) out[k] = fmaf(w13 * y00, x[k], out[k]);
#pragma unroll
        for (int k = 9; k < 16; ++k) out[k] = fmaf(w24 * y00, x[k], out[k]);
      }
      // all reads of slot s and of edge entry m are done
      mbar_arrive(empty0 + 8 * s);
    }
    n += deg;
    // group partials -> shared memory; thread (c, g) sums outputs k in its share
    float* rb = red + buf * (K::EG * 16 * C);
#pragma unroll
    for (int k = 0; k < 16; ++k) rb[(g * 16 + k) * C + c] = out[k];
    named_barrier(1, K::NCONS);
    constexpr int KPER = 16 / K::EG > 0 ? 16 / K::EG : 1;
    const bool head = cr.head_cut && r == r_begin;    // piece handed to the CTA before
    const bool tail = cr.tail_cut && r == r_end - 1;  // the CTA after holds the rest
    float o[16];
    if (g * KPER < 16) {
#pragma unroll
      for (int i = 0; i < KPER; ++i) {
        float sum = 0.0f;
#pragma unroll
        for (int gg = 0; gg < K::EG; ++gg) sum += rb[(gg * 16 + g * KPER + i) * C + c];
        o[i] = sum;
      }
    }
    if (tail) {
      // own piece first, then the next CTA's (which already holds the pieces after it)
      if (!failed && !mbar_wait_cluster(xfull, 0, a.watchdog, 8)) failed = true;
      if (!failed && g * KPER < 16) {
        const uint32_t rex = map_rank(smem_u32(ex + (g * KPER) * C + c), rank + 1);
#pragma unroll
        for (int i = 0; i < KPER; ++i) o[i] += ld_cluster_f32(rex + 4u * (uint32_t)(i * C));
      }
    }
    if (head) {
      if (g * KPER < 16) {
#pragma unroll
        for (int i = 0; i < KPER; ++i) ex[(g * KPER + i) * C + c] = o[i];
      }
      fence_cluster();
      named_barrier(3, K::NCONS);  // the whole piece is in ex
      if (tid == 0) mbar_arrive_remote(map_rank(xfull, rank - 1));
    } else if (g * KPER < 16) {
      if constexpr (sizeof(XT) == 4) {
        float* op = reinterpret_cast<float*>(a.out) + ((size_t)r * C + c) * 16 + g * KPER;
#pragma unroll
        for (int i = 0; i < KPER; ++i) op[i] = o[i];
      } else {
        __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(a.out) + ((size_t)r * C + c) * 16 + g * KPER;
#pragma unroll
        for (int i = 0; i < KPER; ++i) op[i] = __float2bfloat16_rn(o[i]);
      }
    }
    buf ^= 1;
  }
  cluster_arrive();
  cluster_wait();
}

}  // namespace eqmp
