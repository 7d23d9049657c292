// Backward of the fused layer: gradients with respect to the sender
// features, the weights (shared w, or radial R and M) and the edge vectors.
//
//   gx[j,c,k1] = sum_{e: src_e=j} sum_p W[e,p,c] sum_{k3,k2} C_p[k3,k1,k2] g[dst_e,c,k3] Y_e[k2]
//   s[e,p,c]   = sum_{k3,k1,k2} C_p[k3,k1,k2] g[dst_e,c,k3] x[src_e,c,k1] Y_e[k2]
//   gw[p,c]    = sum_e s[e,p,c];  gR[e,k] = sum_{p,c} M[k,pC+c] s[e,p,c];  gM = R^T s
//   dY[e,k2]   = sum_{c,p} W[e,p,c] sum_{k3,k1} C_p[k3,k1,k2] g[dst_e,c,k3] x[src_e,c,k1]
//   gvec[e]    = dY[e,:] . dY(vec_e)/dvec_e
//
// Mapping: a group of G = min(C, 32) lanes owns one node (sender for gx,
// receiver for the rest); lane l handles channels l, l+G, ...  Edge loops
// run in CSR order; every reduction (over channels by warp shuffles, over
// receiver groups and edges through the caller's workspace) has a fixed
// order, so results are deterministic.  No waits; shared memory holds only
// the per-group partial weight gradients.
#pragma once

#include "common.cuh"
#include "layer_args.cuh"

namespace eqmp {

struct BwdArgs {
  const float* vec;
  const float* x;           // [N_src][C][16] fp32
  const int32_t* off;       // [N+1] receiver CSR (absolute)
  const int32_t* src;       // [E]
  const int32_t* dst;       // [E]
  const int32_t* send_off;  // [N_src+1] sender CSR into send_edges
  const int32_t* send_edges;  // edge ids sorted by sender
  const float* w;           // [34][C] or nullptr
  const float* R;           // [E][8] or nullptr
  const float* M;           // [8][34C] or nullptr
  const float* g;           // [N][C][16] dL/dout
  float* gx;                // [N_src][C][16] or nullptr
  float* gvec;              // [E][3] or nullptr
  float* gR;                // [E][8] or nullptr
  float* ws;                // workspace (see eqmp_fused_backward)
  int N, E, N_src, n_send;  // n_send = length of send_edges
};

constexpr float sh_dcoef(int l, int m, int p) { return (p + 1) * tables::kShPoly[l][m][p + 1]; }

template <int L, int M>
__device__ __forceinline__ float sh_dpoly(float z) {
  constexpr float d0 = sh_dcoef(L, M, 0), d1 = sh_dcoef(L, M, 1), d2 = sh_dcoef(L, M, 2);
  return fmaf(fmaf(d2, z, d1), z, d0);
}

// (x + i y)^m as (c[m], s[m]), m = 0..3.
struct Pow3 {
  float c[4], s[4];
};

template <int L, int M>
__device__ __forceinline__ void sh_vjp_term(const float (&dY)[16], float z, const Pow3& pw, float& gx,
                                            float& gy, float& gz) {
  constexpr int kc = L * L + L + M, ks = L * L + L - M;
  const float P = sh_poly<L, M>(z), dP = sh_dpoly<L, M>(z);
  if constexpr (M == 0) {
    gz = fmaf(dY[kc], dP, gz);
  } else {
    // d/dx (x+iy)^m = m (x+iy)^(m-1); d/dy = i m (x+iy)^(m-1)
    const float mc = M * pw.c[M - 1], ms = M * pw.s[M - 1];
    gx = fmaf(dY[kc], P * mc, fmaf(dY[ks], P * ms, gx));
    gy = fmaf(dY[kc], -P * ms, fmaf(dY[ks], P * mc, gy));
    gz = fmaf(dY[kc], dP * pw.c[M], fmaf(dY[ks], dP * pw.s[M], gz));
  }
}

// Gradient of sum_k dY[k] Y_k(v/|v|) with respect to v (0 for |v|^2 < 1e-30).
__device__ __forceinline__ void real_sh16_vjp(float vx, float vy, float vz, const float (&dY)[16],
                                              float& ox, float& oy, float& oz) {
  const float r2 = fmaf(vx, vx, fmaf(vy, vy, vz * vz));
  if (!(r2 >= 1e-30f)) { ox = oy = oz = 0.0f; return; }
  const float inv = rsqrtf(r2);
  const float x = vx * inv, y = vy * inv, z = vz * inv;
  Pow3 pw;
  pw.c[0] = 1.0f; pw.s[0] = 0.0f;
  pw.c[1] = x; pw.s[1] = y;
  pw.c[2] = fmaf(x, x, -y * y); pw.s[2] = 2.0f * x * y;
  pw.c[3] = fmaf(x, pw.c[2], -y * pw.s[2]); pw.s[3] = fmaf(x, pw.s[2], y * pw.c[2]);
  float gx = 0.0f, gy = 0.0f, gz = 0.0f;
  sh_vjp_term<1, 0>(dY, z, pw, gx, gy, gz); sh_vjp_term<1, 1>(dY, z, pw, gx, gy, gz);
  sh_vjp_term<2, 0>(dY, z, pw, gx, gy, gz); sh_vjp_term<2, 1>(dY, z, pw, gx, gy, gz);
  sh_vjp_term<2, 2>(dY, z, pw, gx, gy, gz);
  sh_vjp_term<3, 0>(dY, z, pw, gx, gy, gz); sh_vjp_term<3, 1>(dY, z, pw, gx, gy, gz);
  sh_vjp_term<3, 2>(dY, z, pw, gx, gy, gz); sh_vjp_term<3, 3>(dY, z, pw, gx, gy, gz);
  // project out the radial direction, divide by |v|
  const float nd = x * gx + y * gy + z * gz;
  ox = (gx - x * nd) * inv;
  oy = (gy - y * nd) * inv;
  oz = (gz - z * nd) * inv;
}

__device__ __forceinline__ void load16(const float* p, float (&v)[16]) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float4 t = __ldg(q + h);
    v[4 * h] = t.x; v[4 * h + 1] = t.y; v[4 * h + 2] = t.z; v[4 * h + 3] = t.w;
  }
}

// ---- dL/dx: per path, gx[k1] += W * sum_{k3,k2} C g[k3] Y[k2] -------------
template <int I>
__device__ __forceinline__ void bx_term(const float (&gv)[16], const float (&yv)[16], float (&tmp)[16]) {
  constexpr tables::Term t = term_at(I);
  tmp[t.k1] = fmaf(t.c * gv[t.k3], yv[t.k2], tmp[t.k1]);
}
template <int First, int... Is>
__device__ __forceinline__ void bx_terms(const float (&gv)[16], const float (&yv)[16], float (&tmp)[16],
                                         std::integer_sequence<int, Is...>) {
  (bx_term<First + Is>(gv, yv, tmp), ...);
}
template <int P>
__device__ __forceinline__ void bx_path(const float (&gv)[16], const float (&yv)[16], float wp, float (&acc)[16]) {
  constexpr tables::Path path = path_at(P);
  float tmp[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) tmp[k] = 0.0f;
  bx_terms<path.first>(gv, yv, tmp, std::make_integer_sequence<int, path.count>{});
  constexpr int lo = path.l1 * path.l1, hi = (path.l1 + 1) * (path.l1 + 1);
#pragma unroll
  for (int k = lo; k < hi; ++k) acc[k] = fmaf(wp, tmp[k], acc[k]);
}

// ---- s and dY: a = C g[k3] x[k1]; s += a Y[k2]; dYp[k2] += a -----------------
template <int I>
__device__ __forceinline__ void bs_term(const float (&gv)[16], const float (&xv)[16], const float (&yv)[16],
                                        float& s, float (&dyp)[16]) {
  constexpr tables::Term t = term_at(I);
  const float a = (t.c * gv[t.k3]) * xv[t.k1];
  s = fmaf(a, yv[t.k2], s);
  dyp[t.k2] += a;
}
template <int First, int... Is>
__device__ __forceinline__ void bs_terms(const float (&gv)[16], const float (&xv)[16], const float (&yv)[16],
                                         float& s, float (&dyp)[16], std::integer_sequence<int, Is...>) {
  (bs_term<First + Is>(gv, xv, yv, s, dyp), ...);
}

template <int C, bool RADIAL>
struct BwdCfg {
  static constexpr int G = C < 32 ? C : 32;   // lanes per node group
  static constexpr int CPL = C / G;           // channels per lane
  static constexpr int NT = 128;
  static constexpr int GROUPS = NT / G;       // node groups per block
  // Radial weights with whole-warp groups: the block's four warps share one
  // node and take every fourth of its edges (four times the warps in
  // flight; a node's edges are independent work, and the sender sums of
  // dL/dx are added over the four warps in order).
  static constexpr int SPLIT = RADIAL && G == 32 ? GROUPS : 1;
  static constexpr int NODES = GROUPS / SPLIT;  // nodes per block at a time
};

// Weight of path P for channel c of edge e.
template <int C, bool RADIAL, int P>
__device__ __forceinline__ float path_weight(const BwdArgs& a, int c, const float (&rk)[8]) {
  if constexpr (RADIAL) {
    float wp = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) wp = fmaf(rk[k], __ldg(a.M + (size_t)k * 34 * C + P * C + c), wp);
    return wp;
  } else {
    return __ldg(a.w + P * C + c);
  }
}

template <int C, bool RADIAL, int... Ps>
__device__ __forceinline__ void bx_all(const BwdArgs& a, int c, const float (&rk)[8], const float (&gv)[16],
                                       const float (&yv)[16], float (&acc)[16], std::integer_sequence<int, Ps...>) {
  (bx_path<Ps>(gv, yv, path_weight<C, RADIAL, Ps>(a, c, rk), acc), ...);
}

template <int C, bool RADIAL>
__global__ void __launch_bounds__(128) k_bwd_x(const BwdArgs a) {
  using K = BwdCfg<C, RADIAL>;
  __shared__ float xred[K::SPLIT > 1 ? K::SPLIT * 16 * 32 : 1];
  const int grp = threadIdx.x / K::G, lane = threadIdx.x % K::G;
  const int node = grp / K::SPLIT, sub = grp % K::SPLIT;
  for (int jb = blockIdx.x * K::NODES; jb < a.N_src; jb += gridDim.x * K::NODES) {  // block-uniform
    const int j = jb + node;
    const bool live = j < a.N_src;
    const int a0 = live ? min(max(__ldg(a.send_off + j), 0), a.n_send) : 0;
    const int a1 = live ? min(max(__ldg(a.send_off + j + 1), 0), a.n_send) : 0;
#pragma unroll 1
    for (int cc = 0; cc < K::CPL; ++cc) {
      const int c = lane + cc * K::G;
      float acc[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
      for (int q = a0 + sub; q < a1; q += K::SPLIT) {
        const int e = __ldg(a.send_edges + q);
        if (e < 0 || e >= a.E) continue;
        const int i = __ldg(a.dst + e);
        if (i < 0 || i >= a.N) continue;
        float yv[16], gv[16], rk[8];
        const float* v = a.vec + 3 * (size_t)e;
        real_sh16(__ldg(v), __ldg(v + 1), __ldg(v + 2), yv);
        load16(a.g + ((size_t)i * C + c) * 16, gv);
        if constexpr (RADIAL) {
          const float4* rp = reinterpret_cast<const float4*>(a.R) + 2 * (size_t)e;
          const float4 r0 = __ldg(rp), r1 = __ldg(rp + 1);
          rk[0] = r0.x; rk[1] = r0.y; rk[2] = r0.z; rk[3] = r0.w;
          rk[4] = r1.x; rk[5] = r1.y; rk[6] = r1.z; rk[7] = r1.w;
        }
        bx_all<C, RADIAL>(a, c, rk, gv, yv, acc, std::make_integer_sequence<int, tables::kNumPaths>{});
      }
      if constexpr (K::SPLIT > 1) {
        // the warps' partial sums, added in warp order by warp 0
#pragma unroll
        for (int k = 0; k < 16; ++k) xred[(sub * 16 + k) * 32 + lane] = acc[k];
        __syncthreads();
        if (sub == 0) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            float t = xred[k * 32 + lane];
#pragma unroll
            for (int w = 1; w < K::SPLIT; ++w) t += xred[(w * 16 + k) * 32 + lane];
            acc[k] = t;
          }
        }
        __syncthreads();
      }
      if (live && sub == 0) {
        float4* o = reinterpret_cast<float4*>(a.gx + ((size_t)j * C + c) * 16);
#pragma unroll
        for (int h = 0; h < 4; ++h) o[h] = make_float4(acc[4 * h], acc[4 * h + 1], acc[4 * h + 2], acc[4 * h + 3]);
      }
    }
  }
}

// Per path P for one channel: s_P and dY contribution; shared-weight path
// sums go to gw[P], radial ones to the workspace row of edge e and to gR.
template <int C, bool RADIAL, int P>
__device__ __forceinline__ void bwv_path(const BwdArgs& a, int c, int e, const float (&rk)[8],
                                         const float (&gv)[16], const float (&xv)[16], const float (&yv)[16],
                                         float (&dY)[16], float* gw, float (&gr)[8]) {
  constexpr tables::Path path = path_at(P);
  float s = 0.0f, dyp[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) dyp[k] = 0.0f;
  bs_terms<path.first>(gv, xv, yv, s, dyp, std::make_integer_sequence<int, path.count>{});
  const float wp = path_weight<C, RADIAL, P>(a, c, rk);
  constexpr int lo = path.l2 * path.l2, hi = (path.l2 + 1) * (path.l2 + 1);
#pragma unroll
  for (int k = lo; k < hi; ++k) dY[k] = fmaf(wp, dyp[k], dY[k]);
  if constexpr (RADIAL) {
    a.ws[(size_t)e * 34 * C + P * C + c] = s;
#pragma unroll
    for (int k = 0; k < 8; ++k) gr[k] = fmaf(__ldg(a.M + (size_t)k * 34 * C + P * C + c), s, gr[k]);
  } else {
    gw[P * C + c] += s;  // this group's row; (P, c) is written by one lane only
  }
}

template <int C, bool RADIAL, int... Ps>
__device__ __forceinline__ void bwv_all(const BwdArgs& a, int c, int e, const float (&rk)[8],
                                        const float (&gv)[16], const float (&xv)[16], const float (&yv)[16],
                                        float (&dY)[16], float* gw, float (&gr)[8],
                                        std::integer_sequence<int, Ps...>) {
  (bwv_path<C, RADIAL, Ps>(a, c, e, rk, gv, xv, yv, dY, gw, gr), ...);
}

// Sum over the G lanes of a node group (xor butterfly inside the group).
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o, G);
  return v;
}

template <int C, bool RADIAL>
__global__ void __launch_bounds__(128) k_bwd_wv(const BwdArgs a) {
  using K = BwdCfg<C, RADIAL>;
  const int grp = threadIdx.x / K::G, lane = threadIdx.x % K::G;
  // Shared weights: per-group partial dL/dw in shared memory [GROUPS][34][C].
  extern __shared__ float gws[];
  float* gw = gws + (size_t)grp * 34 * C;
  if constexpr (!RADIAL) {
    for (int i = threadIdx.x; i < K::GROUPS * 34 * C; i += blockDim.x) gws[i] = 0.0f;
    __syncthreads();
  }
  // Every lane of a warp runs the same number of edge iterations (the
  // group-sum shuffles need the whole warp): groups whose receiver has
  // fewer edges idle through the extra ones.
  // Radial weights (SPLIT > 1): the block's warps share a receiver and take
  // every SPLIT-th edge; each edge's outputs are its own.
  const int warp_groups = 32 / K::G;
  const int sub = K::SPLIT > 1 ? grp % K::SPLIT : 0;
  const int r_first = K::SPLIT > 1 ? blockIdx.x * K::NODES + grp / K::SPLIT
                                   : blockIdx.x * K::GROUPS + (grp / warp_groups) * warp_groups;
  const int r_step = K::SPLIT > 1 ? gridDim.x * K::NODES : gridDim.x * K::GROUPS;
  for (int rbase = r_first; rbase < a.N; rbase += r_step) {
    const int r = K::SPLIT > 1 ? rbase : rbase + grp % warp_groups;
    const bool live = r < a.N;
    const int a0 = live ? min(max(__ldg(a.off + r), 0), a.E) : 0;
    const int a1 = live ? max(a0, min(max(__ldg(a.off + r + 1), 0), a.E)) : 0;
    int deg = a1 - a0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) deg = max(deg, __shfl_xor_sync(0xffffffffu, deg, o));
    for (int t = sub; t < deg; t += K::SPLIT) {
      const int e = a0 + t;
      const bool on = e < a1;
      float dY[16], gr[8];
#pragma unroll
      for (int k = 0; k < 16; ++k) dY[k] = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) gr[k] = 0.0f;
      float vx = 0.0f, vy = 0.0f, vz = 0.0f;
      if (on) {
        const int j = __ldg(a.src + e);
        const float* v = a.vec + 3 * (size_t)e;
        vx = __ldg(v); vy = __ldg(v + 1); vz = __ldg(v + 2);
        if (j >= 0 && j < a.N_src) {
          float yv[16], rk[8];
          real_sh16(vx, vy, vz, yv);
          if constexpr (RADIAL) {
            const float4* rp = reinterpret_cast<const float4*>(a.R) + 2 * (size_t)e;
            const float4 r0 = __ldg(rp), r1 = __ldg(rp + 1);
            rk[0] = r0.x; rk[1] = r0.y; rk[2] = r0.z; rk[3] = r0.w;
            rk[4] = r1.x; rk[5] = r1.y; rk[6] = r1.z; rk[7] = r1.w;
          }
#pragma unroll 1
          for (int cc = 0; cc < K::CPL; ++cc) {
            const int c = lane + cc * K::G;
            float gv[16], xv[16];
            load16(a.g + ((size_t)r * C + c) * 16, gv);
            load16(a.x + ((size_t)j * C + c) * 16, xv);
            bwv_all<C, RADIAL>(a, c, e, rk, gv, xv, yv, dY, gw, gr,
                               std::make_integer_sequence<int, tables::kNumPaths>{});
          }
        } else if constexpr (RADIAL) {
#pragma unroll 1
          for (int cc = 0; cc < K::CPL; ++cc)
            for (int p = 0; p < 34; ++p) a.ws[(size_t)e * 34 * C + p * C + lane + cc * K::G] = 0.0f;
        }
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) dY[k] = group_sum<K::G>(dY[k]);
      if constexpr (RADIAL) {
#pragma unroll
        for (int k = 0; k < 8; ++k) gr[k] = group_sum<K::G>(gr[k]);
      }
      if (on && lane == 0) {
        if (a.gvec) {
          float ox, oy, oz;
          real_sh16_vjp(vx, vy, vz, dY, ox, oy, oz);
          a.gvec[3 * (size_t)e] = ox;
          a.gvec[3 * (size_t)e + 1] = oy;
          a.gvec[3 * (size_t)e + 2] = oz;
        }
        if constexpr (RADIAL) {
          if (a.gR) {
            float4* gp = reinterpret_cast<float4*>(a.gR) + 2 * (size_t)e;
            gp[0] = make_float4(gr[0], gr[1], gr[2], gr[3]);
            gp[1] = make_float4(gr[4], gr[5], gr[6], gr[7]);
          }
        }
      }
    }
  }
  if constexpr (!RADIAL) {
    // per-slot partial dL/dw (slot = block * GROUPS + group), summed over
    // slots in order by k_bwd_reduce_w
    __syncthreads();
    float* dstp = a.ws + (size_t)blockIdx.x * K::GROUPS * 34 * C;
    for (int i = threadIdx.x; i < K::GROUPS * 34 * C; i += blockDim.x) dstp[i] = gws[i];
  }
}

// Column sums of a [rows][cols] fp32 matrix (optionally weighted by a
// column of R), deterministic: block (32 columns x 16 row partitions); thread
// (x, y) sums rows y, y+16, ... of column x in order, then the 16 partials
// are added in partition order.
constexpr int kRedX = 32, kRedY = 16;

// dL/dw[i] = sum over slots k of ws[k][i], i = p*C + c (34*C columns).
__global__ void __launch_bounds__(kRedX* kRedY) k_bwd_reduce_w(const float* ws, int slots, int cols, float* gw) {
  __shared__ float part[kRedY][kRedX];
  const int col = blockIdx.x * kRedX + threadIdx.x;
  float s = 0.0f;
  if (col < cols)
    for (int k = threadIdx.y; k < slots; k += kRedY) s += ws[(size_t)k * cols + col];
  part[threadIdx.y][threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.y == 0 && col < cols) {
    float t = 0.0f;
#pragma unroll
    for (int y = 0; y < kRedY; ++y) t += part[y][threadIdx.x];
    gw[col] = t;
  }
}

// dL/dM[k][col] = sum over this call's edges e of R[e][k] S[e][col], in two
// fixed-order stages.  Stage 1 (k_bwd_partial_M): the edge range
// [off[0], off[N]) (read on the device, clamped) is cut into kRmChunks
// equal chunks; block (column tile, chunk) has thread (x, y) sum the edges
// y, y+16, ... of its chunk for column x and all 8 k at once (each S entry
// is read once), then the 16 partials are added in y order and written to
// part[chunk][k][col].  Stage 2 (k_bwd_reduce_w over kRmChunks slots)
// adds the chunks in order.  An empty range gives zeros.
constexpr int kRmChunks = 16;

__global__ void __launch_bounds__(kRedX* kRedY) k_bwd_partial_M(const float* __restrict__ R,
                                                               const float* __restrict__ S,
                                                               const int32_t* __restrict__ off, int N, int E,
                                                               int cols, float* __restrict__ part) {
  __shared__ float red[kRedY][8][kRedX];
  const int col = blockIdx.x * kRedX + threadIdx.x;
  const int chunk = blockIdx.y;
  const int e0 = min(max(__ldg(off), 0), E);
  const int e1 = max(e0, min(max(__ldg(off + N), 0), E));
  const long long span = e1 - e0;
  const int c0 = e0 + (int)(span * chunk / kRmChunks), c1 = e0 + (int)(span * (chunk + 1) / kRmChunks);
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
  if (col < cols) {
    for (int e = c0 + threadIdx.y; e < c1; e += kRedY) {
      const float sv = __ldg(S + (size_t)e * cols + col);
      const float4 r0 = __ldg(reinterpret_cast<const float4*>(R) + 2 * (size_t)e);
      const float4 r1 = __ldg(reinterpret_cast<const float4*>(R) + 2 * (size_t)e + 1);
      acc[0] = fmaf(r0.x, sv, acc[0]); acc[1] = fmaf(r0.y, sv, acc[1]);
      acc[2] = fmaf(r0.z, sv, acc[2]); acc[3] = fmaf(r0.w, sv, acc[3]);
      acc[4] = fmaf(r1.x, sv, acc[4]); acc[5] = fmaf(r1.y, sv, acc[5]);
      acc[6] = fmaf(r1.z, sv, acc[6]); acc[7] = fmaf(r1.w, sv, acc[7]);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) red[threadIdx.y][k][threadIdx.x] = acc[k];
  __syncthreads();
  if (threadIdx.y < 8 && col < cols) {  // thread (x, k) adds the 16 partials of (k, col) in order
    const int k = threadIdx.y;
    float t = 0.0f;
#pragma unroll
    for (int y = 0; y < kRedY; ++y) t += red[y][k][threadIdx.x];
    part[((size_t)chunk * 8 + k) * cols + col] = t;
  }
}

}  // namespace eqmp
