// Gradients of the weights and of the edge vectors for shared weights, in
// the fused forward kernel's schedule.
//
// With g = dL/dout and W[e,p,c] = w[p,c] the chain rule gives
//   dw[p,c]   = sum_i sum_{k3,k1,k2} C_p[k3,k1,k2] g[i,c,k3] A[i,c,k1,k2],
//               A[i,c,k1,k2] = sum_{e -> i} x[src_e,c,k1] Y_e[k2]   (the forward's sums)
//   dY[e,k2]  = sum_c sum_k1 x[src_e,c,k1] H[i,c,k1,k2],
//               H[i,c,k1,k2] = sum_p w[p,c] sum_k3 C_p[k3,k1,k2] g[i,c,k3]
//   dvec[e]   = dY[e,:] . dY(vec_e)/dvec_e
// so per receiver i the kernel forms H once (from g[i] and w), and per edge
// it adds x (x) Y into A (as the forward does) and x . H into the edge's dY,
// both with the paired FP32 FMA.  dY of an edge is summed over all consumer
// threads: a reduce-scatter inside each warp (16 values over 32 lanes), then
// the warps' partials go to the slot's entry of a shared-memory dY ring.
// The producer lane that next claims the slot has just seen the edge
// released, so it finishes that edge first: the sum over warps and the
// harmonics' derivative (the last S edges are finished at the end).  The
// consumers never wait on it.  At the end of a receiver the thread
// contracts its A with g into per-path partial dw (in shared memory, one
// entry per thread and path); at the end of the CTA the partials of the four
// k1 quads are added (fixed order) into one workspace row per CTA, which the
// fixed-order column sum turns into dw.
//
// Pipeline, slot ownership, parity waits, tail and watchdog are the fused
// forward kernel's (k_shared.cuh): the producer warpgroup gathers x[src]
// rows by TMA into an S-slot ring and writes the edge harmonics into the SH
// ring; the consumers run two edges ahead.  Thread (c, q) owns k1 in
// [4q, 4q + 4) of channel c (KQ = 4 for every C, so A and H fit together).
#pragma once

#include "k_bwd.cuh"
#include "k_shared.cuh"

namespace eqmp {

// KQ_ k1 values per thread; DW: accumulate A and form dw; DV: form H and
// each edge's dY (dvec).  Both at KQ = 4 (A and H fit together), or one of
// them at KQ = 8 (a kernel each, half the threads in every dY reduction).
template <int C, int KQ_ = 4, bool DW = true, bool DV = true>
struct BwdSwCfg {
  using B = SharedCfg<C, KQ_, float, true>;
  static constexpr int KQ = KQ_, NQ = B::NQ, NCONS = B::NCONS, NCW = B::NCW;
  static constexpr bool WS = B::WS;
  static_assert(WS, "the shared-weight gradient kernel is warp-specialised (C >= 32)");
  static_assert(DW || DV, "nothing to compute");
  static_assert(KQ == 4 || !(DW && DV), "A and H together fit only at KQ = 4");
  static constexpr int CONS0 = B::CONS0, NTHREADS = B::NTHREADS, MIN_BLOCKS = B::MIN_BLOCKS;
  static constexpr int RP = B::RP, RC = B::RC, NP = B::NP, YR = B::YR, ROWS = B::ROWS;
  static constexpr int ROW_BYTES = B::ROW_BYTES, SLOT = B::SLOT, XBYTES = B::XBYTES;
  // shared memory: x slots, SH ring, dY ring [S][NCW][16] (one entry per
  // slot; DV), per-thread dw partials [NQ][34][C] (DW), weights [34][C]
  // (DV), barriers
  static constexpr int FIXED_NO_S = YR * 64 + (DW ? NQ * 34 * C * 4 : 0) + (DV ? 34 * C * 4 : 0) + 1024 + 1024;
  static constexpr int PER_SLOT = SLOT + (DV ? NCW * 16 * 4 : 0) + 2 * 8;
  static constexpr int S_FIT = (227 * 1024 / MIN_BLOCKS - FIXED_NO_S) / PER_SLOT;
  static constexpr int S = S_FIT >= 32 ? 32 : S_FIT >= 16 ? 16 : S_FIT >= 8 ? 8 : 4;
  static_assert(S_FIT >= 4, "not even four slots fit");
  static constexpr int OFF_X = 0;
  static constexpr int OFF_Y = OFF_X + S * SLOT;
  static constexpr int OFF_DY = OFF_Y + YR * 64;
  static constexpr int OFF_DW = OFF_DY + (DV ? S * NCW * 16 * 4 : 0);
  static constexpr int OFF_W = OFF_DW + (DW ? NQ * 34 * C * 4 : 0);
  static constexpr int OFF_BAR = OFF_W + (DV ? 34 * C * 4 : 0);
  static constexpr int SMEM_BYTES = OFF_BAR + 2 * S * 8 + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// ---- per-receiver H from g[i] and w: H[k1][k2] over the quad's k1 --------
template <int KQ, int Q, int I>
__device__ __forceinline__ void h_term(const float (&gp)[16], float2 (&H)[KQ][8]) {
  constexpr tables::Term t = term_at(I);
  if constexpr (t.k1 >= Q * KQ && t.k1 < Q * KQ + KQ) {
    constexpr int i = t.k1 - Q * KQ;
    if constexpr (t.k2 & 1)
      H[i][t.k2 >> 1].y = fmaf(t.c, gp[t.k3], H[i][t.k2 >> 1].y);
    else
      H[i][t.k2 >> 1].x = fmaf(t.c, gp[t.k3], H[i][t.k2 >> 1].x);
  }
}
template <int KQ, int Q, int First, int... Is>
__device__ __forceinline__ void h_terms(const float (&gp)[16], float2 (&H)[KQ][8], std::integer_sequence<int, Is...>) {
  (h_term<KQ, Q, First + Is>(gp, H), ...);
}
// Bit k3 set when path P has a term from the quad's k1 to output k3 (a
// compile-time constant: the tables are host constants, never read at run
// time on the device).
constexpr unsigned path_mask(int P, int k1lo, int n) {
  unsigned m = 0;
  for (int k3 = 0; k3 < 16; ++k3)
    if (path_has(P, k1lo, n, k3)) m |= 1u << k3;
  return m;
}

// gp[k3] = w[p,c] g[k3] over the outputs the path reaches from this quad
template <int C, int KQ, int Q, int P>
__device__ __forceinline__ void h_path(const float (&g)[16], const float* wcol, float2 (&H)[KQ][8]) {
  if constexpr (path_touches(P, Q * KQ, KQ)) {
    constexpr tables::Path path = path_at(P);
    constexpr unsigned mask = path_mask(P, Q * KQ, KQ);
    const float w = wcol[P * C];
    float gp[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) gp[k] = ((mask >> k) & 1u) ? w * g[k] : 0.0f;
    h_terms<KQ, Q, path.first>(gp, H, std::make_integer_sequence<int, path.count>{});
  }
}
template <int C, int KQ, int Q, int... Ps>
__device__ __forceinline__ void h_quad(const float (&g)[16], const float* wcol, float2 (&H)[KQ][8],
                                       std::integer_sequence<int, Ps...>) {
  (h_path<C, KQ, Q, Ps>(g, wcol, H), ...);
}

// ---- end of receiver: dw partials += sum_k3 g[k3] sum_{k1,k2} C A ---------
template <int KQ, int Q, int I>
__device__ __forceinline__ void dw_term(const float2 (&acc)[KQ][8], float (&tmp)[16]) {
  constexpr tables::Term t = term_at(I);
  if constexpr (t.k1 >= Q * KQ && t.k1 < Q * KQ + KQ) {
    constexpr int i = t.k1 - Q * KQ;
    const float a = (t.k2 & 1) ? acc[i][t.k2 >> 1].y : acc[i][t.k2 >> 1].x;
    tmp[t.k3] = fmaf(t.c, a, tmp[t.k3]);
  }
}
template <int KQ, int Q, int First, int... Is>
__device__ __forceinline__ void dw_terms(const float2 (&acc)[KQ][8], float (&tmp)[16],
                                         std::integer_sequence<int, Is...>) {
  (dw_term<KQ, Q, First + Is>(acc, tmp), ...);
}
template <int KQ, int Q, int P, int... K3>
__device__ __forceinline__ float dw_dot(const float (&g)[16], const float (&tmp)[16], std::integer_sequence<int, K3...>) {
  constexpr unsigned mask = path_mask(P, Q * KQ, KQ);
  float s = 0.0f;
  ((((mask >> K3) & 1u) ? (void)(s = fmaf(g[K3], tmp[K3], s)) : (void)0), ...);
  return s;
}
template <int C, int KQ, int Q, int P>
__device__ __forceinline__ void dw_path(const float2 (&acc)[KQ][8], const float (&g)[16], float* dwp) {
  if constexpr (path_touches(P, Q * KQ, KQ)) {
    constexpr tables::Path path = path_at(P);
    float tmp[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) tmp[k] = 0.0f;
    dw_terms<KQ, Q, path.first>(acc, tmp, std::make_integer_sequence<int, path.count>{});
    dwp[P * C] += dw_dot<KQ, Q, P>(g, tmp, std::make_integer_sequence<int, 16>{});
  }
}
template <int C, int KQ, int Q, int... Ps>
__device__ __forceinline__ void dw_quad(const float2 (&acc)[KQ][8], const float (&g)[16], float* dwp,
                                        std::integer_sequence<int, Ps...>) {
  (dw_path<C, KQ, Q, Ps>(acc, g, dwp), ...);
}

// q-dispatch of a quad template (NQ = 16 / KQ quads per channel).
template <int KQ, typename F>
__device__ __forceinline__ void on_quad(int q, F&& f) {
  if constexpr (KQ == 4) {
    switch (q) {
      case 0: f(std::integral_constant<int, 0>{}); break;
      case 1: f(std::integral_constant<int, 1>{}); break;
      case 2: f(std::integral_constant<int, 2>{}); break;
      default: f(std::integral_constant<int, 3>{}); break;
    }
  } else {
    if (q == 0) f(std::integral_constant<int, 0>{});
    else f(std::integral_constant<int, 1>{});
  }
}

template <int C, int KQ_ = 4, bool DW = true, bool DV = true>
__global__ void __launch_bounds__(BwdSwCfg<C, KQ_, DW, DV>::NTHREADS, BwdSwCfg<C, KQ_, DW, DV>::MIN_BLOCKS)
    k_bwd_sw(const __grid_constant__ CUtensorMap tmap, const BwdArgs a, int* watchdog) {
  using K = BwdSwCfg<C, KQ_, DW, DV>;
  constexpr int S = K::S, KQ = K::KQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align<1024>(smem_raw);
  float4* ys = reinterpret_cast<float4*>(smem + K::OFF_Y);
  float* dyr = reinterpret_cast<float*>(smem + K::OFF_DY);  // [S][NCW][16]
  float* dwq = reinterpret_cast<float*>(smem + K::OFF_DW);  // [NQ][34][C]
  float* ws = reinterpret_cast<float*>(smem + K::OFF_W);
  const uint32_t full0 = smem_u32(smem + K::OFF_BAR);
  const uint32_t empty0 = full0 + 8 * S;
  const int tid = threadIdx.x;

  const int4 rr = balanced_range_off(a.off, a.N, gridDim.x, blockIdx.x, kReceiverCost);
  const int r_begin = rr.x, r_end = rr.y;
  if (tid < S) {
    mbar_init(full0 + 8 * tid, 1);
    mbar_init(empty0 + 8 * tid, K::NCONS);
    fence_mbar_init();
  }
  __syncthreads();
  const int e_begin = min(max(rr.z, 0), a.E);
  const int e_end = max(e_begin, min(max(rr.w, 0), a.E));
  const int total = e_end - e_begin;

  if (tid < K::CONS0) {
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<K::RP>();
    constexpr int CH = S / K::NP;
    static_assert(CH >= 1 && 32 % CH == 0 && K::YR >= 32 * K::NP + S, "producer layout");
    const int pw = tid >> 5, lane = tid & 31;
    if (pw >= K::NP) return;
    if (lane == 0 && pw == 0) prefetch_tmap(&tmap);
    auto ordinal = [&](int g) {
      return (uint32_t)((pw + K::NP * (g * (32 / CH) + lane / CH)) * CH + lane % CH);
    };
    auto load_edge = [&](uint32_t n, int& node, float& vx, float& vy, float& vz) {
      node = 0; vx = vy = vz = 0.0f;
      if (n < (uint32_t)total) {
        const int e = e_begin + (int)n;
        node = __ldg(a.src + e);
        const float* v = a.vec + 3 * (size_t)e;
        vx = __ldg(v); vy = __ldg(v + 1); vz = __ldg(v + 2);
      }
    };
    // dvec of ordinal m from the consumers' partials, once m is released
    // (its dY entry is rewritten only by ordinal m + S, issued after this)
    auto finish = [&](uint32_t m) {
      const float* p = dyr + (size_t)(m % S) * K::NCW * 16;
      float d[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) d[k] = 0.0f;
#pragma unroll
      for (int w = 0; w < K::NCW; ++w) {
        const float4* q = reinterpret_cast<const float4*>(p + w * 16);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float4 v = q[h];
          d[4 * h] += v.x; d[4 * h + 1] += v.y; d[4 * h + 2] += v.z; d[4 * h + 3] += v.w;
        }
      }
      const int e = e_begin + (int)m;
      const float* v = a.vec + 3 * (size_t)e;
      float ox, oy, oz;
      real_sh16_vjp(__ldg(v), __ldg(v + 1), __ldg(v + 2), d, ox, oy, oz);
      a.gvec[3 * (size_t)e] = ox;
      a.gvec[3 * (size_t)e + 1] = oy;
      a.gvec[3 * (size_t)e + 2] = oz;
    };
    const bool want_vec = DV && a.gvec != nullptr;
    bool ok = true;
    int node_nx;
    float vx_nx, vy_nx, vz_nx;
    load_edge(ordinal(0), node_nx, vx_nx, vy_nx, vz_nx);
    uint32_t last = 0;
    for (int g = 0; ok; ++g) {
      const uint32_t n = ordinal(g);
      const uint32_t cnt = (uint32_t)__popc(__ballot_sync(0xffffffffu, n < (uint32_t)total));
      if (cnt == 0) break;
      const int node = node_nx;
      float4* yd = ys + 4 * (n % K::YR);
      {
        float y[16];
        real_sh16(vx_nx, vy_nx, vz_nx, y);
        yd[0] = make_float4(y[0], y[1], y[2], y[3]);
        yd[1] = make_float4(y[4], y[5], y[6], y[7]);
        yd[2] = make_float4(y[8], y[9], y[10], y[11]);
        yd[3] = make_float4(y[12], y[13], y[14], y[15]);
      }
      load_edge(ordinal(g + 1), node_nx, vx_nx, vy_nx, vz_nx);
      for (uint32_t j = 0; j < cnt; ++j) {
        int good = 1;
        if ((uint32_t)lane == j) {
          const uint32_t s = n % S, par = ((n / S) & 1u) ^ 1u;
          if (mbar_try_wait(empty0 + 8 * s, par) || mbar_wait(empty0 + 8 * s, par, watchdog, 2)) {
            if (want_vec && n >= (uint32_t)S) finish(n - S);  // the slot's previous edge
            mbar_arrive_expect_tx(full0 + 8 * s, K::ROW_BYTES);
            tma_load_2d(smem_u32(smem + K::OFF_X + s * K::SLOT), &tmap, 0, node * K::ROWS, full0 + 8 * s);
          } else {
            good = 0;
          }
        }
        if (!__all_sync(0xffffffffu, good)) { ok = false; break; }
      }
      if (!ok) break;
      last = __shfl_sync(0xffffffffu, n, (int)cnt - 1) + 1;
    }
#pragma unroll
    for (uint32_t t = 0; t < kLookAhead; ++t) {
      const uint32_t n = (uint32_t)total + t;
      if (ok && pw == (int)((n / CH) % K::NP)) {
        if (lane == 0) {
          const uint32_t s = n % S, par = ((n / S) & 1u) ^ 1u;
          if (mbar_try_wait(empty0 + 8 * s, par) || mbar_wait(empty0 + 8 * s, par, watchdog, 2))
            mbar_arrive(full0 + 8 * s);
        }
        last = n + 1;
      }
    }
    // Drain: this warp's real ordinals among the last S wait for their
    // release (so their loads have landed and their dY partials are
    // complete), then get their dvec.  Each was issued after its slot's
    // previous ordinal was released, so every parity wait here is for the
    // current phase.
    if (ok) {
      const uint32_t first = (uint32_t)total > (uint32_t)S ? (uint32_t)total - S : 0u;
      for (uint32_t i0 = first; i0 < (uint32_t)total; i0 += 32) {
        const uint32_t i = i0 + lane;
        bool mine = i < (uint32_t)total && (i / CH) % K::NP == (uint32_t)pw;
        if (mine) {
          if (!mbar_wait(empty0 + 8 * (i % S), (i / S) & 1u, watchdog, 3)) mine = false;
          else if (want_vec) finish(i);
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  setmaxnreg_inc<K::RC>();
  const int ct = tid - K::CONS0;
  const int c = ct % C, q = ct / C, lane = tid & 31, cw = ct >> 5;
  if constexpr (DV) {
    constexpr int PER = (34 * C + K::NCONS - 1) / K::NCONS;
    float wv[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = ct + k * K::NCONS;
      wv[k] = i < 34 * C ? __ldg(a.w + i) : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = ct + k * K::NCONS;
      if (i < 34 * C) ws[i] = wv[k];
    }
  }
  auto load_off = [&](int base) {
    const int i = base + lane;
    return i <= r_end ? min(max(__ldg(a.off + i), 0), a.E) : a.E;
  };
  int chunk = r_begin;
  int off_cur = load_off(chunk);
  int off_nxt = load_off(chunk + 32);
  named_barrier(2, K::NCONS);
  const uint32_t xlog = (uint32_t)(c * 16 * 4 + q * K::XBYTES);
  const uint32_t xo[2] = {swz128(xlog), swz128(xlog + 16)};
  const float* wcol = ws + c;
  uint32_t n = 0;
  bool failed = false;
  float* dwp = dwq + (size_t)q * 34 * C + c;  // this thread's partials, path p at dwp[p * C]
  if constexpr (DW) {
#pragma unroll
    for (int p = 0; p < 34; ++p) dwp[p * C] = 0.0f;
  }

  auto full_bar = [&](uint32_t m) { return full0 + 8 * (m % S); };
  auto full_par = [&](uint32_t m) { return (m / S) & 1u; };
  auto wait_full = [&](uint32_t m) {
    if (!mbar_try_wait(full_bar(m), full_par(m)))
      if (!mbar_wait_slow(full_bar(m), full_par(m), watchdog, 1, failed)) failed = true;
  };
  auto load_edge = [&](uint32_t m, float2 (&yv)[8], float (&xv)[KQ]) {
    const float4* yp = ys + 4 * (m % K::YR);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float4 t = yp[h];
      yv[2 * h] = make_float2(t.x, t.y);
      yv[2 * h + 1] = make_float2(t.z, t.w);
    }
    load_x<float, KQ>(smem + K::OFF_X + (m % S) * K::SLOT, xo, xv);
  };
  // One edge: A += x (x) Y; dY partial = x . H, summed over the warp
  // (reduce-scatter: lane l ends with value l >> 1), into the dY ring;
  // then release the slot.
  auto edge = [&](float2 (&acc)[KQ][8], const float2 (&H)[KQ][8], uint32_t m, const float2 (&yv)[8],
                  const float (&xv)[KQ]) {
    if constexpr (DW) fma_edge<KQ>(acc, yv, xv);
    if constexpr (!DV) {
      mbar_arrive(empty0 + 8 * (m % S));
      return;
    }
    float2 dy[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) dy[k] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < KQ; ++i) {
      const float2 xx = make_float2(xv[i], xv[i]);
#pragma unroll
      for (int k = 0; k < 8; ++k) dy[k] = __ffma2_rn(xx, H[i][k], dy[k]);
    }
    float v[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) { v[2 * k] = dy[k].x; v[2 * k + 1] = dy[k].y; }
    // halving steps: keep the upper half when the lane bit is set
#pragma unroll
    for (int o = 16, h = 8; o >= 2; o >>= 1, h >>= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < h; ++i) {
        const float send = up ? v[i] : v[i + h];
        const float keep = up ? v[i + h] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    if ((lane & 1) == 0) dyr[((size_t)(m % S) * K::NCW + cw) * 16 + (lane >> 1)] = v[0];
    mbar_arrive(empty0 + 8 * (m % S));
  };
  float2 yA[8], yB[8];
  float xA[KQ], xB[KQ];
  wait_full(0);
  load_edge(0, yA, xA);
  wait_full(1);
  load_edge(1, yB, xB);
  for (int r = r_begin; r < r_end; ++r) {
    if (r - chunk == 32) {
      chunk += 32;
      off_cur = off_nxt;
      off_nxt = load_off(chunk + 32);
    }
    const int j0 = r - chunk;
    const int a0 = __shfl_sync(0xffffffffu, off_cur, j0);
    const int a1n = __shfl_sync(0xffffffffu, off_cur, (j0 + 1) & 31);
    const int a1x = __shfl_sync(0xffffffffu, off_nxt, 0);
    const int a1 = j0 == 31 ? a1x : a1n;
    const int deg = min(max(a1 - a0, 0), total - (int)n);
    // g[r, c, :] (read again at the end of the receiver) and H
    const float4* grow = reinterpret_cast<const float4*>(a.g + ((size_t)r * C + c) * 16);
    auto load_g = [&](float (&g)[16]) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float4 t = __ldg(grow + h);
        g[4 * h] = t.x; g[4 * h + 1] = t.y; g[4 * h + 2] = t.z; g[4 * h + 3] = t.w;
      }
    };
    float g[16];
    float2 H[KQ][8];
    using Seq = std::make_integer_sequence<int, tables::kNumPaths>;
    if constexpr (DV) {
      load_g(g);
#pragma unroll
      for (int i = 0; i < KQ; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) H[i][k] = make_float2(0.0f, 0.0f);
      on_quad<KQ>(q, [&](auto Qc) { h_quad<C, KQ, decltype(Qc)::value>(g, wcol, H, Seq{}); });
    }
    float2 acc[KQ][8];
    if constexpr (DW) {
#pragma unroll
      for (int i = 0; i < KQ; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[i][k] = make_float2(0.0f, 0.0f);
    }
    int j = 0;
    for (; j + 2 <= deg; j += 2, n += 2) {
      {
        const bool ready = mbar_test_wait(full_bar(n + 2), full_par(n + 2));
        edge(acc, H, n, yA, xA);
        if (!ready) wait_full(n + 2);
        load_edge(n + 2, yA, xA);
      }
      {
        const bool ready = mbar_test_wait(full_bar(n + 3), full_par(n + 3));
        edge(acc, H, n + 1, yB, xB);
        if (!ready) wait_full(n + 3);
        load_edge(n + 3, yB, xB);
      }
    }
    if (j < deg) {
      const bool ready = mbar_test_wait(full_bar(n + 2), full_par(n + 2));
      edge(acc, H, n, yA, xA);
#pragma unroll
      for (int k = 0; k < 8; ++k) yA[k] = yB[k];
#pragma unroll
      for (int i = 0; i < KQ; ++i) xA[i] = xB[i];
      if (!ready) wait_full(n + 2);
      load_edge(n + 2, yB, xB);
      ++n;
    }
    if constexpr (DW) {
      load_g(g);
      on_quad<KQ>(q, [&](auto Qc) { dw_quad<C, KQ, decltype(Qc)::value>(acc, g, dwp, Seq{}); });
    }
  }
  if constexpr (!DW) return;
  // quad partials -> one workspace row [34][C] per CTA, quads added in order
  named_barrier(1, K::NCONS);
  float* row = a.ws + (size_t)blockIdx.x * 34 * C;
  for (int i = ct; i < 34 * C; i += K::NCONS) {
    float s = 0.0f;
#pragma unroll
    for (int qq = 0; qq < K::NQ; ++qq) s += dwq[(size_t)qq * 34 * C + i];
    row[i] = s;
  }
}

}  // namespace eqmp
