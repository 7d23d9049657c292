// Fused SH + CG tensor product + receiver sum, per-edge radial weights.
//
//   out[i,c,k3] = sum_{e->i} sum_p W[e,p,c] sum_{k1,k2} C_p[k3,k1,k2] x[src_e,c,k1] Y_e[k2]
//   W[e,p,c]    = sum_{k<8} R[e,k] M[k, p*C + c]
//
// With per-edge weights the edge sum cannot be taken before the
// contraction, so every edge does the full tensor product (Batmobile blog
// "Batmobile CUDA内核优化", section "3. 操作融合": SH in registers, gather of
// the sender's row, tensor product in registers, one write per output).
//
// Mapping: a group of C threads owns one receiver at a time, thread = channel.
// Per edge each thread evaluates the 16 SH (registers), reads its 16
// features (the group reads the 16*C-element row contiguously), forms the
// 34 weights from R (broadcast) and M (L1-resident), and applies the 611 CG
// terms with compile-time coefficients.  Accumulation is in registers in
// CSR order; one store per output row.  No shared memory, no waits.
#pragma once

#include "common.cuh"
#include "layer_args.cuh"

namespace eqmp {

template <int I>
__device__ __forceinline__ void radial_term(const float (&xv)[16], const float (&yv)[16],
                                            float (&tmp)[16]) {
  constexpr tables::Term t = term_at(I);
  tmp[t.k3] = fmaf(t.c * xv[t.k1], yv[t.k2], tmp[t.k3]);
}

template <int First, int... Is>
__device__ __forceinline__ void radial_terms(const float (&xv)[16], const float (&yv)[16],
                                             float (&tmp)[16], std::integer_sequence<int, Is...>) {
  (radial_term<First + Is>(xv, yv, tmp), ...);
}

template <int C, int P>
__device__ __forceinline__ void radial_path(const float (&xv)[16], const float (&yv)[16],
                                            const float (&rk)[8], const float* __restrict__ Mc,
                                            float (&o)[16]) {
  constexpr tables::Path path = path_at(P);
  float wp = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) wp = fmaf(rk[k], __ldg(Mc + (size_t)k * 34 * C + P * C), wp);
  float tmp[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) tmp[k] = 0.0f;
  radial_terms<path.first>(xv, yv, tmp, std::make_integer_sequence<int, path.count>{});
  constexpr int lo = path.l3 * path.l3, hi = (path.l3 + 1) * (path.l3 + 1);
#pragma unroll
  for (int k = lo; k < hi; ++k) o[k] = fmaf(wp, tmp[k], o[k]);
}

template <int C, int... Ps>
__device__ __forceinline__ void radial_all(const float (&xv)[16], const float (&yv)[16],
                                           const float (&rk)[8], const float* Mc, float (&o)[16],
                                           std::integer_sequence<int, Ps...>) {
  (radial_path<C, Ps>(xv, yv, rk, Mc, o), ...);
}

template <typename XT>
__device__ __forceinline__ void load_row16(const void* x, size_t elem, float (&xv)[16]) {
  if constexpr (sizeof(XT) == 4) {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + elem);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float4 v = __ldg(p + h);
      xv[4 * h] = v.x; xv[4 * h + 1] = v.y; xv[4 * h + 2] = v.z; xv[4 * h + 3] = v.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(x) + elem);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 v = __ldg(p + h);
      xv[8 * h + 0] = bf16_lo(v.x); xv[8 * h + 1] = bf16_hi(v.x);
      xv[8 * h + 2] = bf16_lo(v.y); xv[8 * h + 3] = bf16_hi(v.y);
      xv[8 * h + 4] = bf16_lo(v.z); xv[8 * h + 5] = bf16_hi(v.z);
      xv[8 * h + 6] = bf16_lo(v.w); xv[8 * h + 7] = bf16_hi(v.w);
    }
  }
}

template <typename XT>
__device__ __forceinline__ void store_row16(void* out, size_t elem, const float (&o)[16]) {
  if constexpr (sizeof(XT) == 4) {
    float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + elem);
#pragma unroll
    for (int h = 0; h < 4; ++h) p[h] = make_float4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]);
  } else {
    uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + elem);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 v;
      v.x = pack_bf16x2(o[8 * h + 0], o[8 * h + 1]); v.y = pack_bf16x2(o[8 * h + 2], o[8 * h + 3]);
      v.z = pack_bf16x2(o[8 * h + 4], o[8 * h + 5]); v.w = pack_bf16x2(o[8 * h + 6], o[8 * h + 7]);
      p[h] = v;
    }
  }
}

constexpr int kRadialThreads = 128;

template <int C, typename XT, bool FROM_VEC>
__global__ void __launch_bounds__(C > kRadialThreads ? C : kRadialThreads)
    k_radial(const LayerArgs a) {
  constexpr int NT = C > kRadialThreads ? C : kRadialThreads;
  constexpr int GROUPS = NT / C;
  const int g = threadIdx.x / C, c = threadIdx.x % C;
  const float* Mc = a.M + c;
  for (int r = blockIdx.x * GROUPS + g; r < a.N; r += gridDim.x * GROUPS) {
    const int a0 = min(max(__ldg(a.off + r), 0), a.E);
    const int a1 = min(max(__ldg(a.off + r + 1), 0), a.E);
    float o[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = 0.0f;
    for (int e = a0; e < a1; ++e) {
      const int node = __ldg(a.src + e);
      if (node < 0 || node >= a.N_src) continue;  // out-of-range sender reads as zero
      float yv[16];
      if constexpr (FROM_VEC) {
        const float* v = a.vec + 3 * (size_t)e;
        real_sh16(__ldg(v), __ldg(v + 1), __ldg(v + 2), yv);
      } else {
        const float4* yp = reinterpret_cast<const float4*>(a.Y) + 4 * (size_t)e;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float4 t = __ldg(yp + h);
          yv[4 * h] = t.x; yv[4 * h + 1] = t.y; yv[4 * h + 2] = t.z; yv[4 * h + 3] = t.w;
        }
      }
      float xv[16];
      load_row16<XT>(a.x, ((size_t)node * C + c) * 16, xv);
      float rk[8];
      const float4* rp = reinterpret_cast<const float4*>(a.R) + 2 * (size_t)e;
      const float4 r0 = __ldg(rp), r1 = __ldg(rp + 1);
      rk[0] = r0.x; rk[1] = r0.y; rk[2] = r0.z; rk[3] = r0.w;
      rk[4] = r1.x; rk[5] = r1.y; rk[6] = r1.z; rk[7] = r1.w;
      radial_all<C>(xv, yv, rk, Mc, o, std::make_integer_sequence<int, tables::kNumPaths>{});
    }
    store_row16<XT>(a.out, ((size_t)r * C + c) * 16, o);
  }
}

}  // namespace eqmp
