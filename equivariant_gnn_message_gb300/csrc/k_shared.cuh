// Fused SH + CG tensor product + receiver sum, shared per-path weights.
//
// What it computes (Batmobile blog "Batmobile CUDA内核优化", section
// "3. 操作融合", extended with the receiver sum):
//   out[i,c,k3] = sum_p w[p,c] sum_{k1,k2} C_p[k3,k1,k2] sum_{e->i} x[src_e,c,k1] Y_e[k2]
// Because the weights do not depend on the edge, the edge sum is taken
// first: A[c,k1,k2] = sum_{e->i} x[src_e,c,k1] Y_e[k2] (256 FMAs per edge
// and channel), then contracted once per receiver with the 611 CG terms and
// the 34 path weights.  The result is the same sum in another order.
//
// Organisation of one CTA (persistent; owns a contiguous receiver range,
// balanced on edges plus a per-receiver cost):
//   * producer warps: for their edges, in CSR order, compute the 16 SH in
//     registers (or read them, for the unfused tp_scatter entry point),
//     store them in an SH ring and issue ONE TMA tensor load of the sender's
//     feature row x[src] (C*16 elements) per edge into a ring slot, with
//     128-byte swizzle.  The ring's slots come in pairs, each pair with one
//     full and one empty mbarrier.
//   * consumer warps: thread (c, q) holds A[c, q*KQ .. q*KQ+KQ-1, 0..15] in
//     registers.  Per edge: 4 broadcast LDS.128 of Y, conflict-free swizzled
//     LDS of x, KQ*8 paired FFMAs; per pair of edges: one wait, one release.
//     At the end of a receiver: contraction with compile-time CG constants,
//     partial sums over the NQ quads through shared memory, one store per
//     output.
//   * the receiver sum is in CSR order, deterministic, with no atomics.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "layer_args.cuh"

namespace eqmp {

// Tuning: thread (c, q) owns KQ values of k1 (8 from C = 64: 128
// accumulators; 4 below).  When the consumer warps fill whole warpgroups the
// CTA is warp-specialised: warpgroup 0 is the producer (one active warp) and
// gives registers away with setmaxnreg, the consumer warpgroups take them.
// The EQMP_TUNE_* macros override the defaults for experiments with a
// separately built library.
template <int C, typename XT>
struct SharedTune {
#ifdef EQMP_TUNE_KQ
  static constexpr int KQ = C >= 64 ? EQMP_TUNE_KQ : 4;
#else
  static constexpr int KQ = C >= 64 ? 8 : 4;
#endif
#ifdef EQMP_TUNE_S
  static constexpr int S_MAX = EQMP_TUNE_S;
#else
  // Slots in flight hide the row-gather latency (Little's law: about
  // 16 x 4 KB per CTA at two CTAs per SM); capped by the shared-memory budget.
  static constexpr int S_MAX = 32;
#endif
};

template <int C, int KQ, typename XT, bool FROM_VEC>
struct SharedCfg {
  static constexpr int NQ = 16 / KQ;                 // quads of k1 per channel
  static constexpr int NCONS = C * NQ;               // consumer threads
  static constexpr int NCW = NCONS / 32;             // consumer warps
  static constexpr bool WS = NCW % 4 == 0;           // warp-specialised with setmaxnreg
  static constexpr int CONS0 = WS ? 128 : 0;         // first consumer thread
  static constexpr int NTHREADS = WS ? 128 + NCONS : NCONS + 32;
#ifdef EQMP_TUNE_MINB
  static constexpr int MIN_BLOCKS = WS ? (NCONS >= 256 ? 1 : KQ == 4 ? EQMP_TUNE_MINB : 2) : 4;
#else
  static constexpr int MIN_BLOCKS = WS ? (NCONS >= 256 ? 1 : 2) : 4;
#endif
  // Registers: the launch gives every thread R0 (per-SMSP file of 16K
  // registers shared by the warps resident on it); the producer warpgroup
  // drops to RP and the consumer warpgroups rise to RC within that pool.
  static constexpr int WARPS_PER_SMSP = (NTHREADS / 32 * MIN_BLOCKS + 3) / 4;
  static constexpr int R0_RAW = 16384 / (32 * WARPS_PER_SMSP);
  static constexpr int R0 = (R0_RAW > 255 ? 255 : R0_RAW) & ~7;
#ifdef EQMP_TUNE_RP
  static constexpr int RP = EQMP_TUNE_RP;
#else
  static constexpr int RP = 40;
#endif
  static constexpr int RC_RAW = WS ? (R0 * NTHREADS - RP * 128) / NCONS : R0;
  static constexpr int RC = (RC_RAW > 256 ? 256 : RC_RAW) & ~7;
  static_assert(!WS || RP * 128 + RC * NCONS <= R0 * NTHREADS, "register split exceeds the pool");
  static constexpr int ROW_BYTES = C * 16 * (int)sizeof(XT);
  static constexpr int ROWS = ROW_BYTES / 128;        // 128-byte TMA box rows per node
  static constexpr int INNER = 128 / (int)sizeof(XT);  // elements per box row
  static constexpr int SLOT = ROW_BYTES < 1024 ? 1024 : ROW_BYTES;  // swizzle atom aligned
  // Shared memory besides the x slots: SH ring, partial sums, weights,
  // barriers and alignment slack.  The slots take what is left of the
  // per-CTA share of the SM's 227 KB, rounded down to a power of two.
#ifdef EQMP_TUNE_NP
  static_assert(EQMP_TUNE_NP >= 1 && EQMP_TUNE_NP <= 4, "at most the four warps of warpgroup 0");
  static constexpr int NP = WS ? EQMP_TUNE_NP : 1;
#else
  static constexpr int NP = WS ? 4 : 1;              // producer warps (chunks of S/NP edges, round robin)
#endif
  static constexpr int YR = 64 * NP;                 // SH ring entries (2 batches per producer warp)
  static constexpr int FIXED = YR * 64 + 2 * NQ * 16 * C * 4 + 34 * C * 4 + 2 * 32 * 8 + 1024;
  static constexpr int BUDGET = 227 * 1024 / MIN_BLOCKS - 1024 - FIXED;
  static constexpr int S_FIT = BUDGET / SLOT;
  static constexpr int S_CAP = S_FIT < SharedTune<C, XT>::S_MAX ? S_FIT : SharedTune<C, XT>::S_MAX;
  static constexpr int S = S_CAP >= 32 ? 32 : S_CAP >= 16 ? 16 : S_CAP >= 8 ? 8 : 4;
  static_assert(S_CAP >= 4, "not even four slots fit");
  static_assert((S & (S - 1)) == 0 && S <= 32, "ring size: power of two, at most one batch");
  static constexpr int OFF_X = 0;
  static constexpr int OFF_Y = OFF_X + S * SLOT;            // SH ring, YR entries of 16 floats
  static constexpr int OFF_RED = OFF_Y + YR * 64;
  static constexpr int OFF_W = OFF_RED + 2 * NQ * 16 * C * 4;
  static constexpr int OFF_BAR = OFF_W + 34 * C * 4;
  static constexpr int SMEM_BYTES = OFF_BAR + 2 * S * 8 + 1024;  // + base alignment slack
  static constexpr int XBYTES = KQ * (int)sizeof(XT);              // bytes of x per thread per edge
  static_assert(NCONS % 32 == 0, "consumer threads must fill warps");
  static_assert(XBYTES == 8 || XBYTES == 16 || XBYTES == 32, "unsupported x chunk");
  static_assert(ROW_BYTES % 128 == 0, "row must be whole 128-byte lines");
};

// The backward kernel's consumers read ahead this many edges (its producer pads as many empty
// edges after the last real one).
constexpr uint32_t kLookAhead = 2;

template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Byte offset of logical byte o of a node row inside its 128B-swizzled slot.
__device__ __forceinline__ uint32_t swz128(uint32_t o) {
  return (o & ~0x7Fu) | ((((o >> 4) ^ (o >> 7)) & 7u) << 4) | (o & 15u);
}

// ---- compile-time contraction: partial outputs of quad Q -----------------
template <int KQ, int Q, int I, bool T>
__device__ __forceinline__ void apply_term(const float2 (&acc)[KQ][8], float (&tmp)[16]) {
  constexpr tables::Term t = term_t<T>(I);
  if constexpr (t.k1 >= Q * KQ && t.k1 < Q * KQ + KQ) {
    constexpr int i = t.k1 - Q * KQ;
    const float a = (t.k2 & 1) ? acc[i][t.k2 >> 1].y : acc[i][t.k2 >> 1].x;
    tmp[t.k3] = fmaf(t.c, a, tmp[t.k3]);
  }
}

template <int KQ, int Q, int First, bool T, int... Is>
__device__ __forceinline__ void apply_terms(const float2 (&acc)[KQ][8], float (&tmp)[16],
                                            std::integer_sequence<int, Is...>) {
  (apply_term<KQ, Q, First + Is, T>(acc, tmp), ...);
}

// Bit k3 set when path P reaches output k3 from k1 in [k1lo, k1lo + n);
// used only in constant expressions (the tables are host constants).
template <bool T>
constexpr unsigned path_mask_t(int P, int k1lo, int n) {
  unsigned m = 0;
  for (int k3 = 0; k3 < 16; ++k3)
    if (path_has_t<T>(P, k1lo, n, k3)) m |= 1u << k3;
  return m;
}

template <int KQ, int Q, int P, bool T, int... K3>
__device__ __forceinline__ void weight_outputs(float w, const float (&tmp)[16], float (&part)[16],
                                               std::integer_sequence<int, K3...>) {
  constexpr unsigned mask = path_mask_t<T>(P, Q * KQ, KQ);
  ((((mask >> K3) & 1u) ? (void)(part[K3] = fmaf(w, tmp[K3], part[K3])) : (void)0), ...);
}

template <int C, int KQ, int Q, int P, bool T>
__device__ __forceinline__ void contract_path(const float2 (&acc)[KQ][8], const float* wcol,
                                              float (&part)[16]) {
  if constexpr (path_touches_t<T>(P, Q * KQ, KQ)) {
    constexpr tables::Path path = path_at(P);
    float tmp[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) tmp[k] = 0.0f;
    apply_terms<KQ, Q, path.first, T>(acc, tmp, std::make_integer_sequence<int, path.count>{});
    const float w = wcol[P * C];
    weight_outputs<KQ, Q, P, T>(w, tmp, part, std::make_integer_sequence<int, 16>{});
  }
}

template <int C, int KQ, int Q, bool T, int... Ps>
__device__ __forceinline__ void contract_quad(const float2 (&acc)[KQ][8], const float* wcol,
                                              float (&part)[16], std::integer_sequence<int, Ps...>) {
  (contract_path<C, KQ, Q, Ps, T>(acc, wcol, part), ...);
}

// T = true contracts with the transposed tables (gradient of x).
template <int C, int KQ, bool T>
__device__ __forceinline__ void contract(int q, const float2 (&acc)[KQ][8], const float* wcol,
                                         float (&part)[16]) {
  using Seq = std::make_integer_sequence<int, tables::kNumPaths>;
  if constexpr (KQ == 4) {
    switch (q) {
      case 0: contract_quad<C, KQ, 0, T>(acc, wcol, part, Seq{}); break;
      case 1: contract_quad<C, KQ, 1, T>(acc, wcol, part, Seq{}); break;
      case 2: contract_quad<C, KQ, 2, T>(acc, wcol, part, Seq{}); break;
      default: contract_quad<C, KQ, 3, T>(acc, wcol, part, Seq{}); break;
    }
  } else {
    if (q == 0) contract_quad<C, KQ, 0, T>(acc, wcol, part, Seq{});
    else contract_quad<C, KQ, 1, T>(acc, wcol, part, Seq{});
  }
}

// A[i][k] += x[i] * Y[k] for one edge with the paired FP32 FMA of sm_100+
// (two IEEE round-to-nearest FMAs per instruction, identical to fmaf):
// acc[i][kk] holds (A[i][2kk], A[i][2kk+1]).
template <int KQ>
__device__ __forceinline__ void fma_edge(float2 (&acc)[KQ][8], const float2 (&yv)[8],
                                         const float (&xv)[KQ]) {
#pragma unroll
  for (int i = 0; i < KQ; ++i) {
    const float2 xx = make_float2(xv[i], xv[i]);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) acc[i][kk] = __ffma2_rn(xx, yv[kk], acc[i][kk]);
  }
}

template <int KQ>
__device__ __forceinline__ float acc_at(const float2 (&acc)[KQ][8], int i, int k) {
  return (k & 1) ? acc[i][k >> 1].y : acc[i][k >> 1].x;
}

// ---- x chunk load (KQ elements of one channel) from a swizzled slot -------
// xo[h]: swizzled byte offsets of the thread's 16-byte chunk(s) in a slot.
template <typename XT, int KQ>
__device__ __forceinline__ void load_x(const uint8_t* slot, const uint32_t (&xo)[2], float (&xv)[KQ]) {
  if constexpr (sizeof(XT) == 4) {
#pragma unroll
    for (int h = 0; h < KQ / 4; ++h) {
      const float4 v = *reinterpret_cast<const float4*>(slot + xo[h]);
      xv[4 * h + 0] = v.x; xv[4 * h + 1] = v.y; xv[4 * h + 2] = v.z; xv[4 * h + 3] = v.w;
    }
  } else if constexpr (KQ == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(slot + xo[0]);
    xv[0] = bf16_lo(v.x); xv[1] = bf16_hi(v.x); xv[2] = bf16_lo(v.y); xv[3] = bf16_hi(v.y);
    xv[4] = bf16_lo(v.z); xv[5] = bf16_hi(v.z); xv[6] = bf16_lo(v.w); xv[7] = bf16_hi(v.w);
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(slot + xo[0]);
    xv[0] = bf16_lo(v.x); xv[1] = bf16_hi(v.x); xv[2] = bf16_lo(v.y); xv[3] = bf16_hi(v.y);
  }
}

template <typename XT, int KQ>
__device__ __forceinline__ void store_out(void* out, size_t elem, const float (&o)[KQ]) {
  if constexpr (sizeof(XT) == 4) {
    float* p = reinterpret_cast<float*>(out) + elem;
#pragma unroll
    for (int h = 0; h < KQ / 4; ++h)
      reinterpret_cast<float4*>(p)[h] = make_float4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]);
  } else if constexpr (KQ == 8) {
    uint4 v;
    v.x = pack_bf16x2(o[0], o[1]); v.y = pack_bf16x2(o[2], o[3]);
    v.z = pack_bf16x2(o[4], o[5]); v.w = pack_bf16x2(o[6], o[7]);
    *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + elem) = v;
  } else {
    uint2 v;
    v.x = pack_bf16x2(o[0], o[1]); v.y = pack_bf16x2(o[2], o[3]);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + elem) = v;
  }
}

// TRANS = true: the transposed walk of the gradient of x (rows are senders,
// edges come through a.perm, rows gathered from the upstream gradient by
// the edge's receiver, contraction with the transposed tables).
template <int C, int KQ, typename XT, bool FROM_VEC, bool TRANS>
__global__ void __launch_bounds__(SharedCfg<C, KQ, XT, FROM_VEC>::NTHREADS,
                                  SharedCfg<C, KQ, XT, FROM_VEC>::MIN_BLOCKS)
    k_shared(const __grid_constant__ CUtensorMap tmap, const LayerArgs a) {
  static_assert(!TRANS || FROM_VEC, "the transposed walk computes the harmonics");
  using K = SharedCfg<C, KQ, XT, FROM_VEC>;
  constexpr int S = K::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align<1024>(smem_raw);
  float4* ys = reinterpret_cast<float4*>(smem + K::OFF_Y);
  float* red = reinterpret_cast<float*>(smem + K::OFF_RED);
  float* ws = reinterpret_cast<float*>(smem + K::OFF_W);
  constexpr int SP = S / 2;  // slot pairs: ordinals 2p and 2p+1 share one full and one empty barrier
  const uint32_t full0 = smem_u32(smem + K::OFF_BAR);
  const uint32_t empty0 = full0 + 8 * SP;
  const int tid = threadIdx.x;

  // Contiguous receiver range of this CTA, balanced on edges + 3 per
  // receiver (the contraction and store of a receiver cost about three
  // edges' accumulation).
  const int4 rr = balanced_range_off(a.off, a.N, gridDim.x, blockIdx.x, kReceiverCost);
  const int r_begin = rr.x, r_end = rr.y;

  if (tid < SP) {
    mbar_init(full0 + 8 * tid, 1);          // the even ordinal's arrive (+ the rows' bytes)
    mbar_init(empty0 + 8 * tid, K::NCONS);  // every consumer thread releases the pair
    fence_mbar_init();
  }
  __syncthreads();  // barriers initialised; the producer starts at once

  // Edge range, clamped into [0, E]: a malformed CSR cannot send a load
  // out of bounds, and producer and consumers agree on the count.
  const int e_begin = min(max(rr.z, 0), a.E);
  const int e_end = max(e_begin, min(max(rr.w, 0), a.E));
  const int total = e_end - e_begin;

  if (K::WS ? tid < K::CONS0 : tid >= K::NCONS) {
    // ------------------------------------------------------------ producer
    if constexpr (K::WS) setmaxnreg_dec<K::RP>();
    // NP producer warps.  Ordinals come in chunks of CH = S / NP edges and
    // chunk c belongs to warp c % NP, so slot s = ordinal % S always belongs
    // to warp (s / CH) and every warp issues its own edges in increasing
    // order: a warp is never more than one phase ahead on any of its slots,
    // which is what parity waits require.  A warp works on 32 of its edges at
    // a time (lane l: chunk w + NP (32g/CH + l/CH), element l % CH): the sender
    // indices (and edge vectors) of its next 32 are loaded while these are
    // issued; all lanes compute their 16 SH at once into the SH ring (entry =
    // ordinal % YR); then lanes take turns to claim their slot and launch the
    // row copy of x[src] (tp_scatter: plus a 64-byte copy of the stored SH
    // row).  SH ring reuse: entry n was last used by ordinal n - YR; before
    // this round the warp issued its previous 32 edges (up to 32 NP ordinals
    // back), whose empty-waits proved every ordinal up to that point minus S
    // released; YR >= 32 NP + S.  Each lane's arrive publishes its own SH.
    // Slots come in pairs (ordinals 2p, 2p+1, one full and one empty barrier
    // per pair): CH is even, so a pair always falls to one warp, on lanes
    // 2i and 2i+1 of the same batch, and the even lane (which runs first)
    // waits for the pair to be free, arms its full barrier with the bytes
    // of both rows (one row if the odd ordinal is past the end), and the odd
    // lane only adds its copy.
    constexpr int CH = S / K::NP;
    static_assert(CH >= 2 && CH % 2 == 0 && 32 % CH == 0 && K::YR >= 32 * K::NP + S, "producer layout");
    const int pw = K::WS ? tid >> 5 : 0;  // producer warp index (the non-specialised CTA has one)
    if (pw >= K::NP) return;              // warpgroup 0 has 4 warps; NP of them produce
    const int lane = tid & 31;
    if (lane == 0 && pw == 0) prefetch_tmap(&tmap);
    auto ordinal = [&](int g) {
      return (uint32_t)((pw + K::NP * (g * (32 / CH) + lane / CH)) * CH + lane % CH);
    };
    auto load_edge = [&](uint32_t n, int& node, float& vx, float& vy, float& vz) {
      node = 0; vx = vy = vz = 0.0f;
      if (n < (uint32_t)total) {
        int e = e_begin + (int)n;
        if constexpr (TRANS) {
          e = __ldg(a.perm + e);
          if ((unsigned)e >= (unsigned)a.E_edges) {
            node = -1;  // a bad edge id gathers the zero fill and adds nothing
            return;
          }
          node = __ldg(a.dst + e);
        } else {
          node = __ldg(a.src + e);
        }
        if constexpr (FROM_VEC) {
          const float* v = a.vec + 3 * (size_t)e;
          vx = __ldg(v); vy = __ldg(v + 1); vz = __ldg(v + 2);
        }
      }
    };
    constexpr uint32_t TX = K::ROW_BYTES + (FROM_VEC ? 0 : 64);
    bool ok = true;
    int node_nx;
    float vx_nx, vy_nx, vz_nx;
    load_edge(ordinal(0), node_nx, vx_nx, vy_nx, vz_nx);
    uint32_t lastp = 0;  // this warp's last issued pair + 1 (0: none)
    for (int g = 0; ok; ++g) {
      const uint32_t n = ordinal(g);
      const uint32_t cnt = (uint32_t)__popc(__ballot_sync(0xffffffffu, n < (uint32_t)total));
      if (cnt == 0) break;  // valid lanes are a prefix
      const int node = node_nx;
      float4* yd = ys + 4 * (n % K::YR);
      if constexpr (FROM_VEC) {
        float y[16];
        real_sh16(vx_nx, vy_nx, vz_nx, y);
        yd[0] = make_float4(y[0], y[1], y[2], y[3]);
        yd[1] = make_float4(y[4], y[5], y[6], y[7]);
        yd[2] = make_float4(y[8], y[9], y[10], y[11]);
        yd[3] = make_float4(y[12], y[13], y[14], y[15]);
      }
      load_edge(ordinal(g + 1), node_nx, vx_nx, vy_nx, vz_nx);  // next 32 of this warp, in flight
      for (uint32_t j = 0; j < cnt; ++j) {
        int good = 1;
        if ((uint32_t)lane == j) {
          const uint32_t pr = n >> 1, sp = pr % SP, par = ((pr / SP) & 1u) ^ 1u;
          const uint32_t fb = full0 + 8 * sp;
          bool go = true;
          if ((n & 1u) == 0) {
            go = mbar_try_wait(empty0 + 8 * sp, par) || mbar_wait(empty0 + 8 * sp, par, a.watchdog, 2);
            if (go) mbar_arrive_expect_tx(fb, n + 1 < (uint32_t)total ? 2 * TX : TX);
          }
          if (go) {
            tma_load_2d(smem_u32(smem + K::OFF_X + (n % S) * K::SLOT), &tmap, 0, node * K::ROWS, fb);
            if constexpr (!FROM_VEC)
              bulk_load(smem_u32(yd), a.Y + 16 * (size_t)(e_begin + (int)n), 64, fb);
          } else {
            good = 0;
          }
        }
        if (!__all_sync(0xffffffffu, good)) { ok = false; break; }
      }
      if (ok) lastp = (__shfl_sync(0xffffffffu, n, (int)cnt - 1) >> 1) + 1;
    }
    // Tail: one empty pair after the last pair holding a real edge (phase
    // completed by a plain arrive, no data), issued by the warp that owns it
    // after all its real edges, so the consumers' one-pair look-ahead never
    // waits on a pair that is not coming.
    {
      const uint32_t pr = ((uint32_t)total + 1) >> 1;
      if (ok && pw == (int)((2 * pr / CH) % K::NP)) {
        if (lane == 0) {
          const uint32_t sp = pr % SP, par = ((pr / SP) & 1u) ^ 1u;
          if (mbar_try_wait(empty0 + 8 * sp, par) || mbar_wait(empty0 + 8 * sp, par, a.watchdog, 2))
            mbar_arrive(full0 + 8 * sp);
        }
        lastp = pr + 1;  // the tail is this warp's latest pair on its barriers
      }
    }
    // Drain: wait until this warp's loads among the last SP pairs have
    // landed, so no bulk copy of this warp is in flight when it leaves.  The
    // window [lastp - SP, lastp) holds exactly the latest pair of each
    // barrier, so every phase waited for is the current or the one just
    // completed.
    if (lane == 0 && lastp > 0) {
      const uint32_t first = lastp > (uint32_t)SP ? lastp - SP : 0;
      for (uint32_t i = first; i < lastp; ++i)
        if ((2 * i / CH) % K::NP == (uint32_t)pw)
          if (!mbar_wait(full0 + 8 * (i % SP), (i / SP) & 1u, a.watchdog, 3)) break;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  if constexpr (K::WS) setmaxnreg_inc<K::RC>();
  const int ct = tid - K::CONS0;  // consumer index
  const int c = ct % C, q = ct / C, lane = tid & 31;
  // Path weights to shared memory: every load issued before any store.
  {
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
  // CSR offsets, 32 receivers per warp-wide load, one chunk prefetched ahead:
  // lane i holds off[chunk_base + i]; off[r] and off[r+1] come by shuffle.
  auto load_off = [&](int base) {
    const int i = base + lane;
    return i <= r_end ? min(max(__ldg(a.off + i), 0), a.E) : a.E;
  };
  int chunk = r_begin;
  int off_cur = load_off(chunk);
  int off_nxt = load_off(chunk + 32);
  named_barrier(2, K::NCONS);  // weights visible to all consumers
  const uint32_t xlog = (uint32_t)(c * 16 * (int)sizeof(XT) + q * K::XBYTES);
  const uint32_t xo[2] = {swz128(xlog), swz128(xlog + 16)};
  const float* wcol = ws + c;
  uint32_t n = 0;  // ordinal of the CTA's next edge
  int buf = 0;
  bool failed = false;
  // Edge m lives in slot m % S with its SH in ring entry m % YR; edges 2p
  // and 2p+1 share the barriers of pair p (index p % SP, phase (p / SP) & 1).
  // A cursor holds these for one pair (full barrier address, parity, byte
  // offsets of the even edge's slot and SH entry; the odd edge's are one
  // slot and one entry further) and steps to the next pair with a few
  // warp-uniform adds and selects.
  struct Cursor {
    uint32_t bar, par, xs, ys;
  };
  auto advance = [&](Cursor& u) {
    u.bar += 8;
    u.xs += 2 * K::SLOT;
    u.ys += 128;
    if (u.bar == full0 + 8 * SP) {
      u.bar = full0;
      u.xs = K::OFF_X;
      u.par ^= 1u;
    }
    if (u.ys == (uint32_t)(K::OFF_Y + 64 * K::YR)) u.ys = K::OFF_Y;
  };
  auto wait_cur = [&](const Cursor& u) {
    if (!mbar_try_wait(u.bar, u.par))
      if (!mbar_wait_slow(u.bar, u.par, a.watchdog, 1, failed)) failed = true;
  };
  // Registers of one edge of the pair at the cursor (h = 0 even, 1 odd).
  auto load_half = [&](const Cursor& u, int h, float2 (&yv)[8], float (&xv)[KQ]) {
    const float4* yp = reinterpret_cast<const float4*>(smem + u.ys + 64 * h);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 t = yp[k];
      yv[2 * k] = make_float2(t.x, t.y);
      yv[2 * k + 1] = make_float2(t.z, t.w);
    }
    load_x<XT, KQ>(smem + u.xs + K::SLOT * h, xo, xv);
  };
  // Registers A hold the even edge of the current pair, B the odd one; `la`
  // is the next pair (the look-ahead).  A whole pair: test (non-blocking)
  // that the next pair has landed, run A's FMAs, (waiting only if the test
  // failed) load the next even edge into A, run B's FMAs, release the pair
  // (every consumer thread arrives on its empty barrier, 8 SP bytes past the
  // full one), load the next odd edge into B, step the cursor.  A receiver
  // that starts or ends inside a pair runs the half of it that is its own;
  // the pair is released once both halves are summed.
  Cursor la = {full0, 0u, (uint32_t)K::OFF_X, (uint32_t)K::OFF_Y};
  float2 yA[8], yB[8];
  float xA[KQ], xB[KQ];
  wait_cur(la);
  load_half(la, 0, yA, xA);
  load_half(la, 1, yB, xB);
  uint32_t barP = la.bar;
  advance(la);
  bool half = false;  // the next edge is the odd one of the loaded pair
  for (int r = r_begin; r < r_end; ++r) {
    if (r - chunk == 32) {
      chunk += 32;
      off_cur = off_nxt;
      off_nxt = load_off(chunk + 32);
    }
    const int j0 = r - chunk;  // 0..31; off[r+1] is lane j0+1, or lane 0 of the next chunk
    const int a0 = __shfl_sync(0xffffffffu, off_cur, j0);
    const int a1n = __shfl_sync(0xffffffffu, off_cur, (j0 + 1) & 31);
    const int a1x = __shfl_sync(0xffffffffu, off_nxt, 0);
    const int a1 = j0 == 31 ? a1x : a1n;
    const int deg = min(max(a1 - a0, 0), total - (int)n);
    float2 acc[KQ][8];
#pragma unroll
    for (int i = 0; i < KQ; ++i)
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[i][k] = make_float2(0.0f, 0.0f);

    int j = 0;
    if (half && deg > 0) {  // the receiver starts on the odd edge: finish that pair
      const bool ready = mbar_test_wait(la.bar, la.par);
      fma_edge(acc, yB, xB);
      mbar_arrive(barP + 8 * SP);
      if (!ready) wait_cur(la);
      load_half(la, 0, yA, xA);
      load_half(la, 1, yB, xB);
      barP = la.bar;
      advance(la);
      half = false;
      j = 1;
    }
    for (; j + 2 <= deg; j += 2) {
      const bool ready = mbar_test_wait(la.bar, la.par);
      fma_edge(acc, yA, xA);
      if (!ready) wait_cur(la);
      load_half(la, 0, yA, xA);
      fma_edge(acc, yB, xB);
      mbar_arrive(barP + 8 * SP);
      load_half(la, 1, yB, xB);
      barP = la.bar;
      advance(la);
    }
    if (j < deg) {  // the receiver ends on an even edge: the odd one is the next receiver's
      fma_edge(acc, yA, xA);
      half = true;
    }
    n += (uint32_t)deg;

    float part[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) part[k] = 0.0f;
    contract<C, KQ, TRANS>(q, acc, wcol, part);

    float* rb = red + buf * (K::NQ * 16 * C);
#pragma unroll
    for (int k = 0; k < 16; ++k) rb[(q * 16 + k) * C + c] = part[k];
    named_barrier(1, K::NCONS);
    float o[KQ];
#pragma unroll
    for (int i = 0; i < KQ; ++i) {
      float sum = 0.0f;
#pragma unroll
      for (int qq = 0; qq < K::NQ; ++qq) sum += rb[(qq * 16 + q * KQ + i) * C + c];
      o[i] = sum;
    }
    store_out<XT, KQ>(a.out, ((size_t)r * C + c) * 16 + q * KQ, o);
    buf ^= 1;
  }
}

}  // namespace eqmp
