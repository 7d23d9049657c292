// Device helpers shared by the eqmp kernels (sm_103a).
//
//  * inline-PTX wrappers for mbarriers and TMA tensor loads, every wait
//    bounded by the global nanosecond timer (a wait that gives up records a
//    code in the device watchdog word and returns false; nothing traps);
//  * the register-resident real spherical harmonics, l <= 3 (Batmobile blog
//    "Batmobile CUDA内核优化", section "2. 寄存器中间计算");
//  * compile-time expansion of the generated CG tables (section
//    "1. 编译时常量": coefficients folded into the instruction stream).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "eqmp_tables.h"

namespace eqmp {

// ---------------------------------------------------------------- watchdog
// The watchdog word lives in device memory owned by the library (one per
// device); kernels receive its address.  It becomes nonzero once any
// bounded wait has given up and is read and cleared by eqmp_device_error().
// Codes: 1 consumer full-wait, 2 producer empty-wait, 3 producer drain,
// 4 grid barrier of the single-launch radius graph, 5 the watchdog self-test,
// 7 the look-back of the radius graph's single-pass scan, 8 a CTA waiting
// for the piece of a receiver cut between it and the next CTA of its cluster.

constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void watchdog_trip(int* wd, int code) { atomicCAS(wd, 0, code); }

// ---------------------------------------------------------------- work split
// Receiver range [x, y) of CTA b out of G, balancing the work
//   work(r) = (off[r] - off[0]) + alpha * r
// (edges plus a per-receiver cost in edge units): the range starts at the
// first r with work(r) >= b T / G and ends at the first r with
// work(r) >= (b+1) T / G, T = work(N).  Found by a warp-wide 32-ary search:
// the candidates lo..hi are cut into 32 groups, lane l probes the last
// candidate of group l (lane 31 probes hi, true by construction), and the
// first lane whose probe reaches the target names the group that holds the
// answer; about log32 N dependent loads.  Every warp of a CTA computes the
// same range.  The interval shrinks every round whatever the offsets hold,
// so a malformed CSR still ends in a range inside [0, N].
constexpr int kReceiverCost = 3;  // per-receiver work of the fused kernels, in edges

__device__ __forceinline__ int split_probe(int lo, int hi, int lane) {
  const long long d = (long long)hi - lo + 1;
  return lo + (int)(((lane + 1) * d + 31) / 32) - 1;
}

// Returns (x, y, off[x], off[y]); the offsets are as loaded, unclamped.  The
// search has loaded them already, so the caller's edge range costs no
// further dependent load.
__device__ __forceinline__ int4 balanced_range_off(const int* __restrict__ off, int N, int G, int b, int alpha) {
  const int lane = threadIdx.x & 31;
  // round 1: the probes of both bounds coincide; off[0] and off[N] load with them
  const int p1 = split_probe(0, N, lane);
  const int o_p1 = __ldg(off + p1);
  const int o0 = __ldg(off), oN = __ldg(off + N);
  const long long total = (long long)max(oN - o0, 0) + (long long)alpha * N;
  const long long tgt[2] = {total * b / G, total * (b + 1) / G};
  int lo[2], hi[2], ohi[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const long long w = (long long)(o_p1 - o0) + (long long)alpha * p1;
    const unsigned ge = __ballot_sync(0xffffffffu, p1 == N || w >= tgt[k]);
    const int f = __ffs(ge) - 1;
    hi[k] = __shfl_sync(0xffffffffu, p1, f);
    ohi[k] = __shfl_sync(0xffffffffu, o_p1, f);
    const int prev = __shfl_sync(0xffffffffu, p1, f > 0 ? f - 1 : 0);
    lo[k] = f == 0 ? 0 : prev + 1;
  }
  if (b == 0) { lo[0] = hi[0] = 0; ohi[0] = o0; }
  if (b == G - 1) { lo[1] = hi[1] = N; ohi[1] = oN; }
  while (lo[0] < hi[0] || lo[1] < hi[1]) {
    int p[2], o[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      p[k] = split_probe(lo[k], hi[k], lane);
      o[k] = lo[k] < hi[k] && p[k] < hi[k] ? __ldg(off + p[k]) : 0;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (lo[k] >= hi[k]) continue;  // warp-uniform
      const long long w = (long long)(o[k] - o0) + (long long)alpha * p[k];
      const unsigned ge = __ballot_sync(0xffffffffu, p[k] == hi[k] || w >= tgt[k]);
      const int f = __ffs(ge) - 1;
      const int nh = __shfl_sync(0xffffffffu, p[k], f);
      const int of = __shfl_sync(0xffffffffu, o[k], f);
      const int prev = __shfl_sync(0xffffffffu, p[k], f > 0 ? f - 1 : 0);
      lo[k] = f == 0 ? lo[k] : prev + 1;
      if (nh != hi[k]) ohi[k] = of;  // a probe below hi was loaded; hi itself keeps its value
      hi[k] = nh;
    }
  }
  const bool up = hi[1] >= hi[0];
  return make_int4(hi[0], up ? hi[1] : hi[0], ohi[0], up ? ohi[1] : ohi[0]);
}

// The CTA's range searched by warp 0 alone and written to `slot` (shared
// memory, 16 bytes); the other warps read it after the caller's next
// __syncthreads.  Every CTA's first-round probes hit the same few lines of
// the offsets; one warp per CTA instead of every warp sends fewer of those
// requests (the aligned-frame kernel: 41.0 -> 38.9 us on the 1000-atom
// radial workload; the shared-weight kernel measured slower with it and
// keeps the per-warp search).
__device__ __forceinline__ void balanced_range_publish(int4* slot, const int* __restrict__ off, int N, int G, int b,
                                                       int alpha) {
  if (threadIdx.x < 32) {
    const int4 r = balanced_range_off(off, N, G, b, alpha);
    if (threadIdx.x == 0) *slot = r;
  }
}

// Edge-granular split inside clusters of Q CTAs.  Cluster k (CTAs kQ ..
// kQ+Q-1) takes the whole receivers [R0, R1) between the cuts of targets
// T kQ / G and T (k+1)Q / G, as above.  Its own work W0 = work(R0) ..
// W1 = work(R1) is then cut evenly: CTA kQ+i starts at t = W0 + (W1-W0) i/Q,
// which falls in receiver r with work(r) < t <= work(r+1), at edge
// off[r] + (t - work(r)) when that is below off[r+1] (the receiver is then
// shared by the CTAs on both sides), else at the receiver boundary r+1.
// Both CTAs beside a cut compute it from the same target with the same
// search, so they agree on it bit for bit.  A receiver cut this way is
// summed in pieces: the CTA after a cut hands its piece to the CTA before
// it (head_cut), which adds it to its own piece (tail_cut); a CTA inside
// one long receiver has both.
struct CutRange {
  int r_begin, r_end;  // receivers touched, [r_begin, r_end)
  int e_begin, e_end;  // edges, [e_begin, e_end), as loaded (unclamped)
  bool head_cut;       // receiver r_begin started before e_begin
  bool tail_cut;       // receiver r_end - 1 continues past e_end
};

// First r in [lo0, hi0] with work(r) >= tgt[k] for two targets (hi0 counts
// as reaching both), with ohi = off[r] and olo = off[r - 1] (olo is only
// meaningful when r > lo0).  The warp's 32-ary search from above, sharing
// the first round's probes between the targets.
__device__ __forceinline__ void work_search2(const int* __restrict__ off, int lo0, int hi0, int ohi0, int o0,
                                             int alpha, const long long (&tgt)[2], int (&hi)[2], int (&ohi)[2],
                                             int (&olo)[2]) {
  const int lane = threadIdx.x & 31;
  const int p1 = split_probe(lo0, hi0, lane);
  const int o_p1 = p1 < hi0 ? __ldg(off + p1) : ohi0;
  int lo[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const long long w = (long long)(o_p1 - o0) + (long long)alpha * p1;
    const unsigned ge = __ballot_sync(0xffffffffu, p1 == hi0 || w >= tgt[k]);
    const int f = __ffs(ge) - 1;
    const int g = f > 0 ? f - 1 : 0;
    hi[k] = __shfl_sync(0xffffffffu, p1, f);
    ohi[k] = __shfl_sync(0xffffffffu, o_p1, f);
    const int prev = __shfl_sync(0xffffffffu, p1, g);
    const int oprev = __shfl_sync(0xffffffffu, o_p1, g);
    lo[k] = f == 0 ? lo0 : prev + 1;
    olo[k] = f == 0 ? 0 : oprev;
  }
  while (lo[0] < hi[0] || lo[1] < hi[1]) {
    int p[2], o[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      p[k] = split_probe(lo[k], hi[k], lane);
      o[k] = lo[k] < hi[k] && p[k] < hi[k] ? __ldg(off + p[k]) : 0;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (lo[k] >= hi[k]) continue;  // warp-uniform
      const long long w = (long long)(o[k] - o0) + (long long)alpha * p[k];
      const unsigned ge = __ballot_sync(0xffffffffu, p[k] == hi[k] || w >= tgt[k]);
      const int f = __ffs(ge) - 1;
      const int g = f > 0 ? f - 1 : 0;
      const int nh = __shfl_sync(0xffffffffu, p[k], f);
      const int of = __shfl_sync(0xffffffffu, o[k], f);
      const int prev = __shfl_sync(0xffffffffu, p[k], g);
      const int oprev = __shfl_sync(0xffffffffu, o[k], g);
      if (f > 0) { lo[k] = prev + 1; olo[k] = oprev; }
      if (nh != hi[k]) ohi[k] = of;
      hi[k] = nh;
    }
  }
}

__device__ __forceinline__ CutRange cluster_cut_range(const int* __restrict__ off, int N, int G, int b, int Q,
                                                      int alpha) {
  const int o0 = __ldg(off), oN = __ldg(off + N);
  const long long total = (long long)max(oN - o0, 0) + (long long)alpha * N;
  const int k0 = b - b % Q, i = b - k0;  // the cluster's first CTA; this CTA's rank in it
  // phase 1: the cluster's whole receivers [R0, R1)
  int hi[2], ohi[2], olo[2];
  {
    const long long tgt[2] = {total * k0 / G, total * (k0 + Q) / G};
    work_search2(off, 0, N, oN, o0, alpha, tgt, hi, ohi, olo);
  }
  if (k0 == 0) { hi[0] = 0; ohi[0] = o0; }
  if (k0 + Q >= G) { hi[1] = N; ohi[1] = oN; }
  const int R0 = hi[0], E0 = ohi[0];
  const int R1 = max(hi[1], R0), E1 = max(ohi[1], E0);
  // phase 2: this CTA's cuts inside [R0, R1]
  const long long W0 = (long long)(E0 - o0) + (long long)alpha * R0;
  const long long W1 = max((long long)(E1 - o0) + (long long)alpha * R1, W0);
  const long long tgt[2] = {W0 + (W1 - W0) * i / Q, W0 + (W1 - W0) * (i + 1) / Q};
  work_search2(off, R0, R1, E1, o0, alpha, tgt, hi, ohi, olo);
  // cut k as (receiver, edge, inside)
  auto place = [&](int k, int& r, int& e, bool& inside) {
    r = hi[k]; e = ohi[k]; inside = false;
    if (hi[k] > R0) {
      const long long wprev = (long long)(olo[k] - o0) + (long long)alpha * (hi[k] - 1);
      const long long ee = (long long)olo[k] + (tgt[k] - wprev);
      if (ee < (long long)ohi[k]) { r = hi[k] - 1; e = (int)ee; inside = true; }
    }
    if (e <= E0) { r = R0; e = E0; inside = false; }
    if (e >= E1) { r = R1; e = E1; inside = false; }
  };
  int rb = R0, eb = E0, re = R1, ee = E1;
  bool ib = false, ie = false;
  if (i != 0) place(0, rb, eb, ib);
  if (i != Q - 1) place(1, re, ee, ie);
  CutRange c;
  c.r_begin = rb;
  c.e_begin = eb;
  c.e_end = max(ee, eb);
  c.r_end = max(ie ? re + 1 : re, rb);
  c.head_cut = ib;
  c.tail_cut = ie;
  return c;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The dynamic shared-memory array advanced to the next multiple of A bytes.
// The result is the array plus an offset (not a pointer rebuilt from an
// integer), so the compiler still knows it points into shared memory and
// addresses it with 32-bit shared loads and stores.
template <uint32_t A>
__device__ __forceinline__ uint8_t* smem_align(uint8_t* raw) {
  const uint32_t base = smem_u32(raw);
  return raw + (((base + (A - 1)) & ~(A - 1)) - base);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// One test of the phase.  A thread whose phase is not yet complete is
// suspended by the hardware (up to the hint, 1 ms) instead of spinning, so a
// waiting warp takes no issue slots from the warps doing the arithmetic.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `parity` to complete; false (and the watchdog
// set to `code`) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* wd, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      watchdog_trip(wd, code);
      return false;
    }
  }
}

// Non-blocking test of the phase (no suspension): issue early, branch late.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of another CTA of the cluster (address from map_rank),
// releasing this thread's earlier writes (and those ordered before them) at
// cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void fence_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }
// Bounded wait on a local mbarrier that other CTAs of the cluster arrive on,
// acquiring at cluster scope.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, int* wd, int code) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      watchdog_trip(wd, code);
      return false;
    }
  }
}

// Out-of-line slow path of a wait whose first try failed: keeps the hot loop
// small.  Skips waiting once `failed` is set (the kernel then finishes its
// loop structure without blocking and exits).
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, int* wd, int code,
                                            bool failed) {
  if (failed) return false;
  return mbar_wait(bar, parity, wd, code);
}

// ---------------------------------------------------------------- TMA
// 2-D tiled tensor load global -> shared, completion on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size a
// multiple of 16), completion on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Named barrier over `count` threads (count a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------- storage
template <typename T>
struct Storage;

template <>
struct Storage<float> {
  static __device__ __forceinline__ float load(float v) { return v; }
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round-to-nearest-even pack of two floats into bf16x2 (lo in low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- SH
// Real SH for one edge vector: Y_lm = poly_lm(z) * {Re, Im}(x + i y)^|m| on
// the unit sphere, poly coefficients (normalisation folded in) from the
// generated table.  Zero-length vectors give n = 0 and Y_{l>=1} = 0.
constexpr float sh_coef(int l, int m, int p) { return tables::kShPoly[l][m][p]; }

template <int L, int M>
__device__ __forceinline__ float sh_poly(float z) {
  constexpr float c0 = sh_coef(L, M, 0);
  constexpr float c1 = sh_coef(L, M, 1);
  constexpr float c2 = sh_coef(L, M, 2);
  constexpr float c3 = sh_coef(L, M, 3);
  // Horner; zero coefficients fold away.
  return fmaf(fmaf(fmaf(c3, z, c2), z, c1), z, c0);
}

__device__ __forceinline__ void real_sh16(float vx, float vy, float vz, float (&Y)[16]) {
  const float r2 = fmaf(vx, vx, fmaf(vy, vy, vz * vz));
  const bool nonzero = r2 >= 1e-30f;
  const float inv = nonzero ? rsqrtf(r2) : 0.0f;
  const float x = vx * inv, y = vy * inv, z = vz * inv;
  // (x + i y)^m
  const float c1 = x, s1 = y;
  const float c2 = fmaf(x, x, -y * y), s2 = 2.0f * x * y;
  const float c3 = fmaf(x, c2, -y * s2), s3 = fmaf(x, s2, y * c2);
  Y[0] = sh_poly<0, 0>(z);
  Y[2] = sh_poly<1, 0>(z);
  { const float p = sh_poly<1, 1>(z); Y[3] = p * c1; Y[1] = p * s1; }
  Y[6] = sh_poly<2, 0>(z);
  { const float p = sh_poly<2, 1>(z); Y[7] = p * c1; Y[5] = p * s1; }
  { const float p = sh_poly<2, 2>(z); Y[8] = p * c2; Y[4] = p * s2; }
  Y[12] = sh_poly<3, 0>(z);
  { const float p = sh_poly<3, 1>(z); Y[13] = p * c1; Y[11] = p * s1; }
  { const float p = sh_poly<3, 2>(z); Y[14] = p * c2; Y[10] = p * s2; }
  { const float p = sh_poly<3, 3>(z); Y[15] = p * c3; Y[9] = p * s3; }
  if (!nonzero) {
#pragma unroll
    for (int k = 1; k < 16; ++k) Y[k] = 0.0f;
  }
}

// ---------------------------------------------------------------- CG tables
// Compile-time accessors and queries over the generated term list.
constexpr tables::Term term_at(int i) { return tables::kTerms[i]; }
constexpr tables::Path path_at(int p) { return tables::kPaths[p]; }

constexpr int l_of_k(int k) { return k < 1 ? 0 : (k < 4 ? 1 : (k < 9 ? 2 : 3)); }

// Does path P have a term with k1 in [k1lo, k1lo + n) and output k3?
constexpr bool path_has(int P, int k1lo, int n, int k3) {
  for (int i = tables::kPaths[P].first; i < tables::kPaths[P].first + tables::kPaths[P].count; ++i)
    if (tables::kTerms[i].k3 == k3 && tables::kTerms[i].k1 >= k1lo && tables::kTerms[i].k1 < k1lo + n)
      return true;
  return false;
}

constexpr bool path_touches(int P, int k1lo, int n) {
  for (int k3 = 0; k3 < 16; ++k3)
    if (path_has(P, k1lo, n, k3)) return true;
  return false;
}

// The same tables with the roles of k1 and k3 exchanged (T = true): the
// transposed product sum_{k3,k2} C_p[k3,k1,k2] g[k3] Y[k2] -> out[k1] that
// the gradient of x needs.  Same paths, same coefficients.
template <bool T>
constexpr tables::Term term_t(int i) {
  tables::Term t = tables::kTerms[i];
  if (T) {
    const int k = t.k1;
    t.k1 = t.k3;
    t.k3 = k;
  }
  return t;
}

template <bool T>
constexpr bool path_has_t(int P, int k1lo, int n, int k3) {
  for (int i = tables::kPaths[P].first; i < tables::kPaths[P].first + tables::kPaths[P].count; ++i)
    if (term_t<T>(i).k3 == k3 && term_t<T>(i).k1 >= k1lo && term_t<T>(i).k1 < k1lo + n) return true;
  return false;
}

template <bool T>
constexpr bool path_touches_t(int P, int k1lo, int n) {
  for (int k3 = 0; k3 < 16; ++k3)
    if (path_has_t<T>(P, k1lo, n, k3)) return true;
  return false;
}

}  // namespace eqmp
