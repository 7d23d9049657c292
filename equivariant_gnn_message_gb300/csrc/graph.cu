// Radius graph on the GPU: every ordered pair i != j with |p_j - p_i| < r_c,
// as CSR rows by receiver with senders ascending, plus the edge vectors
// p_j - p_i.  E2Former-V2 (section 4.2) builds neighbour lists by a radius
// cutoff; the Batmobile blog (monitoring section) uses 4-6 Angstrom.
//
// The cutoff decision is taken in float32 in one fixed order, each operation
// rounded on its own (no contraction into FMA):
//     d_a = p_j[a] - p_i[a];  d2 = (d_x*d_x + d_y*d_y) + d_z*d_z;  edge iff d2 < r_c*r_c.
//
// Pipeline (all on the caller's stream, no host synchronisation; one
// cooperative launch of k_graph_coop runs every phase with grid barriers in
// between, or, where cooperative launches are unavailable, one kernel each):
//   k_clear    zero the bucket counters
//   k_bin      cell of each atom (cell side = r_c (1 + 2^-10)), hashed into
//              H = 2^k >= 2N buckets; count atoms per bucket
//   scan       bucket starts (exclusive prefix sum)
//   k_scatter  atoms (and a copy of their positions) listed bucket by bucket
//   k_neigh    (count) one warp per receiver, visited in bucket order so
//              neighbouring warps read the same buckets: the lanes test the
//              atoms of the 27 surrounding cells' buckets (each bucket once)
//   scan       degrees -> row_offsets, E_total
//   k_neigh    (fill) the same walk writes each receiver's senders, unsorted
//   k_sort     one warp per receiver: rank sort of its senders, writes
//              src, vec (and dst) at the sorted position
//   k_rev      (optional) position of the reverse edge, by binary search
// Bucket order and fill order depend on atomics; the output does not: the
// degree is a count and each row is sorted, so the result is bitwise
// deterministic.
//
// Periodic boundaries (eqmp_radius_graph_pbc; E2Former-V2 section 4.2:
// periodic systems by expanded cells, one image per direction): positions
// in an orthorhombic box [0, L), r_c <= min(L); edges (j, image s) -> i for
// s in {-1, 0, 1}^3 with d_a = (p_j[a] - p_i[a]) + s_a L_a below the cutoff
// (same test), except j = i with s = 0.  The cells tile the box (n_a per
// axis, side >= r_c (1 + 2^-10)); an axis shorter than three cells is one
// cell whose three images are walked explicitly.  Wrapped cells are hashed
// into the same bucket table; the walk keys each of its 27 lanes by
// (bucket, image), so one bucket visited under two images is walked twice
// and under one image once.  The fill writes j * 27 + image; the row sort
// ranks by that key (sender, then image index sigma = (s_x + 1) +
// 3 (s_y + 1) + 9 (s_z + 1)) and writes src, img and vec.
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "eqmp.h"
#include "launch.h"

namespace eqmp {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;
constexpr int kScanTile = kScanThreads * kScanItems;
constexpr int kNeighThreads = 256;
constexpr int kSortWarps = 8;
constexpr int kSortCap = 512;          // row length sorted in shared memory
// Walk modes of the neighbour pass (neigh_row) and the per-row scratch of
// the single-walk path: rows up to kRowScratch senders are kept from the
// counting walk, longer ones are walked again.  Used up to kScratchMaxAtoms
// (the scratch is kRowScratch ints per atom).
constexpr int kWalkCount = 0, kWalkFill = 1, kWalkScratch = 2;
constexpr int kRowScratch = 96;
constexpr long long kScratchMaxAtoms = 1ll << 21;
constexpr float kCellRange = 4096.0f;  // |p| / cell side must stay below this
constexpr long long kGraphMaxAtoms = 1ll << 30;  // keeps the bucket count <= 2^31
constexpr long long kGraphMaxAtomsPbc = 1ll << 26;  // keys sender * 27 + image stay below 2^31
constexpr int kCoopMaxBlocks = 2048;              // cooperative grid cap (block totals it can hold)
constexpr long long kCoopMaxAtoms = 16384;        // the single launch is used up to this many atoms
constexpr unsigned long long kGridWaitNs = 4000000000ull;

// Cell coordinates hashed as in Teschner et al. 2003 (optimised spatial
// hashing: XOR of coordinates times three large primes), then mixed by the
// MurmurHash3 finaliser so that masking to the low bits stays uniform.
__device__ __forceinline__ uint32_t cell_hash(int cx, int cy, int cz, uint32_t mask) {
  uint32_t h = (uint32_t)cx * 73856093u ^ (uint32_t)cy * 19349663u ^ (uint32_t)cz * 83492791u;
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h & mask;
}

__device__ __forceinline__ int cell_of(float p, float inv) {
  const float c = floorf(__fmul_rn(p, inv));
  return (int)fminf(fmaxf(c, -kCellRange - 2.0f), kCellRange + 2.0f);
}

// Periodic box: sides, cells per axis (1: one cell spanning the axis, its
// images walked explicitly), cells per unit length.
struct Box {
  float L[3];
  float inv[3];
  int n[3];
};
constexpr int kImages = 27;
constexpr int kSelfImage = 13;  // s = (0, 0, 0)

__device__ __forceinline__ int pbc_cell(float p, float inv, int n) {
  if (n == 1) return 0;
  const int c = (int)floorf(__fmul_rn(p, inv));
  return min(max(c, 0), n - 1);
}

// image shift of component a of image index sigma
__device__ __forceinline__ int image_shift(int sigma, int a) {
  return (a == 0 ? sigma : a == 1 ? sigma / 3 : sigma / 9) % 3 - 1;
}

// d_a = (p_j[a] - p_i[a]) + s_a L_a, each operation rounded on its own
__device__ __forceinline__ float3 image_vec(float3 pi, float3 pj, int sigma, const Box& box) {
  return make_float3(__fadd_rn(__fsub_rn(pj.x, pi.x), (float)image_shift(sigma, 0) * box.L[0]),
                     __fadd_rn(__fsub_rn(pj.y, pi.y), (float)image_shift(sigma, 1) * box.L[1]),
                     __fadd_rn(__fsub_rn(pj.z, pi.z), (float)image_shift(sigma, 2) * box.L[2]));
}

__device__ __forceinline__ float norm2(float3 d) {
  return __fadd_rn(__fadd_rn(__fmul_rn(d.x, d.x), __fmul_rn(d.y, d.y)), __fmul_rn(d.z, d.z));
}

__device__ __forceinline__ float dist2(float3 a, float3 b) {
  const float dx = __fsub_rn(b.x, a.x), dy = __fsub_rn(b.y, a.y), dz = __fsub_rn(b.z, a.z);
  return __fadd_rn(__fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy)), __fmul_rn(dz, dz));
}

__device__ __forceinline__ float3 load_pos(const float* __restrict__ pos, int i) {
  return make_float3(__ldg(pos + 3 * (size_t)i), __ldg(pos + 3 * (size_t)i + 1), __ldg(pos + 3 * (size_t)i + 2));
}

// ------------------------------------------------------------ scan
// Exclusive prefix sum of int32 data in place, with 64-bit block totals so
// that the grand total is exact even where the int32 prefix would wrap.
__device__ __forceinline__ long long block_exclusive(long long v, long long* warp_tot, long long* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    long long w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
    long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    warp_tot[lane] = wi - w;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const long long r = warp_tot[wid] + incl - v;
  __syncthreads();
  return r;
}

// Single-pass exclusive scan (decoupled look-back): each block takes the
// next tile in launch order from a ticket counter, scans it, publishes its
// aggregate, and adds up its predecessors' published values until it meets
// an inclusive prefix (tile 0 publishes one at once), 32 predecessors per
// read; then it publishes its own inclusive prefix and writes its tile.  A block waits only for tiles
// that earlier blocks hold, so the scan completes whatever the residency;
// every wait is bounded (watchdog code 7).  Status words: bits 63..62 flag
// (1 aggregate, 2 inclusive), 61..0 the value (saturated; a sum that large is
// reported as too many edges anyway).  status[] and the ticket start at zero
// (k_clear).
constexpr unsigned long long kScanAgg = 1ull << 62, kScanIncl = 2ull << 62, kScanVal = (1ull << 62) - 1;

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64g(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_1p(int32_t* __restrict__ data, long long n,
                                                          unsigned long long* __restrict__ status,
                                                          unsigned* __restrict__ ticket, const int* __restrict__ bad,
                                                          long long* __restrict__ e_total, int* watchdog) {
  __shared__ long long warp_tot[32];
  __shared__ long long total, prefix_s;
  __shared__ unsigned tile_s;
  if (threadIdx.x == 0) tile_s = atomicAdd(ticket, 1u);
  __syncthreads();
  const long long t = tile_s;
  const long long base = t * kScanTile + (long long)threadIdx.x * kScanItems;
  int v[kScanItems];
  long long s = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    v[k] = base + k < n ? data[base + k] : 0;
    s += v[k];
  }
  long long run = block_exclusive(s, warp_tot, &total);
  if (threadIdx.x < 32) {
    // Look-back by warp 0, 32 predecessors per round: lane i reads tile
    // j - i.  If one of them holds an inclusive prefix, the values from
    // lane 0 up to the nearest such lane make up the prefix; otherwise all
    // 32 are aggregates and the window moves 32 tiles back.  A round whose
    // needed words are not all published yet is read again.
    const int lane = threadIdx.x;
    const unsigned long long agg = (unsigned long long)min(total, (long long)kScanVal);
    long long prefix = 0;
    if (t == 0) {
      if (lane == 0) st_release_u64(status, kScanIncl | agg);
    } else {
      if (lane == 0) st_release_u64(status + t, kScanAgg | agg);
      long long j = t - 1;
      const unsigned long long t0 = global_ns();
      while (j >= 0) {
        const long long idx = j - lane;
        const unsigned long long w = idx >= 0 ? ld_acquire_u64g(status + idx) : 0ull;
        const unsigned incl = __ballot_sync(0xffffffffu, idx >= 0 && (w & kScanIncl) != 0ull);
        const unsigned zero = __ballot_sync(0xffffffffu, idx >= 0 && w == 0ull);
        const unsigned need = incl ? (2u << (__ffs(incl) - 1)) - 1u : 0xffffffffu;  // lanes 0 .. nearest inclusive
        if (zero & need) {
          // the give-up decision is the warp's, so every lane leaves together
          if (__any_sync(0xffffffffu, global_ns() - t0 > kWaitLimitNs)) {
            if (lane == 0) watchdog_trip(watchdog, 7);
            break;
          }
          continue;
        }
        long long v = ((need >> lane) & 1u) && idx >= 0 ? (long long)(w & kScanVal) : 0ll;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
        prefix += __shfl_sync(0xffffffffu, v, 0);
        if (incl) break;
        j -= 32;
      }
      if (lane == 0) st_release_u64(status + t, kScanIncl | (unsigned long long)min(prefix + total, (long long)kScanVal));
    }
    if (lane == 0) {
      prefix_s = prefix;
      if (e_total && t == (long long)gridDim.x - 1) {  // the last tile knows the grand total
        long long e = prefix + total;
        if (e > INT32_MAX) e = -2;
        if (*bad) e = -1;
        *e_total = e;
      }
    }
  }
  __syncthreads();
  run += prefix_s;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    if (base + k < n) data[base + k] = (int32_t)run;
    run += v[k];
  }
}

cudaError_t exclusive_scan(int32_t* data, long long n, unsigned long long* status, unsigned* ticket, const int* bad,
                           long long* e_total, int* watchdog, cudaStream_t st) {
  const long long nb = (n + kScanTile - 1) / kScanTile;
  k_scan_1p<<<(unsigned)nb, kScanThreads, 0, st>>>(data, n, status, ticket, bad, e_total, watchdog);
  return cudaGetLastError();
}

// ------------------------------------------------------------ binning
__global__ void k_clear(int32_t* __restrict__ a, long long n, int* __restrict__ bad) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    a[i] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) *bad = 0;
}

template <bool PBC>
__device__ __forceinline__ void bin_one(int i, const float* __restrict__ pos, float inv, uint32_t mask,
                                        int32_t* __restrict__ atom_bucket, int32_t* __restrict__ count,
                                        int* __restrict__ bad, const Box& box) {
  const float3 p = load_pos(pos, i);
  uint32_t h;
  if constexpr (PBC) {
    // inside the box (false for NaN as well)
    const bool ok = p.x >= 0.0f && p.x < box.L[0] && p.y >= 0.0f && p.y < box.L[1] && p.z >= 0.0f && p.z < box.L[2];
    if (!ok) atomicOr(bad, 1);
    h = cell_hash(pbc_cell(p.x, box.inv[0], box.n[0]), pbc_cell(p.y, box.inv[1], box.n[1]),
                  pbc_cell(p.z, box.inv[2], box.n[2]), mask);
  } else {
    const float qx = __fmul_rn(p.x, inv), qy = __fmul_rn(p.y, inv), qz = __fmul_rn(p.z, inv);
    // false for NaN as well as for out-of-range coordinates
    const bool ok = fabsf(qx) < kCellRange && fabsf(qy) < kCellRange && fabsf(qz) < kCellRange;
    if (!ok) atomicOr(bad, 1);
    h = cell_hash(cell_of(p.x, inv), cell_of(p.y, inv), cell_of(p.z, inv), mask);
  }
  atom_bucket[i] = (int32_t)h;
  atomicAdd(count + h, 1);
}

template <bool PBC>
__global__ void k_bin(const float* __restrict__ pos, int N, float inv, uint32_t mask, int32_t* __restrict__ atom_bucket,
                      int32_t* __restrict__ count, int* __restrict__ bad, const Box box) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < N) bin_one<PBC>(i, pos, inv, mask, atom_bucket, count, bad, box);
}

// Atoms listed bucket by bucket, with a copy of their positions in the same
// order, so that the neighbour walk reads candidates' positions contiguously.
__device__ __forceinline__ void scatter_one(int i, const float* __restrict__ pos, const int32_t* __restrict__ atom_bucket,
                                            const int32_t* __restrict__ start, int32_t* __restrict__ fill,
                                            int32_t* __restrict__ bucket_atoms, float4* __restrict__ bucket_pos) {
  const int h = atom_bucket[i];
  const int slot = start[h] + atomicAdd(fill + h, 1);
  bucket_atoms[slot] = i;
  const float3 p = load_pos(pos, i);
  bucket_pos[slot] = make_float4(p.x, p.y, p.z, 0.0f);
}

__global__ void k_scatter(const float* __restrict__ pos, int N, const int32_t* __restrict__ atom_bucket,
                          const int32_t* __restrict__ start, int32_t* __restrict__ fill,
                          int32_t* __restrict__ bucket_atoms, float4* __restrict__ bucket_pos) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < N) scatter_one(i, pos, atom_bucket, start, fill, bucket_atoms, bucket_pos);
}

// ------------------------------------------------------------ neighbour walk
// One warp per receiver, receivers taken in bucket order so that the warps
// of a CTA read the same buckets.  Lanes 0..26 each name one of the 27
// surrounding cells' buckets (a bucket two cells hash to is kept once, by
// its lowest lane); the warp then walks the concatenation of those buckets,
// one candidate per lane per round, finding each candidate's bucket by a
// binary search over the lanes' running sizes.
// MODE kWalkCount:   row_offsets[i] = degree of i (row_offsets[N] = 0).
// MODE kWalkFill:    senders of i written, unsorted, to src[off[i] .. off[i+1]).
// MODE kWalkScratch: the count of kWalkCount, and the first kRowScratch
//                    senders (in walk order) into cand[i * kRowScratch ..],
//                    so that rows that fit need no second walk.
// (The rows longer than kRowScratch are filled afterwards by fixup_rows.)
// PBC: each lane names a (wrapped cell, image) pair; duplicates are merged
// on (bucket, image); a candidate is tested with its lane's image shift and
// the fill writes sender * 27 + image.
template <int MODE, bool PBC>
__device__ __forceinline__ void neigh_row(long long wg, int lane, const float4* __restrict__ bucket_pos, float inv,
                                          float rc2, uint32_t mask, const int32_t* __restrict__ start,
                                          const int32_t* __restrict__ bucket_atoms,
                                          int32_t* __restrict__ row_offsets, int32_t* __restrict__ src,
                                          long long e_cap, const Box& box, int32_t* __restrict__ cand = nullptr) {
  constexpr bool FILL = MODE == kWalkFill;
  const int i = bucket_atoms[wg];  // the receiver sits at slot wg of the bucket order
  const float4 pw = bucket_pos[wg];
  const float3 pi = make_float3(pw.x, pw.y, pw.z);
  long long w = 0, w_end = 0;
  if (FILL) {
    w = row_offsets[i];
    w_end = row_offsets[i + 1];
    if (w < 0 || w_end > e_cap || w_end < w) return;  // row outside the caller's capacity
  }
  uint32_t h;
  int sigma = kSelfImage;  // this lane's image (PBC)
  unsigned same;
  if constexpr (PBC) {
    const int dc[3] = {lane % 3 - 1, (lane / 3) % 3 - 1, lane / 9 - 1};
    const float pc[3] = {pi.x, pi.y, pi.z};
    int wc[3], sh[3];
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      if (box.n[a] == 1) {  // one cell: the neighbour "cells" are its images
        wc[a] = 0;
        sh[a] = dc[a];
      } else {
        const int t = pbc_cell(pc[a], box.inv[a], box.n[a]) + dc[a];
        sh[a] = t < 0 ? -1 : (t >= box.n[a] ? 1 : 0);
        wc[a] = t - sh[a] * box.n[a];
      }
    }
    sigma = (sh[0] + 1) + 3 * (sh[1] + 1) + 9 * (sh[2] + 1);
    h = lane < 27 ? cell_hash(wc[0], wc[1], wc[2], mask) : 0xffffffffu;
    same = __match_any_sync(0xffffffffu, ((unsigned long long)h << 5) | (unsigned)sigma);
  } else {
    const int cx = cell_of(pi.x, inv), cy = cell_of(pi.y, inv), cz = cell_of(pi.z, inv);
    h = lane < 27 ? cell_hash(cx + lane % 3 - 1, cy + (lane / 3) % 3 - 1, cz + lane / 9 - 1, mask) : 0xffffffffu;
    same = __match_any_sync(0xffffffffu, h);
  }
  const bool keep = lane < 27 && (same & ((1u << lane) - 1u)) == 0u;
  const int b0 = keep ? start[h] : 0;
  const int nb = keep ? start[h + 1] - b0 : 0;
  int incl = nb;  // running size of the buckets of lanes 0..lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  int count = 0;
  for (int base = 0; base < total; base += 32) {
    const int t = base + lane;
    // smallest lane L with incl[L] > t
    int L = 0;
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) {
      const int v = __shfl_sync(0xffffffffu, incl, L + step - 1);
      if (v <= t) L += step;
    }
    L = min(L, 31);
    const int lb0 = __shfl_sync(0xffffffffu, b0, L);
    const int lex = __shfl_sync(0xffffffffu, incl - nb, L);
    const int lsig = PBC ? __shfl_sync(0xffffffffu, sigma, L) : kSelfImage;
    bool hit = false;
    const int slot = lb0 + (t - lex);
    if (t < total) {
      const float4 q = bucket_pos[slot];
      if constexpr (PBC)
        hit = (slot != wg || lsig != kSelfImage) && norm2(image_vec(pi, make_float3(q.x, q.y, q.z), lsig, box)) < rc2;
      else
        hit = slot != wg && dist2(pi, make_float3(q.x, q.y, q.z)) < rc2;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    if (FILL) {
      const long long at = w + __popc(bal & ((1u << lane) - 1u));
      if (hit && at < w_end) src[at] = PBC ? bucket_atoms[slot] * kImages + lsig : bucket_atoms[slot];
      w += __popc(bal);
    } else {
      if (MODE == kWalkScratch) {
        const int at = count + __popc(bal & ((1u << lane) - 1u));
        if (hit && at < kRowScratch)
          cand[(size_t)i * kRowScratch + at] = PBC ? bucket_atoms[slot] * kImages + lsig : bucket_atoms[slot];
      }
      count += __popc(bal);
    }
  }
  if (!FILL && lane == 0) row_offsets[i] = count;
}

template <int MODE, bool PBC>
__global__ void __launch_bounds__(kNeighThreads) k_neigh(const float4* __restrict__ bucket_pos, int N, float inv,
                                                         float rc2, uint32_t mask, const int32_t* __restrict__ start,
                                                         const int32_t* __restrict__ bucket_atoms,
                                                         int32_t* __restrict__ row_offsets,
                                                         int32_t* __restrict__ src, long long e_cap, const Box box,
                                                         int32_t* __restrict__ cand) {
  constexpr bool FILL = MODE == kWalkFill;
  const int lane = threadIdx.x & 31;
  const long long wg = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (!FILL && wg == 0 && lane == 0) row_offsets[N] = 0;
  if (wg < N)
    neigh_row<MODE, PBC>(wg, lane, bucket_pos, inv, rc2, mask, start, bucket_atoms, row_offsets, src, e_cap, box,
                         cand);
}

// Second walk of the single-walk path: thread t checks the receiver at slot
// t of the bucket order, and its warp walks together (kWalkFill) each of
// its 32 receivers whose row is longer than the scratch row.
template <bool PBC>
__device__ __forceinline__ void fixup_rows(long long base, int lane, long long n, const float4* __restrict__ bucket_pos,
                                           float inv, float rc2, uint32_t mask, const int32_t* __restrict__ start,
                                           const int32_t* __restrict__ bucket_atoms,
                                           int32_t* __restrict__ row_offsets, int32_t* __restrict__ src,
                                           long long e_cap, const Box& box) {
  const long long wg = base + lane;
  bool longer = false;
  if (wg < n) {
    const int i = bucket_atoms[wg];
    longer = (long long)row_offsets[i + 1] - row_offsets[i] > kRowScratch;
  }
  unsigned todo = __ballot_sync(0xffffffffu, longer);
  while (todo) {
    const int l = __ffs(todo) - 1;
    todo &= todo - 1;
    neigh_row<kWalkFill, PBC>(base + l, lane, bucket_pos, inv, rc2, mask, start, bucket_atoms, row_offsets, src,
                              e_cap, box);
  }
}

template <bool PBC>
__global__ void __launch_bounds__(kNeighThreads) k_fixup(const float4* __restrict__ bucket_pos, int N, float inv,
                                                         float rc2, uint32_t mask, const int32_t* __restrict__ start,
                                                         const int32_t* __restrict__ bucket_atoms,
                                                         int32_t* __restrict__ row_offsets,
                                                         int32_t* __restrict__ src, long long e_cap, const Box box) {
  const long long base = ((long long)blockIdx.x * blockDim.x + threadIdx.x) & ~31ll;
  fixup_rows<PBC>(base, threadIdx.x & 31, N, bucket_pos, inv, rc2, mask, start, bucket_atoms, row_offsets, src,
                  e_cap, box);
}

// ------------------------------------------------------------ row sort
// One warp per receiver.  Senders in a row are distinct, so the rank of a
// sender (the number of smaller ones) is its sorted position.  Rows up to
// kSortCap are ranked from shared memory; longer rows are staged in the
// row's own vec storage (3 words per edge, so it holds the row) and ranked
// from there before vec is written.
// PBC: the row holds keys sender * 27 + image (distinct); ranked the same
// way, then written as src (sender), img (image) and vec (the image's d).
template <bool PBC>
__device__ __forceinline__ void put_edge(long long e, int key, int i, float3 pi, const float* __restrict__ pos,
                                         int32_t* __restrict__ src, int32_t* __restrict__ img,
                                         float* __restrict__ vec, int32_t* __restrict__ dst, const Box& box) {
  float* o = vec + 3 * e;
  if constexpr (PBC) {
    const int j = key / kImages, sigma = key - j * kImages;
    const float3 d = image_vec(pi, load_pos(pos, j), sigma, box);
    src[e] = j;
    img[e] = sigma;
    o[0] = d.x;
    o[1] = d.y;
    o[2] = d.z;
  } else {
    const float3 pj = load_pos(pos, key);
    src[e] = key;
    o[0] = __fsub_rn(pj.x, pi.x);
    o[1] = __fsub_rn(pj.y, pi.y);
    o[2] = __fsub_rn(pj.z, pi.z);
  }
  if (dst) dst[e] = i;
}

// cand (single-walk path): rows of at most kRowScratch senders come from
// the counting walk's scratch row instead of src.
template <bool PBC>
__device__ __forceinline__ void sort_row(int i, int lane, int32_t* sm, const float* __restrict__ pos,
                                         const int32_t* __restrict__ row_offsets, int32_t* __restrict__ src,
                                         int32_t* __restrict__ img, float* __restrict__ vec,
                                         int32_t* __restrict__ dst, long long e_cap, const Box& box,
                                         const int32_t* __restrict__ cand = nullptr) {
  const long long beg = row_offsets[i], end = row_offsets[i + 1];
  if (beg < 0 || end > e_cap || end < beg) return;
  const int k = (int)(end - beg);
  const float3 pi = load_pos(pos, i);
  int32_t* row = src + beg;
  const int32_t* from = cand && k <= kRowScratch ? cand + (size_t)i * kRowScratch : row;
  if (k <= kSortCap) {
    for (int a = lane; a < k; a += 32) sm[a] = from[a];
    __syncwarp();
    for (int a = lane; a < k; a += 32) {
      const int v = sm[a];
      int r = 0;
      for (int b = 0; b < k; ++b) r += sm[b] < v;
      put_edge<PBC>(beg + r, v, i, pi, pos, src, img, vec, dst, box);
    }
    return;
  }
  int32_t* stage = reinterpret_cast<int32_t*>(vec + 3 * beg);
  for (int a = lane; a < k; a += 32) stage[a] = row[a];
  __syncwarp();
  for (int a = lane; a < k; a += 32) {
    const int v = stage[a];
    int r = 0;
    for (int b = 0; b < k; ++b) r += stage[b] < v;
    row[r] = v;
  }
  __syncwarp();
  for (int a = lane; a < k; a += 32) put_edge<PBC>(beg + a, row[a], i, pi, pos, src, img, vec, dst, box);
}

template <bool PBC>
__global__ void __launch_bounds__(kSortWarps * 32) k_sort(const float* __restrict__ pos, int N,
                                                          const int32_t* __restrict__ row_offsets,
                                                          int32_t* __restrict__ src, int32_t* __restrict__ img,
                                                          float* __restrict__ vec, int32_t* __restrict__ dst,
                                                          long long e_cap, const Box box,
                                                          const int32_t* __restrict__ cand) {
  __shared__ int32_t rows[kSortWarps][kSortCap];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int i = blockIdx.x * kSortWarps + wid;
  if (i < N) sort_row<PBC>(i, lane, rows[wid], pos, row_offsets, src, img, vec, dst, e_cap, box, cand);
}

// rev[e] for e = (i <- j): the position of (j <- i) in row j (binary search;
// the relation is symmetric, so it exists).
// PBC: the reverse of (i <- j, image s) is (j <- i, image -s), i.e. the key
// i * 27 + (26 - sigma) in row j.
template <bool PBC>
__device__ __forceinline__ void rev_row(int i, int lane, const int32_t* __restrict__ row_offsets,
                                        const int32_t* __restrict__ src, const int32_t* __restrict__ img,
                                        int32_t* __restrict__ rev, long long e_cap) {
  const long long beg = row_offsets[i], end = row_offsets[i + 1];
  if (beg < 0 || end > e_cap || end < beg) return;
  for (long long e = beg + lane; e < end; e += 32) {
    const int j = src[e];
    long long lo = row_offsets[j], hi = row_offsets[j + 1];
    if (lo < 0 || hi > e_cap || hi < lo) {
      rev[e] = -1;
      continue;
    }
    const long long want = PBC ? (long long)i * kImages + (kImages - 1 - img[e]) : i;
    while (lo < hi) {
      const long long mid = (lo + hi) >> 1;
      const long long key = PBC ? (long long)src[mid] * kImages + img[mid] : src[mid];
      if (key < want) lo = mid + 1;
      else hi = mid;
    }
    const long long got = lo < row_offsets[j + 1] ? (PBC ? (long long)src[lo] * kImages + img[lo] : src[lo]) : -1;
    rev[e] = got == want ? (int32_t)lo : -1;
  }
}

template <bool PBC>
__global__ void k_rev(int N, const int32_t* __restrict__ row_offsets, const int32_t* __restrict__ src,
                      const int32_t* __restrict__ img, int32_t* __restrict__ rev, long long e_cap) {
  const int lane = threadIdx.x & 31;
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (i < N) rev_row<PBC>(i, lane, row_offsets, src, img, rev, e_cap);
}

// ------------------------------------------------------------ one launch
// The whole pipeline in one cooperative launch (every CTA resident), the
// phases separated by grid barriers: for small systems the twelve launches
// of the multi-kernel path cost more than their work.
struct CoopArgs {
  const float* pos;
  int N;
  float inv, rc2;
  uint32_t mask;
  long long H, n_clear, e_cap;
  int32_t *atom_bucket, *start, *fill, *bucket_atoms;
  float4* bucket_pos;
  int* bad;
  long long* sums;     // [gridDim.x] block totals
  unsigned* bar;       // [2]: arrivals, completed generations (zeroed before the launch)
  int32_t *row_offsets, *src, *dst, *rev, *img;
  float* vec;
  long long* e_total;
  int* watchdog;
  Box box;  // periodic box (k_graph_coop<true>)
  int32_t* cand;  // per-row scratch of the single walk, or nullptr
};

// Grid barrier with a bounded wait: false (and the watchdog set) if the
// other CTAs did not all arrive within kGridWaitNs.
__device__ __forceinline__ bool grid_sync(unsigned* bar, unsigned& gen, int* watchdog) {
  __shared__ int ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    ++gen;
    ok = 1;
    __threadfence();
    const unsigned arrived = atomicAdd(bar, 1u) + 1u;
    if (arrived == gen * gridDim.x) {
      __threadfence();
      atomicExch(bar + 1, gen);
    } else {
      const unsigned long long t0 = global_ns();
      while (*reinterpret_cast<volatile unsigned*>(bar + 1) < gen) {
        if (global_ns() - t0 > kGridWaitNs) {
          watchdog_trip(watchdog, 4);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
  return ok != 0;
}

// Exclusive scan of data[0..n) across the grid: each CTA scans a contiguous
// chunk (tiles of 1024 with a running carry), a barrier, then each CTA adds
// the totals of the CTAs before it.  64-bit totals; *total_out (if given) =
// the grand total, reported as for the multi-kernel path.
__device__ bool grid_scan(int32_t* data, long long n, long long* sums, unsigned* bar, unsigned& gen, int* watchdog,
                          const int* bad, long long* total_out) {
  __shared__ long long warp_tot[32];
  __shared__ long long total;
  const long long chunk = (n + gridDim.x - 1) / gridDim.x;
  const long long lo = min(n, (long long)blockIdx.x * chunk), hi = min(n, lo + chunk);
  long long carry = 0;
  for (long long base = lo; base < hi; base += 4 * blockDim.x) {
    const long long i0 = base + 4 * threadIdx.x;
    int v[4];
    long long s = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[k] = i0 + k < hi ? data[i0 + k] : 0;
      s += v[k];
    }
    long long run = carry + block_exclusive(s, warp_tot, &total);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (i0 + k < hi) data[i0 + k] = (int32_t)run;
      run += v[k];
    }
    carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) sums[blockIdx.x] = carry;
  if (!grid_sync(bar, gen, watchdog)) return false;
  long long before = 0, all = 0;
  for (unsigned b = threadIdx.x; b < gridDim.x; b += blockDim.x) {
    const long long t = sums[b];
    all += t;
    if (b < blockIdx.x) before += t;
  }
  // block sums of `before` and `all` (fixed-order tree: integers, exact)
  before = block_exclusive(before, warp_tot, &total), before = total;
  __syncthreads();
  all = block_exclusive(all, warp_tot, &total), all = total;
  for (long long i = lo + threadIdx.x; i < hi; i += blockDim.x) data[i] += (int32_t)before;
  if (total_out && blockIdx.x == 0 && threadIdx.x == 0) {
    long long e = all;
    if (e > INT32_MAX) e = -2;
    if (*bad) e = -1;
    *total_out = e;
  }
  return grid_sync(bar, gen, watchdog);
}

template <bool PBC>
__global__ void __launch_bounds__(kSortWarps * 32) k_graph_coop(const CoopArgs g) {
  __shared__ int32_t rows[kSortWarps][kSortCap];
  unsigned gen = 0;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const long long warp0 = (long long)blockIdx.x * kSortWarps + wid, nwarps = (long long)gridDim.x * kSortWarps;
  for (long long i = tid; i < g.n_clear; i += nthreads) g.start[i] = 0;
  if (tid == 0) *g.bad = 0;
  if (!grid_sync(g.bar, gen, g.watchdog)) return;
  for (long long i = tid; i < g.N; i += nthreads)
    bin_one<PBC>((int)i, g.pos, g.inv, g.mask, g.atom_bucket, g.start, g.bad, g.box);
  if (!grid_sync(g.bar, gen, g.watchdog)) return;
  if (!grid_scan(g.start, g.H + 1, g.sums, g.bar, gen, g.watchdog, g.bad, nullptr)) return;
  for (long long i = tid; i < g.N; i += nthreads)
    scatter_one((int)i, g.pos, g.atom_bucket, g.start, g.fill, g.bucket_atoms, g.bucket_pos);
  if (!grid_sync(g.bar, gen, g.watchdog)) return;
  if (tid == 0) g.row_offsets[g.N] = 0;
  // one walk counts each row and keeps its first kRowScratch senders; the
  // second walk fills only longer rows (see radius_graph_run)
  for (long long w = warp0; w < g.N; w += nwarps) {
    if (g.cand)
      neigh_row<kWalkScratch, PBC>(w, lane, g.bucket_pos, g.inv, g.rc2, g.mask, g.start, g.bucket_atoms,
                                   g.row_offsets, nullptr, g.e_cap, g.box, g.cand);
    else
      neigh_row<kWalkCount, PBC>(w, lane, g.bucket_pos, g.inv, g.rc2, g.mask, g.start, g.bucket_atoms,
                                 g.row_offsets, nullptr, g.e_cap, g.box);
  }
  if (!grid_sync(g.bar, gen, g.watchdog)) return;
  if (!grid_scan(g.row_offsets, (long long)g.N + 1, g.sums, g.bar, gen, g.watchdog, g.bad, g.e_total)) return;
  if (g.e_cap <= 0) return;
  if (g.cand) {
    for (long long b = warp0 * 32; b < g.N; b += nwarps * 32)
      fixup_rows<PBC>(b, lane, g.N, g.bucket_pos, g.inv, g.rc2, g.mask, g.start, g.bucket_atoms, g.row_offsets,
                      g.src, g.e_cap, g.box);
  } else {
    for (long long w = warp0; w < g.N; w += nwarps)
      neigh_row<kWalkFill, PBC>(w, lane, g.bucket_pos, g.inv, g.rc2, g.mask, g.start, g.bucket_atoms,
                                g.row_offsets, g.src, g.e_cap, g.box);
  }
  if (!grid_sync(g.bar, gen, g.watchdog)) return;
  for (long long i = warp0; i < g.N; i += nwarps)
    sort_row<PBC>((int)i, lane, rows[wid], g.pos, g.row_offsets, g.src, g.img, g.vec, g.dst, g.e_cap, g.box,
                  g.cand);
  if (!g.rev) return;
  if (!grid_sync(g.bar, gen, g.watchdog)) return;
  for (long long i = warp0; i < g.N; i += nwarps)
    rev_row<PBC>((int)i, lane, g.row_offsets, g.src, g.img, g.rev, g.e_cap);
}

// ------------------------------------------------------------ workspace
struct GraphWs {
  long long H = 0;
  size_t atom_bucket = 0, start = 0, fill = 0, scan_a = 0, scan_b = 0, tickets = 0, bucket_atoms = 0, bucket_pos = 0,
         bad = 0, coop = 0, cand = 0, bytes = 0;
  bool scratch = false;  // the single-walk path's per-row scratch is present
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

GraphWs graph_ws(long long N) {
  GraphWs w;
  long long H = 64;
  while (H < 2 * N) H <<= 1;
  w.H = H;
  const long long scan_n = (H + 1 > N + 1 ? H + 1 : N + 1);
  const long long nb = (scan_n + kScanTile - 1) / kScanTile;
  size_t o = 0;
  w.atom_bucket = o; o = align256(o + 4 * (size_t)N);
  w.start = o;       o = align256(o + 4 * (size_t)(H + 1));
  w.fill = o;        o = align256(o + 4 * (size_t)H);
  // single-pass scan status (bucket starts, row offsets) and tickets; zeroed
  // with start and fill
  w.scan_a = o;      o = align256(o + 8 * (size_t)nb);
  w.scan_b = o;      o = align256(o + 8 * (size_t)nb);
  w.tickets = o;     o = align256(o + 8);
  w.bucket_atoms = o; o = align256(o + 4 * (size_t)N);
  w.bucket_pos = o;  o = align256(o + 16 * (size_t)N);
  w.bad = o;         o = align256(o + 4);
  w.coop = o;        o = align256(o + 8 * (size_t)kCoopMaxBlocks + 16);  // block totals + barrier words
  // single-walk scratch rows
  w.scratch = N <= kScratchMaxAtoms;
  w.cand = o;        o = align256(o + (w.scratch ? 4 * (size_t)kRowScratch * (size_t)N : 0));
  w.bytes = o;
  return w;
}

}  // namespace
}  // namespace eqmp

using namespace eqmp;

extern "C" {

size_t eqmp_radius_graph_workspace_size(int64_t N) {
  if (N < 0 || N > kGraphMaxAtoms) return 0;
  return graph_ws(N).bytes;
}

}  // extern "C"

namespace eqmp {
namespace {

// Both entry points: argument checks done, box set up when PBC.
template <bool PBC>
eqmp_status radius_graph_run(const float* pos, int64_t N, float cutoff, const Box& box, int32_t* row_offsets,
                             int32_t* src, float* vec, int32_t* img, int32_t* dst, int32_t* rev, int64_t E_cap,
                             int64_t* E_total, void* workspace, size_t workspace_bytes, cudaStream_t st) {
  const GraphWs w = graph_ws(N);
  if (!workspace || workspace_bytes < w.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return EQMP_ERR_INVALID_ARG;
  char* base = static_cast<char*>(workspace);
  int32_t* atom_bucket = reinterpret_cast<int32_t*>(base + w.atom_bucket);
  int32_t* start = reinterpret_cast<int32_t*>(base + w.start);
  int32_t* fill = reinterpret_cast<int32_t*>(base + w.fill);
  int32_t* bucket_atoms = reinterpret_cast<int32_t*>(base + w.bucket_atoms);
  float4* bucket_pos = reinterpret_cast<float4*>(base + w.bucket_pos);
  int* bad = reinterpret_cast<int*>(base + w.bad);
  // start and fill are adjacent: one clear covers both
  const long long n_clear = (long long)((w.bucket_atoms - w.start) / 4);

  const double cell = (double)cutoff * (1.0 + 1.0 / 1024.0);
  const float inv = (float)(1.0 / cell);
  const float rc2 = cutoff * cutoff;
  const uint32_t mask = (uint32_t)(w.H - 1);
  const int nblk = (int)((N + kNeighThreads - 1) / kNeighThreads);

  // One cooperative launch when the device allows it (grid sized to the
  // work: one warp per receiver, at most what is resident at once).
  {
    static int occ_cache[64] = {0};
    int d = 0;
    cudaGetDevice(&d);
    int occ = __atomic_load_n(&occ_cache[d & 63], __ATOMIC_RELAXED);
    if (occ == 0) {
      int coop = 0;
      if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, d) != cudaSuccess) return EQMP_ERR_CUDA;
      if (!coop || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_graph_coop<PBC>, kSortWarps * 32, 0) !=
                       cudaSuccess || occ < 1)
        occ = -1;  // multi-kernel path only
      __atomic_store_n(&occ_cache[d & 63], occ, __ATOMIC_RELAXED);
    }
    DeviceInfo dev;
    // measured: one launch wins while the launches dominate (up to ~10k
    // atoms); above that the per-phase launch shapes of the multi-kernel
    // path are faster
    if (occ > 0 && N <= kCoopMaxAtoms && device_info(&dev) == EQMP_OK) {
      long long grid = (long long)dev.sms * occ;
      const long long want = (N + kSortWarps - 1) / kSortWarps;
      if (grid > want) grid = want > 0 ? want : 1;
      if (grid > kCoopMaxBlocks) grid = kCoopMaxBlocks;
      CoopArgs g{};
      g.pos = pos; g.N = (int)N; g.inv = inv; g.rc2 = rc2; g.mask = mask; g.H = w.H; g.n_clear = n_clear;
      g.e_cap = E_cap; g.atom_bucket = atom_bucket; g.start = start; g.fill = fill; g.bucket_atoms = bucket_atoms;
      g.bucket_pos = bucket_pos; g.bad = bad;
      g.sums = reinterpret_cast<long long*>(base + w.coop);
      g.bar = reinterpret_cast<unsigned*>(base + w.coop + 8 * (size_t)kCoopMaxBlocks);
      g.row_offsets = row_offsets; g.src = src; g.dst = dst; g.rev = rev; g.img = img; g.vec = vec;
      g.e_total = reinterpret_cast<long long*>(E_total);
      g.watchdog = dev.watchdog;
      g.box = box;
      g.cand = w.scratch ? reinterpret_cast<int32_t*>(base + w.cand) : nullptr;
      if (cudaMemsetAsync(g.bar, 0, 2 * sizeof(unsigned), st) != cudaSuccess) return EQMP_ERR_CUDA;
      void* params[] = {&g};
      const cudaError_t err = cudaLaunchCooperativeKernel((const void*)k_graph_coop<PBC>, dim3((unsigned)grid),
                                                          dim3(kSortWarps * 32), params, 0, st);
      if (err == cudaSuccess) return EQMP_OK;
      (void)cudaGetLastError();  // fall through to the multi-kernel path
    }
  }

  k_clear<<<256, 256, 0, st>>>(start, n_clear, bad);
  if (N > 0) {
    k_bin<PBC><<<nblk, kNeighThreads, 0, st>>>(pos, (int)N, inv, mask, atom_bucket, start, bad, box);
  }
  DeviceInfo sdev;
  if (device_info(&sdev) != EQMP_OK) return EQMP_ERR_CUDA;
  unsigned* tickets = reinterpret_cast<unsigned*>(base + w.tickets);
  cudaError_t err = exclusive_scan(start, w.H + 1, reinterpret_cast<unsigned long long*>(base + w.scan_a), tickets,
                                   bad, nullptr, sdev.watchdog, st);
  if (err != cudaSuccess) return EQMP_ERR_CUDA;
  if (N > 0)
    k_scatter<<<nblk, kNeighThreads, 0, st>>>(pos, (int)N, atom_bucket, start, fill, bucket_atoms, bucket_pos);
  // One walk counts each row and keeps its first kRowScratch senders; after
  // the scan a second walk fills only the rows longer than that (without the
  // scratch: a counting walk, then a filling walk of every row).
  const long long wblk = (N * 32 + kNeighThreads - 1) / kNeighThreads;  // one warp per receiver
  int32_t* cand = w.scratch ? reinterpret_cast<int32_t*>(base + w.cand) : nullptr;
  if (cand)
    k_neigh<kWalkScratch, PBC><<<(unsigned)(wblk > 0 ? wblk : 1), kNeighThreads, 0, st>>>(
        bucket_pos, (int)N, inv, rc2, mask, start, bucket_atoms, row_offsets, nullptr, E_cap, box, cand);
  else
    k_neigh<kWalkCount, PBC><<<(unsigned)(wblk > 0 ? wblk : 1), kNeighThreads, 0, st>>>(
        bucket_pos, (int)N, inv, rc2, mask, start, bucket_atoms, row_offsets, nullptr, E_cap, box, nullptr);
  err = exclusive_scan(row_offsets, N + 1, reinterpret_cast<unsigned long long*>(base + w.scan_b), tickets + 1, bad,
                       reinterpret_cast<long long*>(E_total), sdev.watchdog, st);
  if (err != cudaSuccess) return EQMP_ERR_CUDA;
  if (N > 0 && E_cap > 0) {
    if (cand)
      k_fixup<PBC><<<(unsigned)((N + kNeighThreads - 1) / kNeighThreads), kNeighThreads, 0, st>>>(
          bucket_pos, (int)N, inv, rc2, mask, start, bucket_atoms, row_offsets, src, E_cap, box);
    else
      k_neigh<kWalkFill, PBC><<<(unsigned)wblk, kNeighThreads, 0, st>>>(
          bucket_pos, (int)N, inv, rc2, mask, start, bucket_atoms, row_offsets, src, E_cap, box, nullptr);
    const int sblk = (int)((N + kSortWarps - 1) / kSortWarps);
    k_sort<PBC><<<sblk, kSortWarps * 32, 0, st>>>(pos, (int)N, row_offsets, src, img, vec, dst, E_cap, box, cand);
    if (rev) k_rev<PBC><<<sblk, kSortWarps * 32, 0, st>>>((int)N, row_offsets, src, img, rev, E_cap);
  }
  return cuda_status(cudaGetLastError());
}

eqmp_status graph_args_ok(const float* pos, int64_t N, float cutoff, const int32_t* row_offsets, const int32_t* src,
                          const float* vec, int64_t E_cap, const int64_t* E_total, int64_t n_max) {
  if (N < 0 || E_cap < 0) return EQMP_ERR_INVALID_ARG;
  if (N > n_max) return EQMP_ERR_UNSUPPORTED;
  if (!(cutoff > 0.0f) || !isfinite(cutoff)) return EQMP_ERR_INVALID_ARG;
  if (!row_offsets || !E_total) return EQMP_ERR_INVALID_ARG;
  if (N > 0 && !pos) return EQMP_ERR_INVALID_ARG;
  if (E_cap > 0 && (!src || !vec)) return EQMP_ERR_INVALID_ARG;
  return EQMP_OK;
}

}  // namespace
}  // namespace eqmp

extern "C" {

eqmp_status eqmp_radius_graph(const float* pos, int64_t N, float cutoff, int32_t* row_offsets, int32_t* src,
                              float* vec, int32_t* dst, int32_t* rev, int64_t E_cap, int64_t* E_total,
                              void* workspace, size_t workspace_bytes, eqmp_stream_t stream) {
  const eqmp_status s = graph_args_ok(pos, N, cutoff, row_offsets, src, vec, E_cap, E_total, kGraphMaxAtoms);
  if (s != EQMP_OK) return s;
  return radius_graph_run<false>(pos, N, cutoff, Box{}, row_offsets, src, vec, nullptr, dst, rev, E_cap, E_total,
                                 workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

eqmp_status eqmp_radius_graph_pbc(const float* pos, int64_t N, float cutoff, const float* box_lengths,
                                  int32_t* row_offsets, int32_t* src, float* vec, int32_t* img, int32_t* dst,
                                  int32_t* rev, int64_t E_cap, int64_t* E_total, void* workspace,
                                  size_t workspace_bytes, eqmp_stream_t stream) {
  const eqmp_status s = graph_args_ok(pos, N, cutoff, row_offsets, src, vec, E_cap, E_total, kGraphMaxAtomsPbc);
  if (s != EQMP_OK) return s;
  if (!box_lengths || (E_cap > 0 && !img)) return EQMP_ERR_INVALID_ARG;
  Box box{};
  for (int a = 0; a < 3; ++a) {
    const float L = box_lengths[a];
    if (!(L > 0.0f) || !isfinite(L)) return EQMP_ERR_INVALID_ARG;
    if (cutoff > L) return EQMP_ERR_UNSUPPORTED;  // more than one image per direction
    box.L[a] = L;
    // cells of side >= r_c (1 + 2^-10) tile the axis; fewer than three
    // become one cell whose images are walked; at most kCellRange per axis
    // (the cell index of a coordinate is then exact to well within the margin)
    double n = floor((double)L / ((double)cutoff * (1.0 + 1.0 / 1024.0)));
    if (n > (double)kCellRange) n = (double)kCellRange;
    box.n[a] = n < 3.0 ? 1 : (int)n;
    box.inv[a] = (float)((double)box.n[a] / (double)L);
  }
  return radius_graph_run<true>(pos, N, cutoff, box, row_offsets, src, vec, img, dst, rev, E_cap, E_total,
                                workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
