// Kernel argument block shared by the layer kernels.
#pragma once
#include <stdint.h>

namespace eqmp {

struct LayerArgs {
  const float* vec;       // [E][3]  (fused) or nullptr
  const float* Y;         // [E][16] (tp_scatter) or nullptr
  const void* x;          // [N_src][C][16] fp32 or bf16
  const int32_t* off;     // [N+1] absolute CSR offsets
  const int32_t* src;     // [E]
  const float* w;         // [34][C]       shared weights, or nullptr
  const float* R;         // [E][8]        radial features, or nullptr
  const float* M;         // [8][34*C]     radial mixing matrix, or nullptr
  void* out;              // [N][C][16] fp32 or bf16
  int* watchdog;          // device watchdog word
  int N;                  // receivers
  int E;                  // edges in vec / Y / src / R
  int N_src;              // rows of x
  // Transposed pass (gradient of x): row r of the walk is sender r; its
  // edges are perm[off[r] .. off[r+1]) (edge ids), each gathering the row
  // x[dst[e]] with the harmonics of vec[e].  E counts perm; E_edges counts
  // the edge arrays vec and dst.
  const int32_t* perm;    // [E] edge ids, or nullptr
  const int32_t* dst;     // [E_edges] receiver of each edge, or nullptr
  int E_edges;
};

__host__ __device__ constexpr int round_up(int v, int m) { return (v + m - 1) / m * m; }

}  // namespace eqmp
