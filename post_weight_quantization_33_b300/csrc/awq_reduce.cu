// Per-row and per-grid-point losses, and the argmin over the grid.
//
// AWQ Explained (multigrid.ai), "How the scale is chosen": alpha* is the
// argmin over the grid of the layer-output error.  The error is the squared
// norm divided by N*T; weights sharing one X add their losses.  Every sum
// here runs in a fixed order in fp64, so the result is deterministic; the
// argmin takes the first minimum and treats NaN as +inf.
#include "awq_internal.h"

namespace awq {
namespace {

// row_losses[a][compact row] = sum over token tiles of partials[a][tile][virtual row].
__global__ void k_row_losses(const float* __restrict__ partials, int n_tiles, int64_t n_pad,
                             RowMap map, int64_t n_total, double* __restrict__ row_losses) {
  const int a = blockIdx.y;
  const int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (v >= n_pad) return;
  int w = 0;
  while (w + 1 < map.n_w && v >= map.pad_off[w + 1]) ++w;
  const int64_t n = v - map.pad_off[w];
  if (n >= map.rows[w]) return;   // padding row
  double s = 0.0;
  for (int t = 0; t < n_tiles; ++t)
    s += static_cast<double>(partials[(static_cast<int64_t>(a) * n_tiles + t) * n_pad + v]);
  row_losses[static_cast<int64_t>(a) * n_total + map.cum[w] + n] = s;
}

// losses[a] = sum_w (sum_n row_losses[a][w, n]) / (N_w * T); one block per a.
__global__ void k_grid_losses(const double* __restrict__ row_losses, RowMap map, int64_t n_total,
                              int64_t T, double* __restrict__ losses) {
  __shared__ double red[256];
  const int a = blockIdx.x;
  const double* rl = row_losses + static_cast<int64_t>(a) * n_total;
  double total = 0.0;
  for (int w = 0; w < map.n_w; ++w) {
    double s = 0.0;
    for (int64_t n = threadIdx.x; n < map.rows[w]; n += blockDim.x) s += rl[map.cum[w] + n];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int off = blockDim.x / 2; off; off >>= 1) {
      if (threadIdx.x < off) red[threadIdx.x] += red[threadIdx.x + off];
      __syncthreads();
    }
    if (threadIdx.x == 0)
      total += red[0] / (static_cast<double>(map.rows[w]) * static_cast<double>(T));
    __syncthreads();
  }
  if (threadIdx.x == 0) losses[a] = total;
}

__global__ void k_argmin(const double* __restrict__ losses, int n_grid, int* __restrict__ best,
                         double* __restrict__ alpha_out) {
  if (threadIdx.x != 0) return;
  int bi = 0;
  double bv = 0.0;
  for (int i = 0; i < n_grid; ++i) {
    const double v = isnan(losses[i]) ? INFINITY : losses[i];
    if (i == 0 || v < bv) {
      bi = i;
      bv = v;
    }
  }
  *best = bi;
  *alpha_out = static_cast<double>(bi) / static_cast<double>(n_grid);
}

}  // namespace

cudaError_t launch_loss_reduce(const float* partials, int n_alpha, int n_tiles, int64_t n_pad,
                               int64_t T, const RowMap& map, int64_t n_total,
                               double* row_losses, double* losses, int* best,
                               double* alpha_out, cudaStream_t st) {
  const dim3 g1(static_cast<unsigned>(ceil_div(n_pad, 256)), static_cast<unsigned>(n_alpha));
  k_row_losses<<<g1, 256, 0, st>>>(partials, n_tiles, n_pad, map, n_total, row_losses);
  k_grid_losses<<<n_alpha, 256, 0, st>>>(row_losses, map, n_total, T, losses);
  k_argmin<<<1, 32, 0, st>>>(losses, n_alpha, best, alpha_out);
  return cudaGetLastError();
}

}  // namespace awq
