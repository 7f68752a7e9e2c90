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
                             RowMap map, int64_t n_total, double* __restrict__ row_losses,
                             unsigned int* __restrict__ counter) {
  const int a = blockIdx.y;
  if (a == 0 && blockIdx.x == 0 && threadIdx.x == 0) *counter = 0u;
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
// The last block to finish (counted on *counter, zeroed by k_row_losses)
// takes the argmin -- first minimum, NaN as +inf -- and copies the chosen
// scale vector to s_out.
__global__ void k_grid_losses(const double* __restrict__ row_losses, RowMap map, int64_t n_total,
                              int64_t T, double* __restrict__ losses, int* __restrict__ best,
                              double* __restrict__ alpha_out, const float* __restrict__ s_grid,
                              int64_t K, float* __restrict__ s_out,
                              unsigned int* __restrict__ counter) {
  __shared__ double red[256];
  __shared__ int last, chosen;
  const int a = blockIdx.x;
  const int n_grid = gridDim.x;
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
  if (threadIdx.x == 0) {
    losses[a] = total;
    __threadfence();
    last = (atomicAdd(counter, 1u) == static_cast<unsigned>(n_grid) - 1u);
  }
  __syncthreads();
  if (!last) return;
  if (threadIdx.x == 0) {
    __threadfence();
    const volatile double* lv = losses;
    int bi = 0;
    double bv = 0.0;
    for (int i = 0; i < n_grid; ++i) {
      const double v = isnan(lv[i]) ? INFINITY : lv[i];
      if (i == 0 || v < bv) {
        bi = i;
        bv = v;
      }
    }
    *best = bi;
    *alpha_out = static_cast<double>(bi) / static_cast<double>(n_grid);
    chosen = bi;
  }
  __syncthreads();
  const float* src = s_grid + static_cast<int64_t>(chosen) * K;
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x) s_out[k] = src[k];
}

}  // namespace

cudaError_t launch_loss_reduce(const float* partials, int n_alpha, int n_tiles, int64_t n_pad,
                               int64_t T, const RowMap& map, int64_t n_total,
                               double* row_losses, double* losses, int* best,
                               double* alpha_out, const float* s_grid, int64_t K, float* s_out,
                               unsigned int* counter, cudaStream_t st) {
  const dim3 g1(static_cast<unsigned>(ceil_div(n_pad, 256)), static_cast<unsigned>(n_alpha));
  k_row_losses<<<g1, 256, 0, st>>>(partials, n_tiles, n_pad, map, n_total, row_losses, counter);
  k_grid_losses<<<n_alpha, 256, 0, st>>>(row_losses, map, n_total, T, losses, best, alpha_out,
                                         s_grid, K, s_out, counter);
  return cudaGetLastError();
}

}  // namespace awq
