// Per-row and per-grid-point losses, and the argmin over the grid.
//
// AWQ Explained (multigrid.ai), "How the scale is chosen": alpha* is the
// argmin over the grid of the layer-output error.  The error is the squared
// norm divided by N*T; weights sharing one X add their losses.  Every sum
// here runs in a fixed order, so the result is deterministic: in fp64, except
// the per-row sums over token tiles, which are compensated fp32 (about 2^-48
// relative) because this part has little fp64 throughput.  The argmin takes
// the first minimum and treats NaN as +inf.
#include "awq_bounds.cuh"
#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kLossRows = 256;   // rows per block (a chunk)

// Block (c, a): rows [256c, 256c + 256) of the padded row space, grid point
// a.  Per row: the sum over token tiles of partials[a][tile][row], in tile
// order (compensated fp32, then fp64), times *row_scale when given (the Gram form's scale), written to
// row_losses; per weight present in the chunk: the sum of
// its rows by a fixed tree, written to chunk_sums[a][c][w].  The last block
// to finish (counted on *counter, zeroed by the caller) adds the chunks of
// every grid point in chunk order, divides by N_w * T, sums the weights, takes
// the argmin -- first minimum, NaN as +inf -- and copies the chosen scale
// vector to s_out.  Every sum has a fixed order: the result is deterministic.
// A grid point whose loss is not finite sets *status to kDevNonFinite.
__global__ void __launch_bounds__(kLossRows)
    k_losses(const float* __restrict__ partials, int n_tiles, int64_t n_pad, RowMap map,
             int64_t n_total, int64_t T, double* __restrict__ chunk_sums,
             double* __restrict__ row_losses, double* __restrict__ losses,
             int* __restrict__ best, double* __restrict__ alpha_out,
             const float* __restrict__ s_grid, int64_t K, float* __restrict__ s_out,
             unsigned int* __restrict__ counter, const double* __restrict__ row_scale,
             int* __restrict__ status) {
  __shared__ double red[kLossRows];
  __shared__ int last, chosen;
  const int c = blockIdx.x;
  const int a = blockIdx.y;
  const int n_chunks = gridDim.x;
  const int n_grid = gridDim.y;
  const int64_t v = static_cast<int64_t>(c) * kLossRows + threadIdx.x;   // padded row
  int w = 0;
  while (w + 1 < map.n_w && v >= map.pad_off[w + 1]) ++w;
  const int64_t n = v - map.pad_off[w];
  const bool real = v < n_pad && n < map.rows[w];
  double row = 0.0;
  if (real) {
    // Sum over token tiles in tile order, compensated: s + c carries the
    // sum to about 2^-48 relative (each TwoSum error term is exact), and only
    // one fp64 add per row remains -- this part has little fp64 throughput.
    const float* pa = partials + static_cast<int64_t>(a) * n_tiles * n_pad + v;
    float s = 0.f, c = 0.f;
    for (int t = 0; t < n_tiles; ++t) {
      const float x = pa[static_cast<int64_t>(t) * n_pad];
      const float sn = __fadd_rn(s, x);
      const float bp = __fsub_rn(sn, s);
      c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, __fsub_rn(sn, bp)), __fsub_rn(x, bp)));
      s = sn;
    }
    row = static_cast<double>(s) + static_cast<double>(c);
    if (row_scale != nullptr) row *= *row_scale;
    const int64_t ri = static_cast<int64_t>(a) * n_total + map.cum[w] + n;
    if (in_bounds(kSiteLosses, ri, static_cast<int64_t>(n_grid) * n_total)) row_losses[ri] = row;
  }
  // Per-weight chunk sums (a chunk of 256 rows meets at most a few weights).
  const int64_t v0 = static_cast<int64_t>(c) * kLossRows;
  double* cs = chunk_sums + (static_cast<int64_t>(a) * n_chunks + c) * map.n_w;
  for (int wi = 0; wi < map.n_w; ++wi) {
    const int64_t lo = map.pad_off[wi];
    const int64_t hi = lo + map.rows[wi];
    if (hi <= v0 || lo >= v0 + kLossRows) {   // block-uniform: weight absent from the chunk
      if (threadIdx.x == 0) cs[wi] = 0.0;
      continue;
    }
    red[threadIdx.x] = (real && w == wi) ? row : 0.0;
    __syncthreads();
    for (int off = kLossRows / 2; off; off >>= 1) {
      if (threadIdx.x < off) red[threadIdx.x] += red[threadIdx.x + off];
      __syncthreads();
    }
    if (threadIdx.x == 0) cs[wi] = red[0];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    __threadfence();
    last = (atomicAdd(counter, 1u) == static_cast<unsigned>(n_chunks * n_grid) - 1u);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  // Final reduction: thread i handles grid point i (n_grid <= 64 <= 256).
  // The other blocks' chunk sums are read from L2 (__ldcg: not through this
  // SM's L1), several loads in flight, added in chunk order.
  if (threadIdx.x < n_grid) {
    const int ga = threadIdx.x;
    double total = 0.0;
    for (int wi = 0; wi < map.n_w; ++wi) {
      double sw = 0.0;
#pragma unroll 8
      for (int ci = 0; ci < n_chunks; ++ci)
        sw += __ldcg(chunk_sums + (static_cast<int64_t>(ga) * n_chunks + ci) * map.n_w + wi);
      total += sw / (static_cast<double>(map.rows[wi]) * static_cast<double>(T));
    }
    losses[ga] = total;
    red[ga] = total;
    // Finite inputs give finite losses; an infinity or NaN in X or W reaches
    // every grid point's loss (through s, the residual or the product).
    if (!isfinite(total)) atomicCAS(status, 0, kDevNonFinite);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int bi = 0;
    double bv = 0.0;
    for (int i = 0; i < n_grid; ++i) {
      const double x = isnan(red[i]) ? INFINITY : red[i];
      if (i == 0 || x < bv) {
        bi = i;
        bv = x;
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

int64_t loss_chunks(int64_t n_pad) { return ceil_div(n_pad, kLossRows); }

cudaError_t launch_loss_reduce(const float* partials, int n_alpha, int n_tiles, int64_t n_pad,
                               int64_t T, const RowMap& map, int64_t n_total,
                               double* chunk_sums, double* row_losses, double* losses, int* best,
                               double* alpha_out, const float* s_grid, int64_t K, float* s_out,
                               unsigned int* counter, const double* row_scale, int* status,
                               cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(loss_chunks(n_pad)), static_cast<unsigned>(n_alpha));
  k_losses<<<grid, kLossRows, 0, st>>>(partials, n_tiles, n_pad, map, n_total, T, chunk_sums,
                                       row_losses, losses, best, alpha_out, s_grid, K, s_out,
                                       counter, row_scale, status);
  return cudaGetLastError();
}

AWQ_BOUNDS_READER(bounds_reduce)

}  // namespace awq
