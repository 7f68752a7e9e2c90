// Per-input-channel activation statistic and the per-alpha scale vectors.
//
// AWQ explained (hungho77.github.io), "Scaling instead of mixed precision":
// sX is the average activation magnitude per input channel and s = sX^alpha.
// AWQ Explained (multigrid.ai), "How the scale is chosen": s = mean(|x_j|)^alpha
// over a small grid of alpha in [0, 1].
//
// The channel sums are exact: |x| of an fp16 value is an integer multiple of
// 2^-24 below 2^40 units, so the sums are kept as 64-bit integers in those
// units (order-independent, deterministic, no rounding), and the mean is a
// single correctly rounded fp64 division.
#include <algorithm>

#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kStatsThreads = 256;   // 8 warps; a warp covers 256 channels

// |h| of an fp16 bit pattern, in units of 2^-24, exactly.
__device__ __forceinline__ unsigned long long abs_half_units(uint32_t h) {
  const uint32_t b = h & 0x7FFFu;
  const uint32_t e = b >> 10;
  const uint32_t m = b & 0x3FFu;
  const uint32_t mant = e ? (m | 0x400u) : m;
  const uint32_t sh = e ? e - 1u : 0u;
  return static_cast<unsigned long long>(mant) << sh;
}

__device__ __forceinline__ void add_chunk(unsigned long long (&acc)[8], const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] += abs_half_units(w[i] & 0xFFFFu);
    acc[2 * i + 1] += abs_half_units(w[i] >> 16);
  }
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Block (x, y): channel chunks [32*x, 32*x + 32) (8 channels each), tokens
// [y*rows, (y+1)*rows).  Warp w walks tokens w, w+8, ...; the 8 warps are
// then summed in shared memory and added to acc with one 64-bit atomic per
// channel (integer addition: the result does not depend on the order).
__global__ void __launch_bounds__(kStatsThreads)
    k_stats_accumulate(const uint4* __restrict__ X, int64_t T, int64_t kchunks,
                       int64_t rows_per_block, unsigned long long* __restrict__ acc) {
  __shared__ unsigned long long red[8][8][33];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t chunk = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * rows_per_block;
  const int64_t t1 = min(T, t0 + rows_per_block);
  unsigned long long s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (chunk < kchunks) {
    int64_t t = t0 + warp;
    for (; t + 24 < t1; t += 32) {
      const uint4 v0 = ldg_stream(X + t * kchunks + chunk);
      const uint4 v1 = ldg_stream(X + (t + 8) * kchunks + chunk);
      const uint4 v2 = ldg_stream(X + (t + 16) * kchunks + chunk);
      const uint4 v3 = ldg_stream(X + (t + 24) * kchunks + chunk);
      add_chunk(s, v0);
      add_chunk(s, v1);
      add_chunk(s, v2);
      add_chunk(s, v3);
    }
    for (; t < t1; t += 8) add_chunk(s, ldg_stream(X + t * kchunks + chunk));
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) red[warp][j][lane] = s[j];
  __syncthreads();
  if (warp == 0 && chunk < kchunks) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      unsigned long long tot = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) tot += red[w][j][lane];
      if (tot) atomicAdd(acc + chunk * 8 + j, tot);
    }
  }
}

__global__ void k_stats_finalize(const unsigned long long* __restrict__ acc, int64_t T,
                                 int64_t K, double* __restrict__ sX,
                                 unsigned long long* __restrict__ maxmin, int n_grid) {
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k < K) sX[k] = (static_cast<double>(acc[k]) * 0x1p-24) / static_cast<double>(T);
  // Starting values of the per-grid-point max/min of the scale kernels
  // (block 0 has 256 threads >= n_grid).
  if (maxmin != nullptr && k < n_grid) {
    maxmin[2 * k] = 0ull;
    maxmin[2 * k + 1] = ~0ull;
  }
}

// u[a][k] = max(sX_k, 1e-4)^(a / n_grid) in fp64; per-grid-point max and min
// of u kept as the (order-preserving, u > 0) bit patterns of the doubles.
__global__ void k_scale_pow(const double* __restrict__ sX, int64_t K, int n_grid,
                            double* __restrict__ u, unsigned long long* __restrict__ maxmin) {
  __shared__ unsigned long long smax[8], smin[8];
  const int a = blockIdx.y;
  const double alpha = static_cast<double>(a) / static_cast<double>(n_grid);
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  unsigned long long mx = 0ull, mn = ~0ull;
  if (k < K) {
    const double v = pow(fmax(sX[k], 1e-4), alpha);
    u[static_cast<int64_t>(a) * K + k] = v;
    mx = mn = static_cast<unsigned long long>(__double_as_longlong(v));
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    smax[warp] = mx;
    smin[warp] = mn;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) {
      mx = max(mx, smax[w]);
      mn = min(mn, smin[w]);
    }
    atomicMax(maxmin + 2 * a, mx);
    atomicMin(maxmin + 2 * a + 1, mn);
  }
}

// s = fp32(u / sqrt(max u * min u)); r = fp32(1/s) (nullable) for the residual.
__global__ void k_scale_norm(const double* __restrict__ u, int64_t K,
                             const unsigned long long* __restrict__ maxmin,
                             float* __restrict__ s, float* __restrict__ r) {
  const int a = blockIdx.y;
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k >= K) return;
  const double umax = __longlong_as_double(static_cast<long long>(maxmin[2 * a]));
  const double umin = __longlong_as_double(static_cast<long long>(maxmin[2 * a + 1]));
  const double norm = sqrt(umax * umin);
  const int64_t i = static_cast<int64_t>(a) * K + k;
  const float sv = __double2float_rn(u[i] / norm);
  s[i] = sv;
  if (r != nullptr) r[i] = __frcp_rn(sv);
}

__global__ void k_init_maxmin(unsigned long long* maxmin, int n_grid) {
  const int a = threadIdx.x;
  if (a < n_grid) {
    maxmin[2 * a] = 0ull;
    maxmin[2 * a + 1] = ~0ull;
  }
}

}  // namespace

cudaError_t launch_stats_accumulate(const __half* X, int64_t T, int64_t K,
                                    unsigned long long* acc, cudaStream_t st) {
  const int64_t kchunks = K / 8;
  const int64_t gx = ceil_div(kchunks, 32);
  // Enough row slices for ~8 blocks per SM (148 SMs), at least 32 rows each.
  int64_t gy = ceil_div(148 * 8, gx);
  int64_t rows = ceil_div(T, gy);
  rows = std::max<int64_t>(32, ceil_div(rows, 8) * 8);
  gy = ceil_div(T, rows);
  cudaError_t e = cudaMemsetAsync(acc, 0, sizeof(unsigned long long) * K, st);
  if (e != cudaSuccess) return e;
  k_stats_accumulate<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)),
                       kStatsThreads, 0, st>>>(reinterpret_cast<const uint4*>(X), T, kchunks,
                                               rows, acc);
  return cudaGetLastError();
}

cudaError_t launch_stats_finalize(const unsigned long long* acc, int64_t T, int64_t K,
                                  double* sX, cudaStream_t st, unsigned long long* maxmin,
                                  int n_grid) {
  k_stats_finalize<<<static_cast<unsigned>(ceil_div(K, 256)), 256, 0, st>>>(acc, T, K, sX,
                                                                            maxmin, n_grid);
  return cudaGetLastError();
}

cudaError_t launch_scales(const double* sX, int64_t K, int n_grid, double* u_ws,
                          unsigned long long* maxmin_ws, float* s, float* r, cudaStream_t st,
                          bool maxmin_ready) {
  if (!maxmin_ready) k_init_maxmin<<<1, kMaxGrid, 0, st>>>(maxmin_ws, n_grid);
  const dim3 grid(static_cast<unsigned>(ceil_div(K, 256)), static_cast<unsigned>(n_grid));
  k_scale_pow<<<grid, 256, 0, st>>>(sX, K, n_grid, u_ws, maxmin_ws);
  k_scale_norm<<<grid, 256, 0, st>>>(u_ws, K, maxmin_ws, s, r);
  return cudaGetLastError();
}

}  // namespace awq
