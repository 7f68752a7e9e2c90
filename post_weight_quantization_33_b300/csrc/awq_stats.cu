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

#include "awq_async.cuh"
#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kStatsThreads = 256;   // 8 warps; a warp covers 256 channels

// Exact sums on the FMA pipe.  For an fp16 value x, u = |x| * 2^24 is an
// integer below 2^40.  One fma against C = 1.5 * 2^43 rounds u to a multiple
// of 2^20 (the ulp of [2^43, 2^44)); the two parts
//   hi = (round(u) - C) / 2^20   (an integer <= 2^20)
//   lo = u - round(u)            (an integer, |lo| <= 2^19)
// are exact in fp32, and so are their sums over 16 tokens (|hi sum| <= 2^24,
// |lo sum| <= 2^23).  Every 16 tokens the two fp32 sums are converted to
// integers and added to 64-bit totals: the result is the exact integer sum,
// independent of order.
constexpr float kSplitC = 13194139533312.0f;   // 1.5 * 2^43
constexpr int kFlushTokens = 16;
constexpr int kStatStages = 4;                                   // steps of 4 tokens
constexpr int kStatSmem = (kStatsThreads / 32) * kStatStages * 4 * 32 * 16;   // 64 KB
static_assert(kStatSmem >= 8 * 8 * 33 * 8, "the ring also holds the cross-warp sums");

__device__ __forceinline__ void add_half_exact(float v, float& hi, float& lo) {
  const float r = __fmaf_rn(v, 16777216.0f, kSplitC);        // round(u) + C
  const float fh = __fsub_rn(r, kSplitC);                     // round(u)
  lo = __fadd_rn(lo, __fmaf_rn(v, 16777216.0f, -fh));         // u - round(u), exact
  hi = __fmaf_rn(fh, 0x1p-20f, hi);                           // round(u) / 2^20, exact
}

__device__ __forceinline__ void add_chunk(float (&hi)[8], float (&lo)[8], const uint4 v) {
  const uint32_t w[4] = {v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu, v.z & 0x7FFF7FFFu,
                         v.w & 0x7FFF7FFFu};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    add_half_exact(f.x, hi[2 * i], lo[2 * i]);
    add_half_exact(f.y, hi[2 * i + 1], lo[2 * i + 1]);
  }
}

// Block (x, y): channel chunks [32*x, 32*x + 32) (8 channels each), tokens
// [y*rows, (y+1)*rows).  Warp w walks tokens w, w+8, ... four at a time
// (a step); every 16 of its tokens (and at the end) the fp32 part sums are
// flushed to 64-bit totals.  Loads go through a per-warp ring of
// kStatStages steps in shared memory filled with cp.async (token q of lane l
// at [stage][q][l]: conflict-free; each lane reads back only its own
// copies), so kStatStages - 1 steps of loads are in flight without holding
// registers.  The 8 warps are then summed in shared memory and added to acc
// with one 64-bit atomic per channel (integer addition: the result does not
// depend on the order).
__global__ void __launch_bounds__(kStatsThreads)
    k_stats_accumulate(const uint4* __restrict__ X, int64_t T, int64_t kchunks,
                       int64_t rows_per_block, unsigned long long* __restrict__ acc) {
  extern __shared__ uint4 ring_smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t chunk = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const bool live = chunk < kchunks;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * rows_per_block;
  const int64_t t1 = min(T, t0 + rows_per_block);
  uint4* ring = ring_smem + warp * (kStatStages * 4 * 32);
  const uint32_t ring_u32 = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  const int64_t steps = t1 > t0 + warp ? (t1 - t0 - warp + 31) / 32 : 0;
  auto issue = [&](int64_t step) {
    if (step < steps && live) {
      const int st = static_cast<int>(step % kStatStages);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t t = t0 + warp + 32 * step + 8 * q;
        const bool in = t < t1;
        cp_async16(ring_u32 + ((st * 4 + q) * 32 + lane) * 16, in ? X + t * kchunks + chunk : X,
                   in ? 16 : 0);
      }
    }
    cp_async_commit();   // possibly empty: one group per step
  };
  long long tot[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  float hi[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float lo[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kStatStages - 1; ++i) issue(i);
  int since_flush = 0;
  for (int64_t step = 0; step < steps; ++step) {
    issue(step + kStatStages - 1);
    cp_async_wait<kStatStages - 1>();
    if (live) {
      const int st = static_cast<int>(step % kStatStages);
#pragma unroll
      for (int q = 0; q < 4; ++q) add_chunk(hi, lo, ring[(st * 4 + q) * 32 + lane]);
    }
    since_flush += 4;
    if (since_flush == kFlushTokens || step + 1 == steps) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        tot[j] += (static_cast<long long>(__float2int_rn(hi[j])) << 20) +
                  static_cast<long long>(__float2int_rn(lo[j]));
        hi[j] = 0.f;
        lo[j] = 0.f;
      }
      since_flush = 0;
    }
  }
  cp_async_wait<0>();
  __syncthreads();   // the ring is reused for the cross-warp sum
  auto red = reinterpret_cast<unsigned long long(*)[8][33]>(ring_smem);
#pragma unroll
  for (int j = 0; j < 8; ++j) red[warp][j][lane] = static_cast<unsigned long long>(tot[j]);
  __syncthreads();
  if (warp == 0 && live) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      unsigned long long sum = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) sum += red[w][j][lane];
      if (sum) atomicAdd(acc + chunk * 8 + j, sum);
    }
  }
}

// Order-preserving update of the scale range: for the positive doubles used
// here the IEEE bit pattern is monotone, so range[0] = max bits (atomicMax)
// and range[1] = ~(min bits) (atomicMax of the complement); both start at 0.
__device__ __forceinline__ void range_update(unsigned long long* range, double v) {
  const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(v));
  atomicMax(range, b);
  atomicMax(range + 1, ~b);
}

__device__ __forceinline__ void block_range(double x, bool valid, unsigned long long* range) {
  __shared__ unsigned long long smax[32], smin[32];
  unsigned long long mx = valid ? static_cast<unsigned long long>(__double_as_longlong(x)) : 0ull;
  unsigned long long mn = valid ? ~static_cast<unsigned long long>(__double_as_longlong(x)) : 0ull;
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    mn = max(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
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
      mn = max(mn, smin[w]);
    }
    if (mx) atomicMax(range, mx);
    if (mn) atomicMax(range + 1, mn);
  }
}

// sX = (sum of |x| in units of 2^-24) * 2^-24 / T, one correctly rounded fp64
// division; with `range`, also the range of max(sX, 1e-4) over the channels.
__global__ void k_stats_finalize(const unsigned long long* __restrict__ acc, int64_t T,
                                 int64_t K, double* __restrict__ sX,
                                 unsigned long long* __restrict__ range) {
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  double v = 0.0;
  if (k < K) {
    v = (static_cast<double>(acc[k]) * 0x1p-24) / static_cast<double>(T);
    sX[k] = v;
  }
  if (range != nullptr) block_range(fmax(v, 1e-4), k < K, range);
}

__global__ void k_sx_range(const double* __restrict__ sX, int64_t K,
                           unsigned long long* __restrict__ range) {
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  block_range(k < K ? fmax(sX[k], 1e-4) : 0.0, k < K, range);
}

// s[a][k] = fp32(u / sqrt(u(x_max) * u(x_min))) with u = x^(a / n_grid),
// x = max(sX_k, 1e-4); r[a][k] = fp32 1 / s[a][k] (nullable).
//
// Mathematically s = y^(a/n) with y = x / sqrt(x_max * x_min) (x^alpha is
// increasing in x, so the largest and smallest u are those of the largest
// and smallest x; the range comes from k_stats_finalize / k_sx_range).  It is
// formed as e^a with e = exp((ln x - (ln x_max + ln x_min) / 2) / n) by
// repeated fp64 multiplication: a few logs and one exp per channel instead of
// n powers, a square root and a divide per grid point (this part has little
// fp64 throughput).  The relative error stays near a * 2^-52 (below 2^-47
// for a < 64), far under the half ulp of the fp32 result.
__global__ void k_scales(const double* __restrict__ sX, int64_t K, int n_grid,
                         const unsigned long long* __restrict__ range, float* __restrict__ s,
                         float* __restrict__ r) {
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k >= K) return;
  const double xmax = __longlong_as_double(static_cast<long long>(range[0]));
  const double xmin = __longlong_as_double(static_cast<long long>(~range[1]));
  const double centre = 0.5 * (log(xmax) + log(xmin));
  const double e = exp((log(fmax(sX[k], 1e-4)) - centre) / static_cast<double>(n_grid));
  double u = 1.0;
  for (int a = 0; a < n_grid; ++a) {
    const float sv = __double2float_rn(u);
    s[static_cast<int64_t>(a) * K + k] = sv;
    if (r != nullptr) r[static_cast<int64_t>(a) * K + k] = __frcp_rn(sv);
    u *= e;
  }
}

}  // namespace

cudaError_t launch_stats_accumulate(const __half* X, int64_t T, int64_t K,
                                    unsigned long long* acc, cudaStream_t st) {
  LaunchFacts lf;
  cudaError_t e = launch_facts(reinterpret_cast<const void*>(k_stats_accumulate), kStatsThreads,
                               kStatSmem, &lf);
  if (e != cudaSuccess) return e;
  const int64_t kchunks = K / 8;
  const int64_t gx = ceil_div(kchunks, 32);
  // About one wave of resident blocks (64 KB of ring each); token slices a
  // multiple of 32 rows (8 warps x 4 tokens per step).
  int64_t gy = std::max<int64_t>(1, ceil_div(static_cast<int64_t>(lf.per_sm) * lf.sms, gx));
  int64_t rows = ceil_div(T, gy);
  rows = std::max<int64_t>(32, ceil_div(rows, 32) * 32);
  gy = ceil_div(T, rows);
  e = cudaMemsetAsync(acc, 0, sizeof(unsigned long long) * K, st);
  if (e != cudaSuccess) return e;
  k_stats_accumulate<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)),
                       kStatsThreads, kStatSmem, st>>>(reinterpret_cast<const uint4*>(X), T,
                                                       kchunks, rows, acc);
  return cudaGetLastError();
}

cudaError_t launch_stats_finalize(const unsigned long long* acc, int64_t T, int64_t K,
                                  double* sX, cudaStream_t st, unsigned long long* range) {
  k_stats_finalize<<<static_cast<unsigned>(ceil_div(K, 256)), 256, 0, st>>>(acc, T, K, sX,
                                                                            range);
  return cudaGetLastError();
}

cudaError_t launch_sx_range(const double* sX, int64_t K, unsigned long long* range,
                            cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(range, 0, 2 * sizeof(unsigned long long), st);
  if (e != cudaSuccess) return e;
  k_sx_range<<<static_cast<unsigned>(ceil_div(K, 256)), 256, 0, st>>>(sX, K, range);
  return cudaGetLastError();
}

cudaError_t launch_scales(const double* sX, int64_t K, int n_grid,
                          const unsigned long long* range, float* s, float* r, cudaStream_t st) {
  // One warp per block: the fp64 logs and exps run on as many SMs as possible.
  k_scales<<<static_cast<unsigned>(ceil_div(K, 32)), 32, 0, st>>>(sX, K, n_grid, range, s, r);
  return cudaGetLastError();
}

}  // namespace awq
