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
// single correctly rounded fp64 division.  With at most 2^22 tokens a sum
// stays below 2^62, which leaves the top two bits of each 64-bit word for
// flags: bit 62 = the channel held an infinity, bit 63 = it held a NaN.  The
// mean of such a channel is +inf or NaN, as an IEEE fp64 sum would give it.
#include <algorithm>

#include "awq_bounds.cuh"
#include "awq_f32x2.cuh"
#include "awq_internal.h"
#include "awq_ptx.cuh"

namespace awq {
namespace {

// ---- accumulate: X streamed by TMA in boxes of 32 tokens x 256 channels
constexpr int kStatWarps = 8;                         // consumer warps
constexpr int kStatThreads = (kStatWarps + 1) * 32;   // + one producer warp
constexpr int kBoxTokens = 32;
constexpr int kSlab = 256;                            // channels per box (8 per lane)
constexpr int kBoxBytes = kBoxTokens * kSlab * 2;     // 16 KB
constexpr int kStatStages = 4;
constexpr int kTokensPerWarp = kBoxTokens / kStatWarps;   // per box
constexpr int kFlushBoxes = 16 / kTokensPerWarp;          // 16 tokens per lane per window
constexpr int kRedBytes = kStatWarps * 8 * 32 * 8;        // cross-warp sums
constexpr int kFlagBytes = kStatWarps * 32 * 4;
constexpr int kStatSmem = 1024 + kStatStages * kBoxBytes + kRedBytes + kFlagBytes + 256;
constexpr unsigned long long kFlagInf = 1ull << 62;
constexpr unsigned long long kFlagNan = 1ull << 63;

// Exact sums on the FMA pipe, two channels per packed operation.  For an
// fp16 value x, u = |x| * 2^24 is an integer below 2^40.  One fma against
// C = 1.5 * 2^43 rounds u to a multiple of 2^20 (the ulp of [2^43, 2^44));
// the two parts
//   fh = round(u) = r - C        (a multiple of 2^20, below 2^41)
//   lo = u - fh                  (an integer, |lo| <= 2^19)
// are exact in fp32, and so are their sums over 16 tokens (the fh sum is a
// multiple of 2^20 below 2^45: 24 significant bits; |lo sum| <= 2^23).
// Every 16 tokens the two fp32 sums are converted to integers and added to
// 64-bit totals: the result is the exact integer sum, independent of order.
// An infinity makes fh infinite, a NaN makes it NaN; the running sum of the
// windows' fh keeps that mark for the flags.
constexpr float kSplitC = 13194139533312.0f;   // 1.5 * 2^43

struct LaneSums {
  f32x2 hi[4], lo[4];          // channel pairs (2i, 2i+1)
  unsigned long long tot[8];   // exact sums (wrapping: a flagged channel's is ignored)
  float mark[8];               // sum of the windows' fh sums: finite unless inf/NaN seen
};

__device__ __forceinline__ void add_chunk(LaneSums& a, const uint4 v) {
  const uint32_t w[4] = {v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu, v.z & 0x7FFF7FFFu,
                         v.w & 0x7FFF7FFFu};
  const f32x2 k24 = pack2(16777216.0f, 16777216.0f);
  const f32x2 c = pack2(kSplitC, kSplitC);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    const f32x2 x = pack2(f.x, f.y);
    const f32x2 r = fma2(x, k24, c);                          // round(u) + C
    const f32x2 nfh = sub2(c, r);                             // -round(u), exact
    a.lo[i] = add2(a.lo[i], fma2(x, k24, nfh));               // u - round(u), exact
    a.hi[i] = sub2(a.hi[i], nfh);                             // + round(u)
  }
}

__device__ __forceinline__ unsigned long long window_total(float h, float l) {
  return static_cast<unsigned long long>(
      (static_cast<long long>(__float2int_rn(__fmul_rn(h, 0x1p-20f))) << 20) +
      static_cast<long long>(__float2int_rn(l)));
}

__device__ __forceinline__ void flush_window(LaneSums& a) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float h0 = lo2(a.hi[i]), h1 = hi2(a.hi[i]);
    a.mark[2 * i] = __fadd_rn(a.mark[2 * i], h0);
    a.mark[2 * i + 1] = __fadd_rn(a.mark[2 * i + 1], h1);
    a.tot[2 * i] += window_total(h0, lo2(a.lo[i]));
    a.tot[2 * i + 1] += window_total(h1, hi2(a.lo[i]));
    a.hi[i] = 0ull;
    a.lo[i] = 0ull;
  }
}

// Shared state of one accumulate block.
struct StatSmem {
  uint32_t full0, empty0;     // ring barriers (stage i at +8i)
  uint32_t red_full;          // the consumer warps' partial sums are written (count kStatWarps)
  uint32_t red_free;          // warp 0 has added them up (count 1)
  unsigned long long (*red)[8][32];
  uint32_t* flags;
  volatile int* abort_flag;
};

// Round `round` of the cross-warp sum: every consumer warp writes its lanes'
// sums of one 256-channel slab (and the inf / NaN marks) and clears its
// registers; warp 0 adds the warps' sums and adds them to acc with one
// 64-bit atomic per channel (a flagged channel gets its flag bit instead of
// a sum).  The rounds are ordered by two mbarriers with bounded waits, so a
// warp that gave up cannot leave the others waiting.  Returns false if a
// wait gave up.
__device__ __forceinline__ bool flush_slab(LaneSums& a, int64_t slab, int64_t kchunks,
                                           uint32_t round, const StatSmem& sm, int* status,
                                           unsigned long long* __restrict__ acc) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (round > 0 && !mbar_wait_bounded(sm.red_free, (round - 1) & 1u, sm.abort_flag, status,
                                      kDevTimeoutEmpty))
    return false;
  uint32_t fl = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sm.red[warp][j][lane] = a.tot[j];
    if (isnan(a.mark[j])) fl |= 2u << (2 * j);
    else if (isinf(a.mark[j])) fl |= 1u << (2 * j);
    a.tot[j] = 0;
    a.mark[j] = 0.f;
  }
  sm.flags[warp * 32 + lane] = fl;
  __syncwarp();
  if (lane == 0) mbar_arrive(sm.red_full);
  if (warp != 0) return true;
  if (!mbar_wait_bounded(sm.red_full, round & 1u, sm.abort_flag, status, kDevTimeoutFull))
    return false;
  // The sums were zeroed by the previous kernel, which this one may overlap.
  if (round == 0) grid_dependency_wait();
  const int64_t chunk = slab * 32 + lane;
  if (chunk < kchunks) {
    uint32_t f = 0;
#pragma unroll
    for (int w = 0; w < kStatWarps; ++w) f |= sm.flags[w * 32 + lane];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      unsigned long long sum = 0;
#pragma unroll
      for (int w = 0; w < kStatWarps; ++w) sum += sm.red[w][j][lane];
      const uint32_t fj = (f >> (2 * j)) & 3u;
      if (!in_bounds(kSiteStatsAcc, chunk * 8 + j, kchunks * 8)) continue;
      if (fj) atomicOr(acc + chunk * 8 + j, (fj & 2u) ? kFlagNan : kFlagInf);
      else if (sum) atomicAdd(acc + chunk * 8 + j, sum);
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(sm.red_free);
  return true;
}

// Block b of the grid takes units [b*U/G, (b+1)*U/G) of the U = slabs x
// token-boxes units, slab-major, so a block meets few slabs.  Warp
// kStatWarps (one thread) loads the units' boxes by TMA into a ring of
// kStatStages stages; consumer warp w takes tokens w, w+8, w+16, w+24 of each
// box, lane l its channels 8l..8l+7 (a warp reads one 512-byte row per load:
// conflict-free).  Boxes reaching past K or T are zero-filled by the TMA.
// Every wait is bounded; on expiry the kernel records a code in *status and
// ends (its copies in flight drained), and the finalize kernel turns the
// whole sX into NaN.
__global__ void __launch_bounds__(kStatThreads)
    k_stats_accumulate(const __grid_constant__ CUtensorMap tmap, int64_t kchunks,
                       int64_t tboxes, int64_t units, unsigned long long* __restrict__ acc,
                       int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* ring = base;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kStatStages * kBoxBytes + kRedBytes +
                                               kFlagBytes);
  StatSmem sm;
  sm.red = reinterpret_cast<unsigned long long(*)[8][32]>(base + kStatStages * kBoxBytes);
  sm.flags = reinterpret_cast<uint32_t*>(base + kStatStages * kBoxBytes + kRedBytes);
  sm.full0 = smem_u32(bars);
  sm.empty0 = smem_u32(bars + kStatStages);
  sm.red_full = smem_u32(bars + 2 * kStatStages);
  sm.red_free = smem_u32(bars + 2 * kStatStages + 1);
  sm.abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStatStages + 2);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStatStages; ++i) {
      mbar_init(sm.full0 + 8 * i, 1);
      mbar_init(sm.empty0 + 8 * i, kStatWarps);
    }
    mbar_init(sm.red_full, kStatWarps);
    mbar_init(sm.red_free, 1);
    *sm.abort_flag = 0;
    fence_barrier_init();
    grid_dependents_launch();   // the finalize kernel may start (it waits for this one)
  }
  __syncthreads();
  const int64_t G = gridDim.x;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * units / G;
  const int64_t u1 = (static_cast<int64_t>(blockIdx.x) + 1) * units / G;
  if (warp == kStatWarps) {
    if (lane != 0) return;
    prefetch_tmap(&tmap);
    // X may be written by the kernel before the zeroing kernel: its first
    // load waits for that chain to complete.
    grid_dependency_wait();
    int64_t issued = 0;
    int64_t slab = u0 / tboxes, tb = u0 - slab * tboxes;
    for (int64_t u = u0; u < u1; ++u, ++issued, ++tb) {
      if (tb == tboxes) {
        tb = 0;
        ++slab;
      }
      const int st = static_cast<int>(issued % kStatStages);
      if (issued >= kStatStages &&
          !mbar_wait_bounded(sm.empty0 + 8 * st,
                             static_cast<uint32_t>((issued / kStatStages - 1) & 1),
                             sm.abort_flag, status, kDevTimeoutEmpty))
        break;
      mbar_arrive_expect_tx(sm.full0 + 8 * st, kBoxBytes);
      tma_load_2d(smem_u32(ring + st * kBoxBytes), &tmap, sm.full0 + 8 * st,
                  static_cast<int>(slab * kSlab), static_cast<int>(tb * kBoxTokens));
    }
    // Before the CTA may end, the copies of the last stages issued must have
    // landed (they have, unless the consumers gave up).
    for (int64_t j = issued > kStatStages ? issued - kStatStages : 0; j < issued; ++j) {
      const int st = static_cast<int>(j % kStatStages);
      mbar_wait_bounded(sm.full0 + 8 * st, static_cast<uint32_t>((j / kStatStages) & 1), nullptr,
                        status, kDevTimeoutDrain, kDrainLimitNs);
    }
    return;
  }
  LaneSums a;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    a.tot[j] = 0;
    a.mark[j] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) a.hi[i] = a.lo[i] = 0ull;
  // The unit's slab and token box, advanced without dividing (one division
  // at the start).
  int64_t cur_slab = u0 < u1 ? u0 / tboxes : 0;
  int64_t tb = u0 - cur_slab * tboxes;
  uint32_t round = 0;
  int in_window = 0;
  int st = 0;
  uint32_t phase = 0;
  for (int64_t u = u0; u < u1; ++u, ++tb) {
    if (tb == tboxes) {   // next slab
      tb = 0;
      flush_window(a);
      in_window = 0;
      if (!flush_slab(a, cur_slab, kchunks, round++, sm, status, acc)) return;
      ++cur_slab;
    }
    if (!mbar_wait_bounded(sm.full0 + 8 * st, phase, sm.abort_flag, status, kDevTimeoutFull))
      return;
    const uint4* box = reinterpret_cast<const uint4*>(ring + st * kBoxBytes);
#pragma unroll
    for (int q = 0; q < kTokensPerWarp; ++q)
      add_chunk(a, box[(warp + kStatWarps * q) * 32 + lane]);
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.empty0 + 8 * st);
    if (++st == kStatStages) {
      st = 0;
      phase ^= 1u;
    }
    if (++in_window == kFlushBoxes) {
      flush_window(a);
      in_window = 0;
    }
  }
  if (u0 < u1) {
    flush_window(a);
    flush_slab(a, cur_slab, kchunks, round, sm, status, acc);
  }
}

// The range of the positive doubles x over the block's threads, merged into
// range[0] = max bits and range[1] = ~(min bits) with atomicMax: for positive
// doubles the IEEE bit pattern is monotone; both words start at 0.
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
// division; +inf or NaN for a flagged channel; NaN everywhere if the
// accumulation gave up (*status set).  With `range`, also the range of
// max(sX, 1e-4) over the channels.
__global__ void k_stats_finalize(const unsigned long long* __restrict__ acc, int64_t T,
                                 int64_t K, double* __restrict__ sX,
                                 unsigned long long* __restrict__ range,
                                 const int* __restrict__ status) {
  grid_dependency_wait();   // the accumulation, which this kernel may overlap, is complete
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  double v = 0.0;
  if (k < K && in_bounds(kSiteStatsOut, k, K)) {
    const unsigned long long w = acc[k];
    if ((status != nullptr && *status != 0) || (w & kFlagNan)) v = __longlong_as_double(0x7FF8000000000000ll);
    else if (w & kFlagInf) v = __longlong_as_double(0x7FF0000000000000ll);
    else v = (static_cast<double>(w) * 0x1p-24) / static_cast<double>(T);
    sX[k] = v;
  }
  if (range != nullptr) block_range(fmax(v, 1e-4), k < K, range);
}

// Zeroes the sums (and the word after them) and lets the accumulation start
// behind it.  Launched behind the stream's previous kernel (which may still
// read the memory it zeroes), it waits for that kernel before writing.
__global__ void k_zero_sums(unsigned long long* __restrict__ acc, int64_t n) {
  grid_dependents_launch();
  grid_dependency_wait();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    acc[i] = 0ull;
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
    const int64_t i = static_cast<int64_t>(a) * K + k;
    if (in_bounds(kSiteScalesOut, i, static_cast<int64_t>(n_grid) * K)) {
      s[i] = sv;
      if (r != nullptr) r[i] = __frcp_rn(sv);
    }
    u *= e;
  }
}

}  // namespace

cudaError_t launch_stats_accumulate(const __half* X, int64_t T, int64_t K,
                                    unsigned long long* acc, int* status, cudaStream_t st) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  LaunchFacts lf;
  cudaError_t e = launch_facts(reinterpret_cast<const void*>(k_stats_accumulate), kStatThreads,
                               kStatSmem, &lf);
  if (e != cudaSuccess) return e;
  // X as a 2-D tensor [T][K], boxes of 256 channels x 32 tokens, no swizzle;
  // the parts of a box past K or T read as zeros.
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {kSlab, kBoxTokens};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(X), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int64_t kchunks = K / 8;
  const int64_t slabs = ceil_div(K, kSlab);
  const int64_t tboxes = ceil_div(T, kBoxTokens);
  const int64_t units = slabs * tboxes;
  // One wave of resident blocks (each with a 64 KB ring), or fewer for small inputs.
  const int64_t grid = std::max<int64_t>(
      1, std::min<int64_t>(units, static_cast<int64_t>(lf.per_sm) * lf.sms));
  // The sums, and the status word when it directly follows them, zeroed by
  // a kernel the accumulation is launched behind; that kernel is itself
  // launched behind the stream's previous kernel, so the chain's launches
  // overlap the kernels before them.
  const bool status_next = status == reinterpret_cast<int*>(acc + K);
  const int64_t nz = K + (status_next ? 1 : 0);
  e = launch_dependent(k_zero_sums, std::min<int64_t>(ceil_div(nz, 256), 4 * lf.sms), 256, 0, st,
                       acc, nz);
  if (e != cudaSuccess) return e;
  return launch_dependent(k_stats_accumulate, grid, kStatThreads, kStatSmem, st, tmap, kchunks,
                          tboxes, units, acc, status);
}

cudaError_t launch_stats_finalize(const unsigned long long* acc, int64_t T, int64_t K,
                                  double* sX, const int* status, cudaStream_t st,
                                  unsigned long long* range) {
  // Launched behind the accumulation, which lets it start early; it waits.
  // 64-thread blocks spread the fp64 divisions over as many SMs as possible.
  return launch_dependent(k_stats_finalize, ceil_div(K, 64), 64, 0, st,
                          static_cast<const unsigned long long*>(acc), T, K, sX, range, status);
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

AWQ_BOUNDS_READER(bounds_stats)

}  // namespace awq
