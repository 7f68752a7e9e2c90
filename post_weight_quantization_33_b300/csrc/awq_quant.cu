// Scale -> group min/max -> round-to-nearest -> pack, one HBM pass over W.
//
// AWQ explained (hungho77.github.io), "Scaling instead of mixed precision":
// W' = W diag(s) is quantized instead of W.  AWQ Explained (multigrid.ai),
// "Scaling instead of mixed precision": the grid step is the group's range
// divided by the number of levels; "How the scale is chosen": AwqConfig
// bits / group_size / zero_point.  AWQ (ai360xpert.com), "How It Works"
// step 4: plain round-to-nearest.  activation-aware weight quantization (AWQ)
// (realpython.com): codes packed at 3 or 4 bits in groups of 128.
//
// Arithmetic (fp32, each operation correctly rounded, nothing fused):
//   w' = w * s;  rng = max - min;  step = max(rng, 1e-5) / (2^b - 1);
//   scale = fp16_rn(step);  rcp = 1 / float(scale);
//   z = clamp(rn(-min * rcp), 0, 2^b - 1);  q = clamp(rn(w' * rcp) + z, 0, 2^b - 1)
// where rn rounds half to even.
//
// One thread owns 8 consecutive weights of a row (one 16-byte load); a group
// of 64 or 128 weights is 8 or 16 adjacent lanes, reduced with shuffles.
#include <algorithm>

#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

struct Quant8 {
  uint32_t q[8];
  __half scale;
  int zero;
};

// Quantize the thread's 8 weights; every lane of the warp must call this
// (shuffles), GLANES = group / 8 adjacent lanes form one group.
template <int GLANES>
__device__ __forceinline__ Quant8 quantize8(const uint4 wv, const float* __restrict__ s8,
                                            const int levels) {
  const float4 sa = __ldg(reinterpret_cast<const float4*>(s8));
  const float4 sb = __ldg(reinterpret_cast<const float4*>(s8) + 1);
  const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
  const uint32_t wv32[4] = {wv.x, wv.y, wv.z, wv.w};
  float w[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = *reinterpret_cast<const __half2*>(&wv32[i]);
    w[2 * i] = __fmul_rn(__low2float(h), sv[2 * i]);
    w[2 * i + 1] = __fmul_rn(__high2float(h), sv[2 * i + 1]);
  }
  float mn = w[0], mx = w[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    mn = fminf(mn, w[i]);
    mx = fmaxf(mx, w[i]);
  }
#pragma unroll
  for (int off = GLANES / 2; off; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  }
  const float rng = __fsub_rn(mx, mn);
  const float step = __fdiv_rn(fmaxf(rng, 1e-5f), static_cast<float>(levels));
  Quant8 r;
  r.scale = __float2half_rn(step);
  const float rcp = __frcp_rn(__half2float(r.scale));
  int z = __float2int_rn(__fmul_rn(-mn, rcp));
  z = min(max(z, 0), levels);
  r.zero = z;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int q = __float2int_rn(__fmul_rn(w[i], rcp));
    q = min(max(q, -levels), levels) + z;
    r.q[i] = static_cast<uint32_t>(min(max(q, 0), levels));
  }
  return r;
}

__device__ __forceinline__ uint32_t pack4(const Quant8& r) {
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) word |= r.q[i] << (4 * i);
  return word;
}

__device__ __forceinline__ uint32_t pack3_bits24(const Quant8& r) {
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) bits |= r.q[i] << (3 * i);
  return bits;
}

// Round half to even without the conversion unit: adding and removing
// 1.5 * 2^23 leaves rne(t) for |t| <= 2^22 (the sum's ulp is 1, and the
// addition rounds half to even).  The map is monotone, so for larger |t| the
// result keeps the side of [-2^22, 2^22] that t is on, which is all the
// clamps below ever look at.
__device__ __forceinline__ float rne_small(float t) {
  return __fsub_rn(__fadd_rn(t, 12582912.0f), 12582912.0f);
}

__device__ __forceinline__ void ld_v8f(const float* p, float* v) {
  uint32_t r[8];
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st_v8(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// Packed fp32 pairs (sm_100 f32x2 arithmetic, both lanes rounded to nearest
// even).  ptxas fuses a packed multiply into a following packed add even with
// .rn, so packed ops are used here only where no add consumes a product:
// every "product, then add" of the quantizer stays in scalar intrinsics.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack2(float a, float b) {
  return static_cast<f32x2>(__float_as_uint(a)) | (static_cast<f32x2>(__float_as_uint(b)) << 32);
}
__device__ __forceinline__ float lo2(f32x2 v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi2(f32x2 v) {
  return __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// Three-input min / max (exact, like fminf / fmaxf).
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Search output: the quantization residual of every grid point, in the units
// of W,
//   delta[a][row_off + n][k] = fp16( w - ((q - z) * scale) / s_k ),
// i.e. W - deq(Q(W diag(s))) diag(s)^-1 row by row.  The codes and zero
// points are those of quantize8 (same fp32 steps, same rounding); only the
// rounding itself uses rne_small instead of a float-to-int conversion, with
// the clamp applied to (q - z) directly:
//   q - z = clamp(rne(w' * rcp), -z, L - z).
// (q - z) * scale is exact in fp32 (a 4-bit integer times an 11-bit
// significand); w - that * (1/s_k) is one fused multiply-add, and the one
// coarse rounding is the final one to fp16, relative to the residual.
//
// Work split: a lane owns 16 consecutive channels of two consecutive rows (a
// group of 128 is 8 lanes, of 64 is 4), loads s and 1/s of a grid point once
// for both rows, and evaluates every grid point, so W is read and converted
// to fp32 once.  A warp covers 512 channels of its row pair; the 8 warps of a
// block take 16 consecutive rows at the same channels, so their 256-bit loads
// of s and 1/s hit the same L1 lines.  Warps are numbered row panel (64
// rows), channel chunk, row pair.  Each lane writes one whole 32-byte sector
// per row and grid point.
constexpr int kResPanel = 64;
constexpr int kResPerLane = 16;
constexpr int kResRowsPerLane = 2;

template <int GROUP>
__global__ void __launch_bounds__(kQuantThreads)
    k_quant_residual(const __half* __restrict__ W, int64_t N, int64_t K, int levels,
                     const float* __restrict__ s_grid, const float* __restrict__ r_grid,
                     int n_alpha, int64_t row_off, int64_t n_pad, __half* __restrict__ delta) {
  constexpr int EPL = kResPerLane, RPT = kResRowsPerLane;
  constexpr int GLANES = GROUP / EPL;
  constexpr int SUBS = kResPanel / RPT;
  const int64_t lanes_per_row = K / EPL;
  const int64_t kw = (lanes_per_row + 31) / 32;      // warp chunks per row
  const int64_t panels = (N + kResPanel - 1) / kResPanel;
  const int64_t total_warps = panels * SUBS * kw;
  const int lane = threadIdx.x & 31;
  const float L = static_cast<float>(levels);
  const int64_t slab = n_pad * K;                     // halves per grid point
  for (int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       gw < total_warps; gw += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
    const int64_t pn = gw / (SUBS * kw);
    const int64_t rem = gw - pn * (SUBS * kw);
    const int64_t j = rem / SUBS;
    const int64_t row0 = pn * kResPanel + (rem - j * SUBS) * RPT;
    if (row0 >= N) continue;                          // whole warp: no shuffle mixes rows
    // Lanes past the end of the row form whole groups (K % GROUP == 0), so
    // their dummy values never meet real ones in a reduction.
    const int64_t lc = j * 32 + lane;
    const bool active = lc < lanes_per_row;
    const int64_t k0 = (active ? lc : lanes_per_row - 1) * EPL;
    float w[RPT][EPL];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int64_t row = min(row0 + r, N - 1);       // a lone last row loads itself twice
      const uint4* wp = reinterpret_cast<const uint4*>(W + row * K + k0);
#pragma unroll
      for (int v = 0; v < EPL / 8; ++v) {
        const uint4 q = __ldg(wp + v);
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
          w[r][8 * v + 2 * i] = f.x;
          w[r][8 * v + 2 * i + 1] = f.y;
        }
      }
    }
#pragma unroll 1
    for (int a = 0; a < n_alpha; ++a) {
      float sv[EPL], rv[EPL];
      const float* sp = s_grid + static_cast<int64_t>(a) * K + k0;
      const float* rp = r_grid + static_cast<int64_t>(a) * K + k0;
#pragma unroll
      for (int v = 0; v < EPL / 8; ++v) {
        ld_v8f(sp + 8 * v, sv + 8 * v);
        ld_v8f(rp + 8 * v, rv + 8 * v);
      }
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        float ws[EPL];
#pragma unroll
        for (int i = 0; i < EPL; i += 2) {
          const f32x2 p = mul2(pack2(w[r][i], w[r][i + 1]), pack2(sv[i], sv[i + 1]));
          ws[i] = lo2(p);
          ws[i + 1] = hi2(p);
        }
        float mnA = fminf(ws[0], ws[1]), mxA = fmaxf(ws[0], ws[1]);
        float mnB = fminf(ws[2], ws[3]), mxB = fmaxf(ws[2], ws[3]);
#pragma unroll
        for (int i = 4; i < EPL; i += 4) {
          mnA = min3f(mnA, ws[i], ws[i + 1]);
          mxA = max3f(mxA, ws[i], ws[i + 1]);
          mnB = min3f(mnB, ws[i + 2], ws[i + 3]);
          mxB = max3f(mxB, ws[i + 2], ws[i + 3]);
        }
        float mn = fminf(mnA, mnB), mx = fmaxf(mxA, mxB);
#pragma unroll
        for (int off = GLANES / 2; off; off >>= 1) {
          mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
          mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        }
        const float step = __fdiv_rn(fmaxf(__fsub_rn(mx, mn), 1e-5f), L);
        const float sf = __half2float(__float2half_rn(step));
        const float rcp = __frcp_rn(sf);
        const float z = fminf(fmaxf(rne_small(__fmul_rn(-mn, rcp)), 0.0f), L);
        const float lo = -z, hi = L - z;
        const f32x2 nsf = pack2(-sf, -sf);
        uint32_t o[EPL / 2];
#pragma unroll
        for (int i = 0; i < EPL; i += 2) {
          const float d0 = fminf(fmaxf(rne_small(__fmul_rn(ws[i], rcp)), lo), hi);
          const float d1 = fminf(fmaxf(rne_small(__fmul_rn(ws[i + 1], rcp)), lo), hi);
          // w - (d * sf) * (1/s): the product d * sf is exact.
          const f32x2 e = fma2(mul2(pack2(d0, d1), nsf), pack2(rv[i], rv[i + 1]),
                               pack2(w[r][i], w[r][i + 1]));
          const __half2 hv = __floats2half2_rn(lo2(e), hi2(e));
          o[i / 2] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        const int64_t row = row0 + r;
        if (active && row < N) st_v8(delta + a * slab + (row_off + row) * K + k0, o);
      }
    }
  }
}

// Result layout: INT4 codes [N][K/8] (code 8j+m in nibble m of word j);
// INT3 codes [N][3K/32] (bit stream, code k in bits [3k, 3k+3));
// scales fp16 [N][K/group]; zeros u8 [N][K/group].
template <int BITS, int GROUP>
__global__ void __launch_bounds__(kQuantThreads)
    k_quant_final(const uint4* __restrict__ W, int64_t N, int64_t K, const float* __restrict__ s_base,
                  const int* __restrict__ sel, uint32_t* __restrict__ codes,
                  __half* __restrict__ scales, uint8_t* __restrict__ zeros) {
  constexpr int GLANES = GROUP / 8;
  constexpr int LEVELS = (1 << BITS) - 1;
  const int64_t kc = K / 8;
  const int64_t total = N * kc;
  const int64_t groups = K / GROUP;
  const float* s = s_base + (sel ? static_cast<int64_t>(*sel) * K : 0);
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
       base < total; base += stride) {
    const int64_t item = base + lane;
    const bool active = item < total;
    const int64_t it = active ? item : 0;
    const int64_t row = it / kc;
    const int64_t c = it - row * kc;
    const uint4 wv = active ? ldg_stream(W + it) : make_uint4(0, 0, 0, 0);
    const Quant8 r = quantize8<GLANES>(wv, s + c * 8, LEVELS);
    if (BITS == 4) {
      if (active) codes[it] = pack4(r);
    } else {
      // Four threads hold 4 x 24 bits = 3 words; thread j of the quad writes
      // word j from its own bits and those of thread j+1.
      const uint32_t own = pack3_bits24(r);
      const uint32_t next = __shfl_down_sync(0xFFFFFFFFu, own, 1);
      const int j = static_cast<int>(c & 3);
      if (active && j < 3) {
        const uint32_t word = (own >> (8 * j)) | (next << (24 - 8 * j));
        codes[row * (3 * K / 32) + (c >> 2) * 3 + j] = word;
      }
    }
    if (active && (lane % GLANES) == 0) {
      const int64_t g = (c * 8) / GROUP;
      scales[row * groups + g] = r.scale;
      zeros[row * groups + g] = static_cast<uint8_t>(r.zero);
    }
  }
}

__global__ void k_unpack(const uint32_t* __restrict__ codes, int64_t N, int64_t K, int bits,
                         uint8_t* __restrict__ q) {
  const int64_t total = N * K;
  const int64_t words = bits == 4 ? K / 8 : 3 * K / 32;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / K;
    const int64_t k = i - row * K;
    const uint32_t* rw = codes + row * words;
    const int64_t bit = static_cast<int64_t>(bits) * k;
    const int64_t w = bit >> 5;
    const int off = static_cast<int>(bit & 31);
    uint32_t v = rw[w] >> off;
    if (off + bits > 32) v |= rw[w + 1] << (32 - off);
    q[i] = static_cast<uint8_t>(v & ((1u << bits) - 1u));
  }
}

unsigned grid_for(int64_t items) {
  const int64_t blocks = ceil_div(items, kQuantThreads);
  return static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(blocks, 148 * 16)));
}

}  // namespace

cudaError_t launch_quant_residual(const __half* W, int64_t N, int64_t K, int bits, int group,
                                  const float* s_grid, const float* r_grid, int n_alpha,
                                  int64_t row_off, int64_t n_pad, __half* delta,
                                  cudaStream_t st) {
  const int levels = (1 << bits) - 1;
  const int64_t warps = ceil_div(N, kResPanel) * (kResPanel / kResRowsPerLane) *
                        ceil_div(K / kResPerLane, 32);
  const int64_t blocks = ceil_div(warps * 32, kQuantThreads);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(blocks, int64_t(1) << 30));
  if (group == 128)
    k_quant_residual<128><<<grid, kQuantThreads, 0, st>>>(W, N, K, levels, s_grid, r_grid,
                                                          n_alpha, row_off, n_pad, delta);
  else
    k_quant_residual<64><<<grid, kQuantThreads, 0, st>>>(W, N, K, levels, s_grid, r_grid,
                                                         n_alpha, row_off, n_pad, delta);
  return cudaGetLastError();
}

cudaError_t launch_quant_final(const __half* W, int64_t N, int64_t K, int bits, int group,
                               const float* s, const int* sel, uint32_t* codes,
                               __half* scales, uint8_t* zeros, cudaStream_t st) {
  const unsigned grid = grid_for(N * (K / 8));
  const uint4* w = reinterpret_cast<const uint4*>(W);
  if (bits == 4 && group == 128)
    k_quant_final<4, 128><<<grid, kQuantThreads, 0, st>>>(w, N, K, s, sel, codes, scales, zeros);
  else if (bits == 4 && group == 64)
    k_quant_final<4, 64><<<grid, kQuantThreads, 0, st>>>(w, N, K, s, sel, codes, scales, zeros);
  else if (bits == 3 && group == 128)
    k_quant_final<3, 128><<<grid, kQuantThreads, 0, st>>>(w, N, K, s, sel, codes, scales, zeros);
  else
    k_quant_final<3, 64><<<grid, kQuantThreads, 0, st>>>(w, N, K, s, sel, codes, scales, zeros);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* codes, int64_t N, int64_t K, int bits, uint8_t* q,
                          cudaStream_t st) {
  k_unpack<<<grid_for(N * K), kQuantThreads, 0, st>>>(codes, N, K, bits, q);
  return cudaGetLastError();
}

}  // namespace awq
