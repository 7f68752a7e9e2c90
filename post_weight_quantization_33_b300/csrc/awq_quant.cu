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

// Search output (one launch per weight, blockIdx.y = grid point a): the
// quantization residual in the units of W,
//   delta[a][row_off + n][k] = fp16( w - ((q - z) * scale) * (1/s_k) ),
// i.e. W - deq(Q(W diag(s))) diag(s)^-1 row by row.  (q - z) * scale is exact
// in fp32 (a 5-bit integer times an 11-bit significand); the product with the
// fp32 reciprocal and the difference are single fp32 roundings, and the only
// coarse rounding is the final one to fp16, relative to the residual itself.
template <int GROUP>
__global__ void __launch_bounds__(kQuantThreads)
    k_quant_residual(const uint4* __restrict__ W, int64_t N, int64_t K, int levels,
                     const float* __restrict__ s_grid, const float* __restrict__ r_grid,
                     int64_t row_off, int64_t n_pad, uint4* __restrict__ delta) {
  constexpr int GLANES = GROUP / 8;
  const int a = blockIdx.y;
  const int64_t kc = K / 8;
  const int64_t total = N * kc;
  const float* s = s_grid + static_cast<int64_t>(a) * K;
  const float* r = r_grid + static_cast<int64_t>(a) * K;
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
    const Quant8 q = quantize8<GLANES>(wv, s + c * 8, levels);
    if (active) {
      const float4 ra = __ldg(reinterpret_cast<const float4*>(r + c * 8));
      const float4 rb = __ldg(reinterpret_cast<const float4*>(r + c * 8) + 1);
      const float rv[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
      const float sf = __half2float(q.scale);
      const uint32_t w32[4] = {wv.x, wv.y, wv.z, wv.w};
      uint32_t out[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h = *reinterpret_cast<const __half2*>(&w32[i]);
        const float d0 = __fmul_rn(static_cast<float>(static_cast<int>(q.q[2 * i]) - q.zero), sf);
        const float d1 =
            __fmul_rn(static_cast<float>(static_cast<int>(q.q[2 * i + 1]) - q.zero), sf);
        const float e0 = __fsub_rn(__low2float(h), __fmul_rn(d0, rv[2 * i]));
        const float e1 = __fsub_rn(__high2float(h), __fmul_rn(d1, rv[2 * i + 1]));
        const __half2 e = __floats2half2_rn(e0, e1);
        out[i] = *reinterpret_cast<const uint32_t*>(&e);
      }
      delta[(static_cast<int64_t>(a) * n_pad + row_off + row) * kc + c] =
          make_uint4(out[0], out[1], out[2], out[3]);
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
  const dim3 grid(grid_for(N * (K / 8)), static_cast<unsigned>(n_alpha));
  const uint4* w = reinterpret_cast<const uint4*>(W);
  uint4* d = reinterpret_cast<uint4*>(delta);
  if (group == 128)
    k_quant_residual<128><<<grid, kQuantThreads, 0, st>>>(w, N, K, levels, s_grid, r_grid,
                                                          row_off, n_pad, d);
  else
    k_quant_residual<64><<<grid, kQuantThreads, 0, st>>>(w, N, K, levels, s_grid, r_grid,
                                                         row_off, n_pad, d);
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
