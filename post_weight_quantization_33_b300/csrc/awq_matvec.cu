// W4A16 decode product with the packed output of the search.
//
// AWQ explained (hungho77.github.io), "Why weight-only quantization fits
// decoding": generating a token at small batch reads every weight once while
// the activations are tiny, so the step is bound by weight traffic; 4-bit
// weights with 16-bit activations cut that traffic about four times.
//
//   y[m][n] = sum_g scale[n][g] * sum_{k in g} (code[n][k] - zero[n][g]) * x[m][k]
//
// HBM-bound for M <= 8: per weight 0.5 byte of codes plus 3 bytes per group.
// A warp takes two rows; per step a lane reads 32 consecutive codes (16
// bytes) of each row, two steps ahead; x is staged once per block in shared
// memory as fp32 ([M][Kc], chunked along K, swizzled) and shared by all 16
// rows of the block.  (code - zero) is formed exactly as a float: the code's
// 4 bits placed in the significand of 2^23 by a byte permute, minus the
// constant 2^23 + zero, two codes at a time (packed f32x2).  Each lane sums
// even and odd codes of a 32-code piece separately (packed fma), scales the
// piece's dot product by the group's scale as it goes and keeps one fp32 sum
// per (row, token); the warp adds its 32 lanes at the end.  All sums are fp32.
#include <algorithm>

#include "awq_f32x2.cuh"
#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kMvThreads = 256;
constexpr int kMvRowsPerWarp = 2;
constexpr int kMvRowsPerBlock = (kMvThreads / 32) * kMvRowsPerWarp;
constexpr int kMvSmemBytes = 96 * 1024;   // x chunk: M * Kc fp32
constexpr int kMvSteps = 2;               // 16-byte code loads in flight per lane and row

// x lives in shared memory as fp32, [M][kc], in 16-byte chunks with the chunk
// index XOR-swizzled by (chunk / 8) % 8: a lane reads 8 consecutive chunks
// (32 channels) and lanes are 8 chunks apart, so without the swizzle the 8
// lanes of a quarter-warp would hit the same banks.
__device__ __forceinline__ int64_t xs_chunk(int64_t c) { return c ^ ((c >> 3) & 7); }

// 2^23 + code as a float, for the code in the low nibble of byte k of `nib`
// (a byte permute places that byte under 0x4B0000).
template <int k>
__device__ __forceinline__ float magic_code(uint32_t nib) {
  return __uint_as_float(__byte_perm(nib, 0x4B000000u, 0x7640 + k));
}

// GROUP: 64, 128, or 0 (one group per row).  A lane takes 32 consecutive
// channels (one 16-byte load of 4 code words) of each of its warp's two rows
// per step, so its group scale and zero are loaded once per 32 codes; a warp
// covers 1024 channels per step.
template <int M, int GROUP>
__global__ void __launch_bounds__(kMvThreads)
    k_w4_matvec(const uint32_t* __restrict__ codes, const __half* __restrict__ scales,
                const uint8_t* __restrict__ zeros, int64_t N, int64_t K,
                const __half* __restrict__ x, float* __restrict__ y, int64_t kc) {
  extern __shared__ float4 xs4[];            // [M][kc / 4] swizzled 16-byte chunks
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t words = K / 8;
  const int64_t groups = GROUP ? K / GROUP : 1;
  const int64_t n_chunks = (K + kc - 1) / kc;
  const int64_t cpr = kc / 4;                // 16-byte chunks per x row in shared memory
  int it = 0;
  // Block-uniform loop over 16-row tiles: every warp runs the same iterations
  // and meets the same barriers (rows past N idle).
  for (int64_t tile = static_cast<int64_t>(blockIdx.x) * kMvRowsPerBlock; tile < N;
       tile += static_cast<int64_t>(gridDim.x) * kMvRowsPerBlock, ++it) {
    const int64_t n0 = tile + warp * kMvRowsPerWarp;
    const bool live = n0 < N;
    const int64_t n1 = min(n0 + 1, N - 1);   // a lone last row is computed twice
    float acc[kMvRowsPerWarp][M];
#pragma unroll
    for (int r = 0; r < kMvRowsPerWarp; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[r][m] = 0.f;
    for (int64_t c = 0; c < n_chunks; ++c) {
      const int64_t k0 = c * kc;
      const int64_t klen = min(kc, K - k0);
      if (n_chunks > 1 || it == 0) {        // one chunk: x is staged once per block
        __syncthreads();
        for (int64_t i = threadIdx.x; i < M * (klen / 4); i += blockDim.x) {
          const int64_t m = i / (klen / 4), q4 = i - m * (klen / 4);
          const __half2* src = reinterpret_cast<const __half2*>(x + m * K + k0 + 4 * q4);
          const float2 a = __half22float2(src[0]), b = __half22float2(src[1]);
          xs4[m * cpr + xs_chunk(q4)] = make_float4(a.x, a.y, b.x, b.y);
        }
        __syncthreads();
      }
      if (!live) continue;
      const uint4* r0 = reinterpret_cast<const uint4*>(codes + n0 * words + k0 / 8);
      const uint4* r1 = reinterpret_cast<const uint4*>(codes + n1 * words + k0 / 8);
      const int64_t nq = klen / 32;          // 32-channel pieces in the chunk
      for (int64_t pb = lane; pb < nq; pb += 32 * kMvSteps) {
        uint4 wv[kMvSteps][kMvRowsPerWarp];
        float sf[kMvSteps][kMvRowsPerWarp], zo[kMvSteps][kMvRowsPerWarp];
#pragma unroll
        for (int u = 0; u < kMvSteps; ++u) {
          const int64_t p = pb + 32 * u;
          const bool in = p < nq;
          const int64_t pp = in ? p : 0;
          const int64_t g = GROUP ? (k0 + 32 * pp) / GROUP : 0;
          wv[u][0] = in ? __ldg(r0 + pp) : make_uint4(0, 0, 0, 0);
          wv[u][1] = in ? __ldg(r1 + pp) : make_uint4(0, 0, 0, 0);
          sf[u][0] = __half2float(scales[n0 * groups + g]);
          sf[u][1] = __half2float(scales[n1 * groups + g]);
          zo[u][0] = 8388608.0f + static_cast<float>(zeros[n0 * groups + g]);
          zo[u][1] = 8388608.0f + static_cast<float>(zeros[n1 * groups + g]);
        }
#pragma unroll
        for (int u = 0; u < kMvSteps; ++u) {
          const int64_t p = pb + 32 * u;
          if (p >= nq) break;
          // Packed pairs (even code, odd code): (2^23 + code) - (2^23 + zero)
          // is exact, then one packed fma per pair of weights.
          f32x2 d2[kMvRowsPerWarp][M];
#pragma unroll
          for (int r = 0; r < kMvRowsPerWarp; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) d2[r][m] = 0ull;
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {   // word wi: channels 32p + 8wi .. + 8
            f32x2 q2[kMvRowsPerWarp][4];     // pair b: codes 2b, 2b + 1 of the word
#pragma unroll
            for (int r = 0; r < kMvRowsPerWarp; ++r) {
              const uint32_t wd = wi == 0 ? wv[u][r].x : wi == 1 ? wv[u][r].y
                                : wi == 2 ? wv[u][r].z : wv[u][r].w;
              const uint32_t ev = wd & 0x0F0F0F0Fu, od = (wd >> 4) & 0x0F0F0F0Fu;
              const f32x2 nz = pack2(-zo[u][r], -zo[u][r]);
              q2[r][0] = add2(pack2(magic_code<0>(ev), magic_code<0>(od)), nz);
              q2[r][1] = add2(pack2(magic_code<1>(ev), magic_code<1>(od)), nz);
              q2[r][2] = add2(pack2(magic_code<2>(ev), magic_code<2>(od)), nz);
              q2[r][3] = add2(pack2(magic_code<3>(ev), magic_code<3>(od)), nz);
            }
#pragma unroll
            for (int m = 0; m < M; ++m) {
              const int64_t cidx = 8 * p + 2 * wi;          // first 16-byte chunk of the word
              const float4 xa = xs4[m * cpr + xs_chunk(cidx)];
              const float4 xb = xs4[m * cpr + xs_chunk(cidx + 1)];
              const f32x2 x2[4] = {pack2(xa.x, xa.y), pack2(xa.z, xa.w), pack2(xb.x, xb.y),
                                   pack2(xb.z, xb.w)};
#pragma unroll
              for (int r = 0; r < kMvRowsPerWarp; ++r)
#pragma unroll
                for (int b = 0; b < 4; ++b) d2[r][m] = fma2(q2[r][b], x2[b], d2[r][m]);
            }
          }
          float d[kMvRowsPerWarp][M];
#pragma unroll
          for (int r = 0; r < kMvRowsPerWarp; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) d[r][m] = __fadd_rn(lo2(d2[r][m]), hi2(d2[r][m]));
#pragma unroll
          for (int r = 0; r < kMvRowsPerWarp; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) acc[r][m] = __fmaf_rn(sf[u][r], d[r][m], acc[r][m]);
        }
      }
    }
    if (!live) continue;
#pragma unroll
    for (int r = 0; r < kMvRowsPerWarp; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float v = acc[r][m];
#pragma unroll
        for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        acc[r][m] = v;
      }
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < M; ++m) {
        y[m * N + n0] = acc[0][m];
        if (n0 + 1 < N) y[m * N + n0 + 1] = acc[1][m];
      }
    }
  }
}

template <int M>
cudaError_t launch_mv_m(int group, const uint32_t* codes, const __half* scales,
                        const uint8_t* zeros, int64_t N, int64_t K, const __half* x, float* y,
                        cudaStream_t st) {
  // x chunk: as many channels as fit, a multiple of 256 (whole 32-channel
  // pieces, whole groups, whole swizzle periods of 8 chunks).
  int64_t kc = (kMvSmemBytes / (M * 4)) / 256 * 256;
  if (kc >= K) kc = K;
  const int smem = static_cast<int>(M * kc * 4);
  auto go = [&](auto kern) -> cudaError_t {
    LaunchFacts lf;   // resident blocks per SM: one wave of persistent blocks
    cudaError_t e = launch_facts(reinterpret_cast<const void*>(kern), kMvThreads, smem, &lf);
    if (e != cudaSuccess) return e;
    const int64_t blocks =
        std::min<int64_t>(ceil_div(N, kMvRowsPerBlock), static_cast<int64_t>(lf.per_sm) * lf.sms);
    kern<<<static_cast<unsigned>(blocks), kMvThreads, smem, st>>>(codes, scales, zeros, N, K, x, y,
                                                                  kc);
    return cudaGetLastError();
  };
  if (group == 128) return go(k_w4_matvec<M, 128>);
  if (group == 64) return go(k_w4_matvec<M, 64>);
  return go(k_w4_matvec<M, 0>);
}

}  // namespace

cudaError_t launch_w4_matvec(const uint32_t* codes, const __half* scales, const uint8_t* zeros,
                             int64_t N, int64_t K, int group, const __half* x, int M, float* y,
                             cudaStream_t st) {
  switch (M) {
    case 1: return launch_mv_m<1>(group, codes, scales, zeros, N, K, x, y, st);
    case 2: return launch_mv_m<2>(group, codes, scales, zeros, N, K, x, y, st);
    case 3: return launch_mv_m<3>(group, codes, scales, zeros, N, K, x, y, st);
    case 4: return launch_mv_m<4>(group, codes, scales, zeros, N, K, x, y, st);
    case 5: return launch_mv_m<5>(group, codes, scales, zeros, N, K, x, y, st);
    case 6: return launch_mv_m<6>(group, codes, scales, zeros, N, K, x, y, st);
    case 7: return launch_mv_m<7>(group, codes, scales, zeros, N, K, x, y, st);
    case 8: return launch_mv_m<8>(group, codes, scales, zeros, N, K, x, y, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace awq
