// Gram form of the layer-output loss (a faster evaluation of the same
// objective when calibration tokens outnumber input channels).
//
// AWQ Explained (multigrid.ai), "How the scale is chosen": the loss is
// || W x - Q(W diag(s)) diag(s)^-1 x ||^2 over the calibration tokens.  With
// the residual d_n of output row n, sum_t (d_n . x_t)^2 = d_n^T G d_n where
// G = X^T X (K x K) does not depend on alpha: one GEMM of T K^2 flops, after
// which each grid point costs N K^2 instead of N K T.
//
// This file prepares G for the tensor cores: X^T (fp16 [K][Tp], tokens
// zero-padded to a multiple of 64), then -- after G = X^T (X^T)^T in fp32 on
// the reference GEMM -- the fp16 operand Gs = G * (c / T) with c a power of
// two chosen from max |G| so that |Gs| <= 32768 (fp16 cannot hold G itself
// once channels carry outliers), and row_scale = T / c to undo it.
#include <algorithm>

#include "awq_internal.h"

namespace awq {
namespace {

// X [T][K] -> XT [K][Tp]; columns T..Tp-1 are zero.  32 x 32 tiles through
// shared memory (the +1 column avoids bank conflicts).
__global__ void k_transpose(const __half* __restrict__ X, int64_t T, int64_t K, int64_t Tp,
                            __half* __restrict__ XT) {
  __shared__ __half tile[32][33];
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int64_t k0 = static_cast<int64_t>(blockIdx.y) * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t t = t0 + i, k = k0 + threadIdx.x;
    tile[i][threadIdx.x] = (t < T && k < K) ? X[t * K + k] : __float2half(0.f);
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t k = k0 + i, t = t0 + threadIdx.x;
    if (k < K && t < Tp) XT[k * Tp + t] = tile[threadIdx.x][i];
  }
}

// max |G| as the bit pattern of a non-negative float (monotone as unsigned).
__global__ void k_absmax(const float* __restrict__ G, int64_t n, unsigned int* __restrict__ mx) {
  float m = 0.f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    m = fmaxf(m, fabsf(G[i]));
#pragma unroll
  for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if ((threadIdx.x & 31) == 0) atomicMax(mx, __float_as_uint(m));
}

// Gs = fp16(G * (c / T)), c = 2^e the largest power of two with
// max|G| * c / T <= 32768; row_scale = T / c.
__global__ void k_gram_half(const float* __restrict__ G, int64_t n, int64_t T,
                            const unsigned int* __restrict__ mx, __half* __restrict__ Gs,
                            double* __restrict__ row_scale) {
  const float gmax = __uint_as_float(*mx);
  // exponent e with gmax * 2^e / T <= 2^15 (e may be negative); gmax == 0 -> e = 0
  int e = 0;
  if (gmax > 0.f) {
    const double r = 32768.0 * static_cast<double>(T) / static_cast<double>(gmax);
    e = static_cast<int>(floor(log2(r)));
    e = max(-120, min(120, e));
  }
  const float cs = static_cast<float>(ldexp(1.0, e) / static_cast<double>(T));
  if (blockIdx.x == 0 && threadIdx.x == 0) *row_scale = static_cast<double>(T) / ldexp(1.0, e);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    Gs[i] = __float2half_rn(G[i] * cs);
}

}  // namespace

cudaError_t launch_gram_prepare(const __half* X, int64_t T, int64_t K, __half* XT, int64_t Tp,
                                float* G, unsigned int* mx, __half* Gs, double* row_scale,
                                int* status, cudaStream_t st, int* launches) {
  const dim3 tgrid(static_cast<unsigned>(ceil_div(Tp, 32)), static_cast<unsigned>(ceil_div(K, 32)));
  k_transpose<<<tgrid, dim3(32, 8), 0, st>>>(X, T, K, Tp, XT);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_gemm_reference(XT, K, XT, K, Tp, G, status, st);   // G = X^T X, fp32 [K][K]
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(mx, 0, sizeof(unsigned int), st);
  if (e != cudaSuccess) return e;
  const int64_t n = K * K;
  const unsigned blocks = static_cast<unsigned>(std::min<int64_t>(ceil_div(n, 256), static_cast<int64_t>(device_sm_count()) * 8));
  k_absmax<<<blocks, 256, 0, st>>>(G, n, mx);
  k_gram_half<<<blocks, 256, 0, st>>>(G, n, T, mx, Gs, row_scale);
  *launches += 4;
  return cudaGetLastError();
}

}  // namespace awq
