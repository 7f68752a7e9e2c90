// Deploy step: fold diag(s)^-1 into the producer of the layer's input.
//
// AWQ Explained (multigrid.ai), "Scaling instead of mixed precision": the
// division on the activation side costs nothing at run time, because
// diag(s)^-1 folds offline into the operation before the layer -- the
// preceding LayerNorm / RMSNorm weight, or a preceding linear layer -- and
// what ships is the quantized matrix plus that modified operation.
//
//   out[i][j] = fp16_rne( fp32(V[i][j]) / s[i] )   (correctly rounded fp32
//   division; row i of V feeds input channel i of the quantized layer).
//
// One HBM pass: 2 bytes read and 2 written per element.
#include <algorithm>

#include "awq_bounds.cuh"
#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kFoldThreads = 256;

__device__ __forceinline__ __half fold1(__half v, float s) {
  return __float2half_rn(__fdiv_rn(__half2float(v), s));
}

// Vector (a norm weight or a bias): element i uses s[i].
__global__ void __launch_bounds__(kFoldThreads)
    k_fold_vec(const __half* __restrict__ V, int64_t n, const float* __restrict__ s,
               __half* __restrict__ out) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = fold1(V[i], s[i]);
}

// Matrix [rows][cols]: block (x, y) takes columns [2048x, 2048x + 2048) of
// rows y, y + gridDim.y, ...; a thread takes 8 consecutive columns (one
// 16-byte access when VEC: cols % 8 == 0 and both pointers 16-byte aligned).
template <bool VEC>
__global__ void __launch_bounds__(kFoldThreads)
    k_fold_rows(const __half* V, int64_t rows, int64_t cols, const float* __restrict__ s,
                __half* out) {
  const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  if (c0 >= cols) return;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    const float sr = __ldg(s + r);
    const int64_t base = r * cols + c0;
    if (!in_bounds(kSiteFold, base + (VEC ? 8 : std::min<int64_t>(cols - c0, 8)) - 1,
                   rows * cols))
      continue;
    if (VEC) {
      const uint4 v = *reinterpret_cast<const uint4*>(V + base);
      uint4 o;
      const __half* h = reinterpret_cast<const __half*>(&v);
      __half* g = reinterpret_cast<__half*>(&o);
#pragma unroll
      for (int j = 0; j < 8; ++j) g[j] = fold1(h[j], sr);
      *reinterpret_cast<uint4*>(out + base) = o;
    } else {
      const int64_t m = cols - c0 < 8 ? cols - c0 : 8;
      for (int64_t j = 0; j < m; ++j) out[base + j] = fold1(V[base + j], sr);
    }
  }
}

}  // namespace

cudaError_t launch_fold(const __half* V, int64_t rows, int64_t cols, const float* s, __half* out,
                        cudaStream_t st) {
  if (cols == 1) {
    const int64_t blocks = std::min<int64_t>(ceil_div(rows, kFoldThreads), static_cast<int64_t>(device_sm_count()) * 8);
    k_fold_vec<<<static_cast<unsigned>(blocks), kFoldThreads, 0, st>>>(V, rows, s, out);
    return cudaGetLastError();
  }
  const bool vec = cols % 8 == 0 && reinterpret_cast<uintptr_t>(V) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(out) % 16 == 0;
  const int64_t gx = ceil_div(ceil_div(cols, 8), kFoldThreads);
  // Enough blocks for ~8 per SM in total, rows walked grid-stride.
  const int64_t gy = std::max<int64_t>(1, std::min<int64_t>({rows, 65535, ceil_div(static_cast<int64_t>(device_sm_count()) * 8, gx)}));
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  if (vec)
    k_fold_rows<true><<<grid, kFoldThreads, 0, st>>>(V, rows, cols, s, out);
  else
    k_fold_rows<false><<<grid, kFoldThreads, 0, st>>>(V, rows, cols, s, out);
  return cudaGetLastError();
}

AWQ_BOUNDS_READER(bounds_fold)

}  // namespace awq
