// Decode product with the packed output of the search: y = deq(Q) x for a
// batch of 1 to 16 tokens, INT4 or INT3 codes.
//
// AWQ explained (hungho77.github.io), "Why weight-only quantization fits
// decoding": generating tokens at small batch reads every weight once while
// the activations are tiny, so the step is bound by weight traffic; 3- or
// 4-bit weights with 16-bit activations cut that traffic four times or more.
//
//   y[m][n] = sum_g scale[n][g] * sum_{k in g} (code[n][k] - zero[n][g]) * x[m][k]
//
// HBM-bound: per weight b/8 byte of codes plus 3 bytes per group.  The
// multiply-adds run on the tensor cores (mma.sync m16n8k16, fp16 operands,
// fp32 accumulation): A is a 16-row tile of the weight as exact fp16
// (code - zero) values built in registers, B holds 8 tokens of x.  A warp
// reads 16 rows x 64 channels (a "unit") per step and issues 4 MMAs per 8
// tokens; at each group's end the fp32 sums are scaled by the group's fp16
// scale (in fp32) and added to the row's accumulator.
//
// Channel order.  The dot product over a group does not depend on the order
// of its channels, so each thread of a quad takes 16 consecutive codes of its
// two rows (one 8-byte load per row for INT4) and feeds them to the four
// MMAs of the unit: in step j, thread c supplies channels 16c+j, 16c+j+4,
// 16c+8+j and 16c+12+j in the slots the fragment layout gives it (2c, 2c+1,
// 2c+8, 2c+9).  The B fragment of thread (token t, c) holds x at the same
// channels, taken from its own 32-byte load of x[t][16c .. 16c+15] by byte
// permutes.  (code - zero) is formed exactly in fp16: 0x6400 | code is
// 1024 + code, minus 1024 + zero.
//
// Work split.  One block per SM; the (row tile, unit) items, tile-major, are
// cut into equal contiguous ranges, one per warp, each at least one row tile
// long, so every SM gets the same work and at most two warps add into an
// output (y is zeroed first; two fp32 additions onto zero commute, so the
// result does not depend on their order).
#include <algorithm>

#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kUnit = 64;        // channels per unit
constexpr int kPrefetch = 8;     // units of codes in flight per warp
constexpr int kMaxWarps = 12;    // per block (one block per SM)

__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream_u64(const uint32_t* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a),
                            *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// The 16 codes of one row that thread c uses in a unit, as two 32-bit
// fields holding codes 0..7 and 8..15 in consecutive b-bit slots.
template <int BITS>
struct RowCodes {
  uint32_t lo, hi;
};

// INT4: codes 16c .. 16c+15 of the unit are words 2c, 2c+1 (8 codes each).
// INT3: they are bits [48c, 48c+48) of the unit's 6 words.
template <int BITS>
__device__ __forceinline__ RowCodes<BITS> load_codes(const uint32_t* row, int64_t unit, int c) {
  RowCodes<BITS> r;
  if (BITS == 4) {
    const uint2 v = ld_stream_u64(row + unit * 8 + 2 * c);
    r.lo = v.x;
    r.hi = v.y;
  } else {
    const uint32_t* u = row + unit * 6 + (3 * c) / 2;
    const uint32_t w0 = ld_stream_u32(u), w1 = ld_stream_u32(u + 1);
    if (c & 1) {   // the 48 bits start at bit 16 of w0
      r.lo = __funnelshift_r(w0, w1, 16) & 0xFFFFFFu;
      r.hi = w1 >> 8;
    } else {
      r.lo = w0 & 0xFFFFFFu;
      r.hi = __funnelshift_r(w0, w1, 24) & 0xFFFFFFu;
    }
  }
  return r;
}

// 1024 + code_j (low half) and 1024 + code_{j+4} (high half) of a field.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(uint32_t f, int j) {
  if (BITS == 4) return ((f >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
  const uint32_t t = f >> (3 * j);
  return (t & 0x7u) | ((t << 4) & 0x70000u) | 0x64006400u;
}

template <int NT, int GROUP, int BITS>
__global__ void __launch_bounds__(kMaxWarps * 32)
    k_wq_mma(const uint32_t* __restrict__ codes, const __half* __restrict__ scales,
             const uint8_t* __restrict__ zeros, int64_t N, int64_t K,
             const __half* __restrict__ x, int M, float* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t upr = K / kUnit;                        // units per row
  const int64_t tiles = (N + 15) / 16;
  const int64_t items = tiles * upr;
  const int64_t i0 = w * items / warps, i1 = (w + 1) * items / warps;
  const int64_t words_per_row = K * BITS / 32;
  const int64_t groups = GROUP ? K / GROUP : 1;
  constexpr int kUnitsPerGroup = GROUP ? GROUP / kUnit : 1;

  int64_t i = i0;
  while (i < i1) {
    const int64_t tile = i / upr;
    const int64_t u0 = i - tile * upr;
    const int64_t u1 = min(upr, u0 + (i1 - i));
    const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
    const int64_t l0 = min(r0, N - 1), l1 = min(r1, N - 1);
    const uint32_t* row0 = codes + l0 * words_per_row;
    const uint32_t* row1 = codes + l1 * words_per_row;
    float acc[NT][4], part[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] = part[t][e] = 0.f;
    // Codes of the next kPrefetch units in flight.
    RowCodes<BITS> q0[kPrefetch], q1[kPrefetch];
#pragma unroll
    for (int p = 0; p < kPrefetch; ++p)
      if (u0 + p < u1) {
        q0[p] = load_codes<BITS>(row0, u0 + p, c);
        q1[p] = load_codes<BITS>(row1, u0 + p, c);
      }
    for (int64_t u = u0; u < u1; u += kPrefetch) {
#pragma unroll
      for (int p = 0; p < kPrefetch; ++p) {
        const int64_t uu = u + p;
        if (uu >= u1) break;
        const RowCodes<BITS> a0 = q0[p], a1 = q1[p];
        if (uu + kPrefetch < u1) {
          q0[p] = load_codes<BITS>(row0, uu + kPrefetch, c);
          q1[p] = load_codes<BITS>(row1, uu + kPrefetch, c);
        }
        const int64_t k0 = uu * kUnit;
        int64_t grp = 0;
        if constexpr (GROUP != 0) grp = k0 / GROUP;
        // 1024 + zero of each row in both halves (exact: fp16 bits 0x6400 + z).
        const uint32_t z0 = 0x6400u + zeros[l0 * groups + grp];
        const uint32_t z1 = 0x6400u + zeros[l1 * groups + grp];
        const uint32_t zp0 = z0 | (z0 << 16), zp1 = z1 | (z1 << 16);
        // x of this thread's tokens at channels k0 + 16c .. + 15.
        uint4 xv[NT][2];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int tok = t * 8 + g;
          if (tok < M) {
            const uint4* xp = reinterpret_cast<const uint4*>(x + tok * K + k0 + 16 * c);
            xv[t][0] = __ldg(xp);
            xv[t][1] = __ldg(xp + 1);
          } else {
            xv[t][0] = xv[t][1] = make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t a[4];
          a[0] = hsub2_u32(code_pair<BITS>(a0.lo, j), zp0);   // row g,   slots 2c, 2c+1
          a[1] = hsub2_u32(code_pair<BITS>(a1.lo, j), zp1);   // row g+8
          a[2] = hsub2_u32(code_pair<BITS>(a0.hi, j), zp0);   // row g,   slots 2c+8, 2c+9
          a[3] = hsub2_u32(code_pair<BITS>(a1.hi, j), zp1);   // row g+8
          const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const uint32_t X[8] = {xv[t][0].x, xv[t][0].y, xv[t][0].z, xv[t][0].w,
                                   xv[t][1].x, xv[t][1].y, xv[t][1].z, xv[t][1].w};
            // x[16c + j], x[16c + j + 4]  and  x[16c + 8 + j], x[16c + 12 + j]
            const uint32_t b0 = __byte_perm(X[j >> 1], X[(j >> 1) + 2], sel);
            const uint32_t b1 = __byte_perm(X[4 + (j >> 1)], X[6 + (j >> 1)], sel);
            mma_16816(part[t], a, b0, b1);
          }
        }
        // End of a group (or of this warp's part of a per-row group).
        bool group_end = uu + 1 == u1;
        if constexpr (GROUP != 0) group_end = (uu + 1) % kUnitsPerGroup == 0;
        if (group_end) {
          const float s0 = __half2float(scales[l0 * groups + grp]);
          const float s1 = __half2float(scales[l1 * groups + grp]);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            acc[t][0] = __fmaf_rn(s0, part[t][0], acc[t][0]);
            acc[t][1] = __fmaf_rn(s0, part[t][1], acc[t][1]);
            acc[t][2] = __fmaf_rn(s1, part[t][2], acc[t][2]);
            acc[t][3] = __fmaf_rn(s1, part[t][3], acc[t][3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) part[t][e] = 0.f;
          }
        }
      }
    }
    // A range may end inside a group (g128: after its first unit): scale
    // the partial sum of that group too.
    if (GROUP != 0 && (u1 % kUnitsPerGroup) != 0) {
      const int64_t grp = (u1 * kUnit - 1) / (GROUP != 0 ? GROUP : 1);
      const float s0 = __half2float(scales[l0 * groups + grp]);
      const float s1 = __half2float(scales[l1 * groups + grp]);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        acc[t][0] = __fmaf_rn(s0, part[t][0], acc[t][0]);
        acc[t][1] = __fmaf_rn(s0, part[t][1], acc[t][1]);
        acc[t][2] = __fmaf_rn(s1, part[t][2], acc[t][2]);
        acc[t][3] = __fmaf_rn(s1, part[t][3], acc[t][3]);
      }
    }
    // C fragment: elements 0, 1 are row g, tokens 2c, 2c+1; 2, 3 row g+8.
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int m0 = t * 8 + 2 * c;
      if (r0 < N) {
        if (m0 < M) atomicAdd(y + m0 * N + r0, acc[t][0]);
        if (m0 + 1 < M) atomicAdd(y + (m0 + 1) * N + r0, acc[t][1]);
      }
      if (r1 < N) {
        if (m0 < M) atomicAdd(y + m0 * N + r1, acc[t][2]);
        if (m0 + 1 < M) atomicAdd(y + (m0 + 1) * N + r1, acc[t][3]);
      }
    }
    i += u1 - u0;
  }
}

template <int NT, int BITS>
cudaError_t launch_wq(int group, const uint32_t* codes, const __half* scales,
                      const uint8_t* zeros, int64_t N, int64_t K, const __half* x, int M,
                      float* y, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * static_cast<size_t>(M) * N, st);
  if (e != cudaSuccess) return e;
  // One block per SM.  Warps: at most one per 16-row tile (every warp's range
  // is then at least a tile long: at most two warps per output), at most 12.
  const int64_t tiles = (N + 15) / 16;
  const int sms = device_sm_count();
  int64_t blocks = std::min<int64_t>(sms, tiles);
  int64_t wpb = std::max<int64_t>(1, std::min<int64_t>(kMaxWarps, tiles / blocks));
  auto go = [&](auto kern) -> cudaError_t {
    kern<<<static_cast<unsigned>(blocks), static_cast<unsigned>(32 * wpb), 0, st>>>(
        codes, scales, zeros, N, K, x, M, y);
    return cudaGetLastError();
  };
  if (group == 128) return go(k_wq_mma<NT, 128, BITS>);
  if (group == 64) return go(k_wq_mma<NT, 64, BITS>);
  return go(k_wq_mma<NT, 0, BITS>);
}

}  // namespace

cudaError_t launch_w4_matvec(const uint32_t* codes, const __half* scales, const uint8_t* zeros,
                             int64_t N, int64_t K, int group, int bits, const __half* x, int M,
                             float* y, cudaStream_t st) {
  if (M < 1 || M > 16 || K % kUnit) return cudaErrorInvalidValue;
  if (bits == 4)
    return M <= 8 ? launch_wq<1, 4>(group, codes, scales, zeros, N, K, x, M, y, st)
                  : launch_wq<2, 4>(group, codes, scales, zeros, N, K, x, M, y, st);
  if (bits == 3)
    return M <= 8 ? launch_wq<1, 3>(group, codes, scales, zeros, N, K, x, M, y, st)
                  : launch_wq<2, 3>(group, codes, scales, zeros, N, K, x, M, y, st);
  return cudaErrorInvalidValue;
}

}  // namespace awq
