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
// Work split.  One block of 16 warps per SM.  The (row tile, unit) items,
// tile-major, are cut into equal contiguous ranges, one per block (each at
// least one row tile long), and a block's range into one contiguous range per
// warp.  A warp streams its units with the codes and group parameters of the
// next kPrefetch units in flight, across row-tile boundaries.  A row tile
// entirely inside one warp's range is added to y at once; the partial sums of
// the tiles at the two ends of a warp's range go to shared memory, and the
// block adds them up in warp order before adding them to y.  y is zeroed
// first and at most two blocks add into an output (two fp32 additions onto
// zero commute), so the result is deterministic.  x is staged once per block
// in shared memory when M x K fits (16-byte chunks swizzled by token, so a
// quad-row read is conflict-free), else read through L1.
#include <algorithm>

#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kUnit = 64;          // channels per unit
constexpr int kMaxWarps = 16;      // per block (one block per SM)
constexpr int kXSmemMax = 192 * 1024;

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

// One unit of one row as thread c needs it: codes 16c .. 16c+15 of the unit
// as two fields (codes 0..7 and 8..15 in consecutive b-bit slots).
struct UnitRow {
  uint32_t lo, hi;
};

template <int BITS>
__device__ __forceinline__ void load_fields(const uint32_t* p, int c, uint32_t& lo, uint32_t& hi) {
  if (BITS == 4) {   // words 2c, 2c+1 of the unit (p points at word 2c)
    const uint2 v = ld_stream_u64(p);
    lo = v.x;
    hi = v.y;
  } else {           // bits [48c, 48c+48) of the unit's 6 words (p at word 3c/2)
    const uint32_t w0 = ld_stream_u32(p), w1 = ld_stream_u32(p + 1);
    if (c & 1) {
      lo = __funnelshift_r(w0, w1, 16) & 0xFFFFFFu;
      hi = w1 >> 8;
    } else {
      lo = w0 & 0xFFFFFFu;
      hi = __funnelshift_r(w0, w1, 24) & 0xFFFFFFu;
    }
  }
}

// 1024 + code_j (low half) and 1024 + code_{j+4} (high half) of a field.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(uint32_t f, int j) {
  if (BITS == 4) return ((f >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
  const uint32_t t = f >> (3 * j);
  return (t & 0x7u) | ((t << 4) & 0x70000u) | 0x64006400u;
}

template <int NT, int GROUP, int BITS, bool XSMEM>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
    k_wq_mma(const uint32_t* __restrict__ codes, const __half* __restrict__ scales,
             const uint8_t* __restrict__ zeros, int64_t N, int64_t K,
             const __half* __restrict__ x, int M, float* __restrict__ y) {
  extern __shared__ uint4 xs[];   // XSMEM: x [M][K/8] 16-byte chunks, chunk j of token t at j ^ (t & 7)
  // Partial sums of the first and last tile of each warp's range.
  __shared__ float part_smem[kMaxWarps][2][16 * 16];
  __shared__ int64_t part_tile[kMaxWarps][2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int upr = static_cast<int>(K / kUnit);          // units per row tile
  const int64_t tiles = (N + 15) / 16;
  const int64_t items = tiles * upr;
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * items / gridDim.x;
  const int64_t b1 = (static_cast<int64_t>(blockIdx.x) + 1) * items / gridDim.x;
  const int64_t i0 = b0 + (b1 - b0) * warp / nwarps;
  const int64_t i1 = b0 + (b1 - b0) * (warp + 1) / nwarps;
  const int64_t words_per_row = K * BITS / 32;
  const int64_t groups = GROUP ? K / GROUP : 1;
  constexpr int kUnitWords = BITS == 4 ? 8 : 6;          // code words per row and unit
  // Units of codes in flight per warp (fewer with 16 tokens: more registers
  // per unit).
  constexpr int kPrefetch = NT == 1 ? 8 : 5;

  if constexpr (XSMEM) {
    const int64_t cpr = K / 8;
    for (int64_t q = threadIdx.x; q < M * cpr; q += blockDim.x) {
      const int64_t t = q / cpr, j = q - t * cpr;
      xs[t * cpr + (j ^ (t & 7))] = __ldg(reinterpret_cast<const uint4*>(x) + q);
    }
  }
  if (lane == 0) {
    part_tile[warp][0] = -1;
    part_tile[warp][1] = -1;
  }
  __syncthreads();
  if (i0 >= i1) goto combine;
  {
    // The first code word this thread reads in a row: INT4 words 2c, 2c+1 of
    // a unit; INT3 bits [48c, 48c+48) of its 6 words.
    const int cw = BITS == 4 ? 2 * c : (3 * c) / 2;
    // Stream of units to load (kPrefetch ahead): tile and unit, and the two
    // rows' code pointers at that unit.  Advanced by pointer increments; a
    // new tile (every upr units) recomputes them.
    int64_t ptile = i0 / upr;
    int punit = static_cast<int>(i0 - ptile * upr);
    const uint32_t* pc0;
    const uint32_t* pc1;
    auto set_load_rows = [&]() {
      const int64_t l0 = min(ptile * 16 + g, N - 1), l1 = min(ptile * 16 + g + 8, N - 1);
      pc0 = codes + l0 * words_per_row + static_cast<int64_t>(punit) * kUnitWords + cw;
      pc1 = codes + l1 * words_per_row + static_cast<int64_t>(punit) * kUnitWords + cw;
    };
    set_load_rows();
    auto load_next = [&](UnitRow& r0, UnitRow& r1) {
      load_fields<BITS>(pc0, c, r0.lo, r0.hi);
      load_fields<BITS>(pc1, c, r1.lo, r1.hi);
      pc0 += kUnitWords;
      pc1 += kUnitWords;
      if (++punit == upr) {
        punit = 0;
        ++ptile;
        set_load_rows();
      }
    };
    const int n = static_cast<int>(i1 - i0);   // units of this warp
    UnitRow q0[kPrefetch], q1[kPrefetch];
#pragma unroll
    for (int p = 0; p < kPrefetch; ++p)
      if (p < n) load_next(q0[p], q1[p]);

    // The unit being computed: its tile, its index in the tile, and the
    // tile's group parameters and x rows.
    int64_t tile = i0 / upr;
    int unit = static_cast<int>(i0 - tile * upr);
    int tile_u0 = unit;   // first unit of the current tile inside this range
    const uint8_t* zr0;
    const uint8_t* zr1;
    const __half* sr0;
    const __half* sr1;
    auto set_rows = [&]() {
      const int64_t l0 = min(tile * 16 + g, N - 1), l1 = min(tile * 16 + g + 8, N - 1);
      zr0 = zeros + l0 * groups;
      zr1 = zeros + l1 * groups;
      sr0 = scales + l0 * groups;
      sr1 = scales + l1 * groups;
    };
    set_rows();
    // x of this thread's tokens (t * 8 + g): 16-byte chunks 2c + 8 unit and
    // the next, swizzled by (token & 7) = g in shared memory.
    const uint4* xrow[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int tok = t * 8 + g;
      if constexpr (XSMEM) xrow[t] = xs + static_cast<int64_t>(min(tok, M - 1)) * (K / 8);
      else xrow[t] = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(min(tok, M - 1)) * K);
    }

    float acc[NT][4], part[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] = part[t][e] = 0.f;
    float last_sf0 = 0.f, last_sf1 = 0.f;   // group scales of the last unit done

    // Close the current tile at unit `end`: scale the group the range leaves
    // open (per-row groups: always), then add the tile to y if this warp did
    // all of it, else park it in shared memory for the block's sum.
    auto finish_tile = [&](int end) {
      if (GROUP == 0 || (GROUP == 128 && (end & 1))) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          acc[t][0] = __fmaf_rn(last_sf0, part[t][0], acc[t][0]);
          acc[t][1] = __fmaf_rn(last_sf0, part[t][1], acc[t][1]);
          acc[t][2] = __fmaf_rn(last_sf1, part[t][2], acc[t][2]);
          acc[t][3] = __fmaf_rn(last_sf1, part[t][3], acc[t][3]);
        }
      }
      if (tile_u0 == 0 && end == upr) {
        const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
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
      } else {
        const int slot = tile == i0 / upr ? 0 : 1;   // the range's first or last tile
        float* ps = part_smem[warp][slot];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int m0 = t * 8 + 2 * c;
          ps[g * 16 + m0] = acc[t][0];
          ps[g * 16 + m0 + 1] = acc[t][1];
          ps[(g + 8) * 16 + m0] = acc[t][2];
          ps[(g + 8) * 16 + m0 + 1] = acc[t][3];
        }
        if (lane == 0) part_tile[warp][slot] = tile;
      }
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = part[t][e] = 0.f;
    };

    for (int base = 0; base < n; base += kPrefetch) {
#pragma unroll
      for (int p = 0; p < kPrefetch; ++p) {
        if (base + p >= n) break;
        if (unit == upr) {   // the previous unit ended a tile
          finish_tile(upr);
          ++tile;
          unit = 0;
          tile_u0 = 0;
          set_rows();
        }
        const UnitRow a0 = q0[p], a1 = q1[p];
        if (base + p + kPrefetch < n) load_next(q0[p], q1[p]);
        int grp = 0;
        if constexpr (GROUP == 128) grp = unit >> 1;
        if constexpr (GROUP == 64) grp = unit;
        // 1024 + zero in both halves (exact: fp16 bits 0x6400 + z), and the scale.
        const uint32_t z0 = 0x6400u + __ldg(zr0 + grp);
        const uint32_t z1 = 0x6400u + __ldg(zr1 + grp);
        const uint32_t zp0 = z0 | (z0 << 16), zp1 = z1 | (z1 << 16);
        const float sf0 = __half2float(__ldg(sr0 + grp));
        const float sf1 = __half2float(__ldg(sr1 + grp));
        uint32_t X[NT][8];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
          if (t * 8 + g < M) {
            const int chunk = unit * 8 + 2 * c;   // 16-byte chunk of x[tok][unit*64 + 16c]
            if constexpr (XSMEM) {
              v0 = xrow[t][chunk ^ g];
              v1 = xrow[t][(chunk + 1) ^ g];
            } else {
              v0 = __ldg(xrow[t] + chunk);
              v1 = __ldg(xrow[t] + chunk + 1);
            }
          }
          X[t][0] = v0.x; X[t][1] = v0.y; X[t][2] = v0.z; X[t][3] = v0.w;
          X[t][4] = v1.x; X[t][5] = v1.y; X[t][6] = v1.z; X[t][7] = v1.w;
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
            // x[16c + j], x[16c + j + 4]  and  x[16c + 8 + j], x[16c + 12 + j]
            const uint32_t bb0 = __byte_perm(X[t][j >> 1], X[t][(j >> 1) + 2], sel);
            const uint32_t bb1 = __byte_perm(X[t][4 + (j >> 1)], X[t][6 + (j >> 1)], sel);
            mma_16816(part[t], a, bb0, bb1);
          }
        }
        last_sf0 = sf0;
        last_sf1 = sf1;
        // End of a group: scale it into the row's sum (per-row groups are
        // scaled when their tile closes).
        if (GROUP == 64 || (GROUP == 128 && (unit & 1))) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            acc[t][0] = __fmaf_rn(sf0, part[t][0], acc[t][0]);
            acc[t][1] = __fmaf_rn(sf0, part[t][1], acc[t][1]);
            acc[t][2] = __fmaf_rn(sf1, part[t][2], acc[t][2]);
            acc[t][3] = __fmaf_rn(sf1, part[t][3], acc[t][3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) part[t][e] = 0.f;
          }
        }
        ++unit;
      }
    }
    finish_tile(unit);
  }
combine:
  __syncthreads();
  // The parked partial sums, in warp order (equal tile ids are consecutive);
  // thread e of the block owns element e of a tile (16 rows x 16 tokens).
  for (int e = threadIdx.x; e < 16 * 16; e += blockDim.x) {
    const int row = e >> 4, tok = e & 15;
    int64_t tl = -1;
    float sum = 0.f;
    for (int w = 0; w < nwarps; ++w) {
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int64_t t = part_tile[w][s2];
        if (t < 0) continue;
        if (t != tl) {
          if (tl >= 0 && tl * 16 + row < N && tok < M) atomicAdd(y + tok * N + tl * 16 + row, sum);
          tl = t;
          sum = 0.f;
        }
        sum = __fadd_rn(sum, part_smem[w][s2][e]);
      }
    }
    if (tl >= 0 && tl * 16 + row < N && tok < M) atomicAdd(y + tok * N + tl * 16 + row, sum);
  }
}

template <int NT, int BITS>
cudaError_t launch_wq(int group, const uint32_t* codes, const __half* scales,
                      const uint8_t* zeros, int64_t N, int64_t K, const __half* x, int M,
                      float* y, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(y, 0, sizeof(float) * static_cast<size_t>(M) * N, st);
  if (e != cudaSuccess) return e;
  // One block per SM, at most one per 16-row tile (every block's range is
  // then at least a tile long: at most two blocks add into an output).
  const int64_t tiles = (N + 15) / 16;
  const int64_t blocks = std::min<int64_t>(device_sm_count(), tiles);
  const int64_t xbytes = static_cast<int64_t>(M) * K * 2;
  const bool xsmem = xbytes <= kXSmemMax;
  const int smem = xsmem ? static_cast<int>(xbytes) : 0;
  auto go = [&](auto kern) -> cudaError_t {
    LaunchFacts lf;   // raises the kernel's dynamic shared memory limit once per device
    cudaError_t err = launch_facts(reinterpret_cast<const void*>(kern), kMaxWarps * 32,
                                   kXSmemMax, &lf);
    if (err != cudaSuccess) return err;
    kern<<<static_cast<unsigned>(blocks), kMaxWarps * 32, smem, st>>>(codes, scales, zeros, N, K,
                                                                      x, M, y);
    return cudaGetLastError();
  };
  if (xsmem) {
    if (group == 128) return go(k_wq_mma<NT, 128, BITS, true>);
    if (group == 64) return go(k_wq_mma<NT, 64, BITS, true>);
    return go(k_wq_mma<NT, 0, BITS, true>);
  }
  if (group == 128) return go(k_wq_mma<NT, 128, BITS, false>);
  if (group == 64) return go(k_wq_mma<NT, 64, BITS, false>);
  return go(k_wq_mma<NT, 0, BITS, false>);
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
