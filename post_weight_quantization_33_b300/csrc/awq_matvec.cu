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
// (code - zero) values built in registers, B holds 8 tokens of x.  At each
// group's end the fp32 sums are scaled by the group's fp16 scale (in fp32)
// and added to the row's accumulator.
//
// Units.  A warp step (a "unit") covers 16 rows x 128 channels when
// K % 128 == 0, else 16 rows x 64 channels, in halves of 64 channels; a half
// is four MMAs per 8 tokens.  In a half, each thread of a quad takes 16
// consecutive codes of its two rows (INT4: one 8-byte load per row; INT3:
// two 4-byte loads) and feeds them to the four MMAs: in MMA j, thread c
// supplies channels 16c+j, 16c+j+4, 16c+8+j and 16c+12+j in the k slots the
// fragment layout gives it (2c, 2c+1, 2c+8, 2c+9).  A group's dot product
// does not depend on the order of its channels, and the two halves of a unit
// never share an MMA, so 64-channel groups stay apart.
//
// (code - zero) in fp16, exactly.  A code masked into the low mantissa bits
// of 1024 (0x6400 | code) is 1024 + code; minus 1024 + zero (HSUB2) is
// code - zero.  A code masked in place at bit offset 4 is 1024 + 16 code; one
// HFMA2 with 1/16 and -(64 + zero) gives code - zero (the product and the sum
// are exact in fp16).  So the eight INT4 codes of a word cost one shift, four
// LOP3s and four HSUB2/HFMA2s; INT3 codes sit at offsets 0, 3, 6, 9 (factors
// 1, 1/8, 1/64, and a shift for the last).
//
// x.  When M x K fp16 fits in shared memory the block stages x once,
// permuted so that a thread's B fragments for the four MMAs of a half are two
// 16-byte loads (no byte permutes in the loop); for odd tokens the two
// 64-byte halves of the staged 128 bytes are swapped, so the quads of a warp
// (8 tokens) spread over all 32 banks.  When only half of it fits (and K is
// a multiple of 1024), the grid is cut in two halves of K, each block staging
// its half (k_wq_tma).  Otherwise x is read through L1 and its B fragments
// are formed by byte permutes.
//
// Work split.  One block of 16 warps per SM (8 for 16 tokens, or x read
// through L1).  The (row tile, unit) items, tile-major, are cut into equal
// contiguous ranges, one per block (each at least one row tile long), and a
// block's range into one contiguous range per warp.  A warp streams its units
// across row-tile boundaries: K % 128 == 0 through a TMA ring in shared
// memory (k_wq_tma below), else with the codes and group parameters of the
// next kPrefetch 64-channel units held in registers (k_wq_mma).  A row tile
// entirely inside one warp's range is added to y at once; the partial sums of
// the tiles at the two ends of a warp's range go to shared memory, and the
// block adds them up in warp order before adding them to y.  y is zeroed
// first and at most two blocks add into an output (two fp32 additions onto
// zero commute), so the result is deterministic.
#include <algorithm>
#include <type_traits>

#include "awq_bounds.cuh"
#include "awq_internal.h"
#include "awq_ptx.cuh"

namespace awq {
namespace {

constexpr int kHalf = 64;          // channels per half unit (four MMAs)
constexpr int kMaxWarps = 16;      // per block (one block per SM)
constexpr int kXSmemMax = 192 * 1024;
constexpr uint32_t kMagic = 0x64006400u;   // fp16 1024 in both halves

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

// Programmatic dependent launch: k_zero_y is launched behind the stream's
// previous kernel and the product behind k_zero_y, so both are resident early
// and start as soon as their predecessor ends (no launch gap between calls).
// k_zero_y waits for the previous kernel before it writes y (that kernel may
// still read it); the product waits for k_zero_y, and so for everything
// before it, before its first load (x, codes and parameters may come from
// the kernel before) and its first access to y.
__device__ __forceinline__ void wait_for_zeroed_y() { grid_dependency_wait(); }

// One fp32 addition into y[i] (y holds n = M x N values).
__device__ __forceinline__ void add_y(float* y, int64_t i, int64_t n, float v) {
  if (in_bounds(kSiteDecodeY, i, n)) atomicAdd(y + i, v);
}

__global__ void k_zero_y(float* __restrict__ y, int64_t n) {
  grid_dependents_launch();
  grid_dependency_wait();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    y[i] = 0.f;
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a),
                            *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a),
                            *reinterpret_cast<const __half2*>(&b),
                            *reinterpret_cast<const __half2*>(&c));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// fp16 pairs made from a row's zero point z (an integer in [0, 2^b - 1]):
// p = 1024 + z, and q1, q2 = -(1024/m + z) for the in-place factors m
// (INT4: 16; INT3: 8 and 64).  Each is exact: 1024/m + z stays inside one
// binade whose spacing is 1/m.
struct ZeroPairs {
  uint32_t p, q1, q2;
};

template <int BITS>
__device__ __forceinline__ ZeroPairs zero_pairs(uint32_t z) {
  ZeroPairs r;
  r.p = z * 0x00010001u + kMagic;                 // 1024 + z (spacing 1)
  if (BITS == 4) {
    r.q1 = z * 0x00100010u + 0xD400D400u;         // -(64 + z)  (spacing 1/16)
    r.q2 = 0;
  } else {
    r.q1 = z * 0x00080008u + 0xD800D800u;         // -(128 + z) (spacing 1/8)
    r.q2 = z * 0x00400040u + 0xCC00CC00u;         // -(16 + z)  (spacing 1/64)
  }
  return r;
}

// (code - zero) of codes j and j + 4 of a field of 8 codes, as an fp16 pair,
// for j = 0..3.  INT4: code i at bits 4i.  INT3: code i at bits 3i (bits
// above 24 are ignored).
// (f & mask) | magic in one LOP3: the mask is the instruction's immediate and
// `magic` (fp16 1024 in both halves) a register.  The kernels take magic as
// an argument so that it stays in a register instead of being folded into a
// second immediate (which would take a second LOP3).
template <uint32_t MASK>
__device__ __forceinline__ uint32_t mask_or(uint32_t f, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(f), "n"(MASK), "r"(magic));
  return d;
}

template <int BITS>
__device__ __forceinline__ void dequant_field(uint32_t f, const ZeroPairs& z, uint32_t magic,
                                              uint32_t (&d)[4]) {
  if (BITS == 4) {
    d[0] = hsub2_u32(mask_or<0x000F000Fu>(f, magic), z.p);
    d[1] = hfma2_u32(mask_or<0x00F000F0u>(f, magic), 0x2C002C00u, z.q1);   // x 1/16
    const uint32_t t = f >> 8;
    d[2] = hsub2_u32(mask_or<0x000F000Fu>(t, magic), z.p);
    d[3] = hfma2_u32(mask_or<0x00F000F0u>(t, magic), 0x2C002C00u, z.q1);
  } else {
    // Codes 0..3 stay at bits 0..11, codes 4..7 move to bits 16..27 (bits
    // 12..15 and 28..31 are left over and never masked in).
    const uint32_t w = (f & 0x00000FFFu) | ((f << 4) & 0xFFFFF000u);
    d[0] = hsub2_u32(mask_or<0x00070007u>(w, magic), z.p);
    d[1] = hfma2_u32(mask_or<0x00380038u>(w, magic), 0x30003000u, z.q1);   // x 1/8
    d[2] = hfma2_u32(mask_or<0x01C001C0u>(w, magic), 0x24002400u, z.q2);   // x 1/64
    d[3] = hsub2_u32(mask_or<0x00070007u>(w >> 9, magic), z.p);
  }
}

// Raw code words of one unit for the two rows of a thread, and the packed
// group parameters of the unit (one or two zeros and fp16 scales per row).
template <int H>
struct UnitWords {
  uint32_t r0[2 * H], r1[2 * H];
  uint32_t z0, z1, s0, s1;
};

// Warps per block: 16, or 8 with twice the registers each when 16 tokens
// are read through L1.
template <int NT, bool XPERM>
__host__ __device__ constexpr int block_warps() {
  return NT == 2 && !XPERM ? 8 : kMaxWarps;
}

template <int NT, int GROUP, int BITS, bool XPERM, int H>
__global__ void __launch_bounds__(block_warps<NT, XPERM>() * 32, 1)
    k_wq_mma(const uint32_t* __restrict__ codes, const __half* __restrict__ scales,
             const uint8_t* __restrict__ zeros, int64_t N, int64_t K,
             const __half* __restrict__ x, int M, float* __restrict__ y, uint32_t magic) {
  // XPERM: x permuted, 8 chunks of 16 bytes per token and half (see above).
  extern __shared__ uint4 xs[];
  // Partial sums of the first and last tile of each warp's range.
  __shared__ float part_smem[kMaxWarps][2][16 * 16];
  __shared__ int64_t part_tile[kMaxWarps][2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  constexpr int kUnitCh = kHalf * H;
  constexpr int kHalfWords = 2 * BITS;              // code words per row and half
  constexpr int kUnitWords = kHalfWords * H;
  constexpr int kGroupsPerUnit = GROUP == 64 ? H : 1;
  // Units in flight per warp: as many as the registers allow (16 tokens, x
  // read through L1, and two groups per unit each take more per unit; 16
  // tokens with x read through L1 run 8 warps with twice the registers).
  constexpr int kPrefetch =
      (H == 2 ? (NT == 1 ? (XPERM ? 4 : (BITS == 4 ? 3 : 2)) : (XPERM ? 3 : 5))
              : (NT == 1 ? (XPERM ? 6 : 5) : (XPERM ? 4 : 8))) -
      (GROUP == 64 ? 1 : 0);
  const int upr = static_cast<int>(K / kUnitCh);   // units per row tile
  const int hcs = static_cast<int>(K / kHalf);     // halves per row
  const int64_t tiles = (N + 15) / 16;
  const int64_t items = tiles * upr;
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * items / gridDim.x;
  const int64_t b1 = (static_cast<int64_t>(blockIdx.x) + 1) * items / gridDim.x;
  const int64_t i0 = b0 + (b1 - b0) * warp / nwarps;
  const int64_t i1 = b0 + (b1 - b0) * (warp + 1) / nwarps;
  const int64_t words_per_row = K * BITS / 32;
  const int64_t groups = GROUP ? K / GROUP : 1;
  wait_for_zeroed_y();

  if constexpr (XPERM) {
    // Item q: token t, half hc, quad slot cc (channels 64 hc + 16 cc .. + 15).
    // Chunk i of the slot holds the B words of MMAs 2i and 2i + 1:
    // {x[j], x[j+4]} and {x[8+j], x[12+j]} of the slot's 16 channels.
    const int per_tok = hcs * 4;
    for (int q = threadIdx.x; q < M * per_tok; q += blockDim.x) {
      const int t = q / per_tok, r = q - t * per_tok;
      const int hc = r >> 2, cc = r & 3;
      const int64_t xi = static_cast<int64_t>(t) * K + hc * kHalf + cc * 16;
      const uint4* src = reinterpret_cast<const uint4*>(x + xi);
      const bool xin = in_bounds(kSiteDecodeX, xi + 15, static_cast<int64_t>(M) * K);
      const uint4 v0 = xin ? __ldg(src) : make_uint4(0, 0, 0, 0);
      const uint4 v1 = xin ? __ldg(src + 1) : make_uint4(0, 0, 0, 0);
      const uint32_t X[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
        o[2 * j] = __byte_perm(X[j >> 1], X[(j >> 1) + 2], sel);
        o[2 * j + 1] = __byte_perm(X[4 + (j >> 1)], X[6 + (j >> 1)], sel);
      }
      const int odd4 = (t & 1) * 4;
      uint4* dst = xs + (static_cast<int64_t>(t) * hcs + hc) * 8;
      dst[cc ^ odd4] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[(4 + cc) ^ odd4] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
  if (lane == 0) {
    part_tile[warp][0] = -1;
    part_tile[warp][1] = -1;
  }
  __syncthreads();
  if (i0 >= i1) goto combine;
  {
    // The first code word of this thread in a half: INT4 words 2c, 2c+1;
    // INT3 bits [48c, 48c+48) of the half's 6 words (c odd: from bit 16 of
    // word (3c)/2).
    const int cw = BITS == 4 ? 2 * c : (3 * c) / 2;
    const bool odd = c & 1;
    // Stream of units to load (kPrefetch ahead): tile and unit, and the two
    // rows' code and group-parameter pointers at that unit.  Advanced by
    // pointer increments; a new tile (every upr units) recomputes them.
    int64_t ptile = i0 / upr;
    int punit = static_cast<int>(i0 - ptile * upr);
    const uint32_t* pc0;
    const uint32_t* pc1;
    const uint8_t* pz0 = nullptr;
    const uint8_t* pz1 = nullptr;
    const __half* ps0 = nullptr;
    const __half* ps1 = nullptr;
    auto set_load_rows = [&]() {
      const int64_t l0 = min(ptile * 16 + g, N - 1), l1 = min(ptile * 16 + g + 8, N - 1);
      pc0 = codes + l0 * words_per_row + static_cast<int64_t>(punit) * kUnitWords + cw;
      pc1 = codes + l1 * words_per_row + static_cast<int64_t>(punit) * kUnitWords + cw;
      if constexpr (GROUP != 0) {
        const int64_t gi = static_cast<int64_t>(punit) * kGroupsPerUnit;
        pz0 = zeros + l0 * groups + gi;
        pz1 = zeros + l1 * groups + gi;
        ps0 = scales + l0 * groups + gi;
        ps1 = scales + l1 * groups + gi;
      }
    };
    set_load_rows();
    auto load_next = [&](UnitWords<H>& u) {
      if (!in_bounds(kSiteDecodeCodes, (pc1 - codes) + (H - 1) * kHalfWords + 1,
                     N * words_per_row) ||
          (GROUP != 0 && !in_bounds(kSiteDecodeParams, (pz1 - zeros) + kGroupsPerUnit - 1,
                                    N * groups))) {
        u = UnitWords<H>{};
        return;
      }
#pragma unroll
      for (int h = 0; h < H; ++h) {
        if constexpr (BITS == 4) {
          const uint2 v0 = ld_stream_u64(pc0 + h * kHalfWords);
          const uint2 v1 = ld_stream_u64(pc1 + h * kHalfWords);
          u.r0[2 * h] = v0.x;
          u.r0[2 * h + 1] = v0.y;
          u.r1[2 * h] = v1.x;
          u.r1[2 * h + 1] = v1.y;
        } else {
          u.r0[2 * h] = ld_stream_u32(pc0 + h * kHalfWords);
          u.r0[2 * h + 1] = ld_stream_u32(pc0 + h * kHalfWords + 1);
          u.r1[2 * h] = ld_stream_u32(pc1 + h * kHalfWords);
          u.r1[2 * h + 1] = ld_stream_u32(pc1 + h * kHalfWords + 1);
        }
      }
      if constexpr (GROUP != 0) {
        if constexpr (kGroupsPerUnit == 2) {   // two groups: 2 zeros, 2 scales per row
          u.z0 = __ldg(reinterpret_cast<const unsigned short*>(pz0));
          u.z1 = __ldg(reinterpret_cast<const unsigned short*>(pz1));
          u.s0 = __ldg(reinterpret_cast<const unsigned int*>(ps0));
          u.s1 = __ldg(reinterpret_cast<const unsigned int*>(ps1));
        } else {
          u.z0 = __ldg(pz0);
          u.z1 = __ldg(pz1);
          u.s0 = __ldg(reinterpret_cast<const unsigned short*>(ps0));
          u.s1 = __ldg(reinterpret_cast<const unsigned short*>(ps1));
        }
        pz0 += kGroupsPerUnit;
        pz1 += kGroupsPerUnit;
        ps0 += kGroupsPerUnit;
        ps1 += kGroupsPerUnit;
      }
      pc0 += kUnitWords;
      pc1 += kUnitWords;
      if (++punit == upr) {
        punit = 0;
        ++ptile;
        set_load_rows();
      }
    };
    const int n = static_cast<int>(i1 - i0);   // units of this warp
    UnitWords<H> q[kPrefetch];
#pragma unroll
    for (int p = 0; p < kPrefetch; ++p)
      if (p < n) load_next(q[p]);

    // The unit being computed: its tile, its index in the tile, and (groups
    // of a whole row) the tile's group parameters.
    int64_t tile = i0 / upr;
    int unit = static_cast<int>(i0 - tile * upr);
    int tile_u0 = unit;   // first unit of the current tile inside this range
    ZeroPairs rz0{}, rz1{};
    float rsf0 = 0.f, rsf1 = 0.f;
    auto set_rows = [&]() {
      if constexpr (GROUP == 0) {
        const int64_t l0 = min(tile * 16 + g, N - 1), l1 = min(tile * 16 + g + 8, N - 1);
        rz0 = zero_pairs<BITS>(__ldg(zeros + l0));
        rz1 = zero_pairs<BITS>(__ldg(zeros + l1));
        rsf0 = __half2float(__ldg(scales + l0));
        rsf1 = __half2float(__ldg(scales + l1));
      }
    };
    set_rows();
    // x of this thread's tokens (t * 8 + g, tokens past M read token M - 1;
    // their output columns are never written).  XPERM: the two chunks of
    // half 0 (add 8 chunks per half); else 16-byte chunk 2c of half 0.
    const uint4* xa[NT];
    const uint4* xb[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int tok = min(t * 8 + g, M - 1);
      if constexpr (XPERM) {
        const int odd4 = (tok & 1) * 4;
        xa[t] = xs + static_cast<int64_t>(tok) * hcs * 8 + (c ^ odd4);
        xb[t] = xs + static_cast<int64_t>(tok) * hcs * 8 + ((4 + c) ^ odd4);
      } else {
        xa[t] = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(tok) * K) + 2 * c;
        xb[t] = xa[t] + 1;
      }
    }

    float acc[NT][4], part[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] = part[t][e] = 0.f;

    // Close the current tile at unit `end`: scale the sums of a whole-row
    // group, then add the tile to y if this warp did all of it, else park it
    // in shared memory for the block's sum.
    auto finish_tile = [&](int end) {
      if constexpr (GROUP == 0) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          acc[t][0] = __fmaf_rn(rsf0, part[t][0], acc[t][0]);
          acc[t][1] = __fmaf_rn(rsf0, part[t][1], acc[t][1]);
          acc[t][2] = __fmaf_rn(rsf1, part[t][2], acc[t][2]);
          acc[t][3] = __fmaf_rn(rsf1, part[t][3], acc[t][3]);
        }
      }
      if (tile_u0 == 0 && end == upr) {
        const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int m0 = t * 8 + 2 * c;
          if (r0 < N) {
            if (m0 < M) add_y(y, m0 * N + r0, static_cast<int64_t>(M) * N, acc[t][0]);
            if (m0 + 1 < M) add_y(y, (m0 + 1) * N + r0, static_cast<int64_t>(M) * N, acc[t][1]);
          }
          if (r1 < N) {
            if (m0 < M) add_y(y, m0 * N + r1, static_cast<int64_t>(M) * N, acc[t][2]);
            if (m0 + 1 < M) add_y(y, (m0 + 1) * N + r1, static_cast<int64_t>(M) * N, acc[t][3]);
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
        const UnitWords<H> u = q[p];
        if (base + p + kPrefetch < n) load_next(q[p]);
        // Group parameters of group k of the unit (whole-row groups: the tile's).
        ZeroPairs z0, z1;
        float sf0 = 0.f, sf1 = 0.f;
        auto group_params = [&](int k) {
          if constexpr (GROUP == 0) {
            z0 = rz0;
            z1 = rz1;
          } else {
            z0 = zero_pairs<BITS>((u.z0 >> (8 * k)) & 0xFFu);
            z1 = zero_pairs<BITS>((u.z1 >> (8 * k)) & 0xFFu);
            sf0 = half_bits_to_float(u.s0 >> (16 * k));
            sf1 = half_bits_to_float(u.s1 >> (16 * k));
          }
        };
        group_params(0);
        const int hc0 = unit * H;
#pragma unroll
        for (int h = 0; h < H; ++h) {
          if (kGroupsPerUnit == 2 && h == 1) group_params(1);
          // B fragments: MMA j takes words 2j and 2j + 1.
          uint32_t B[NT][8];
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int off = (hc0 + h) * 8;
            if constexpr (XPERM) {
              const uint4 v0 = xa[t][off], v1 = xb[t][off];
              B[t][0] = v0.x; B[t][1] = v0.y; B[t][2] = v0.z; B[t][3] = v0.w;
              B[t][4] = v1.x; B[t][5] = v1.y; B[t][6] = v1.z; B[t][7] = v1.w;
            } else {
              const uint4 v0 = __ldg(xa[t] + off), v1 = __ldg(xb[t] + off);
              const uint32_t X[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
                B[t][2 * j] = __byte_perm(X[j >> 1], X[(j >> 1) + 2], sel);
                B[t][2 * j + 1] = __byte_perm(X[4 + (j >> 1)], X[6 + (j >> 1)], sel);
              }
            }
          }
          // The fields (codes 0..7 and 8..15 of this thread's 16) of both rows.
          uint32_t lo0, hi0, lo1, hi1;
          if constexpr (BITS == 4) {
            lo0 = u.r0[2 * h];
            hi0 = u.r0[2 * h + 1];
            lo1 = u.r1[2 * h];
            hi1 = u.r1[2 * h + 1];
          } else {
            const int sl = odd ? 16 : 0, sh = odd ? 8 : 24;
            lo0 = __funnelshift_r(u.r0[2 * h], u.r0[2 * h + 1], sl);
            hi0 = __funnelshift_r(odd ? u.r0[2 * h + 1] : u.r0[2 * h], u.r0[2 * h + 1], sh);
            lo1 = __funnelshift_r(u.r1[2 * h], u.r1[2 * h + 1], sl);
            hi1 = __funnelshift_r(odd ? u.r1[2 * h + 1] : u.r1[2 * h], u.r1[2 * h + 1], sh);
          }
          uint32_t dl0[4], dl1[4], dh0[4], dh1[4];
          dequant_field<BITS>(lo0, z0, magic, dl0);   // row g,   slots 2c, 2c+1
          dequant_field<BITS>(lo1, z1, magic, dl1);   // row g+8
          dequant_field<BITS>(hi0, z0, magic, dh0);   // row g,   slots 2c+8, 2c+9
          dequant_field<BITS>(hi1, z1, magic, dh1);   // row g+8
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t a[4] = {dl0[j], dl1[j], dh0[j], dh1[j]};
#pragma unroll
            for (int t = 0; t < NT; ++t) mma_16816(part[t], a, B[t][2 * j], B[t][2 * j + 1]);
          }
          // End of a group: scale it into the row's sum (whole-row groups
          // are scaled when their tile closes).
          if (GROUP == 64 || (GROUP == 128 && h == H - 1)) {
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
          if (tl >= 0 && tl * 16 + row < N && tok < M) add_y(y, tok * N + tl * 16 + row, static_cast<int64_t>(M) * N, sum);
          tl = t;
          sum = 0.f;
        }
        sum = __fadd_rn(sum, part_smem[w][s2][e]);
      }
    }
    if (tl >= 0 && tl * 16 + row < N && tok < M) add_y(y, tok * N + tl * 16 + row, static_cast<int64_t>(M) * N, sum);
  }
}

// ---------------------------------------------------------------- TMA ring
// K % 128 == 0: each warp streams its units through its own ring of S
// shared-memory stages filled by TMA.  A stage is up to 4 units (512
// channels) of 16 rows in two 2-D boxes of 2 units each (INT4 16 x 128 bytes
// in the 128-byte swizzle, 16-byte chunk j of row r at j ^ (r & 7), so the
// quads' 8-byte reads of 8 rows hit distinct banks; INT3 16 x 96 bytes).
// Stages end at multiples of 4 units of a tile (and at the ends of a warp's
// range), so most are 4 whole units.  Lane 0 issues a stage's two copies and
// their transaction count on the stage's mbarrier; the warp waits on it
// (bounded), reads the codes with shared loads and feeds the MMAs, and lane
// 0 refills the slot with the stage S ahead once every lane has read it.
// When a row's group count is a multiple of 16, a stage also carries two
// small boxes of 16 rows with the group zeros (16 per row) and fp16 scales (8
// per row) whose blocks hold the stage's groups; otherwise the warp reads
// them at the stage's start (before its wait), with one vector load per row
// when the stage is whole and aligned.  The zero's fp16 pairs come from one
// byte permute (0x64 | z in both halves is 1024 + z) and fp16 subtractions.
// A group's first MMA starts from a zero accumulator.  y is zeroed by
// k_zero_y, which the product is launched behind (programmatic dependent
// launch, both chained to the stream's previous kernel: see
// wait_for_zeroed_y).
constexpr int kStageUnits = 4;        // 128-channel units per stage
constexpr int kBoxBytes = 2048;       // one box: 16 rows x (INT4 128, INT3 96) bytes
constexpr int kSlotBytes = 2 * kBoxBytes;
// Stages per warp: measured at one token on W 28672 x 8192 INT4, 2 stages
// (37.3 us) beat 3 (40.1 us; the shared memory they take is the L1 the
// per-stage group-parameter loads then miss) and 1 (39.4 us).
constexpr int kMaxStages = 2;
constexpr int kDecodeSmemMax = 227 * 1024;

template <int BITS>
__host__ __device__ constexpr int box_row_bytes() {
  return BITS == 4 ? 128 : 96;
}

// With the group parameters loaded by TMA as well, a stage also holds two
// boxes of 16 rows: 16 zeros (bytes) and 8 fp16 scales per row, placed so
// that they cover the stage's groups.
constexpr int kParamSlotBytes = 512;

// Dynamic shared memory of the TMA kernel, in this order: the rings
// (1024-byte aligned), the parameter boxes (with pt), x (staged), the parked
// partial sums, their tile ids, the mbarriers, the abort flag.
__host__ __device__ constexpr int64_t tma_smem_bytes(int nwarps, int S, int64_t xbytes, int NT,
                                                     bool pt) {
  return 1024 + static_cast<int64_t>(nwarps) * S * (kSlotBytes + (pt ? kParamSlotBytes : 0)) +
         xbytes +
         static_cast<int64_t>(nwarps) * 2 * 16 * 8 * NT * 4 + nwarps * 2 * 8 +
         static_cast<int64_t>(nwarps) * S * 8 + 16;
}

// D = A B with a zero accumulator input.
__device__ __forceinline__ void mma_16816_first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                uint32_t b1) {
  const float z = 0.f;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

// The zero's fp16 pairs from p = 1024 + z (both halves): q1, q2 by exact fp16
// subtractions (960 - p = -(64 + z); 896 - p = -(128 + z); 1008 - p = -(16 + z)).
template <int BITS>
__device__ __forceinline__ ZeroPairs zero_pairs_from_p(uint32_t p) {
  ZeroPairs r;
  r.p = p;
  if (BITS == 4) {
    r.q1 = hsub2_u32(0x63806380u, p);   // 960
    r.q2 = 0;
  } else {
    r.q1 = hsub2_u32(0x63006300u, p);   // 896
    r.q2 = hsub2_u32(0x63E063E0u, p);   // 1008
  }
  return r;
}

// 1024 + (byte b of w) in both fp16 halves: bytes {w.b, 0x64, w.b, 0x64}.
__device__ __forceinline__ uint32_t magic_pair_of_byte(uint32_t w, int b) {
  return __byte_perm(w, 0x64646464u, static_cast<uint32_t>(b | 0x40 | (b << 8) | 0x4000));
}

// Group parameters of one stage for rows g and g + 8: GS = 4 (groups of 128)
// or 8 (groups of 64) zeros (bytes) and fp16 scales per row.
template <int GS>
struct StageParams {
  uint32_t z0[GS / 4], z1[GS / 4];
  uint32_t s0[GS / 2], s1[GS / 2];
};

// Warps per block of the TMA kernel: 16, or 8 with twice the registers each
// for 16 tokens or x read through L1.
template <int NT, bool XPERM>
__host__ __device__ constexpr int tma_warps() {
  return NT == 2 || !XPERM ? 8 : kMaxWarps;
}

template <int NT, int GROUP, int BITS, bool XPERM, bool PT, bool SPLIT>
__global__ void __launch_bounds__(tma_warps<NT, XPERM>() * 32, 1)
    k_wq_tma(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_z,
             const __grid_constant__ CUtensorMap tmap_s, const __half* __restrict__ scales,
             const uint8_t* __restrict__ zeros, int64_t N, int64_t K,
             const __half* __restrict__ x, int M, float* __restrict__ y, int S, int vec,
             uint32_t magic) {
  extern __shared__ uint8_t dsmem[];
  const uint32_t raw_base = smem_u32(dsmem);
  uint8_t* const sm = dsmem + (((raw_base + 1023u) & ~1023u) - raw_base);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  // The box row that MMA row g takes (row g + 8 takes gr + 8).  INT4 boxes
  // are 128-byte swizzled (16-byte chunk j of row r stored at j ^ (r & 7)),
  // so the 8-byte code loads of lanes 0-15 (g = 0..3) cover all 32 banks
  // when they read rows 0, 2, 4, 6, and only 16 of them (two wavefronts per
  // half-warp) when they read rows 0..3.  INT3 rows (96 bytes, unswizzled)
  // keep g.
  const int gr = BITS == 4 ? ((g & 3) << 1) | (g >> 2) : g;
  constexpr int kRowBytes = box_row_bytes<BITS>();
  constexpr int kUnitBytes = 16 * BITS;               // bytes of a row per 128-channel unit
  constexpr int kTok = 8 * NT;
  constexpr int kGPU = GROUP == 64 ? 2 : 1;           // groups per unit
  constexpr int GS = kStageUnits * kGPU;              // groups per stage
  // SPLIT: block b of the grid's two equal parts takes the part's channels
  // [part K/2, (part + 1) K/2), over whole row tiles, so each output gets
  // one sum per part.
  constexpr int kp = SPLIT ? 2 : 1;
  const int bpp = static_cast<int>(gridDim.x) / kp;
  const int part = SPLIT ? static_cast<int>(blockIdx.x) / bpp : 0;
  const int64_t bb = static_cast<int64_t>(blockIdx.x) - static_cast<int64_t>(part) * bpp;
  const int64_t kpart = K / kp;
  const int upr = static_cast<int>(kpart / 128);     // units per row of the part
  const int ubase = part * upr;                      // the part's first unit of a row
  const int hcs = static_cast<int>(kpart / kHalf);
  const int64_t tiles = (N + 15) / 16;
  const int64_t items = tiles * upr;
  const int64_t b0 = SPLIT ? bb * tiles / bpp * upr : bb * items / bpp;
  const int64_t b1 = SPLIT ? (bb + 1) * tiles / bpp * upr : (bb + 1) * items / bpp;
  const int64_t i0 = b0 + (b1 - b0) * warp / nwarps;
  const int64_t i1 = b0 + (b1 - b0) * (warp + 1) / nwarps;
  const int64_t groups = GROUP ? K / GROUP : 1;

  uint8_t* const ring = sm;
  uint8_t* const pring = ring + static_cast<int64_t>(nwarps) * S * kSlotBytes;   // PT
  uint4* const xs =
      reinterpret_cast<uint4*>(pring + (PT ? static_cast<int64_t>(nwarps) * S * kParamSlotBytes : 0));
  float* const part_all =
      reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xs) + (XPERM ? int64_t(M) * kpart * 2 : 0));
  int64_t* const part_tile = reinterpret_cast<int64_t*>(part_all + nwarps * 2 * 16 * kTok);
  uint64_t* const bars = reinterpret_cast<uint64_t*>(part_tile + nwarps * 2);
  int* const abort_flag = reinterpret_cast<int*>(bars + nwarps * S);

  const uint32_t bar_w = smem_u32(bars + warp * S);
  const uint32_t ring_w = smem_u32(ring) + static_cast<uint32_t>(warp * S * kSlotBytes);
  const uint32_t pring_w = smem_u32(pring) + static_cast<uint32_t>(warp * S * kParamSlotBytes);
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(bar_w + 8 * s, 1);
    part_tile[2 * warp] = -1;
    part_tile[2 * warp + 1] = -1;
  }
  if (threadIdx.x == 0) *abort_flag = 0;
  fence_barrier_init();
  __syncwarp();

  // Units of the stage that starts at `unit` with `left` units of the range
  // to go: to the next multiple of 4, the tile's end or the range's end.
  auto stage_units = [&](int unit, int left) {
    return min(min(kStageUnits - (unit & (kStageUnits - 1)), upr - unit), left);
  };
  // Producer cursor (every lane keeps it; lane 0 issues the copies).
  int ptile = static_cast<int>(i0 / upr);
  int punit = static_cast<int>(i0 - ptile * upr);
  int pleft = static_cast<int>(i1 - i0);
  int issued = 0;
  auto produce = [&](int slot) {
    if (lane == 0) {
      const uint32_t bar = bar_w + 8 * slot;
      const uint32_t dst = ring_w + slot * kSlotBytes;
      const int xw = (ubase + punit) * (kUnitBytes / 4), yr = static_cast<int>(ptile * 16);
      mbar_arrive_expect_tx(bar, 2 * 16 * kRowBytes + (PT ? kParamSlotBytes : 0));
      tma_load_2d(dst, &tmap, bar, xw, yr);
      tma_load_2d(dst + kBoxBytes, &tmap, bar, xw + 2 * kUnitBytes / 4, yr);
      if constexpr (PT) {
        // The 16 zeros and 8 scales per row whose blocks hold the stage's
        // groups (a stage never crosses a multiple of 4 units).
        const int gz = (ubase + punit) * kGPU;
        const uint32_t pdst = pring_w + slot * kParamSlotBytes;
        tma_load_2d(pdst, &tmap_z, bar, gz & ~15, yr);
        tma_load_2d(pdst + kParamSlotBytes / 2, &tmap_s, bar, gz & ~7, yr);
      }
    }
    const int nu = stage_units(punit, pleft);
    punit += nu;
    pleft -= nu;
    if (punit == upr) {
      punit = 0;
      ++ptile;
    }
    ++issued;
  };
  wait_for_zeroed_y();
  // The first S stages go out before x is staged.
  for (int s = 0; s < S && pleft > 0; ++s) produce(s);

  if constexpr (XPERM) {
    // Staged x: for token t and half hc, 8 chunks of 16 bytes; chunk i*4 + cc
    // (stored at (i*4 + cc) ^ ((t & 1) * 4)) holds the B words of MMAs 2i and
    // 2i + 1 of quad slot cc: {x[j], x[j+4]} and {x[8+j], x[12+j]} of the
    // slot's 16 channels 64 hc + 16 cc + (0..15).  One chunk per thread,
    // consecutive threads writing consecutive chunks.
    //
    // In the 9-16 token and K-split kernels the loads of a batch of 8 chunks
    // per thread are all issued before the first is used: at 16 tokens with
    // the K split a thread stages 32 chunks, and staged one at a time, each
    // waiting for its own loads, they made the split slower than reading x
    // through L1.  The 5-8 token split kernels (5-7 chunks per thread at 5-7
    // tokens) then take a batch of 4; the rest go one at a time.  (The
    // one-token kernel stages 2 chunks per thread; compiled into it, the
    // batch loop cost INT3 1.2 us though it never ran.)
    const int per_tok = hcs * 8;
    const int nchunks = M * per_tok;
    const int nthreads = static_cast<int>(blockDim.x);
    auto chunk_src = [&](int q, int& i) -> const uint4* {
      const int t = q / per_tok, r = q - t * per_tok;
      const int hc = r >> 3, pos = r & 7;
      const int within = pos ^ ((t & 1) * 4);
      i = within >> 2;
      const int cc = within & 3;
      const int64_t xi = static_cast<int64_t>(t) * K + part * kpart + hc * kHalf + cc * 16;
      return in_bounds(kSiteDecodeX, xi + 15, static_cast<int64_t>(M) * K)
                 ? reinterpret_cast<const uint4*>(x + xi)
                 : nullptr;
    };
    auto store_chunk = [&](int q, int i, const uint4& v0, const uint4& v1) {
      const uint32_t a0 = i ? v0.y : v0.x, a2 = i ? v0.w : v0.z;
      const uint32_t c0 = i ? v1.y : v1.x, c2 = i ? v1.w : v1.z;
      xs[q] = make_uint4(__byte_perm(a0, a2, 0x5410u), __byte_perm(c0, c2, 0x5410u),
                         __byte_perm(a0, a2, 0x7632u), __byte_perm(c0, c2, 0x7632u));
    };
    int q = threadIdx.x;
    auto stage_batch = [&](auto nb) {
      constexpr int NB = decltype(nb)::value;
      uint4 v0[NB], v1[NB];
      int sel[NB];
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const uint4* src = chunk_src(q + u * nthreads, sel[u]);
        v0[u] = src ? __ldg(src) : make_uint4(0, 0, 0, 0);
        v1[u] = src ? __ldg(src + 1) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < NB; ++u) store_chunk(q + u * nthreads, sel[u], v0[u], v1[u]);
      q += NB * nthreads;
    };
    if constexpr (NT == 2 || SPLIT) {
      while (q + 7 * nthreads < nchunks) stage_batch(std::integral_constant<int, 8>{});
      if constexpr (NT == 1) {
        if (q + 3 * nthreads < nchunks) stage_batch(std::integral_constant<int, 4>{});
      }
    }
    for (; q < nchunks; q += nthreads) {
      int i;
      const uint4* src = chunk_src(q, i);
      const uint4 v0 = src ? __ldg(src) : make_uint4(0, 0, 0, 0);
      const uint4 v1 = src ? __ldg(src + 1) : make_uint4(0, 0, 0, 0);
      store_chunk(q, i, v0, v1);
    }
  }
  __syncthreads();
  bool failed = false;
  if (i0 < i1) {
    // Group parameters: row pointers of one tile (cached) and the loads of a
    // stage.
    int prow_tile = -1;
    const uint8_t* zr0 = zeros;
    const uint8_t* zr1 = zeros;
    const __half* sr0 = scales;
    const __half* sr1 = scales;
    auto load_params = [&](StageParams<GS>& p, int T, int U, int nu) {
      if constexpr (GROUP != 0) {
        if (T != prow_tile) {
          prow_tile = T;
          const int64_t l0 = min(static_cast<int64_t>(T) * 16 + gr, N - 1);
          const int64_t l1 = min(static_cast<int64_t>(T) * 16 + gr + 8, N - 1);
          zr0 = zeros + l0 * groups;
          zr1 = zeros + l1 * groups;
          sr0 = scales + l0 * groups;
          sr1 = scales + l1 * groups;
        }
        const int64_t gi = static_cast<int64_t>(ubase + U) * kGPU;
        if (!in_bounds(kSiteDecodeParams,
                       min(static_cast<int64_t>(T) * 16 + gr + 8, N - 1) * groups + gi +
                           static_cast<int64_t>(nu == kStageUnits && vec ? GS : nu * kGPU) - 1,
                       N * groups))
          return;
        if (nu == kStageUnits && vec) {   // aligned: one load per row and array
          if constexpr (GS == 4) {
            p.z0[0] = __ldg(reinterpret_cast<const unsigned int*>(zr0 + gi));
            p.z1[0] = __ldg(reinterpret_cast<const unsigned int*>(zr1 + gi));
            const uint2 a = __ldg(reinterpret_cast<const uint2*>(sr0 + gi));
            const uint2 b = __ldg(reinterpret_cast<const uint2*>(sr1 + gi));
            p.s0[0] = a.x; p.s0[1] = a.y; p.s1[0] = b.x; p.s1[1] = b.y;
          } else {
            const uint2 za = __ldg(reinterpret_cast<const uint2*>(zr0 + gi));
            const uint2 zb = __ldg(reinterpret_cast<const uint2*>(zr1 + gi));
            p.z0[0] = za.x; p.z0[1] = za.y; p.z1[0] = zb.x; p.z1[1] = zb.y;
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(sr0 + gi));
            const uint4 b = __ldg(reinterpret_cast<const uint4*>(sr1 + gi));
            p.s0[0] = a.x; p.s0[1] = a.y; p.s0[2] = a.z; p.s0[3] = a.w;
            p.s1[0] = b.x; p.s1[1] = b.y; p.s1[2] = b.z; p.s1[3] = b.w;
          }
        } else {   // element by element (groups past the stage repeat its first)
          const int ng = nu * kGPU;
#pragma unroll
          for (int k = 0; k < GS / 4; ++k) p.z0[k] = p.z1[k] = 0;
#pragma unroll
          for (int k = 0; k < GS / 2; ++k) p.s0[k] = p.s1[k] = 0;
#pragma unroll
          for (int k = 0; k < GS; ++k) {
            const int kk = k < ng ? k : 0;
            p.z0[k >> 2] |= static_cast<uint32_t>(__ldg(zr0 + gi + kk)) << (8 * (k & 3));
            p.z1[k >> 2] |= static_cast<uint32_t>(__ldg(zr1 + gi + kk)) << (8 * (k & 3));
            p.s0[k >> 1] |= static_cast<uint32_t>(__half_as_ushort(__ldg(sr0 + gi + kk)))
                            << (16 * (k & 1));
            p.s1[k >> 1] |= static_cast<uint32_t>(__half_as_ushort(__ldg(sr1 + gi + kk)))
                            << (16 * (k & 1));
          }
        }
      } else {
        (void)p; (void)T; (void)U; (void)nu;
      }
    };

    // The stage being computed, and (whole-row groups) the tile's parameters.
    int tile = static_cast<int>(i0 / upr);
    int unit = static_cast<int>(i0 - static_cast<int64_t>(tile) * upr);
    int tile_u0 = unit;
    int left = static_cast<int>(i1 - i0);
    ZeroPairs rz0{}, rz1{};
    float rsf0 = 0.f, rsf1 = 0.f;
    auto set_rows = [&]() {
      if constexpr (GROUP == 0) {
        const int64_t l0 = min(static_cast<int64_t>(tile) * 16 + gr, N - 1);
        const int64_t l1 = min(static_cast<int64_t>(tile) * 16 + gr + 8, N - 1);
        rz0 = zero_pairs_from_p<BITS>(magic_pair_of_byte(__ldg(zeros + l0), 0));
        rz1 = zero_pairs_from_p<BITS>(magic_pair_of_byte(__ldg(zeros + l1), 0));
        rsf0 = __half2float(__ldg(scales + l0));
        rsf1 = __half2float(__ldg(scales + l1));
      }
    };
    set_rows();
    const uint4* xa[NT];
    const uint4* xb[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int tok = min(t * 8 + g, M - 1);
      if constexpr (XPERM) {
        const int odd4 = (tok & 1) * 4;
        xa[t] = xs + static_cast<int64_t>(tok) * hcs * 8 + (c ^ odd4);
        xb[t] = xs + static_cast<int64_t>(tok) * hcs * 8 + ((4 + c) ^ odd4);
      } else {
        xa[t] = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(tok) * K + part * kpart) +
                2 * c;
        xb[t] = xa[t] + 1;
      }
    }
    // Byte offsets of this thread's code words in a box, for row gr (row
    // gr + 8 is 8 rows further), per (unit of the box, half): INT4, its 8
    // bytes in the swizzled layout; INT3, the first of its two words.
    uint32_t coff[4];
#pragma unroll
    for (int uh = 0; uh < 4; ++uh) {
      if constexpr (BITS == 4) {
        const uint32_t chunk = ((static_cast<uint32_t>(uh) << 1) | (c >> 1)) ^ gr;
        coff[uh] = gr * kRowBytes + chunk * 16 + (c & 1) * 8;
      } else {
        coff[uh] = gr * kRowBytes + (uh >> 1) * kUnitBytes + (uh & 1) * 24 + 4 * ((3 * c) / 2);
      }
    }
    const bool odd = c & 1;

    float acc[NT][4], part[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] = part[t][e] = 0.f;

    auto finish_tile = [&](int end) {
      if constexpr (GROUP == 0) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          acc[t][0] = __fmaf_rn(rsf0, part[t][0], acc[t][0]);
          acc[t][1] = __fmaf_rn(rsf0, part[t][1], acc[t][1]);
          acc[t][2] = __fmaf_rn(rsf1, part[t][2], acc[t][2]);
          acc[t][3] = __fmaf_rn(rsf1, part[t][3], acc[t][3]);
        }
      }
      if (tile_u0 == 0 && end == upr) {
        const int64_t r0 = static_cast<int64_t>(tile) * 16 + gr, r1 = r0 + 8;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int m0 = t * 8 + 2 * c;
          if (r0 < N) {
            if (m0 < M) add_y(y, m0 * N + r0, static_cast<int64_t>(M) * N, acc[t][0]);
            if (m0 + 1 < M) add_y(y, (m0 + 1) * N + r0, static_cast<int64_t>(M) * N, acc[t][1]);
          }
          if (r1 < N) {
            if (m0 < M) add_y(y, m0 * N + r1, static_cast<int64_t>(M) * N, acc[t][2]);
            if (m0 + 1 < M) add_y(y, (m0 + 1) * N + r1, static_cast<int64_t>(M) * N, acc[t][3]);
          }
        }
      } else {
        const int slot = tile == i0 / upr ? 0 : 1;   // the range's first or last tile
        float* ps = part_all + (warp * 2 + slot) * 16 * kTok;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int m0 = t * 8 + 2 * c;
          ps[gr * kTok + m0] = acc[t][0];
          ps[gr * kTok + m0 + 1] = acc[t][1];
          ps[(gr + 8) * kTok + m0] = acc[t][2];
          ps[(gr + 8) * kTok + m0 + 1] = acc[t][3];
        }
        if (lane == 0) part_tile[2 * warp + slot] = tile;
      }
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = part[t][e] = 0.f;
    };

    // One stage from slot address sl: FULL (4 units, compiled without
    // per-unit guards) or the first nu units.
    auto run_stage = [&](auto full_tag, uint32_t sl, const StageParams<GS>& pc, int nu) {
      constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
      for (int uu = 0; uu < kStageUnits; ++uu) {
        if (!FULL && uu >= nu) break;
        ZeroPairs z0, z1;
        float sf0 = 0.f, sf1 = 0.f;
        auto group_params = [&](int k) {   // group k of the stage
          if constexpr (GROUP == 0) {
            z0 = rz0;
            z1 = rz1;
          } else {
            z0 = zero_pairs_from_p<BITS>(magic_pair_of_byte(pc.z0[k >> 2], k & 3));
            z1 = zero_pairs_from_p<BITS>(magic_pair_of_byte(pc.z1[k >> 2], k & 3));
            sf0 = half_bits_to_float(pc.s0[k >> 1] >> (16 * (k & 1)));
            sf1 = half_bits_to_float(pc.s1[k >> 1] >> (16 * (k & 1)));
          }
        };
        group_params(uu * kGPU);
        const int hc0 = (unit + uu) * 2;
        const uint32_t box = sl + (uu >> 1) * kBoxBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (kGPU == 2 && h == 1) group_params(uu * 2 + 1);
          uint32_t B[NT][8];
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int off = (hc0 + h) * 8;
            if constexpr (XPERM) {
              const uint4 v0 = xa[t][off], v1 = xb[t][off];
              B[t][0] = v0.x; B[t][1] = v0.y; B[t][2] = v0.z; B[t][3] = v0.w;
              B[t][4] = v1.x; B[t][5] = v1.y; B[t][6] = v1.z; B[t][7] = v1.w;
            } else {
              const uint4 v0 = __ldg(xa[t] + off), v1 = __ldg(xb[t] + off);
              const uint32_t X[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
                B[t][2 * j] = __byte_perm(X[j >> 1], X[(j >> 1) + 2], sel);
                B[t][2 * j + 1] = __byte_perm(X[4 + (j >> 1)], X[6 + (j >> 1)], sel);
              }
            }
          }
          uint32_t lo0, hi0, lo1, hi1;
          const uint32_t a0 = box + coff[(uu & 1) * 2 + h];
          if constexpr (BITS == 4) {
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(lo0), "=r"(hi0) : "r"(a0));
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(lo1), "=r"(hi1)
                         : "r"(a0 + 8 * kRowBytes));
          } else {
            uint32_t w0, w1, v0, v1;
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(a0));
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w1) : "r"(a0 + 4));
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v0) : "r"(a0 + 8 * kRowBytes));
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v1) : "r"(a0 + 8 * kRowBytes + 4));
            const int sl16 = odd ? 16 : 0, sh = odd ? 8 : 24;
            lo0 = __funnelshift_r(w0, w1, sl16);
            hi0 = __funnelshift_r(odd ? w1 : w0, w1, sh);
            lo1 = __funnelshift_r(v0, v1, sl16);
            hi1 = __funnelshift_r(odd ? v1 : v0, v1, sh);
          }
          uint32_t dl0[4], dl1[4], dh0[4], dh1[4];
          dequant_field<BITS>(lo0, z0, magic, dl0);
          dequant_field<BITS>(lo1, z1, magic, dl1);
          dequant_field<BITS>(hi0, z0, magic, dh0);
          dequant_field<BITS>(hi1, z1, magic, dh1);
          // A group's first MMA starts from zero (whole-row groups keep
          // their sum until the tile closes).
          constexpr bool kFresh = GROUP != 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t a[4] = {dl0[j], dl1[j], dh0[j], dh1[j]};
            const bool first = kFresh && j == 0 && (GROUP == 64 || h == 0);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (first) mma_16816_first(part[t], a, B[t][2 * j], B[t][2 * j + 1]);
              else mma_16816(part[t], a, B[t][2 * j], B[t][2 * j + 1]);
            }
          }
          if (GROUP == 64 || (GROUP == 128 && h == 1)) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              acc[t][0] = __fmaf_rn(sf0, part[t][0], acc[t][0]);
              acc[t][1] = __fmaf_rn(sf0, part[t][1], acc[t][1]);
              acc[t][2] = __fmaf_rn(sf1, part[t][2], acc[t][2]);
              acc[t][3] = __fmaf_rn(sf1, part[t][3], acc[t][3]);
            }
          }
        }
      }
    };

    // PT: the stage's group parameters from its parameter boxes (rows gr and
    // gr + 8; box rows of 16 bytes: zeros of groups (gz & ~15) + 0..15, scales
    // of groups (gz & ~7) + 0..7).
    auto smem_params = [&](StageParams<GS>& p, int slot, int U, int n) {
      if constexpr (PT && GROUP != 0) {
        const uint32_t pz = pring_w + slot * kParamSlotBytes, ps = pz + kParamSlotBytes / 2;
        const int gz = (ubase + U) * kGPU, bz = gz & 15, bs = gz & 7;
        const uint32_t rz0 = pz + gr * 16, rz1 = pz + (gr + 8) * 16;
        const uint32_t rs0 = ps + gr * 16, rs1 = ps + (gr + 8) * 16;
        if (n == kStageUnits) {
          if constexpr (GS == 4) {
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(p.z0[0]) : "r"(rz0 + bz));
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(p.z1[0]) : "r"(rz1 + bz));
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(p.s0[0]), "=r"(p.s0[1]) : "r"(rs0 + 2 * bs));
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(p.s1[0]), "=r"(p.s1[1]) : "r"(rs1 + 2 * bs));
          } else {
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(p.z0[0]), "=r"(p.z0[1]) : "r"(rz0 + bz));
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(p.z1[0]), "=r"(p.z1[1]) : "r"(rz1 + bz));
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(p.s0[0]), "=r"(p.s0[1]), "=r"(p.s0[2]), "=r"(p.s0[3]) : "r"(rs0));
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(p.s1[0]), "=r"(p.s1[1]), "=r"(p.s1[2]), "=r"(p.s1[3]) : "r"(rs1));
          }
        } else {   // element by element (groups past the stage repeat its first)
          const int ng = n * kGPU;
#pragma unroll
          for (int k = 0; k < GS / 4; ++k) p.z0[k] = p.z1[k] = 0;
#pragma unroll
          for (int k = 0; k < GS / 2; ++k) p.s0[k] = p.s1[k] = 0;
#pragma unroll
          for (int k = 0; k < GS; ++k) {
            const int kk = k < ng ? k : 0;
            uint32_t a, b, cs, d;
            asm volatile("ld.shared.u8 %0, [%1];" : "=r"(a) : "r"(rz0 + bz + kk));
            asm volatile("ld.shared.u8 %0, [%1];" : "=r"(b) : "r"(rz1 + bz + kk));
            asm volatile("ld.shared.u16 %0, [%1];" : "=r"(cs) : "r"(rs0 + 2 * (bs + kk)));
            asm volatile("ld.shared.u16 %0, [%1];" : "=r"(d) : "r"(rs1 + 2 * (bs + kk)));
            p.z0[k >> 2] |= a << (8 * (k & 3));
            p.z1[k >> 2] |= b << (8 * (k & 3));
            p.s0[k >> 1] |= cs << (16 * (k & 1));
            p.s1[k >> 1] |= d << (16 * (k & 1));
          }
        }
      } else {
        (void)p; (void)slot; (void)U; (void)n;
      }
    };
    StageParams<GS> pcur{};
    int nu = stage_units(unit, left);
    int slot = 0;
    uint32_t phase = 0;
    int consumed = 0;
    while (true) {
      // The next stage's position.
      int nunit = unit + nu;
      const int nleft = left - nu;
      int ntile = tile;
      if (nunit == upr) {
        nunit = 0;
        ++ntile;
      }
      const int nnu = nleft > 0 ? stage_units(nunit, nleft) : 0;
      if constexpr (!PT) load_params(pcur, tile, unit, nu);
      if (!mbar_wait_bounded(bar_w + 8 * slot, phase, abort_flag, nullptr, 0)) {
        failed = true;
        break;
      }
      if constexpr (PT) smem_params(pcur, slot, unit, nu);
      const uint32_t sl = ring_w + slot * kSlotBytes;
      if (nu == kStageUnits) run_stage(std::true_type{}, sl, pcur, nu);
      else run_stage(std::false_type{}, sl, pcur, nu);
      // Every lane has read the slot (its loads fed the MMAs above): refill it.
      __syncwarp();
      ++consumed;
      if (pleft > 0) produce(slot);
      if (++slot == S) {
        slot = 0;
        phase ^= 1;
      }
      if (nleft == 0) {
        finish_tile(unit + nu);
        break;
      }
      if (ntile != tile) {
        finish_tile(upr);
        tile = ntile;
        tile_u0 = 0;
        set_rows();
      }
      unit = nunit;
      left = nleft;
      nu = nnu;
    }
    if (failed) {
      // Let the copies still in flight land before the block can exit.
      for (int k = consumed; k < issued; ++k) {
        mbar_wait_bounded(bar_w + 8 * slot, phase, nullptr, nullptr, 0, kDrainLimitNs);
        if (++slot == S) {
          slot = 0;
          phase ^= 1;
        }
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 16 * kTok; e += blockDim.x) {
    const int row = e / kTok, tok = e - row * kTok;
    int64_t tl = -1;
    float sum = 0.f;
    for (int w = 0; w < nwarps; ++w) {
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int64_t t = part_tile[2 * w + s2];
        if (t < 0) continue;
        if (t != tl) {
          if (tl >= 0 && tl * 16 + row < N && tok < M) add_y(y, tok * N + tl * 16 + row, static_cast<int64_t>(M) * N, sum);
          tl = t;
          sum = 0.f;
        }
        sum = __fadd_rn(sum, part_all[(w * 2 + s2) * 16 * kTok + e]);
      }
    }
    if (tl >= 0 && tl * 16 + row < N && tok < M) add_y(y, tok * N + tl * 16 + row, static_cast<int64_t>(M) * N, sum);
  }
  if (*abort_flag) {
    // A wait expired: every output of the block's rows reads NaN.
    __syncthreads();
    const int64_t r0 = (b0 / upr) * 16, r1 = min(N, ((b1 + upr - 1) / upr) * 16);
    for (int64_t q = threadIdx.x; q < (r1 - r0) * M; q += blockDim.x) {
      const int64_t m = q / (r1 - r0), r = r0 + (q - m * (r1 - r0));
      y[m * N + r] = __int_as_float(0x7FC00000);
    }
  }
}

template <int NT, int BITS, bool XPERM, int H>
cudaError_t launch_wq_h(int group, int64_t blocks, int smem, const uint32_t* codes,
                        const __half* scales, const uint8_t* zeros, int64_t N, int64_t K,
                        const __half* x, int M, float* y, cudaStream_t st) {
  auto go = [&](auto kern) -> cudaError_t {
    LaunchFacts lf;   // raises the kernel's dynamic shared memory limit once per device
    constexpr int threads = block_warps<NT, XPERM>() * 32;
    cudaError_t err = launch_facts(reinterpret_cast<const void*>(kern), threads, kXSmemMax, &lf);
    if (err != cudaSuccess) return err;
    return launch_dependent(kern, blocks, threads, smem, st, codes, scales, zeros, N, K, x, M, y,
                            kMagic);
  };
  if (group == 64) return go(k_wq_mma<NT, 64, BITS, XPERM, H>);
  if (group == 128) return cudaErrorInvalidValue;   // 64-channel units: K % 128 != 0
  return go(k_wq_mma<NT, 0, BITS, XPERM, H>);
}

template <int NT, int BITS, bool XPERM>
cudaError_t launch_tma(int group, int64_t blocks, int S, int64_t smem, int vec, bool pt,
                       bool split, const uint32_t* codes, const __half* scales, const uint8_t* zeros, int64_t N,
                       int64_t K, const __half* x, int M, float* y, cudaStream_t st) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // The codes as a 2-D tensor of 32-bit words [N][K b / 32]; boxes of 16
  // rows x two units (INT4 128 bytes, 128-byte swizzle; INT3 96 bytes).
  // Rows past N and words past a row's end read as zeros.
  CUtensorMap tmap, tmap_z, tmap_s;
  const int64_t words = K * BITS / 32;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(words), static_cast<cuuint64_t>(N)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(words) * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_row_bytes<BITS>() / 4), 16};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(codes), dims, strides,
          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          BITS == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  tmap_z = tmap;
  tmap_s = tmap;
  if (pt) {
    // zeros [N][groups] bytes, boxes of 16 rows x 16 groups; scales [N][groups]
    // fp16, boxes of 16 rows x 8 groups (row strides multiples of 16 bytes).
    const int64_t groups = K / group;
    const cuuint64_t gd[2] = {static_cast<cuuint64_t>(groups), static_cast<cuuint64_t>(N)};
    const cuuint64_t zs[1] = {static_cast<cuuint64_t>(groups)};
    const cuuint64_t ss[1] = {static_cast<cuuint64_t>(groups) * 2};
    const cuuint32_t zb[2] = {16, 16}, sb[2] = {8, 16};
    if (enc(&tmap_z, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(zeros), gd, zs, zb,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&tmap_s, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<__half*>(scales), gd, ss, sb,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto go = [&](auto kern) -> cudaError_t {
    LaunchFacts lf;   // raises the kernel's dynamic shared memory limit once per device
    constexpr int threads = tma_warps<NT, XPERM>() * 32;
    cudaError_t err = launch_facts(reinterpret_cast<const void*>(kern), threads, kDecodeSmemMax,
                                   &lf);
    if (err != cudaSuccess) return err;
    return launch_dependent(kern, blocks, threads, smem, st, tmap, tmap_z, tmap_s, scales, zeros,
                            N, K, x, M, y, S, vec, kMagic);
  };
  // The K split is compiled with x staged only.
  constexpr bool kCanSplit = XPERM;
  if (kCanSplit && split) {
    if (group == 128)
      return pt ? go(k_wq_tma<NT, 128, BITS, XPERM, true, kCanSplit>)
                : go(k_wq_tma<NT, 128, BITS, XPERM, false, kCanSplit>);
    if (group == 64)
      return pt ? go(k_wq_tma<NT, 64, BITS, XPERM, true, kCanSplit>)
                : go(k_wq_tma<NT, 64, BITS, XPERM, false, kCanSplit>);
    return go(k_wq_tma<NT, 0, BITS, XPERM, false, kCanSplit>);
  }
  if (group == 128)
    return pt ? go(k_wq_tma<NT, 128, BITS, XPERM, true, false>)
              : go(k_wq_tma<NT, 128, BITS, XPERM, false, false>);
  if (group == 64)
    return pt ? go(k_wq_tma<NT, 64, BITS, XPERM, true, false>)
              : go(k_wq_tma<NT, 64, BITS, XPERM, false, false>);
  return go(k_wq_tma<NT, 0, BITS, XPERM, false, false>);
}

template <int NT, int BITS>
cudaError_t launch_wq(int group, const uint32_t* codes, const __half* scales,
                      const uint8_t* zeros, int64_t N, int64_t K, const __half* x, int M,
                      float* y, cudaStream_t st) {
  // y is zeroed by a kernel launched behind the stream's previous kernel,
  // and the product is launched behind it (see wait_for_zeroed_y).
  const int64_t ny = static_cast<int64_t>(M) * N;
  cudaError_t e = launch_dependent(
      k_zero_y, std::min<int64_t>(ceil_div(ny, 256), 4 * device_sm_count()), 256, 0, st, y, ny);
  if (e != cudaSuccess) return e;
  // One block per SM, at most one per 16-row tile (every block's range is
  // then at least a tile long: at most two blocks add into an output).
  const int64_t tiles = (N + 15) / 16;
  int64_t blocks = std::min<int64_t>(device_sm_count(), tiles);
  const int64_t xbytes = static_cast<int64_t>(M) * K * 2;
  if (K % 128 == 0) {
    // Stage x when it leaves room for 2 stages per warp; the rest of the
    // shared memory is ring (at most kMaxStages stages per warp).
    // Group parameters by TMA with the codes when their rows are whole
    // multiples of 16 bytes (and the arrays 16-byte aligned); else loaded by
    // the warps, with one vector load per row on whole aligned stages when
    // the arrays allow it.
    const int64_t groups = group > 0 ? K / group : 1;
    const bool pt = group > 0 && groups % 16 == 0 &&
                    reinterpret_cast<uintptr_t>(zeros) % 16 == 0 &&
                    reinterpret_cast<uintptr_t>(scales) % 16 == 0;
    bool xperm = tma_smem_bytes(tma_warps<NT, true>(), 2, xbytes, NT, pt) <= kDecodeSmemMax;
    // When x does not fit but half of it does (K a multiple of 1024, so a
    // half starts on a 4-unit stage boundary): half the blocks take the first
    // K/2 channels and half the rest, each over whole row tiles, so every
    // output gets exactly two sums (deterministic).
    int kp = 1;
    if (!xperm && K % 1024 == 0 && tiles >= 2 &&
        tma_smem_bytes(tma_warps<NT, true>(), 2, xbytes / 2, NT, pt) <= kDecodeSmemMax) {
      kp = 2;
      xperm = true;
      blocks = 2 * std::min<int64_t>(device_sm_count() / 2, tiles);
    }
    const int nw = xperm ? tma_warps<NT, true>() : tma_warps<NT, false>();
    const int64_t xb = xperm ? xbytes / kp : 0;
    int S = 1;
    while (S < kMaxStages && tma_smem_bytes(nw, S + 1, xb, NT, pt) <= kDecodeSmemMax) ++S;
    const int64_t smem = tma_smem_bytes(nw, S, xb, NT, pt);
    const int gs = kStageUnits * (group == 64 ? 2 : 1);
    const int vec = group > 0 && groups % gs == 0 &&
                    reinterpret_cast<uintptr_t>(zeros) % gs == 0 &&
                    reinterpret_cast<uintptr_t>(scales) % (2 * gs) == 0;
    return xperm ? launch_tma<NT, BITS, true>(group, blocks, S, smem, vec, pt, kp == 2, codes,
                                              scales, zeros, N, K, x, M, y, st)
                 : launch_tma<NT, BITS, false>(group, blocks, S, smem, vec, pt, kp == 2, codes,
                                               scales, zeros, N, K, x, M, y, st);
  }
  const bool xperm = xbytes <= kXSmemMax;
  const int smem = xperm ? static_cast<int>(xbytes) : 0;
  return xperm ? launch_wq_h<NT, BITS, true, 1>(group, blocks, smem, codes, scales, zeros, N, K, x,
                                                M, y, st)
               : launch_wq_h<NT, BITS, false, 1>(group, blocks, smem, codes, scales, zeros, N, K, x,
                                                 M, y, st);
}

}  // namespace

cudaError_t launch_w4_matvec(const uint32_t* codes, const __half* scales, const uint8_t* zeros,
                             int64_t N, int64_t K, int group, int bits, const __half* x, int M,
                             float* y, cudaStream_t st) {
  if (M < 1 || M > 16 || K % kHalf) return cudaErrorInvalidValue;
  if (bits == 4)
    return M <= 8 ? launch_wq<1, 4>(group, codes, scales, zeros, N, K, x, M, y, st)
                  : launch_wq<2, 4>(group, codes, scales, zeros, N, K, x, M, y, st);
  if (bits == 3)
    return M <= 8 ? launch_wq<1, 3>(group, codes, scales, zeros, N, K, x, M, y, st)
                  : launch_wq<2, 3>(group, codes, scales, zeros, N, K, x, M, y, st);
  return cudaErrorInvalidValue;
}

AWQ_BOUNDS_READER(bounds_matvec)

}  // namespace awq
