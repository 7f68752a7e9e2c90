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
// Both kernels that quantize (the search's residual pass and the final
// quantize + pack) give a lane 16 consecutive channels of two consecutive
// rows: a group of 128 channels is 8 lanes, of 64 is 4, reduced with
// shuffles, and the per-group step, fp16 scale and reciprocal are paid once
// per 16 weights.  Rounding avoids the float-to-int conversion unit (see
// rne_small).
#include <algorithm>
#include <type_traits>

#include "awq_async.cuh"
#include "awq_bounds.cuh"
#include "awq_f32x2.cuh"
#include "awq_internal.h"
#include "awq_ptx.cuh"

namespace awq {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kPerLane = 16;        // consecutive channels per lane
constexpr int kRowsPerLane = 2;     // rows per lane

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ void st_v8(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// 16 fp16 weights (two raw 16-byte chunks, or 32 bytes of memory) as fp32.
__device__ __forceinline__ void raw_to_f32(const uint4* raw, float* w) {
#pragma unroll
  for (int v = 0; v < 2; ++v) {
    const uint32_t u[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
      w[8 * v + 2 * i] = f.x;
      w[8 * v + 2 * i + 1] = f.y;
    }
  }
}

// Packed fp32 pairs come from awq_f32x2.cuh.  In the quantizer no packed
// add consumes a product directly: the rounding add consumes a clamped value
// (a min / max sits between).
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

// Round half to even without the conversion unit: adding and removing
// 1.5 * 2^23 leaves rne(t) for |t| <= 2^22 (the sum's ulp is 1, and the
// addition rounds half to even).  The map is monotone, so for larger |t| the
// result keeps the side of [-2^22, 2^22] that t is on, which is all the
// clamps below ever look at.
constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23
__device__ __forceinline__ float rne_small(float t) {
  return __fsub_rn(__fadd_rn(t, kMagic), kMagic);
}

// Per-group parameters of the quantizer for the lane's two rows, from the
// lane's 16 scaled weights w' = w * s of each row.  GROUP 64 or 128: GLANES =
// GROUP / 16 adjacent lanes form one group and reduce min / max by shuffles
// (every lane of the warp calls this); the two rows' reductions, shuffles and
// arithmetic are interleaved (independent chains).  GROUP 0 (one group per
// row): the row's min / max come precomputed in `rowmm` (k_row_minmax).
//
// Asymmetric (zero_point): step = max(max - min, 1e-5) / L, z = clamp(rne(-min
// * rcp), 0, L).  Symmetric: step = max(max |w'|, 1e-5) / ((L - 1) / 2) and
// z = (L + 1) / 2, the mid-code.
//
// Only one side of the code clamp can ever act (rne is odd-symmetric and
// fl(x * rcp) is monotone in x): asymmetric with zu = rne(-min * rcp) <= L,
// every code rne(w' * rcp) + z is >= 0 and only the upper bound L can be
// exceeded; with zu > L (z clamped to L, every w' < 0) every code is <= L and
// only 0 can be undershot (`low` marks that case).  Symmetric: |w' * rcp| <=
// (L - 1) / 2 within the fp16 rounding of the step, so no clamp acts; the
// upper one is kept.
struct GroupQ {
  float sf;    // float(fp16 scale)
  float rcp;   // fp32 1 / sf
  float z;     // zero point (an integer in [0, L])
  bool low;    // the clamp that can act is the one at 0 (else the one at L)
  __half scale;
};

// min / max of the 8 (GROUP 128) or 4 (GROUP 64) lanes of each group, for
// both rows; every lane of the warp calls this.
template <int GROUP>
__device__ __forceinline__ void group_reduce2(float (&mn)[kRowsPerLane], float (&mx)[kRowsPerLane]) {
  constexpr int GLANES = GROUP / kPerLane;
#pragma unroll
  for (int off = GLANES / 2; off; off >>= 1) {
#pragma unroll
    for (int r = 0; r < kRowsPerLane; ++r) {
      mn[r] = fminf(mn[r], __shfl_xor_sync(0xFFFFFFFFu, mn[r], off));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xFFFFFFFFu, mx[r], off));
    }
  }
}

// The quantizer's parameters from the group's min / max.  The two lanes
// 2i and 2i + 1 hold the same groups (a group is 4 or 8 whole lanes, or a
// whole row), so each computes the parameters of one row (row lane & 1) and
// takes the other row's from its neighbour: the divide and the reciprocal
// are paid once per lane instead of twice.
template <bool SYM>
__device__ __forceinline__ void group_finish2(const float (&mn)[kRowsPerLane],
                                              const float (&mx)[kRowsPerLane], float L,
                                              GroupQ (&g)[kRowsPerLane]) {
  static_assert(kRowsPerLane == 2, "one row per lane of a pair");
  const bool odd = (threadIdx.x & 1) != 0;
  const float lo_v = odd ? mn[1] : mn[0], hi_v = odd ? mx[1] : mx[0];
  GroupQ q;
  if constexpr (SYM) {
    const float half_levels = 0.5f * (L - 1.0f);   // 7 or 3, exact
    const float step = __fdiv_rn(fmaxf(fmaxf(-lo_v, hi_v), 1e-5f), half_levels);
    q.scale = __float2half_rn(step);
    q.sf = __half2float(q.scale);
    q.rcp = __frcp_rn(q.sf);
    q.low = false;
    q.z = 0.5f * (L + 1.0f);                        // 8 or 4, exact
  } else {
    const float step = __fdiv_rn(fmaxf(__fsub_rn(hi_v, lo_v), 1e-5f), L);
    q.scale = __float2half_rn(step);
    q.sf = __half2float(q.scale);
    q.rcp = __frcp_rn(q.sf);
    const float zu = rne_small(__fmul_rn(-lo_v, q.rcp));
    q.low = zu > L;
    q.z = fminf(fmaxf(zu, 0.0f), L);
  }
  GroupQ o;   // the neighbour's row
  o.sf = __shfl_xor_sync(0xFFFFFFFFu, q.sf, 1);
  o.rcp = __shfl_xor_sync(0xFFFFFFFFu, q.rcp, 1);
  o.z = __shfl_xor_sync(0xFFFFFFFFu, q.z, 1);
  o.low = __shfl_xor_sync(0xFFFFFFFFu, static_cast<int>(q.low), 1) != 0;
  o.scale = __float2half_rn(o.sf);   // exact: sf is an fp16 value
  g[0] = odd ? o : q;
  g[1] = odd ? q : o;
}

template <int GROUP, bool SYM>
__device__ __forceinline__ void group_params2(const float (&ws)[kRowsPerLane][kPerLane], float L,
                                              const float2* rowmm, GroupQ (&g)[kRowsPerLane]) {
  float mn[kRowsPerLane], mx[kRowsPerLane];
  if constexpr (GROUP == 0) {
#pragma unroll
    for (int r = 0; r < kRowsPerLane; ++r) {
      mn[r] = rowmm[r].x;
      mx[r] = rowmm[r].y;
    }
  } else {
#pragma unroll
    for (int r = 0; r < kRowsPerLane; ++r) {
      float mnA = fminf(ws[r][0], ws[r][1]), mxA = fmaxf(ws[r][0], ws[r][1]);
      float mnB = fminf(ws[r][2], ws[r][3]), mxB = fmaxf(ws[r][2], ws[r][3]);
#pragma unroll
      for (int i = 4; i < kPerLane; i += 4) {
        mnA = min3f(mnA, ws[r][i], ws[r][i + 1]);
        mxA = max3f(mxA, ws[r][i], ws[r][i + 1]);
        mnB = min3f(mnB, ws[r][i + 2], ws[r][i + 3]);
        mxB = max3f(mxB, ws[r][i + 2], ws[r][i + 3]);
      }
      mn[r] = fminf(mnA, mnB);
      mx[r] = fmaxf(mxA, mxB);
    }
    group_reduce2<GROUP>(mn, mx);
  }
  group_finish2<SYM>(mn, mx, L, g);
}

// ws[i] = w[i] * s[i], correctly rounded (packed multiplies; no add follows).
__device__ __forceinline__ void scale16(const float* w, const float* s, float* ws) {
#pragma unroll
  for (int i = 0; i < kPerLane; i += 2) {
    const f32x2 p = mul2(pack2(w[i], w[i + 1]), pack2(s[i], s[i + 1]));
    ws[i] = lo2(p);
    ws[i + 1] = hi2(p);
  }
}

// Launch geometry shared by both kernels: blockIdx.x is a chunk of 32 lanes x
// kPerLane channels, and the 8 warps of a block take 16 consecutive rows (two
// per warp) at those channels; blockIdx.y walks 16-row blocks (grid-stride,
// one wave of persistent blocks).  Lanes past the end of a row form whole
// groups (K % GROUP == 0), so their dummy values (they re-read the row's last
// chunk) never meet real ones in a reduction.
constexpr int kRowsPerBlock = (kQuantThreads / 32) * kRowsPerLane;

struct Lane {
  int64_t lc;      // lane chunk along the row (kPerLane channels each)
  int64_t k0;      // first channel (clamped for lanes past the row's end)
  bool active;     // lc is inside the row
};

__device__ __forceinline__ Lane lane_chunk(int64_t K) {
  const int64_t lanes_per_row = K / kPerLane;
  Lane l;
  l.lc = static_cast<int64_t>(blockIdx.x) * 32 + (threadIdx.x & 31);
  l.active = l.lc < lanes_per_row;
  l.k0 = (l.active ? l.lc : lanes_per_row - 1) * kPerLane;
  return l;
}

// ---------------------------------------------------------------- W rings
// Both kernels stream W through per-warp rings in shared memory filled with
// cp.async.  A warp's 512 channels of one row (1 KB) are copied as two fully
// coalesced 512-byte requests (lane l: 16-byte chunks l and 32 + l); lane l
// then reads its own chunks 2l and 2l + 1.  Chunk c is stored at
// c ^ ((c / 8) % 2), so that the copies and the 16-byte reads of each
// quarter-warp hit distinct banks.
constexpr int kRowChunks = 32 * kPerLane / 8;   // 16-byte chunks of a warp's row segment

__device__ __forceinline__ int fin_slot(int c) { return c ^ ((c >> 3) & 1); }

// ---------------------------------------------------------------- residual
// Search output: the quantization residual of every grid point, in the units
// of W,
//   delta[a][row_off + n][k] = fp16( w - ((q - z) * scale) / s_k ),
// i.e. W - deq(Q(W diag(s))) diag(s)^-1 row by row.  The codes and zero
// points are those of the final quantizer (same steps, same rounding), with
// the clamp applied to (q - z) directly:  q - z = clamp(rne(w' * rcp), -z, L - z).
// (q - z) * scale is exact in fp32 (a 4-bit integer times an 11-bit
// significand); w - that * (1/s_k) is one fused multiply-add, and the one
// coarse rounding is the final one to fp16, relative to the residual.
//
//
// Persistent blocks (two per SM) each keep one 512-channel chunk.  s and 1/s
// of up to kResAlphaTile grid points for those channels are staged once per
// block in shared memory; a lane reads its 16 channels' values there (16-byte
// chunk c of a grid point's 512 channels stored at c ^ ((c / 8) % 8): the 8
// lanes of a quarter-warp read distinct banks).  W comes through a per-warp
// ring of kResStages row pairs, so the next row pair's loads are in flight
// while every grid point of the current one is evaluated.  Each lane writes
// one whole 32-byte sector per row and grid point.  More than kResAlphaTile
// grid points are done in tiles (W is read once per tile).
constexpr int kResAlphaTile = 20;
constexpr int kResStages = 2;
constexpr int kResSChunks = 32 * kPerLane / 4;                        // 16-byte chunks of s
constexpr int kResSRBytes = kResAlphaTile * 2 * kResSChunks * 16;     // 80 KB: s and 1/s
constexpr int kResRingBytes = (kQuantThreads / 32) * kResStages * kRowsPerLane * kRowChunks * 16;
constexpr int kResSmem = kResSRBytes + kResRingBytes;                 // 112 KB

__device__ __forceinline__ int res_slot(int c) { return c ^ ((c >> 3) & 7); }

template <int GROUP, bool SYM>
__global__ void __launch_bounds__(kQuantThreads)
    k_quant_residual(const __half* __restrict__ W, int64_t N, int64_t K, int levels,
                     const float* __restrict__ s_grid, const float* __restrict__ r_grid,
                     int n_alpha, int64_t row_off, int64_t n_pad, __half* __restrict__ delta,
                     const float2* __restrict__ rowmm) {
  extern __shared__ uint4 res_smem[];
  float4* s_tile = reinterpret_cast<float4*>(res_smem);      // [kResAlphaTile][kResSChunks]
  float4* r_tile = s_tile + kResAlphaTile * kResSChunks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint4* ring = reinterpret_cast<uint4*>(r_tile + kResAlphaTile * kResSChunks) +
                warp * (kResStages * kRowsPerLane * kRowChunks);
  const uint32_t ring_u32 = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  const float L = static_cast<float>(levels);
  const int64_t slab = n_pad * K;                     // halves per grid point
  const Lane lw = lane_chunk(K);
  const int64_t kbase = static_cast<int64_t>(blockIdx.x) * (32 * kPerLane);
  const int64_t w_rest = (K - kbase) / 8, s_rest = (K - kbase) / 4;
  const int w_valid = static_cast<int>(w_rest < kRowChunks ? w_rest : kRowChunks);
  const int s_valid = static_cast<int>(s_rest < kResSChunks ? s_rest : kResSChunks);
  const int w_mine = static_cast<int>((lw.k0 - kbase) / 8);   // the lane's 2 chunks of W
  const int s_mine = static_cast<int>((lw.k0 - kbase) / 4);   // the lane's 4 chunks of s
  const int64_t row_step = static_cast<int64_t>(gridDim.y) * kRowsPerBlock;
  const int64_t first = (static_cast<int64_t>(blockIdx.y) * (kQuantThreads / 32) + warp) *
                        kRowsPerLane;
  const int64_t iters = first < N ? (N - first + row_step - 1) / row_step : 0;
  auto issue = [&](int64_t it) {
    if (it < iters) {
      const int st = static_cast<int>(it % kResStages);
      const int64_t row0 = first + it * row_step;
#pragma unroll
      for (int r = 0; r < kRowsPerLane; ++r) {   // a lone last row loads itself twice
        const int64_t w_off = min(row0 + r, N - 1) * K + kbase;
        const __half* src = W + w_off;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = 32 * j + lane;
          if (c < w_valid && in_bounds(kSiteResidualW, w_off + 8 * c + 7, N * K))
            cp_async16(ring_u32 + ((st * kRowsPerLane + r) * kRowChunks + fin_slot(c)) * 16,
                       src + 8 * c);
        }
      }
    }
    cp_async_commit();   // possibly empty: one group per row pair
  };
  for (int a0 = 0; a0 < n_alpha; a0 += kResAlphaTile) {
    const int na = n_alpha - a0 < kResAlphaTile ? n_alpha - a0 : kResAlphaTile;
    __syncthreads();   // every warp is done with the previous tile of s and 1/s
    for (int a = warp; a < na; a += kQuantThreads / 32) {
      const float* sp = s_grid + static_cast<int64_t>(a0 + a) * K + kbase;
      const float* rp = r_grid + static_cast<int64_t>(a0 + a) * K + kbase;
      for (int c = lane; c < s_valid; c += 32) {
        if (!in_bounds(kSiteResidualS, static_cast<int64_t>(a0 + a) * K + kbase + 4 * c + 3,
                       static_cast<int64_t>(n_alpha) * K))
          continue;
        cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(
                       s_tile + a * kResSChunks + res_slot(c))), sp + 4 * c);
        cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(
                       r_tile + a * kResSChunks + res_slot(c))), rp + 4 * c);
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();   // the tile of s and 1/s is in place
#pragma unroll
    for (int i = 0; i < kResStages - 1; ++i) issue(i);
    for (int64_t it = 0; it < iters; ++it) {
      issue(it + kResStages - 1);
      cp_async_wait<kResStages - 1>();
      __syncwarp();   // every lane's copies of this row pair have landed
      const int st = static_cast<int>(it % kResStages);
      const int64_t row0 = first + it * row_step;
      float w[kRowsPerLane][kPerLane];
#pragma unroll
      for (int r = 0; r < kRowsPerLane; ++r) {
        const uint4* slot = ring + (st * kRowsPerLane + r) * kRowChunks;
        const uint4 raw[2] = {slot[fin_slot(w_mine)], slot[fin_slot(w_mine + 1)]};
        raw_to_f32(raw, w[r]);
      }
      __syncwarp();   // the slot is refilled at the next row pair
      // Where this row pair's residual goes at the tile's first grid point
      // (advanced by one slab per grid point).
      __half* dst = delta + static_cast<int64_t>(a0) * slab + (row_off + row0) * K + lw.k0;
#pragma unroll 1
      for (int a = 0; a < na; ++a, dst += slab) {
        float sv[kPerLane], rv[kPerLane];
#pragma unroll
        for (int q = 0; q < kPerLane / 4; ++q) {
          const float4 fs = s_tile[a * kResSChunks + res_slot(s_mine + q)];
          const float4 fr = r_tile[a * kResSChunks + res_slot(s_mine + q)];
          sv[4 * q] = fs.x;
          sv[4 * q + 1] = fs.y;
          sv[4 * q + 2] = fs.z;
          sv[4 * q + 3] = fs.w;
          rv[4 * q] = fr.x;
          rv[4 * q + 1] = fr.y;
          rv[4 * q + 2] = fr.z;
          rv[4 * q + 3] = fr.w;
        }
        const int ga = a0 + a;
        // w' = w * s is written out twice (here for the group's min / max,
        // below for the codes); the compiler keeps the products in registers
        // between the two (measured: 4.7 % faster than forcing the second
        // product, which saved registers the kernel does not need).
        float mn[kRowsPerLane], mx[kRowsPerLane];
        if constexpr (GROUP == 0) {   // per-row groups: min / max of this grid point's rows
#pragma unroll
          for (int r = 0; r < kRowsPerLane; ++r) {
            const int64_t im = static_cast<int64_t>(ga) * N + min(row0 + r, N - 1);
            const float2 m = in_bounds(kSiteResidualRowmm, im, static_cast<int64_t>(n_alpha) * N)
                                 ? rowmm[im]
                                 : make_float2(0.f, 0.f);
            mn[r] = m.x;
            mx[r] = m.y;
          }
        } else {
#pragma unroll
          for (int r = 0; r < kRowsPerLane; ++r) {
            float mnA = INFINITY, mxA = -INFINITY, mnB = INFINITY, mxB = -INFINITY;
#pragma unroll
            for (int i = 0; i < kPerLane; i += 4) {
              const f32x2 p = mul2(pack2(w[r][i], w[r][i + 1]), pack2(sv[i], sv[i + 1]));
              const f32x2 q = mul2(pack2(w[r][i + 2], w[r][i + 3]), pack2(sv[i + 2], sv[i + 3]));
              mnA = min3f(mnA, lo2(p), hi2(p));
              mxA = max3f(mxA, lo2(p), hi2(p));
              mnB = min3f(mnB, lo2(q), hi2(q));
              mxB = max3f(mxB, lo2(q), hi2(q));
            }
            mn[r] = fminf(mnA, mnB);
            mx[r] = fmaxf(mxA, mxB);
          }
          group_reduce2<GROUP>(mn, mx);
        }
        GroupQ gq[kRowsPerLane];
        group_finish2<SYM>(mn, mx, L, gq);
        // rare: some group of the warp is all negative (both clamp sides needed)
        const bool low = __any_sync(0xFFFFFFFFu, gq[0].low || gq[1].low);
#pragma unroll
        for (int r = 0; r < kRowsPerLane; ++r) {
          const GroupQ& g = gq[r];
          const float lo = -g.z, hi = L - g.z;
          const f32x2 nsf = pack2(-g.sf, -g.sf);
          // d = clamp(rne(w' * rcp), -z, L - z): the bounds are integers, so
          // the clamp may come before the rounding adds.
          const f32x2 rcp2 = pack2(g.rcp, g.rcp);
          const f32x2 magic2 = pack2(kMagic, kMagic), nmagic2 = pack2(-kMagic, -kMagic);
          float d[kPerLane];
          // The two loops differ only in the lower clamp, needed only where
          // some group of the warp is all negative (a warp-uniform branch
          // around the loop, so the common one has one min per weight).
          if (low) {
#pragma unroll
            for (int i = 0; i < kPerLane; i += 2) {
              const f32x2 ws2 = mul2(pack2(w[r][i], w[r][i + 1]), pack2(sv[i], sv[i + 1]));
              const f32x2 t = mul2(ws2, rcp2);
              const float t0 = fmaxf(fminf(lo2(t), hi), lo), t1 = fmaxf(fminf(hi2(t), hi), lo);
              const f32x2 m = add2(add2(pack2(t0, t1), magic2), nmagic2);
              d[i] = lo2(m);
              d[i + 1] = hi2(m);
            }
          } else {
#pragma unroll
            for (int i = 0; i < kPerLane; i += 2) {
              const f32x2 ws2 = mul2(pack2(w[r][i], w[r][i + 1]), pack2(sv[i], sv[i + 1]));
              const f32x2 t = mul2(ws2, rcp2);
              const float t0 = fminf(lo2(t), hi), t1 = fminf(hi2(t), hi);
              const f32x2 m = add2(add2(pack2(t0, t1), magic2), nmagic2);
              d[i] = lo2(m);
              d[i + 1] = hi2(m);
            }
          }
          uint32_t o[kPerLane / 2];
#pragma unroll
          for (int i = 0; i < kPerLane; i += 2) {
            // w - (d * sf) * (1/s): the product d * sf is exact.
            const f32x2 e = fma2(mul2(pack2(d[i], d[i + 1]), nsf), pack2(rv[i], rv[i + 1]),
                                 pack2(w[r][i], w[r][i + 1]));
            const __half2 hv = __floats2half2_rn(lo2(e), hi2(e));
            o[i / 2] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          if (lw.active && row0 + r < N &&
              in_bounds(kSiteResidualOut,
                        static_cast<int64_t>(ga) * slab + (row_off + row0 + r) * K + lw.k0 + 15,
                        static_cast<int64_t>(n_alpha) * slab))
            st_v8(dst + r * K, o);
        }
      }
    }
    cp_async_wait<0>();
  }
}

// ---------------------------------------------------------------- final
// Result layout: INT4 codes [N][K/8] (code 8j+m in nibble m of word j);
// INT3 codes [N][3K/32] (bit stream, code k in bits [3k, 3k+3));
// scales fp16 [N][K/group]; zeros u8 [N][K/group].
//
// The code is taken in the rounding constant's binade: m = rn(w' * rcp) +
// 1.5 * 2^23 is clamped to [M - z, M + L - z], and the integer code is the
// difference of the bit patterns of m and M - z (consecutive integers in
// [2^23, 2^24) have consecutive patterns).  codes8: the code words are
// 8-byte aligned (INT4 only), so a lane stores its two words at once.
//
// One wave of persistent blocks; a warp keeps its 512 channels (and its
// lanes' s) and walks row pairs.  W reaches registers through a per-warp
// ring of kFinStages row pairs in shared memory filled with cp.async, so
// kFinStages - 1 row pairs of loads are in flight while one is quantized.
// The warp copies a row's 1 KB as two fully coalesced 512-byte requests
// (lane l: 16-byte chunks l and 32 + l); lane l then reads its own chunks
// 2l and 2l + 1, stored at chunk ^ ((chunk / 8) % 2) so that both the
// copies and the 16-byte reads of each quarter-warp hit distinct banks.
constexpr int kFinStages = 4;
constexpr int kFinSmem = (kQuantThreads / 32) * kFinStages * kRowsPerLane * kRowChunks * 16;
static_assert(kFinSmem == 64 * 1024, "ring size");

template <int BITS, int GROUP, bool SYM>
__global__ void __launch_bounds__(kQuantThreads, 3)
    k_quant_final(const __half* __restrict__ W, int64_t N, int64_t K,
                  const float* __restrict__ s_base, const int* __restrict__ sel,
                  uint32_t* __restrict__ codes, __half* __restrict__ scales,
                  uint8_t* __restrict__ zeros, bool codes8, const float2* __restrict__ rowmm) {
  extern __shared__ uint4 fin_ring[];
  // Launched behind the stream's previous kernel (the chosen grid point, W
  // and s may come from it).
  grid_dependency_wait();
  grid_dependents_launch();
  constexpr int LEVELS = (1 << BITS) - 1;
  const float L = static_cast<float>(LEVELS);
  const int64_t groups = GROUP == 0 ? 1 : K / (GROUP == 0 ? 1 : GROUP);
  const int64_t words = BITS == 4 ? K / 8 : 3 * K / 32;
  const float* s = s_base + (sel ? static_cast<int64_t>(*sel) * K : 0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Lane lw = lane_chunk(K);
  const int64_t kbase = static_cast<int64_t>(blockIdx.x) * (32 * kPerLane);
  const int64_t rest = (K - kbase) / 8;
  const int valid = static_cast<int>(rest < kRowChunks ? rest : kRowChunks);
  const int mine = static_cast<int>((lw.k0 - kbase) / 8);   // first of the lane's two chunks
  uint4* ring = fin_ring + warp * (kFinStages * kRowsPerLane * kRowChunks);
  const uint32_t ring_u32 = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  const int64_t row_step = static_cast<int64_t>(gridDim.y) * kRowsPerBlock;
  const int64_t first = (static_cast<int64_t>(blockIdx.y) * (kQuantThreads / 32) + warp) *
                        kRowsPerLane;
  const int64_t iters = first < N ? (N - first + row_step - 1) / row_step : 0;
  auto issue = [&](int64_t it) {
    if (it < iters) {
      const int st = static_cast<int>(it % kFinStages);
      const int64_t row0 = first + it * row_step;
#pragma unroll
      for (int r = 0; r < kRowsPerLane; ++r) {   // a lone last row loads itself twice
        const int64_t w_off = min(row0 + r, N - 1) * K + kbase;
        const __half* src = W + w_off;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = 32 * j + lane;
          if (c < valid && in_bounds(kSiteFinalW, w_off + 8 * c + 7, N * K))
            cp_async16(ring_u32 + ((st * kRowsPerLane + r) * kRowChunks + fin_slot(c)) * 16,
                       src + 8 * c);
        }
      }
    }
    cp_async_commit();   // possibly empty: one group per row pair
  };
#pragma unroll
  for (int i = 0; i < kFinStages - 1; ++i) issue(i);
  // The lane's s: the same 16 channels for every row.
  float sv[kPerLane];
#pragma unroll
  for (int v = 0; v < kPerLane / 4; ++v) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(s + lw.k0) + v);
    sv[4 * v] = f.x;
    sv[4 * v + 1] = f.y;
    sv[4 * v + 2] = f.z;
    sv[4 * v + 3] = f.w;
  }
  for (int64_t it = 0; it < iters; ++it) {
    issue(it + kFinStages - 1);
    cp_async_wait<kFinStages - 1>();
    __syncwarp();   // every lane's copies of this row pair have landed
    const int st = static_cast<int>(it % kFinStages);
    const int64_t row0 = first + it * row_step;
    uint4 raw[kRowsPerLane][2];
#pragma unroll
    for (int r = 0; r < kRowsPerLane; ++r) {
      const uint4* slot = ring + (st * kRowsPerLane + r) * kRowChunks;
      raw[r][0] = slot[fin_slot(mine)];
      raw[r][1] = slot[fin_slot(mine + 1)];
    }
    __syncwarp();   // the slot is refilled at the next row pair
    float ws[kRowsPerLane][kPerLane];
#pragma unroll
    for (int r = 0; r < kRowsPerLane; ++r) {
      float w[kPerLane];
      raw_to_f32(raw[r], w);
      scale16(w, sv, ws[r]);
    }
    float2 mm[kRowsPerLane];
    if constexpr (GROUP == 0) {   // per-row groups: precomputed min / max
#pragma unroll
      for (int r = 0; r < kRowsPerLane; ++r) mm[r] = rowmm[min(row0 + r, N - 1)];
    }
    GroupQ gq[kRowsPerLane];
    group_params2<GROUP, SYM>(ws, L, mm, gq);
    // rare: some group of the warp is all negative (both clamp sides needed)
    const bool low = __any_sync(0xFFFFFFFFu, gq[0].low || gq[1].low);
#pragma unroll
    for (int r = 0; r < kRowsPerLane; ++r) {
      const int64_t row = row0 + r;
      const GroupQ& g = gq[r];
      const uint32_t base = __float_as_uint(__fsub_rn(kMagic, g.z));   // bits of M - z
      // b[i] = bit pattern of M + clamp(rne(w' * rcp), -z, L - z); code = b[i] - base.
      // The bounds are integers, so clamping before the rounding add is the
      // same as clamping after it.
      const float lo = -g.z, hi = L - g.z;
      const f32x2 rcp2 = pack2(g.rcp, g.rcp), magic2 = pack2(kMagic, kMagic);
      uint32_t b[kPerLane];
      // The lower clamp only where some group of the warp is all negative (a
      // warp-uniform branch around the loop: the common one has one min per
      // weight).
      if (low) {
#pragma unroll
        for (int i = 0; i < kPerLane; i += 2) {
          const f32x2 t = mul2(pack2(ws[r][i], ws[r][i + 1]), rcp2);
          const float t0 = fmaxf(fminf(lo2(t), hi), lo), t1 = fmaxf(fminf(hi2(t), hi), lo);
          const f32x2 m = add2(pack2(t0, t1), magic2);
          b[i] = static_cast<uint32_t>(m);
          b[i + 1] = static_cast<uint32_t>(m >> 32);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kPerLane; i += 2) {
          const f32x2 t = mul2(pack2(ws[r][i], ws[r][i + 1]), rcp2);
          const float t0 = fminf(lo2(t), hi), t1 = fminf(hi2(t), hi);
          const f32x2 m = add2(pack2(t0, t1), magic2);
          b[i] = static_cast<uint32_t>(m);
          b[i + 1] = static_cast<uint32_t>(m >> 32);
        }
      }
      const bool store = lw.active && row < N;
      uint32_t* crow = codes + row * words;
      // Packing by multiply-add on the FMA pipe: sum_i code_i * 2^(bits*i) =
      // sum_i b_i * 2^(bits*i) - base * sum_i 2^(bits*i) (mod 2^32), exact
      // because the true packed value fits in 32 bits.
      if (BITS == 4) {
        uint32_t c0 = b[7], c1 = b[15];
#pragma unroll
        for (int i = 6; i >= 0; --i) {
          c0 = c0 * 16u + b[i];
          c1 = c1 * 16u + b[8 + i];
        }
        c0 -= base * 0x11111111u;
        c1 -= base * 0x11111111u;
        if (store && in_bounds(kSiteFinalCodes, row * words + 2 * lw.lc + 1, N * words)) {
          uint32_t* dst = crow + 2 * lw.lc;
          if (codes8) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(c0, c1);
          } else {
            dst[0] = c0;
            dst[1] = c1;
          }
        }
      } else {
        // 16 codes = 48 bits: codes 0..10 in lo32 (code 10 keeps its low 2
        // bits there), code 10's top bit and codes 11..15 in hi16.  An
        // even/odd lane pair holds 96 bits = 3 words (K % 32 == 0, so pairs
        // are never split by the row's end).
        uint32_t lo32 = b[10];
#pragma unroll
        for (int i = 9; i >= 0; --i) lo32 = lo32 * 8u + b[i];
        lo32 -= base * 0x49249249u;                     // sum_{i<=10} 8^i mod 2^32
        uint32_t hi16 = b[15];
#pragma unroll
        for (int i = 14; i >= 11; --i) hi16 = hi16 * 8u + b[i];
        hi16 = (hi16 - base * 0x00001249u) * 2u + ((b[10] - base) >> 2);
        const uint32_t next_lo = __shfl_down_sync(0xFFFFFFFFu, lo32, 1);
        if (store && in_bounds(kSiteFinalCodes, row * words + (lw.lc >> 1) * 3 + 2, N * words)) {
          uint32_t* dst = crow + (lw.lc >> 1) * 3;
          if ((lane & 1) == 0) {
            dst[0] = lo32;
            dst[1] = hi16 | (next_lo << 16);
          } else {
            // this lane's bits 16..47: the pair's word 2
            dst[2] = (lo32 >> 16) | (hi16 << 16);
          }
        }
      }
      bool group_lead;
      int64_t gi;
      if constexpr (GROUP == 0) {
        group_lead = lw.lc == 0;
        gi = row;
      } else {
        group_lead = (lane % (GROUP / kPerLane)) == 0;
        gi = row * groups + lw.k0 / GROUP;
      }
      if (store && group_lead && in_bounds(kSiteFinalParams, gi, N * groups)) {
        scales[gi] = g.scale;
        zeros[gi] = static_cast<uint8_t>(__float2uint_rn(g.z));
      }
    }
  }
}

// ---------------------------------------------------------------- per-row groups
// group_size -1: the min / max of w' = w * s over each row's K channels,
// rowmm[a][n] = {min, max} for grid point a -- or, with `sel`, for the one
// grid point *sel, stored at a = 0.  Block = one row (grid-stride over rows);
// 16-byte loads of W and s.  Min and max are exact, so the order of the
// reduction does not matter.
__global__ void __launch_bounds__(256)
    k_row_minmax(const __half* __restrict__ W, int64_t N, int64_t K,
                 const float* __restrict__ s_grid, const int* __restrict__ sel, int n_alpha,
                 float2* __restrict__ rowmm) {
  __shared__ float smn[8], smx[8];
  grid_dependency_wait();   // launched behind the stream's previous kernel
  grid_dependents_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
    const uint4* wr = reinterpret_cast<const uint4*>(W + row * K);
    for (int a = 0; a < n_alpha; ++a) {
      const float* s = s_grid + static_cast<int64_t>(sel ? *sel : a) * K;
      float mn = INFINITY, mx = -INFINITY;
      for (int64_t c = threadIdx.x; c < K / 8; c += blockDim.x) {
        const uint4 q = __ldg(wr + c);
        const float4 s0 = __ldg(reinterpret_cast<const float4*>(s + 8 * c));
        const float4 s1 = __ldg(reinterpret_cast<const float4*>(s + 8 * c) + 1);
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
        const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
          const float w0 = __fmul_rn(f.x, sv[2 * i]), w1 = __fmul_rn(f.y, sv[2 * i + 1]);
          mn = min3f(mn, w0, w1);
          mx = max3f(mx, w0, w1);
        }
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
      }
      if (lane == 0) {
        smn[warp] = mn;
        smx[warp] = mx;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        for (int w = 1; w < 8; ++w) {
          mn = fminf(mn, smn[w]);
          mx = fmaxf(mx, smx[w]);
        }
        rowmm[static_cast<int64_t>(a) * N + row] = make_float2(mn, mx);
      }
      __syncthreads();
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

// One wave of resident blocks of a quantizer kernel: x = 512-channel chunks,
// y = an equal share of the 16-row blocks for each (at most as many blocks
// as are resident at once).
cudaError_t one_wave_grid(const void* kern, int smem, int64_t N, int64_t K, dim3* grid) {
  LaunchFacts lf;
  const cudaError_t e = launch_facts(kern, kQuantThreads, smem, &lf);
  if (e != cudaSuccess) return e;
  const int64_t gx = ceil_div(K / kPerLane, 32);
  const int64_t row_blocks = ceil_div(N, kRowsPerBlock);
  int64_t gy = std::max<int64_t>(1, (static_cast<int64_t>(lf.per_sm) * lf.sms) / gx);
  gy = std::min<int64_t>(gy, row_blocks);
  gy = ceil_div(row_blocks, ceil_div(row_blocks, gy));
  *grid = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  return cudaSuccess;
}

template <int BITS, int GROUP, bool SYM>
cudaError_t launch_final(const __half* W, int64_t N, int64_t K, const float* s, const int* sel,
                         uint32_t* codes, __half* scales, uint8_t* zeros, const float2* rowmm,
                         cudaStream_t st) {
  auto kern = k_quant_final<BITS, GROUP, SYM>;
  dim3 grid;
  const cudaError_t e = one_wave_grid(reinterpret_cast<const void*>(kern), kFinSmem, N, K, &grid);
  if (e != cudaSuccess) return e;
  const bool c8 = (reinterpret_cast<uintptr_t>(codes) % 8) == 0;
  return launch_dependent(kern, grid, kQuantThreads, kFinSmem, st, W, N, K, s, sel, codes, scales,
                          zeros, c8, rowmm);
}

template <int BITS, bool SYM>
cudaError_t launch_final_g(int group, const __half* W, int64_t N, int64_t K, const float* s,
                           const int* sel, uint32_t* codes, __half* scales, uint8_t* zeros,
                           const float2* rowmm, cudaStream_t st) {
  if (group == 128)
    return launch_final<BITS, 128, SYM>(W, N, K, s, sel, codes, scales, zeros, rowmm, st);
  if (group == 64)
    return launch_final<BITS, 64, SYM>(W, N, K, s, sel, codes, scales, zeros, rowmm, st);
  return launch_final<BITS, 0, SYM>(W, N, K, s, sel, codes, scales, zeros, rowmm, st);
}

cudaError_t launch_row_minmax(const __half* W, int64_t N, int64_t K, const float* s_grid,
                              const int* sel, int n_alpha, float2* rowmm, cudaStream_t st) {
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>(N, static_cast<int64_t>(device_sm_count()) * 8));
  return launch_dependent(k_row_minmax, static_cast<int64_t>(grid), 256, 0, st, W, N, K, s_grid,
                          sel, n_alpha, rowmm);
}

template <int GROUP, bool SYM>
cudaError_t launch_residual_t(cudaStream_t st, const __half* W, int64_t N, int64_t K, int levels,
                              const float* s_grid, const float* r_grid, int n_alpha,
                              int64_t row_off, int64_t n_pad, __half* delta, const float2* rowmm) {
  auto kern = k_quant_residual<GROUP, SYM>;
  dim3 grid;
  const cudaError_t e = one_wave_grid(reinterpret_cast<const void*>(kern), kResSmem, N, K, &grid);
  if (e != cudaSuccess) return e;
  kern<<<grid, kQuantThreads, kResSmem, st>>>(W, N, K, levels, s_grid, r_grid, n_alpha, row_off,
                                              n_pad, delta, rowmm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_residual(const __half* W, int64_t N, int64_t K, int bits, int group,
                                  int zero_point, const float* s_grid, const float* r_grid,
                                  int n_alpha, int64_t row_off, int64_t n_pad, __half* delta,
                                  float2* rowmm, cudaStream_t st) {
  const int levels = (1 << bits) - 1;
  const bool sym = zero_point == 0;
  if (group == -1) {
    cudaError_t e = launch_row_minmax(W, N, K, s_grid, nullptr, n_alpha, rowmm, st);
    if (e != cudaSuccess) return e;
  }
  auto go = [&](auto g, auto y) {
    return launch_residual_t<decltype(g)::value, decltype(y)::value>(
        st, W, N, K, levels, s_grid, r_grid, n_alpha, row_off, n_pad, delta, rowmm);
  };
  using I128 = std::integral_constant<int, 128>;
  using I64 = std::integral_constant<int, 64>;
  using I0 = std::integral_constant<int, 0>;
  using T = std::true_type;
  using F = std::false_type;
  if (group == 128) return sym ? go(I128{}, T{}) : go(I128{}, F{});
  if (group == 64) return sym ? go(I64{}, T{}) : go(I64{}, F{});
  return sym ? go(I0{}, T{}) : go(I0{}, F{});
}

cudaError_t launch_quant_final(const __half* W, int64_t N, int64_t K, int bits, int group,
                               int zero_point, const float* s, const int* sel, uint32_t* codes,
                               __half* scales, uint8_t* zeros, float2* rowmm, cudaStream_t st) {
  if (group == -1) {
    cudaError_t e = launch_row_minmax(W, N, K, s, sel, 1, rowmm, st);
    if (e != cudaSuccess) return e;
  }
  const bool sym = zero_point == 0;
  if (bits == 4)
    return sym ? launch_final_g<4, true>(group, W, N, K, s, sel, codes, scales, zeros, rowmm, st)
               : launch_final_g<4, false>(group, W, N, K, s, sel, codes, scales, zeros, rowmm, st);
  return sym ? launch_final_g<3, true>(group, W, N, K, s, sel, codes, scales, zeros, rowmm, st)
             : launch_final_g<3, false>(group, W, N, K, s, sel, codes, scales, zeros, rowmm, st);
}

cudaError_t launch_unpack(const uint32_t* codes, int64_t N, int64_t K, int bits, uint8_t* q,
                          cudaStream_t st) {
  const int64_t blocks = ceil_div(N * K, kQuantThreads);
  k_unpack<<<static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(blocks, static_cast<int64_t>(device_sm_count()) * 16))),
             kQuantThreads, 0, st>>>(codes, N, K, bits, q);
  return cudaGetLastError();
}

AWQ_BOUNDS_READER(bounds_quant)

}  // namespace awq
