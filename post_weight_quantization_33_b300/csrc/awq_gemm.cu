// The dense contractions of the scale search, on tcgen05 tensor cores.
//
// AWQ Explained (multigrid.ai), "How the scale is chosen": alpha* minimises
// || W x - Q(W diag(s)) diag(s)^-1 x || over the calibration batch.  Written
// as (W - deq(Q(W diag(s))) diag(s)^-1) x, the error of every grid point is
// one GEMM of the fp16 quantization residual (produced by the quantizer pass)
// with the calibration activations: k_gemm_err_pair below, on CTA pairs.
//
// k_gemm_ref computes Y = W X^T in fp32 (the "W x" term, and the Gram matrix
// X^T X of the Gram form) with a single-CTA persistent kernel:
//
//   warp 4      TMA producer: A tile [128 x 64] and B tile [256 x 64], both
//               128-byte swizzled, into a 4-stage shared-memory ring;
//   warp 5      owns TMEM (2 x 256 fp32 columns) and issues tcgen05.mma
//               (M 128, N 256, K 16, fp16 in, fp32 accumulate);
//   warps 0-3   epilogue: tcgen05.ld the finished accumulator (warp w reads
//               lanes 32w..32w+31 = tile rows) and store it row-major.
#include <algorithm>
#include <mutex>

#include "awq_internal.h"
#include "awq_ptx.cuh"

namespace awq {
namespace {

constexpr int BM = kTileM, BN = kTileN, BK = kTileK;
constexpr int STAGES = 4;
constexpr int kEpilogueWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;
constexpr int kEpilogueThreads = 32 * kEpilogueWarps;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t A_BYTES = BM * BK * 2;   // fp16 A tile
constexpr uint32_t B_BYTES = BN * BK * 2;   // fp16 X tile

constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
constexpr uint32_t OFF_BAR = OFF_B + STAGES * B_BYTES;
constexpr uint32_t NUM_BARS = 2 * STAGES + 5;   // full, empty, tfull x2, tempty x2, drain
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;   // slack to align the base to 1024
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_B % 1024 == 0 && A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms");

constexpr uint32_t kIdesc = idesc_f16_f32(BM, BN);

struct GemmArgs {
  int num_m_tiles;   // tiles along rows of W
  int num_n_tiles;   // tiles along rows of X
  int k_blocks;      // K / BK
  int64_t T;         // rows of X
  int64_t n_rows;    // rows of W
  float* y;          // [n_rows][T]
  int* status;
};

__device__ __forceinline__ void decode_tile(int tile, const GemmArgs& p, int& nt, int& mt) {
  nt = tile / p.num_m_tiles;
  mt = tile - nt * p.num_m_tiles;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_ref(const __grid_constant__ CUtensorMap tmap_a,
               const __grid_constant__ CUtensorMap tmap_b, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_tfull = bar_empty + 8 * STAGES;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, kEpilogueThreads);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = p.num_m_tiles * p.num_n_tiles;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, fills = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        int nt, mt;
        decode_tile(tile, p, nt, mt);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status,
                                 kDevTimeoutEmpty)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
          tma_load_2d(sbase + OFF_A + stage * A_BYTES, &tmap_a, fb, kb * BK, mt * BM);
          tma_load_2d(sbase + OFF_B + stage * B_BYTES, &tmap_b, fb, kb * BK, nt * BN);
          ++fills;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every copy already issued land before shared memory is released.
        for (uint32_t s = 0; s < STAGES && s < fills; ++s) {
          const uint32_t n_s = (fills - s + STAGES - 1) / STAGES;   // fills of stage s
          mbar_wait_bounded(bar_full + 8 * s, (n_s - 1u) & 1u, nullptr, p.status,
                            kDevTimeoutDrain, kDrainLimitNs);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true, issued = false;
      int it = 0;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++it) {
        const uint32_t acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_bounded(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag, p.status,
                               kDevTimeoutTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait_bounded(bar_full + 8 * stage, phase, abort_flag, p.status,
                                 kDevTimeoutFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sbase + OFF_A + stage * A_BYTES;
          const uint32_t b_addr = sbase + OFF_B + stage * B_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            umma_f16(d_tmem, smem_desc_sw128(a_addr + 32 * k), smem_desc_sw128(b_addr + 32 * k),
                     kIdesc, (kb | k) != 0 ? 1u : 0u);
          }
          issued = true;
          umma_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(bar_tfull + 8 * acc);
      }
      if (!ok && issued) {
        // Wait for the MMAs in flight before TMEM is released.
        umma_commit(bar_drain);
        mbar_wait_bounded(bar_drain, 0, nullptr, p.status, kDevTimeoutDrain, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp;               // TMEM lane quarter (warps 0-3)
    const int row = q * 32 + lane;    // tile row
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
      int nt, mt;
      decode_tile(tile, p, nt, mt);
      const uint32_t acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      // tcgen05.ld is warp-collective: decide together and reconverge.
      const bool ready = __all_sync(0xFFFFFFFFu,
                                    mbar_wait_bounded(bar_tfull + 8 * acc, acc_phase, abort_flag,
                                                      p.status, kDevTimeoutTmemFull));
      if (!ready) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      const int64_t grow = static_cast<int64_t>(mt) * BM + row;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c * 32, v);
        tmem_ld_wait();
        if (grow < p.n_rows) {
          float* yr = p.y + grow * p.T;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t col = static_cast<int64_t>(nt) * BN + c * 32 + j;
            if (col < p.T) yr[col] = __uint_as_float(v[j]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar_tempty + 8 * acc);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- CTA-pair error GEMM
// The error GEMM proper.  A cluster of two CTAs (one per SM) owns a pair tile
// of 256 residual rows x 256 tokens; the even CTA issues
// tcgen05.mma.cta_group::2 (M 256, N 256, K 16), which reads A from both
// CTAs' shared memories (128 rows each) and B likewise (128 tokens each) and
// leaves each CTA's 128 rows x 256 tokens in its own TMEM.  Per SM and K step
// of 64 this moves 32 KB from L2 into shared memory for 4.2 MFLOP (a single
// CTA with M 128 needs 48 KB), and 6 stages fit instead of 4.
//
//   warp 4 (both CTAs)  TMA producer: own 128 residual rows and own 128
//                       tokens of X into its stage; completion is counted on
//                       the even CTA's `full` barrier;
//   warp 5              TMEM owner in both CTAs (pair allocation of 512
//                       columns: two 256-column accumulators); in the even CTA
//                       lane 0 issues the MMAs and commits to `empty` (both
//                       CTAs: their stages are free) and `tfull` (both CTAs:
//                       the accumulator is ready);
//   warps 0-3 (both)    epilogue as in k_gemm, then one arrival per thread on
//                       the even CTA's `tempty` (256 arrivals free it).
//
// Tile scheduling: the even CTA's producer takes the pair's next tile from a
// global counter (atomicAdd), so the tiles in progress on all pairs at any
// time are about 74 consecutive ones of the tile order, however much pairs
// drift apart over a long launch (with a fixed assignment, pair p taking
// tiles p, p + 74, ..., the pairs drift, and the L2 reuse the tile order is
// built for fades on the large workloads).  The id is published into a ring
// of kTileIdSlots slots in both CTAs' shared memory (tid_full); its readers
// -- the even CTA's MMA thread and epilogue warps, the odd CTA's producer and
// epilogue warps -- release the slot on the even CTA's tid_empty.  Id -1 ends
// the sequence.
//
// Teardown: each producer waits until every stage it filled was released
// (so no MMA still reads its shared memory and no commit still targets its
// barriers), then both CTAs meet at a cluster barrier before TMEM is freed and
// either CTA exits.
constexpr int PM = 128;                 // rows per CTA
constexpr int PN = 256;                 // tokens per pair tile
constexpr int PSTAGES = 6;
constexpr uint32_t PA_BYTES = PM * BK * 2;        // 16 KB
constexpr uint32_t PB_BYTES = (PN / 2) * BK * 2;  // 16 KB (this CTA's half of the tokens)
constexpr uint32_t P_OFF_A = 0;
constexpr uint32_t P_OFF_B = P_OFF_A + PSTAGES * PA_BYTES;
constexpr int kTileIdSlots = 4;
// Readers of a published tile id: the even CTA's MMA thread and 4 epilogue
// warps, the odd CTA's producer and 4 epilogue warps.
constexpr uint32_t kTileIdReaders = 1 + kEpilogueWarps + 1 + kEpilogueWarps;
constexpr uint32_t P_OFF_BAR = P_OFF_B + PSTAGES * PB_BYTES;
// full, empty, tfull x2, tempty x2, drain, tid_full, tid_empty
constexpr uint32_t P_NUM_BARS = 2 * PSTAGES + 5 + 2 * kTileIdSlots;
constexpr uint32_t P_OFF_MISC = P_OFF_BAR + P_NUM_BARS * 8;
constexpr uint32_t P_OFF_TID = P_OFF_MISC + 16;   // tile id ring (int per slot)
constexpr uint32_t P_SMEM_BYTES = P_OFF_TID + 4 * kTileIdSlots + 1024;
static_assert(P_SMEM_BYTES <= 232448, "shared memory budget");
static_assert(P_OFF_B % 1024 == 0 && PA_BYTES % 1024 == 0 && PB_BYTES % 1024 == 0,
              "swizzle atoms");
constexpr uint32_t kIdescPair = idesc_f16_f32(2 * PM, PN);
constexpr uint32_t kPairTmemCols = 512;

struct PairArgs {
  int num_mp;        // pair tiles along residual rows (256 rows each)
  int num_n_tiles;   // column tiles (256 tokens, or 256 channels for the Gram form)
  int num_alpha;     // grid points
  int k_blocks;      // K / 64
  int64_t n_pad;     // rows of the residual and partials layout (multiple of 256)
  float* partials;   // [alpha][n_tiles][n_pad]
  int* status;
  const __half* delta;   // Gram form: the residual [alpha][n_pad][K] (the epilogue's weights)
  int64_t K;             // Gram form: channels (columns of Gs and of delta)
  int group_rows;        // tile order: row tiles per group (see pair_tile_order)
  int keep_rows;         // 1: load residual tiles as evict_last and B as evict_first
                         // in L2 (a group's row tiles are the data read again); 0: no
                         // priority
  unsigned int* tile_counter;   // next tile to hand out (zeroed before the launch)
};

// kGram: the B operand is Gs (K x K) instead of X, and the epilogue forms
// sum_j E[n][j] * delta[n][j] over its 256 columns instead of sum E^2.
template <bool kGram>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_gemm_err_pair(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b, const PairArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + P_OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * PSTAGES;
  const uint32_t bar_tfull = bar_empty + 8 * PSTAGES;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;
  const uint32_t bar_tid_full = bar_drain + 8;
  const uint32_t bar_tid_empty = bar_tid_full + 8 * kTileIdSlots;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + P_OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P_OFF_MISC + 4);
  volatile int* tile_ids = reinterpret_cast<volatile int*>(smem + P_OFF_TID);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 2 * kEpilogueThreads);
    }
    mbar_init(bar_drain, 1);
    for (int s = 0; s < kTileIdSlots; ++s) {
      mbar_init(bar_tid_full + 8 * s, 1);
      mbar_init(bar_tid_empty + 8 * s, kTileIdReaders);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), kPairTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = p.num_mp * p.num_n_tiles * p.num_alpha;
  // Tile order (grid point, group of group_rows row tiles, column tile, row
  // tile in the group): the pairs working at one time share a few residual
  // row tiles and a few column tiles of X (or Gs), each read from HBM about
  // once per group.  group_rows = 1 walks every column tile of one row tile
  // before the next (X stays in L2 when it fits there).
  auto decode = [&](int tile, int& a, int& nt, int& mp) {
    const int per_alpha = p.num_mp * p.num_n_tiles;
    a = tile / per_alpha;
    const int rem = tile - a * per_alpha;
    const int per_group = p.group_rows * p.num_n_tiles;
    const int g = rem / per_group;
    const int r2 = rem - g * per_group;
    const int rows = min(p.group_rows, p.num_mp - g * p.group_rows);
    nt = r2 / rows;
    mp = g * p.group_rows + (r2 - nt * rows);
  };
  // The pair's i-th tile id (ring slot i % kTileIdSlots): published by the
  // even CTA's producer, read here by every other role.  A reader releases
  // the slot on the even CTA's tid_empty (one arrival per reading thread or
  // warp).  Returns -1 at the end of the sequence, -2 if the wait gave up.
  auto read_tile = [&](int i, bool arrive) -> int {
    const int slot = i % kTileIdSlots;
    if (!mbar_wait_cluster_bounded(bar_tid_full + 8 * slot,
                                   static_cast<uint32_t>((i / kTileIdSlots) & 1), abort_flag,
                                   p.status, kDevTimeoutTileId))
      return -2;
    const int t = tile_ids[slot];
    if (arrive) mbar_arrive_cluster(map_shared(bar_tid_empty + 8 * slot, 0));
    return t;
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        int tile;
        if (leader) {
          // Take the next tile and publish it to both CTAs once the slot's
          // previous id has been read by all of its readers.
          const int slot = i % kTileIdSlots;
          if (i >= kTileIdSlots &&
              !mbar_wait_cluster_bounded(bar_tid_empty + 8 * slot,
                                         static_cast<uint32_t>((i / kTileIdSlots - 1) & 1),
                                         abort_flag, p.status, kDevTimeoutTileId)) {
            ok = false;
            break;
          }
          tile = static_cast<int>(atomicAdd(p.tile_counter, 1u));
          if (tile >= total_tiles) tile = -1;
          const uint32_t id_addr = sbase + P_OFF_TID + 4 * slot;
          tile_ids[slot] = tile;
          st_shared_cluster_u32(map_shared(id_addr, 1), static_cast<uint32_t>(tile));
          mbar_arrive_cluster(bar_tid_full + 8 * slot);                    // own CTA
          mbar_arrive_cluster(map_shared(bar_tid_full + 8 * slot, 1));     // the odd CTA
        } else {
          tile = read_tile(i, true);
          if (tile == -2) ok = false;
        }
        if (tile < 0) break;
        int a, nt, mp;
        decode(tile, a, nt, mp);
        const uint64_t pol_a = p.keep_rows ? l2_policy_evict_last() : l2_policy_evict_normal();
        const uint64_t pol_b = p.keep_rows ? l2_policy_evict_first() : l2_policy_evict_normal();
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status,
                                 kDevTimeoutEmpty)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = bar_full + 8 * stage;
          if (leader) mbar_arrive_expect_tx(fb_local, 2 * (PA_BYTES + PB_BYTES));
          const uint32_t fb = map_shared(fb_local, 0);
          tma_load_3d_pair_hint(sbase + P_OFF_A + stage * PA_BYTES, &tmap_a, fb, kb * BK,
                                mp * 2 * PM + static_cast<int>(rank) * PM, a, pol_a);
          tma_load_2d_pair_hint(sbase + P_OFF_B + stage * PB_BYTES, &tmap_b, fb, kb * BK,
                                nt * PN + static_cast<int>(rank) * (PN / 2), pol_b);
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Tail: wait until every stage this CTA filled has been released by the
      // MMAs (a stage never filled passes at once).
      for (int i = 0; i < PSTAGES; ++i) {
        mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, nullptr, p.status, kDevTimeoutDrain,
                          ok ? kWaitLimitNs : kDrainLimitNs);
        if (++stage == PSTAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true, issued = false;
      for (int it = 0; ok; ++it) {
        const int tile = read_tile(it, true);
        if (tile == -2) ok = false;
        if (tile < 0) break;
        const uint32_t acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_bounded(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag, p.status,
                               kDevTimeoutTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * PN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait_bounded(bar_full + 8 * stage, phase, abort_flag, p.status,
                                 kDevTimeoutFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sbase + P_OFF_A + stage * PA_BYTES;
          const uint32_t b_addr = sbase + P_OFF_B + stage * PB_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            umma_f16_pair(d_tmem, smem_desc_sw128(a_addr + 32 * k),
                          smem_desc_sw128(b_addr + 32 * k), kIdescPair, (kb | k) != 0 ? 1u : 0u);
          }
          issued = true;
          umma_commit_pair(bar_empty + 8 * stage, 0x3);
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit_pair(bar_tfull + 8 * acc, 0x3);
      }
      if (!ok && issued) {
        // Wait for the MMAs in flight before TMEM or either CTA's stages go away.
        umma_commit_pair(bar_drain, 0x1);
        mbar_wait_bounded(bar_drain, 0, nullptr, p.status, kDevTimeoutDrain, kDrainLimitNs);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp;               // TMEM lane quarter (warps 0-3)
    const int row = q * 32 + lane;    // row within this CTA's 128
    const uint32_t tempty_leader = map_shared(bar_tempty, 0);
    for (int it = 0;; ++it) {
      const int tile = read_tile(it, false);
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_shared(bar_tid_empty + 8 * (it % kTileIdSlots), 0));
      if (__any_sync(0xFFFFFFFFu, tile < 0)) break;
      int a, nt, mp;
      decode(tile, a, nt, mp);
      const uint32_t acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      // tcgen05.ld is warp-collective: decide together and reconverge.
      const bool ready = __all_sync(0xFFFFFFFFu,
                                    mbar_wait_bounded(bar_tfull + 8 * acc, acc_phase, abort_flag,
                                                      p.status, kDevTimeoutTmemFull));
      if (!ready) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * PN;
      float sum0 = 0.f, sum1 = 0.f;
      const __half* drow =
          kGram ? p.delta + (static_cast<int64_t>(a) * p.n_pad + static_cast<int64_t>(mp) * 2 * PM +
                             static_cast<int64_t>(rank) * PM + row) * p.K
                : nullptr;
#pragma unroll 1
      for (int c = 0; c < PN / 32; ++c) {
        uint4 dv[4];
        const int64_t j0 = static_cast<int64_t>(nt) * PN + c * 32;   // Gram: first column
        const bool in = kGram && j0 < p.K;   // K % 64 == 0: a 32-column chunk is all in or out
        if (in) {
#pragma unroll
          for (int i = 0; i < 4; ++i) dv[i] = __ldg(reinterpret_cast<const uint4*>(drow + j0) + i);
        }
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c * 32, v);
        tmem_ld_wait();
        if (kGram) {
          if (in) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __half2* h = reinterpret_cast<const __half2*>(&dv[i]);
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const float2 d = __half22float2(h[t]);
                sum0 = fmaf(__uint_as_float(v[8 * i + 2 * t]), d.x, sum0);
                sum1 = fmaf(__uint_as_float(v[8 * i + 2 * t + 1]), d.y, sum1);
              }
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float e0 = __uint_as_float(v[j]);
            const float e1 = __uint_as_float(v[j + 1]);
            sum0 = fmaf(e0, e0, sum0);
            sum1 = fmaf(e1, e1, sum1);
          }
        }
      }
      tc_fence_before();
      mbar_arrive_cluster(tempty_leader + 8 * acc);
      p.partials[(static_cast<int64_t>(a) * p.num_n_tiles + nt) * p.n_pad +
                 static_cast<int64_t>(mp) * 2 * PM + static_cast<int64_t>(rank) * PM + row] =
          sum0 + sum1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Error path only: give copies already issued time to land before the
    // pair's shared memory is released.
    const unsigned long long t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  cluster_sync();   // neither CTA leaves while the other may still touch it
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kPairTmemCols);
  }
}

__global__ void k_wait_selftest(unsigned long long limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar_storage;
  const uint32_t bar = smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing ever arrives on this barrier: the wait must give up.
    mbar_wait_bounded(bar, 0, nullptr, status, kDevTimeoutSelfTest, limit_ns);
  }
}

// ---------------------------------------------------------------- host side
EncodeTiledFn encode_fn() { return tensor_map_encoder(); }

// fp16 tensor [depth][rows][cols] (cols contiguous), box 64 x box_rows (x 1),
// 128-byte swizzle; depth 1 gives a 2-D map.
bool make_tmap_f16(CUtensorMap* m, const void* base, int64_t depth, int64_t rows, int64_t cols,
                   int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(depth)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                                 static_cast<cuuint64_t>(cols) * 2 * static_cast<cuuint64_t>(rows)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint32_t rank = depth > 1 ? 3 : 2;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_ref(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& args,
                       cudaStream_t st) {
  LaunchFacts lf;
  cudaError_t e = launch_facts(reinterpret_cast<const void*>(k_gemm_ref), kThreads,
                               static_cast<int>(SMEM_BYTES), &lf);
  if (e != cudaSuccess) return e;
  const int total = args.num_m_tiles * args.num_n_tiles;
  const int grid = total < lf.sms ? total : lf.sms;
  k_gemm_ref<<<grid, kThreads, SMEM_BYTES, st>>>(ta, tb, args);
  return cudaGetLastError();
}

// Residual [alpha][n_pad][K]: box 64 x 128 (one CTA's rows of a pair tile).
bool make_residual_tmap(CUtensorMap* ta, const __half* delta, int64_t K, int64_t n_pad,
                        int n_alpha) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(n_pad),
                              static_cast<cuuint64_t>(n_alpha)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2,
                                 static_cast<cuuint64_t>(K) * 2 * static_cast<cuuint64_t>(n_pad)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(PM), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(delta), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kGram>
cudaError_t launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const PairArgs& a,
                        cudaStream_t st) {
  // One pair per co-resident cluster slot (persistent), at most one per tile.
  const int64_t tiles = static_cast<int64_t>(a.num_mp) * a.num_n_tiles * a.num_alpha;
  int max_clusters = 0;
  cudaError_t e = cluster_facts(reinterpret_cast<const void*>(k_gemm_err_pair<kGram>), kThreads,
                                static_cast<int>(P_SMEM_BYTES), &max_clusters);
  if (e != cudaSuccess) return e;
  const int clusters = std::min(device_sm_count() / 2, max_clusters);
  const int pairs = static_cast<int>(std::min<int64_t>(clusters, tiles));
  if (a.tile_counter == nullptr) return cudaErrorInvalidValue;
  e = cudaMemsetAsync(a.tile_counter, 0, sizeof(unsigned int), st);
  if (e != cudaSuccess) return e;
  k_gemm_err_pair<kGram><<<2 * pairs, kThreads, P_SMEM_BYTES, st>>>(ta, tb, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_reference(const __half* W, int64_t N, const __half* X, int64_t T,
                                  int64_t K, float* y, int* status, cudaStream_t st) {
  CUtensorMap ta, tb;
  if (!make_tmap_f16(&ta, W, 1, N, K, BM) || !make_tmap_f16(&tb, X, 1, T, K, BN))
    return cudaErrorInvalidValue;
  GemmArgs a{};
  a.num_m_tiles = static_cast<int>(ceil_div(N, BM));
  a.num_n_tiles = static_cast<int>(ceil_div(T, BN));
  a.k_blocks = static_cast<int>(K / BK);
  a.T = T;
  a.n_rows = N;
  a.y = y;
  a.status = status;
  return launch_ref(ta, tb, a, st);
}

// Row tiles per group of the tile order.  When the B operand (X, or Gs) fits
// comfortably in L2 it stays there, and one row tile at a time (all its column
// tiles) reads each residual tile once.  Otherwise as many row tiles as fit
// in an L2 budget share each column tile of B, so B is read once per group;
// their loads then carry an L2 priority that keeps the group's residual
// tiles over B's (measured on W 28672 x 8192, T 8192: DRAM reads 57.5 ->
// 55.4 GB per launch).  Ordering by groups of B's column tiles instead (B
// kept, the residual streaming past once per group) was measured too: it
// read more (55.1 to 75.7 GB), with or without the priorities.
static void pair_tile_order(int64_t b_rows, int64_t K, int num_mp, int* group_rows,
                            int* keep_rows) {
  constexpr int64_t kL2Budget = 48ll << 20;   // of the 126 MB L2
  *group_rows = 1;
  *keep_rows = 0;
  if (b_rows * K * 2 <= kL2Budget) return;
  const int64_t row_tile_bytes = 2ll * PM * K * 2;   // one 256-row residual tile
  const int64_t g = std::max<int64_t>(1, kL2Budget / row_tile_bytes);
  *group_rows = static_cast<int>(std::min<int64_t>(g, num_mp));
  *keep_rows = 1;
}

cudaError_t launch_gemm_error(const __half* delta, const __half* X, int64_t T, int64_t K,
                              int64_t n_pad, int n_alpha, float* partials, int* status,
                              unsigned int* tile_counter, cudaStream_t st) {
  if (n_pad % (2 * PM) != 0) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_residual_tmap(&ta, delta, K, n_pad, n_alpha)) return cudaErrorInvalidValue;
  // X [T][K]: box 64 x 128 (this CTA's half of a 256-token tile; tokens past
  // T read as zeros).
  if (!make_tmap_f16(&tb, X, 1, T, K, PN / 2)) return cudaErrorInvalidValue;
  PairArgs a{};
  a.num_mp = static_cast<int>(n_pad / (2 * PM));
  a.num_n_tiles = static_cast<int>(ceil_div(T, PN));
  a.num_alpha = n_alpha;
  a.k_blocks = static_cast<int>(K / BK);
  a.n_pad = n_pad;
  a.partials = partials;
  a.status = status;
  pair_tile_order(T, K, a.num_mp, &a.group_rows, &a.keep_rows);
  a.tile_counter = tile_counter;
  return launch_pair<false>(ta, tb, a, st);
}

cudaError_t launch_gemm_error_gram(const __half* delta, const __half* Gs, int64_t K,
                                   int64_t n_pad, int n_alpha, float* partials, int* status,
                                   unsigned int* tile_counter, cudaStream_t st) {
  if (n_pad % (2 * PM) != 0 || K % BK != 0) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_residual_tmap(&ta, delta, K, n_pad, n_alpha)) return cudaErrorInvalidValue;
  // Gs [K][K] (symmetric): B rows are its columns; box 64 x 128.
  if (!make_tmap_f16(&tb, Gs, 1, K, K, PN / 2)) return cudaErrorInvalidValue;
  PairArgs a{};
  a.num_mp = static_cast<int>(n_pad / (2 * PM));
  a.num_n_tiles = static_cast<int>(ceil_div(K, PN));
  a.num_alpha = n_alpha;
  a.k_blocks = static_cast<int>(K / BK);
  a.n_pad = n_pad;
  a.partials = partials;
  a.status = status;
  a.delta = delta;
  a.K = K;
  pair_tile_order(K, K, a.num_mp, &a.group_rows, &a.keep_rows);
  a.tile_counter = tile_counter;
  return launch_pair<true>(ta, tb, a, st);
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, int* status, cudaStream_t st) {
  k_wait_selftest<<<1, 32, 0, st>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace awq
