// Host-side launchers shared between the C ABI (awq_api.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <nvtx3/nvToolsExt.h>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace awq {

// NVTX ranges on the host thread that enqueues the library's work: a tool
// (Nsight Compute with --nvtx) attributes each kernel to the ranges open at
// its launch, e.g. awq_search_layer/error_gemm.  With no tool attached a push
// or pop does nothing.
class NvtxScope {
 public:
  explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
  ~NvtxScope() { nvtxRangePop(); }
  NvtxScope(const NvtxScope&) = delete;
  NvtxScope& operator=(const NvtxScope&) = delete;
};

// Sibling ranges in sequence: next() closes the open one and opens another.
class NvtxStages {
 public:
  NvtxStages() = default;
  ~NvtxStages() {
    if (open_) nvtxRangePop();
  }
  void next(const char* name) {
    close();
    nvtxRangePushA(name);
    open_ = true;
  }
  void close() {
    if (open_) nvtxRangePop();
    open_ = false;
  }
  NvtxStages(const NvtxStages&) = delete;
  NvtxStages& operator=(const NvtxStages&) = delete;

 private:
  bool open_ = false;
};


// Device status codes written to the per-call status word.
enum DeviceError : int {
  kDevOk = 0,
  kDevTimeoutFull = 1,      // producer data never arrived
  kDevTimeoutEmpty = 2,     // a stage was never released
  kDevTimeoutAReady = 3,    // dequantized operand never arrived
  kDevTimeoutTmemFull = 4,  // accumulator never completed
  kDevTimeoutTmemEmpty = 5, // accumulator never drained
  kDevTimeoutDrain = 6,     // in-flight copies/MMAs did not finish on abort
  kDevTimeoutSelfTest = 7,  // the self-test wait expired (expected there)
  kDevNonFinite = 8,        // a grid point's loss is not finite: X or W holds inf/NaN
  kDevTimeoutTileId = 9,    // a tile id was never published, or its slot never released
};

constexpr int kMaxWeights = 16;
constexpr int kMaxGrid = 64;

// ---- GEMM geometry (one CTA tile = 128 weight rows x 256 tokens; the error
// GEMM runs on CTA pairs, so its row space is padded to 256-row pair tiles)
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kTileK = 64;
constexpr int kPairRows = 2 * kTileM;

// Map from the padded "virtual row" space used by the error GEMM (every
// weight's rows start on a multiple of kTileM) to the compact row order of
// the result (weights concatenated).
struct RowMap {
  int n_w;
  int64_t pad_off[kMaxWeights];   // first virtual row of weight i
  int64_t rows[kMaxWeights];      // N_i
  int64_t cum[kMaxWeights];       // first compact row of weight i
};

// ---- statistics and scales (awq_stats.cu)
// Largest token count of the exact statistic: the 64-bit sums stay below
// 2^62, and the top two bits flag channels that held an infinity or a NaN.
constexpr int64_t kMaxStatTokens = int64_t(1) << 22;
// acc: K 64-bit words of scratch (zeroed here, on the stream); status: a
// device int that receives a code if a bounded wait expired, nullable.  If
// status is the word right after the sums (acc + K) it is zeroed here with
// them; otherwise the caller zeroes it.
cudaError_t launch_stats_accumulate(const __half* X, int64_t T, int64_t K,
                                    unsigned long long* acc, int* status, cudaStream_t st);
// range (nullable, 2 words zeroed by the caller): also the range of
// max(sX, 1e-4) over the channels, for launch_scales.  A non-zero *status
// (nullable) makes every sX NaN.
cudaError_t launch_stats_finalize(const unsigned long long* acc, int64_t T, int64_t K,
                                  double* sX, const int* status, cudaStream_t st,
                                  unsigned long long* range = nullptr);
// The same range for a caller-given sX (zeroes `range` first).
cudaError_t launch_sx_range(const double* sX, int64_t K, unsigned long long* range,
                            cudaStream_t st);
// s: fp32 [n_grid][K]; r (nullable): fp32 1/s [n_grid][K].
cudaError_t launch_scales(const double* sX, int64_t K, int n_grid,
                          const unsigned long long* range, float* s, float* r, cudaStream_t st);

// ---- group quantizer (awq_quant.cu)
// group: 64, 128, or -1 (one group per row); zero_point 1 (asymmetric) or 0
// (symmetric).  rowmm: scratch of n_alpha * N float2 (residual) or N float2
// (final), used only when group is -1.
// Search output: delta[a][row_off + n][k] = fp16(w - (q - z) * scale / s_k)
// for every grid point a, rows of weight i placed at row_off in a row space
// of n_pad rows.
cudaError_t launch_quant_residual(const __half* W, int64_t N, int64_t K, int bits, int group,
                                  int zero_point, const float* s_grid, const float* r_grid,
                                  int n_alpha, int64_t row_off, int64_t n_pad, __half* delta,
                                  float2* rowmm, cudaStream_t st);
// Result layout: packed codes, fp16 scales [N][K/group], u8 zeros [N][K/group]
// (one per row for group -1).  The scale vector is s + (*sel) * K when sel is
// non-null, else s.
cudaError_t launch_quant_final(const __half* W, int64_t N, int64_t K, int bits, int group,
                               int zero_point, const float* s, const int* sel, uint32_t* codes,
                               __half* scales, uint8_t* zeros, float2* rowmm, cudaStream_t st);
cudaError_t launch_unpack(const uint32_t* codes, int64_t N, int64_t K, int bits, uint8_t* q,
                          cudaStream_t st);

// ---- tcgen05 GEMMs (awq_gemm.cu)
// Y = W X^T in fp32, row-major [N][T].
cudaError_t launch_gemm_reference(const __half* W, int64_t N, const __half* X, int64_t T,
                                  int64_t K, float* y, int* status, cudaStream_t st);
// partials[a][n_tile][n_pad] = sum over the tile's tokens of (delta[a] X^T)^2
// for every grid point a (delta: fp16 [n_alpha][n_pad][K], n_pad a multiple
// of kPairRows).
// tile_counter: one device word of scratch (the launch zeroes it) from which
// the CTA pairs take their tiles.
cudaError_t launch_gemm_error(const __half* delta, const __half* X, int64_t T, int64_t K,
                              int64_t n_pad, int n_alpha, float* partials, int* status,
                              unsigned int* tile_counter, cudaStream_t st);
// Self-test of the bounded wait: one CTA waits on an mbarrier nothing
// arrives at; *status receives kDevTimeoutSelfTest after ~limit_ns.
cudaError_t launch_wait_selftest(unsigned long long limit_ns, int* status, cudaStream_t st);

// ---- deploy (awq_fold.cu)
// out[i][j] = fp16(fp32(V[i][j]) / s[i]) for V fp16 [rows][cols] (cols = 1:
// a vector); out may alias V.
cudaError_t launch_fold(const __half* V, int64_t rows, int64_t cols, const float* s, __half* out,
                        cudaStream_t st);

// ---- Gram form (awq_gram.cu)
// XT fp16 [K][Tp] (Tp = T rounded up to 64), G fp32 [K][K], mx one u32,
// Gs fp16 [K][K] = G * (c / T), *row_scale = T / c (c a power of two).
cudaError_t launch_gram_prepare(const __half* X, int64_t T, int64_t K, __half* XT, int64_t Tp,
                                float* G, unsigned int* mx, __half* Gs, double* row_scale,
                                int* status, cudaStream_t st, int* launches);
// partials[a][j_tile][n_pad] = sum over the tile's 256 columns j of
// (delta[a] Gs)[n][j] * delta[a][n][j] (Gs fp16 [K][K], symmetric).
cudaError_t launch_gemm_error_gram(const __half* delta, const __half* Gs, int64_t K,
                                   int64_t n_pad, int n_alpha, float* partials, int* status,
                                   unsigned int* tile_counter,
                                   cudaStream_t st);

// ---- decode product (awq_matvec.cu)
// y[m][n] = sum_k (code - zero) * scale * x[m][k], fp32 [M][N] (zeroed here),
// 1 <= M <= 16, INT4 or INT3 packed codes, group 64, 128 or -1, K % 64 == 0.
cudaError_t launch_w4_matvec(const uint32_t* codes, const __half* scales, const uint8_t* zeros,
                             int64_t N, int64_t K, int group, int bits, const __half* x, int M,
                             float* y, cudaStream_t st);

// ---- loss reduction (awq_reduce.cu)
// Number of 256-row chunks of the padded row space (chunk_sums holds
// n_alpha * loss_chunks(n_pad) * n_w doubles of scratch).
int64_t loss_chunks(int64_t n_pad);
// Also copies s_grid[best] (K floats) to s_out.  counter: one u32 of scratch,
// zeroed by the caller before the launch.  row_scale (nullable, device):
// factor on every row sum (the Gram form's T / c).  status: the call's device
// status word; a non-finite loss sets kDevNonFinite (unless a code is there).
cudaError_t launch_loss_reduce(const float* partials, int n_alpha, int n_tiles, int64_t n_pad,
                               int64_t T, const RowMap& map, int64_t n_total,
                               double* chunk_sums, double* row_losses, double* losses, int* best,
                               double* alpha_out, const float* s_grid, int64_t K, float* s_out,
                               unsigned int* counter, const double* row_scale, int* status,
                               cudaStream_t st);

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Launch facts of a kernel on the current device, looked up once per
// (device, kernel, threads, dynamic shared memory) and cached: the SM count
// and the blocks resident per SM.  The first lookup raises the kernel's
// dynamic shared memory limit to `smem`.
struct LaunchFacts {
  int sms;
  int per_sm;
};
cudaError_t launch_facts(const void* fn, int threads, int smem, LaunchFacts* out);
// Co-resident clusters of a kernel compiled with cluster dimensions (cached).
cudaError_t cluster_facts(const void* fn, int threads, int smem, int* max_clusters);
int device_sm_count();

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime
// (nullptr if the driver lacks it).  Linked statically, the library does not
// need the driver at load time.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// Launches kern with programmatic stream serialization: it may start before
// the stream's previous kernel ends, and must call grid_dependency_wait()
// before it touches anything that kernel writes.
template <typename Kern, typename... Args>
cudaError_t launch_dependent(Kern kern, dim3 grid, int threads, int64_t smem, cudaStream_t st,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename Kern, typename... Args>
cudaError_t launch_dependent(Kern kern, int64_t blocks, int threads, int64_t smem,
                             cudaStream_t st, Args... args) {
  return launch_dependent(kern, dim3(static_cast<unsigned>(blocks)), threads, smem, st, args...);
}

}  // namespace awq
