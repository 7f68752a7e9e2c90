// C ABI of libawq (declarations and contracts in include/awq.h).
//
// Host-side only: argument validation (before any launch), a per-device
// stream-ordered memory pool, and the ordering of the kernels that make up
// the scale search.  All arithmetic runs in the kernels of awq_stats.cu,
// awq_quant.cu, awq_gemm.cu and awq_reduce.cu.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <vector>

#include "awq.h"
#include "awq_bounds.cuh"
#include "awq_internal.h"

using namespace awq;

namespace {

thread_local char g_last_error[512] = "";

awq_status fail(awq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

awq_status ok() {
  g_last_error[0] = '\0';
  return AWQ_OK;
}

awq_status cuda_fail(cudaError_t e, const char* what) {
  const awq_status st = (e == cudaErrorMemoryAllocation) ? AWQ_ERR_OOM : AWQ_ERR_CUDA;
  return fail(st, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define AWQ_CUDA(expr, what)                 \
  do {                                       \
    cudaError_t e_ = (expr);                 \
    if (e_ != cudaSuccess) {                 \
      cleanup();                             \
      return cuda_fail(e_, what);            \
    }                                        \
  } while (0)

// True if p is device or managed memory usable on the current device.
bool device_ptr(const void* p) {
  if (p == nullptr) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  if (a.type != cudaMemoryTypeDevice) return false;
  int dev = -1;
  cudaGetDevice(&dev);
  return a.device == dev;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

awq_status check_dev(const void* p, const char* name, uintptr_t align) {
  if (p == nullptr) return fail(AWQ_ERR_INVALID, "%s is NULL", name);
  if (!aligned(p, align))
    return fail(AWQ_ERR_INVALID, "%s is not %d-byte aligned", name, static_cast<int>(align));
  if (!device_ptr(p))
    return fail(AWQ_ERR_INVALID, "%s is not device memory of the current device", name);
  return AWQ_OK;
}

// K must be a multiple of the group size, and of 64 for one group per row
// (the quantizer's 16-channel lanes and the GEMM's 64-channel K step).
bool k_fits(int64_t K, const awq_qconfig* cfg) {
  const int64_t g = cfg->group_size == -1 ? 64 : cfg->group_size;
  return K >= 1 && K % g == 0;
}

int64_t groups_per_row(int64_t K, const awq_qconfig* cfg) {
  return cfg->group_size == -1 ? 1 : K / cfg->group_size;
}

awq_status check_cfg(const awq_qconfig* cfg) {
  if (cfg == nullptr) return fail(AWQ_ERR_INVALID, "cfg is NULL");
  if (cfg->bits != 3 && cfg->bits != 4)
    return fail(AWQ_ERR_UNSUPPORTED, "bits=%d (supported: 3, 4)", cfg->bits);
  if (cfg->group_size != 64 && cfg->group_size != 128 && cfg->group_size != -1)
    return fail(AWQ_ERR_UNSUPPORTED, "group_size=%d (supported: 64, 128, -1 = per row)",
                cfg->group_size);
  if (cfg->zero_point != 0 && cfg->zero_point != 1)
    return fail(AWQ_ERR_UNSUPPORTED, "zero_point=%d (supported: 1 asymmetric, 0 symmetric)",
                cfg->zero_point);
  if (cfg->n_grid < 1 || cfg->n_grid > kMaxGrid)
    return fail(AWQ_ERR_INVALID, "n_grid=%d (1..%d)", cfg->n_grid, kMaxGrid);
  return AWQ_OK;
}

// ---------------------------------------------------------------- memory pool
cudaMemPool_t pool_for_current_device(cudaError_t* err) {
  static std::mutex mu;
  static std::map<int, cudaMemPool_t> pools;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  auto it = pools.find(dev);
  if (it != pools.end()) return it->second;
  cudaMemPoolProps props;
  memset(&props, 0, sizeof(props));
  props.allocType = cudaMemAllocationTypePinned;
  props.handleTypes = cudaMemHandleTypeNone;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  cudaMemPool_t pool = nullptr;
  *err = cudaMemPoolCreate(&pool, &props);
  if (*err != cudaSuccess) return nullptr;
  uint64_t keep = ~0ull;   // keep freed blocks cached for the next call
  cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
  pools[dev] = pool;
  return pool;
}

// Allocation-failure injection (awq_inject_allocation_failures): the next
// g_alloc_skip pool allocations go through, then g_alloc_fail of them report
// cudaErrorMemoryAllocation without reaching the allocator.
std::mutex g_inject_mu;
int g_alloc_skip = 0, g_alloc_fail = 0;

bool injected_failure() {
  std::lock_guard<std::mutex> lock(g_inject_mu);
  if (g_alloc_fail <= 0) return false;
  if (g_alloc_skip > 0) {
    --g_alloc_skip;
    return false;
  }
  --g_alloc_fail;
  return true;
}

cudaError_t pool_alloc(void** p, size_t bytes, cudaStream_t st) {
  cudaError_t e;
  cudaMemPool_t pool = pool_for_current_device(&e);
  if (pool == nullptr) return e;
  if (injected_failure()) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMallocFromPoolAsync(p, bytes < 256 ? 256 : bytes, pool, st);
}

// Carves 256-byte-aligned pieces out of one allocation.
struct Carver {
  size_t off = 0;
  template <typename T>
  size_t take(int64_t count) {
    const size_t at = off;
    off += (static_cast<size_t>(count) * sizeof(T) + 255) & ~static_cast<size_t>(255);
    return at;
  }
};

// Pinned host mirror of the small outputs, recycled across calls.
struct HostMirror {
  int best;
  int status;
  double alpha;
  double losses[kMaxGrid];
};

std::atomic<int> g_stage_timing{0};

std::mutex g_mirror_mu;
std::vector<HostMirror*> g_mirrors;

HostMirror* take_mirror() {
  {
    std::lock_guard<std::mutex> lock(g_mirror_mu);
    if (!g_mirrors.empty()) {
      HostMirror* m = g_mirrors.back();
      g_mirrors.pop_back();
      return m;
    }
  }
  HostMirror* m = nullptr;
  if (cudaMallocHost(reinterpret_cast<void**>(&m), sizeof(HostMirror)) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return m;
}

void give_mirror(HostMirror* m) {
  if (m == nullptr) return;
  std::lock_guard<std::mutex> lock(g_mirror_mu);
  g_mirrors.push_back(m);
}

}  // namespace

struct awq_result;
static void destroy_events(awq_result* r);

struct awq_result {
  cudaStream_t stream = nullptr;
  int n_grid = 0, n_w = 0, bits = 0, group = 0;
  int64_t K = 0, T = 0, n_total = 0;
  int64_t rows[kMaxWeights] = {};
  void* block = nullptr;
  HostMirror* host = nullptr;
  float* s = nullptr;
  float* s_grid = nullptr;
  int* best = nullptr;
  double* alpha = nullptr;
  double* losses = nullptr;
  double* row_losses = nullptr;
  int* status = nullptr;
  uint32_t* codes[kMaxWeights] = {};
  __half* scales[kMaxWeights] = {};
  uint8_t* zeros[kMaxWeights] = {};
  int launches = 0;                     // kernels this call enqueued
  cudaEvent_t ev[AWQ_NUM_STAGES + 1] = {};   // stage boundaries (timing enabled)
  bool timed = false;
};

static void destroy_events(awq_result* r) {
  for (int e = 0; e <= AWQ_NUM_STAGES; ++e)
    if (r->ev[e]) cudaEventDestroy(r->ev[e]);
}

namespace awq {
namespace {
// One synthetic out-of-range index at site 0 (no memory access): shows the
// record path of the bounds-checked build working.
__global__ void k_bounds_selftest() { (void)in_bounds(kSiteSelfTest, -1, 0); }
}  // namespace

AWQ_BOUNDS_READER(bounds_api)
}  // namespace awq

extern "C" {

int awq_abi_version(void) { return AWQ_ABI_VERSION; }

const char* awq_last_error(void) { return g_last_error; }

const char* awq_status_string(int status) {
  switch (status) {
    case AWQ_OK: return "AWQ_OK";
    case AWQ_ERR_INVALID: return "AWQ_ERR_INVALID";
    case AWQ_ERR_UNSUPPORTED: return "AWQ_ERR_UNSUPPORTED";
    case AWQ_ERR_CUDA: return "AWQ_ERR_CUDA";
    case AWQ_ERR_OOM: return "AWQ_ERR_OOM";
    case AWQ_ERR_TIMEOUT: return "AWQ_ERR_TIMEOUT";
    default: return "AWQ_ERR_UNKNOWN";
  }
}

int64_t awq_packed_words(int64_t N, int64_t K, int bits) {
  if (N < 0 || K <= 0) return -1;
  if (bits == 4) return (K % 8) ? -1 : N * (K / 8);
  if (bits == 3) return (K % 32) ? -1 : N * (3 * K / 32);
  return -1;
}

awq_status awq_stats(const void* X, int64_t T, int64_t K, double* sX, void* stream) {
  NvtxScope nvtx("awq_stats");
  if (T < 1) return fail(AWQ_ERR_INVALID, "T=%lld (must be >= 1)", static_cast<long long>(T));
  if (T > kMaxStatTokens)
    return fail(AWQ_ERR_INVALID,
                "T=%lld exceeds AWQ_MAX_STAT_TOKENS=%lld (the exact 64-bit channel sums)",
                static_cast<long long>(T), static_cast<long long>(kMaxStatTokens));
  if (K < 8 || K % 8) return fail(AWQ_ERR_INVALID, "K=%lld (must be a positive multiple of 8)",
                                  static_cast<long long>(K));
  if (K > (int64_t(1) << 31)) return fail(AWQ_ERR_INVALID, "K too large");
  awq_status st;
  if ((st = check_dev(X, "X", 16)) != AWQ_OK) return st;
  if ((st = check_dev(sX, "sX", 8)) != AWQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  auto cleanup = [&] {
    if (ws) cudaFreeAsync(ws, s);
  };
  // K 64-bit sums, then the status word of the bounded waits.
  AWQ_CUDA(pool_alloc(&ws, sizeof(unsigned long long) * (K + 1), s), "scratch allocation");
  auto* acc = static_cast<unsigned long long*>(ws);
  int* status = reinterpret_cast<int*>(acc + K);   // zeroed with the sums
  AWQ_CUDA(launch_stats_accumulate(static_cast<const __half*>(X), T, K, acc, status, s),
           "stats kernel");
  AWQ_CUDA(launch_stats_finalize(acc, T, K, sX, status, s), "stats finalize kernel");
  AWQ_CUDA(cudaFreeAsync(ws, s), "scratch release");
  return ok();
}

awq_status awq_scales(const double* sX, int64_t K, int n_grid, float* s_out, void* stream) {
  NvtxScope nvtx("awq_scales");
  if (K < 1 || K > (int64_t(1) << 31))
    return fail(AWQ_ERR_INVALID, "K=%lld", static_cast<long long>(K));
  if (n_grid < 1 || n_grid > kMaxGrid)
    return fail(AWQ_ERR_INVALID, "n_grid=%d (1..%d)", n_grid, kMaxGrid);
  awq_status st;
  if ((st = check_dev(sX, "sX", 8)) != AWQ_OK) return st;
  if ((st = check_dev(s_out, "s", 4)) != AWQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  auto cleanup = [&] {
    if (ws) cudaFreeAsync(ws, s);
  };
  AWQ_CUDA(pool_alloc(&ws, 2 * sizeof(unsigned long long), s), "scratch allocation");
  auto* range = static_cast<unsigned long long*>(ws);
  AWQ_CUDA(launch_sx_range(sX, K, range, s), "scale range kernel");
  AWQ_CUDA(launch_scales(sX, K, n_grid, range, s_out, nullptr, s), "scale kernel");
  AWQ_CUDA(cudaFreeAsync(ws, s), "scratch release");
  return ok();
}

awq_status awq_quantize_pack(const void* W, int64_t N, int64_t K, const float* s_vec,
                             const awq_qconfig* cfg, uint32_t* codes, void* scales,
                             uint8_t* zeros, void* stream) {
  NvtxScope nvtx("awq_quantize_pack");
  awq_status st;
  if ((st = check_cfg(cfg)) != AWQ_OK) return st;
  if (N < 0) return fail(AWQ_ERR_INVALID, "N=%lld", static_cast<long long>(N));
  if (!k_fits(K, cfg) || K > (int64_t(1) << 31))
    return fail(AWQ_ERR_INVALID,
                "K=%lld (must be a positive multiple of group_size=%d; of 64 for -1)",
                static_cast<long long>(K), cfg->group_size);
  if (N == 0) return ok();
  if ((st = check_dev(W, "W", 16)) != AWQ_OK) return st;
  if ((st = check_dev(s_vec, "s", 16)) != AWQ_OK) return st;
  if ((st = check_dev(codes, "codes", 4)) != AWQ_OK) return st;
  if ((st = check_dev(scales, "scales", 2)) != AWQ_OK) return st;
  if ((st = check_dev(zeros, "zeros", 1)) != AWQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;   // per-row min / max, for one group per row only
  auto cleanup = [&] {
    if (ws) cudaFreeAsync(ws, s);
  };
  if (cfg->group_size == -1)
    AWQ_CUDA(pool_alloc(&ws, sizeof(float2) * N, s), "scratch allocation");
  AWQ_CUDA(launch_quant_final(static_cast<const __half*>(W), N, K, cfg->bits, cfg->group_size,
                              cfg->zero_point, s_vec, nullptr, codes,
                              static_cast<__half*>(scales), zeros, static_cast<float2*>(ws), s),
           "quantize kernel");
  if (ws) {
    AWQ_CUDA(cudaFreeAsync(ws, s), "scratch release");
    ws = nullptr;
  }
  return ok();
}

awq_status awq_unpack_codes(const uint32_t* codes, int64_t N, int64_t K, int bits, uint8_t* q,
                            void* stream) {
  NvtxScope nvtx("awq_unpack_codes");
  if (awq_packed_words(N, K, bits) < 0)
    return fail(AWQ_ERR_INVALID, "invalid shape N=%lld K=%lld bits=%d",
                static_cast<long long>(N), static_cast<long long>(K), bits);
  if (N == 0) return ok();
  awq_status st;
  if ((st = check_dev(codes, "codes", 4)) != AWQ_OK) return st;
  if ((st = check_dev(q, "q", 1)) != AWQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto cleanup = [] {};
  AWQ_CUDA(launch_unpack(codes, N, K, bits, q, s), "unpack kernel");
  return ok();
}

awq_status awq_w4a16_matvec(const uint32_t* codes, const void* scales, const uint8_t* zeros,
                            int64_t N, int64_t K, const awq_qconfig* cfg, const void* x, int M,
                            float* y, void* stream) {
  NvtxScope nvtx("awq_w4a16_matvec");
  awq_status st;
  if ((st = check_cfg(cfg)) != AWQ_OK) return st;
  if (N < 1 || N > (int64_t(1) << 31) || !k_fits(K, cfg) || K % 64 || K > (int64_t(1) << 31))
    return fail(AWQ_ERR_INVALID, "N=%lld K=%lld (N >= 1; K a multiple of 64 and of the group)",
                static_cast<long long>(N), static_cast<long long>(K));
  if (M < 1 || M > 16) return fail(AWQ_ERR_INVALID, "M=%d (1..16)", M);
  if ((st = check_dev(codes, "codes", 16)) != AWQ_OK) return st;
  if ((st = check_dev(scales, "scales", 2)) != AWQ_OK) return st;
  if ((st = check_dev(zeros, "zeros", 1)) != AWQ_OK) return st;
  if ((st = check_dev(x, "x", 16)) != AWQ_OK) return st;
  if ((st = check_dev(y, "y", 4)) != AWQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto cleanup = [] {};
  AWQ_CUDA(launch_w4_matvec(codes, static_cast<const __half*>(scales), zeros, N, K,
                            cfg->group_size, cfg->bits, static_cast<const __half*>(x), M, y, s),
           "decode product kernel");
  return ok();
}

awq_status awq_fold_scale(const void* V, int64_t rows, int64_t cols, const float* s_vec,
                          void* out, void* stream) {
  NvtxScope nvtx("awq_fold_scale");
  if (rows < 1 || cols < 1 || rows > (int64_t(1) << 40) / cols)
    return fail(AWQ_ERR_INVALID, "rows=%lld cols=%lld (both >= 1)", static_cast<long long>(rows),
                static_cast<long long>(cols));
  awq_status st;
  if ((st = check_dev(V, "V", 2)) != AWQ_OK) return st;
  if ((st = check_dev(s_vec, "s", 4)) != AWQ_OK) return st;
  if ((st = check_dev(out, "out", 2)) != AWQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto cleanup = [] {};
  AWQ_CUDA(launch_fold(static_cast<const __half*>(V), rows, cols, s_vec,
                       static_cast<__half*>(out), s),
           "fold kernel");
  return ok();
}

awq_status awq_reference_output(const void* W, int64_t N, const void* X, int64_t T, int64_t K,
                                float* Y, int* status_dev, void* stream) {
  NvtxScope nvtx("awq_reference_output");
  if (N < 1 || T < 1 || K < 64 || K % 64)
    return fail(AWQ_ERR_INVALID, "N=%lld T=%lld K=%lld (N, T >= 1; K a positive multiple of 64)",
                static_cast<long long>(N), static_cast<long long>(T), static_cast<long long>(K));
  if (N > (int64_t(1) << 30) || T > (int64_t(1) << 30) || K > (int64_t(1) << 30) ||
      ceil_div(N, kTileM) * ceil_div(T, kTileN) > (int64_t(1) << 30))
    return fail(AWQ_ERR_INVALID, "shape too large");
  awq_status st;
  if ((st = check_dev(W, "W", 16)) != AWQ_OK) return st;
  if ((st = check_dev(X, "X", 16)) != AWQ_OK) return st;
  if ((st = check_dev(Y, "Y", 4)) != AWQ_OK) return st;
  if (status_dev != nullptr && (st = check_dev(status_dev, "status_dev", 4)) != AWQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto cleanup = [] {};
  AWQ_CUDA(launch_gemm_reference(static_cast<const __half*>(W), N, static_cast<const __half*>(X),
                                 T, K, Y, status_dev, s),
           "reference GEMM");
  return ok();
}

}  // extern "C"

// The search; gram: evaluate the loss in the Gram form d^T (X^T X) d.
static awq_status search_impl(const void* X, int64_t T, int64_t K, const double* sX,
                              const awq_weight* Ws, int n_w, const awq_qconfig* cfg, void* stream,
                              awq_result** out, bool gram) {
  if (out == nullptr) return fail(AWQ_ERR_INVALID, "out is NULL");
  *out = nullptr;
  awq_status st;
  if ((st = check_cfg(cfg)) != AWQ_OK) return st;
  if (T < 1) return fail(AWQ_ERR_INVALID, "T=%lld (must be >= 1)", static_cast<long long>(T));
  if (sX == nullptr && T > kMaxStatTokens)
    return fail(AWQ_ERR_INVALID,
                "T=%lld exceeds AWQ_MAX_STAT_TOKENS=%lld for the channel statistic (pass sX)",
                static_cast<long long>(T), static_cast<long long>(kMaxStatTokens));
  if (!k_fits(K, cfg))
    return fail(AWQ_ERR_INVALID,
                "K=%lld (must be a positive multiple of group_size=%d; of 64 for -1)",
                static_cast<long long>(K), cfg->group_size);
  if (Ws == nullptr || n_w < 1 || n_w > kMaxWeights)
    return fail(AWQ_ERR_INVALID, "n_w=%d (1..%d) with a non-NULL Ws", n_w, kMaxWeights);
  if ((st = check_dev(X, "X", 16)) != AWQ_OK) return st;
  if (sX != nullptr && (st = check_dev(sX, "sX", 8)) != AWQ_OK) return st;
  RowMap map{};
  map.n_w = n_w;
  int64_t n_pad = 0, n_total = 0;
  for (int i = 0; i < n_w; ++i) {
    if (Ws[i].N < 1)
      return fail(AWQ_ERR_INVALID, "Ws[%d].N=%lld (must be >= 1)", i,
                  static_cast<long long>(Ws[i].N));
    char name[32];
    snprintf(name, sizeof(name), "Ws[%d].W", i);
    if ((st = check_dev(Ws[i].W, name, 16)) != AWQ_OK) return st;
    map.pad_off[i] = n_pad;
    map.rows[i] = Ws[i].N;
    map.cum[i] = n_total;
    n_pad += ceil_div(Ws[i].N, kTileM) * kTileM;
    n_total += Ws[i].N;
  }
  const int64_t n_used = n_pad;                 // rows of the last weight's tiles
  n_pad = ceil_div(n_pad, kPairRows) * kPairRows;   // whole pair tiles for the error GEMM
  const int G = cfg->n_grid;
  const int64_t groups = groups_per_row(K, cfg);
  // Column tiles of the error GEMM: tokens, or channels in the Gram form.
  const int64_t n_tiles = ceil_div(gram ? K : T, kTileN);
  const int64_t Tp = ceil_div(T, kTileK) * kTileK;   // Gram form: tokens padded for X^T
  if (K > (int64_t(1) << 30) || T > (int64_t(1) << 30) || n_pad > (int64_t(1) << 30) ||
      (n_pad / kTileM) * n_tiles * G > (int64_t(1) << 30))
    return fail(AWQ_ERR_INVALID, "shape too large for one call");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  awq_result* r = new (std::nothrow) awq_result();
  if (r == nullptr) return fail(AWQ_ERR_OOM, "host allocation failed");
  void* ws = nullptr;
  auto cleanup = [&] {
    if (ws) cudaFreeAsync(ws, s);
    if (r) {
      if (r->block) cudaFreeAsync(r->block, s);
      give_mirror(r->host);
      destroy_events(r);
      delete r;
      r = nullptr;
    }
  };
  r->stream = s;
  r->n_grid = G;
  r->n_w = n_w;
  r->bits = cfg->bits;
  r->group = cfg->group_size;
  r->K = K;
  r->T = T;
  r->n_total = n_total;
  for (int i = 0; i < n_w; ++i) r->rows[i] = Ws[i].N;
  r->host = take_mirror();
  if (r->host == nullptr) {
    cleanup();
    return fail(AWQ_ERR_OOM, "pinned host allocation failed");
  }

  // Result block.
  Carver rc;
  const size_t o_s = rc.take<float>(K);
  const size_t o_sg = rc.take<float>(int64_t(G) * K);
  const size_t o_best = rc.take<int>(1);
  const size_t o_alpha = rc.take<double>(1);
  const size_t o_loss = rc.take<double>(G);
  const size_t o_rows = rc.take<double>(int64_t(G) * n_total);
  const size_t o_status = rc.take<int>(1);
  size_t o_codes[kMaxWeights], o_scales[kMaxWeights], o_zeros[kMaxWeights];
  for (int i = 0; i < n_w; ++i) {
    o_codes[i] = rc.take<uint32_t>(awq_packed_words(Ws[i].N, K, cfg->bits));
    o_scales[i] = rc.take<__half>(Ws[i].N * groups);
    o_zeros[i] = rc.take<uint8_t>(Ws[i].N * groups);
  }
  // Scratch block.
  Carver wc;
  const size_t o_acc = wc.take<unsigned long long>(K);
  const size_t o_sx = wc.take<double>(K);
  // scale range [2], loss counter, the error GEMM's tile counter
  const size_t o_rng = wc.take<unsigned long long>(4);
  const size_t o_r = wc.take<float>(int64_t(G) * K);
  const size_t o_d = wc.take<__half>(int64_t(G) * n_pad * K);
  const size_t o_pt = wc.take<float>(int64_t(G) * n_tiles * n_pad);
  const size_t o_cs = wc.take<double>(int64_t(G) * loss_chunks(n_pad) * n_w);
  int64_t max_rows = 0;
  for (int i = 0; i < n_w; ++i) max_rows = std::max<int64_t>(max_rows, Ws[i].N);
  const size_t o_mmr = wc.take<float2>(cfg->group_size == -1 ? int64_t(G) * max_rows : 1);
  const size_t o_xt = wc.take<__half>(gram ? K * Tp : 1);
  const size_t o_g32 = wc.take<float>(gram ? K * K : 1);
  const size_t o_gs = wc.take<__half>(gram ? K * K : 1);
  const size_t o_gmx = wc.take<unsigned int>(1);
  const size_t o_rsc = wc.take<double>(1);

  AWQ_CUDA(pool_alloc(&r->block, rc.off, s), "result allocation");
  AWQ_CUDA(pool_alloc(&ws, wc.off, s), "scratch allocation");
  char* rb = static_cast<char*>(r->block);
  char* wb = static_cast<char*>(ws);
  r->s = reinterpret_cast<float*>(rb + o_s);
  r->s_grid = reinterpret_cast<float*>(rb + o_sg);
  r->best = reinterpret_cast<int*>(rb + o_best);
  r->alpha = reinterpret_cast<double*>(rb + o_alpha);
  r->losses = reinterpret_cast<double*>(rb + o_loss);
  r->row_losses = reinterpret_cast<double*>(rb + o_rows);
  r->status = reinterpret_cast<int*>(rb + o_status);
  for (int i = 0; i < n_w; ++i) {
    r->codes[i] = reinterpret_cast<uint32_t*>(rb + o_codes[i]);
    r->scales[i] = reinterpret_cast<__half*>(rb + o_scales[i]);
    r->zeros[i] = reinterpret_cast<uint8_t*>(rb + o_zeros[i]);
  }
  auto* acc = reinterpret_cast<unsigned long long*>(wb + o_acc);
  auto* sx_ws = reinterpret_cast<double*>(wb + o_sx);
  auto* range = reinterpret_cast<unsigned long long*>(wb + o_rng);
  auto* r_ws = reinterpret_cast<float*>(wb + o_r);
  auto* delta = reinterpret_cast<__half*>(wb + o_d);
  auto* partials = reinterpret_cast<float*>(wb + o_pt);
  auto* chunk_sums = reinterpret_cast<double*>(wb + o_cs);
  auto* rowmm = reinterpret_cast<float2*>(wb + o_mmr);   // per-row min / max (group -1)
  auto* xt = reinterpret_cast<__half*>(wb + o_xt);        // Gram form scratch
  auto* g32 = reinterpret_cast<float*>(wb + o_g32);
  auto* gs = reinterpret_cast<__half*>(wb + o_gs);
  auto* gmx = reinterpret_cast<unsigned int*>(wb + o_gmx);
  auto* rsc = reinterpret_cast<double*>(wb + o_rsc);
  auto* counter = reinterpret_cast<unsigned int*>(range + 2);
  auto* tile_counter = reinterpret_cast<unsigned int*>(range + 3);
  const __half* Xh = static_cast<const __half*>(X);

  AWQ_CUDA(cudaMemsetAsync(r->status, 0, sizeof(int), s), "status reset");
  // Padding rows of the residual (between weights) must be exactly 0.
  for (int i = 0; i < n_w; ++i) {
    const int64_t pad_rows = ceil_div(Ws[i].N, kTileM) * kTileM - Ws[i].N;
    if (pad_rows == 0) continue;
    AWQ_CUDA(cudaMemset2DAsync(delta + (map.pad_off[i] + Ws[i].N) * K,
                               sizeof(__half) * n_pad * K, 0, sizeof(__half) * pad_rows * K, G,
                               s),
             "residual padding reset");
  }
  if (n_pad > n_used) {
    AWQ_CUDA(cudaMemset2DAsync(delta + n_used * K, sizeof(__half) * n_pad * K, 0,
                               sizeof(__half) * (n_pad - n_used) * K, G, s),
             "residual tail reset");
  }
  // Optional stage boundaries (awq_set_stage_timing): events on this stream.
  if (g_stage_timing.load()) {
    for (int e = 0; e <= AWQ_NUM_STAGES; ++e)
      AWQ_CUDA(cudaEventCreate(&r->ev[e]), "event creation");
    r->timed = true;
  }
  // Each stage is also an NVTX range (stats, scales, residual, error_gemm,
  // loss, final).
  NvtxStages nvtx_stage;
  static const char* const kStageNames[AWQ_NUM_STAGES] = {"stats", "scales", "residual",
                                                          "error_gemm", "loss", "final"};
  auto mark = [&](int e) -> cudaError_t {
    if (e < AWQ_NUM_STAGES) nvtx_stage.next(kStageNames[e]);
    else nvtx_stage.close();
    return r->timed ? cudaEventRecord(r->ev[e], s) : cudaSuccess;
  };
  AWQ_CUDA(mark(AWQ_STAGE_STATS), "event record");
  // 1. channel statistic (and the range of max(sX, 1e-4) for the scales)
  const double* sxp = sX;
  AWQ_CUDA(cudaMemsetAsync(range, 0, 3 * sizeof(unsigned long long), s), "range reset");
  if (sxp == nullptr) {
    AWQ_CUDA(launch_stats_accumulate(Xh, T, K, acc, r->status, s), "stats kernel");
    AWQ_CUDA(launch_stats_finalize(acc, T, K, sx_ws, r->status, s, range),
             "stats finalize kernel");
    r->launches += 3;   // zeroing, accumulation, finalize
    sxp = sx_ws;
  }
  AWQ_CUDA(mark(AWQ_STAGE_SCALES), "event record");
  // 2. scales (and their fp32 reciprocals) for every grid point
  if (sX != nullptr) {
    AWQ_CUDA(launch_sx_range(sX, K, range, s), "scale range kernel");
    r->launches += 1;
  }
  AWQ_CUDA(launch_scales(sxp, K, G, range, r->s_grid, r_ws, s), "scale kernel");
  r->launches += 1;
  AWQ_CUDA(mark(AWQ_STAGE_RESIDUAL), "event record");
  // 3. quantize every weight at every grid point; keep the fp16 residual
  for (int i = 0; i < n_w; ++i) {
    AWQ_CUDA(launch_quant_residual(static_cast<const __half*>(Ws[i].W), Ws[i].N, K, cfg->bits,
                                   cfg->group_size, cfg->zero_point, r->s_grid, r_ws, G,
                                   map.pad_off[i], n_pad, delta, rowmm, s),
             "quantize kernel (residual)");
    r->launches += cfg->group_size == -1 ? 2 : 1;
  }
  AWQ_CUDA(mark(AWQ_STAGE_ERROR_GEMM), "event record");
  // 4. error GEMM for every grid point: per-row sums of (residual X^T)^2, or
  //    in the Gram form sum_j (residual G)[n][j] residual[n][j] with G = X^T X
  if (gram) {
    AWQ_CUDA(launch_gram_prepare(Xh, T, K, xt, Tp, g32, gmx, gs, rsc, r->status, s,
                                 &r->launches),
             "Gram matrix");
    AWQ_CUDA(launch_gemm_error_gram(delta, gs, K, n_pad, G, partials, r->status, tile_counter, s),
             "error GEMM (Gram form)");
  } else {
    AWQ_CUDA(launch_gemm_error(delta, Xh, T, K, n_pad, G, partials, r->status, tile_counter, s),
             "error GEMM");
  }
  r->launches += 1;
  AWQ_CUDA(mark(AWQ_STAGE_LOSS), "event record");
  // 5. losses and argmin
  AWQ_CUDA(launch_loss_reduce(partials, G, static_cast<int>(n_tiles), n_pad, T, map, n_total,
                              chunk_sums, r->row_losses, r->losses, r->best, r->alpha,
                              r->s_grid, K, r->s, counter, gram ? rsc : nullptr, r->status, s),
           "loss reduction");
  r->launches += 1;
  AWQ_CUDA(mark(AWQ_STAGE_FINAL), "event record");
  // 6. final quantization at the chosen grid point (index read on the device)
  for (int i = 0; i < n_w; ++i) {
    AWQ_CUDA(launch_quant_final(static_cast<const __half*>(Ws[i].W), Ws[i].N, K, cfg->bits,
                                cfg->group_size, cfg->zero_point, r->s_grid, r->best,
                                r->codes[i], r->scales[i], r->zeros[i], rowmm, s),
             "quantize kernel (final)");
    r->launches += cfg->group_size == -1 ? 2 : 1;
  }
  AWQ_CUDA(mark(AWQ_NUM_STAGES), "event record");
  // 7. small outputs to pinned host memory
  AWQ_CUDA(cudaMemcpyAsync(r->host->losses, r->losses, sizeof(double) * G, cudaMemcpyDeviceToHost,
                           s),
           "loss copy");
  AWQ_CUDA(cudaMemcpyAsync(&r->host->best, r->best, sizeof(int), cudaMemcpyDeviceToHost, s),
           "index copy");
  AWQ_CUDA(cudaMemcpyAsync(&r->host->alpha, r->alpha, sizeof(double), cudaMemcpyDeviceToHost, s),
           "alpha copy");
  AWQ_CUDA(cudaMemcpyAsync(&r->host->status, r->status, sizeof(int), cudaMemcpyDeviceToHost, s),
           "status copy");
  AWQ_CUDA(cudaFreeAsync(ws, s), "scratch release");
  ws = nullptr;
  *out = r;
  return ok();
}

extern "C" {

awq_status awq_search_layer(const void* X, int64_t T, int64_t K, const double* sX,
                            const awq_weight* Ws, int n_w, const awq_qconfig* cfg, void* stream,
                            awq_result** out) {
  NvtxScope nvtx("awq_search_layer");
  return search_impl(X, T, K, sX, Ws, n_w, cfg, stream, out, false);
}

awq_status awq_search_layer_gram(const void* X, int64_t T, int64_t K, const double* sX,
                                 const awq_weight* Ws, int n_w, const awq_qconfig* cfg,
                                 void* stream, awq_result** out) {
  NvtxScope nvtx("awq_search_layer_gram");
  return search_impl(X, T, K, sX, Ws, n_w, cfg, stream, out, true);
}

awq_status awq_result_check(const awq_result* r) {
  if (r == nullptr) return fail(AWQ_ERR_INVALID, "result is NULL");
  if (r->host->status == kDevNonFinite)
    return fail(AWQ_ERR_INVALID,
                "X or W holds a non-finite value (a grid point's loss is not finite); "
                "the result is undefined");
  if (r->host->status != 0)
    return fail(AWQ_ERR_TIMEOUT, "a bounded device wait expired (device code %d)",
                r->host->status);
  return ok();
}

int awq_result_n_grid(const awq_result* r) { return r ? r->n_grid : 0; }
int awq_result_n_weights(const awq_result* r) { return r ? r->n_w : 0; }
int awq_result_best_index(const awq_result* r) { return r ? r->host->best : -1; }
double awq_result_alpha(const awq_result* r) { return r ? r->host->alpha : -1.0; }
const double* awq_result_losses(const awq_result* r) { return r ? r->host->losses : nullptr; }
const float* awq_result_s(const awq_result* r) { return r ? r->s : nullptr; }
const float* awq_result_s_grid(const awq_result* r) { return r ? r->s_grid : nullptr; }
const double* awq_result_row_losses(const awq_result* r) { return r ? r->row_losses : nullptr; }
const uint32_t* awq_result_codes(const awq_result* r, int i) {
  return (r && i >= 0 && i < r->n_w) ? r->codes[i] : nullptr;
}
const void* awq_result_scales(const awq_result* r, int i) {
  return (r && i >= 0 && i < r->n_w) ? r->scales[i] : nullptr;
}
const uint8_t* awq_result_zeros(const awq_result* r, int i) {
  return (r && i >= 0 && i < r->n_w) ? r->zeros[i] : nullptr;
}

void awq_free(awq_result* r) {
  if (r == nullptr) return;
  if (r->block) cudaFreeAsync(r->block, r->stream);
  give_mirror(r->host);
  destroy_events(r);
  delete r;
}

void awq_set_stage_timing(int enable) { g_stage_timing.store(enable ? 1 : 0); }

int awq_result_kernel_launches(const awq_result* r) { return r ? r->launches : -1; }

awq_status awq_result_stage_ms(const awq_result* r, int stage, float* ms) {
  if (r == nullptr || ms == nullptr) return fail(AWQ_ERR_INVALID, "result or ms is NULL");
  if (stage < 0 || stage >= AWQ_NUM_STAGES)
    return fail(AWQ_ERR_INVALID, "stage=%d (0..%d)", stage, AWQ_NUM_STAGES - 1);
  if (!r->timed) return fail(AWQ_ERR_INVALID, "stage timing was off during this search");
  const cudaError_t e = cudaEventElapsedTime(ms, r->ev[stage], r->ev[stage + 1]);
  if (e != cudaSuccess) return cuda_fail(e, "event elapsed time");
  return ok();
}

awq_status awq_release_cached_memory(void) {
  cudaError_t e;
  cudaMemPool_t pool = pool_for_current_device(&e);
  if (pool == nullptr) return cuda_fail(e, "pool lookup");
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
  e = cudaMemPoolTrimTo(pool, 0);
  if (e != cudaSuccess) return cuda_fail(e, "pool trim");
  return ok();
}

void awq_inject_allocation_failures(int skip, int count) {
  std::lock_guard<std::mutex> lock(g_inject_mu);
  g_alloc_skip = skip > 0 ? skip : 0;
  g_alloc_fail = count > 0 ? count : 0;
}

awq_status awq_pool_usage(int64_t* used_bytes, int64_t* reserved_bytes) {
  if (used_bytes == nullptr || reserved_bytes == nullptr)
    return fail(AWQ_ERR_INVALID, "used_bytes or reserved_bytes is NULL");
  cudaError_t e;
  cudaMemPool_t pool = pool_for_current_device(&e);
  if (pool == nullptr) return cuda_fail(e, "pool lookup");
  uint64_t used = 0, reserved = 0;
  if ((e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemCurrent, &used)) != cudaSuccess ||
      (e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &reserved)) !=
          cudaSuccess)
    return cuda_fail(e, "pool attribute");
  *used_bytes = static_cast<int64_t>(used);
  *reserved_bytes = static_cast<int64_t>(reserved);
  return ok();
}

awq_status awq_bounds_selftest(void) {
#ifdef AWQ_CHECK_BOUNDS
  NvtxScope nvtx("awq_bounds_selftest");
  auto cleanup = [] {};
  k_bounds_selftest<<<1, 1>>>();
  AWQ_CUDA(cudaGetLastError(), "bounds self-test launch");
  AWQ_CUDA(cudaDeviceSynchronize(), "device synchronisation");
  return ok();
#else
  return fail(AWQ_ERR_UNSUPPORTED, "awq_bounds_selftest: not the bounds-checked build");
#endif
}

int awq_bounds_checked(void) {
#ifdef AWQ_CHECK_BOUNDS
  return 1;
#else
  return 0;
#endif
}

awq_status awq_bounds_report(int64_t* count, int* site, int64_t* index, int64_t* extent,
                             int reset) {
  NvtxScope nvtx("awq_bounds_report");
  auto cleanup = [] {};
  AWQ_CUDA(cudaDeviceSynchronize(), "device synchronisation");
  typedef cudaError_t (*Reader)(BoundsRecord*, bool);
  const Reader readers[] = {bounds_api,    bounds_stats,  bounds_quant,
                            bounds_matvec, bounds_reduce, bounds_fold};
  int64_t total = 0;
  BoundsRecord first{0, -1, -1, -1};
  for (Reader rd : readers) {
    BoundsRecord rec{};
    AWQ_CUDA(rd(&rec, reset != 0), "bounds record read");
    if (rec.count != 0 && total == 0) first = rec;
    total += static_cast<int64_t>(rec.count);
  }
  if (count) *count = total;
  if (site) *site = static_cast<int>(first.site);
  if (index) *index = first.index;
  if (extent) *extent = first.extent;
  return ok();
}

awq_status awq_selftest_bounded_wait(int64_t limit_ns) {
  if (limit_ns < 1000 || limit_ns > 5000000000ll)
    return fail(AWQ_ERR_INVALID, "limit_ns=%lld (1e3..5e9)", static_cast<long long>(limit_ns));
  int* status = nullptr;
  auto cleanup = [&] {
    if (status) cudaFree(status);
  };
  AWQ_CUDA(cudaMalloc(&status, sizeof(int)), "status allocation");
  AWQ_CUDA(cudaMemset(status, 0, sizeof(int)), "status reset");
  AWQ_CUDA(launch_wait_selftest(static_cast<unsigned long long>(limit_ns), status, nullptr),
           "self-test launch");
  AWQ_CUDA(cudaDeviceSynchronize(), "self-test synchronize");
  int h = 0;
  AWQ_CUDA(cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost), "status copy");
  cleanup();
  if (h == kDevTimeoutSelfTest)
    return fail(AWQ_ERR_TIMEOUT, "bounded wait expired as expected (device code %d)", h);
  if (h != 0) return fail(AWQ_ERR_CUDA, "unexpected device code %d", h);
  return ok();
}

}  // extern "C"

// Status helpers for entry points defined in other translation units; they
// share this file's thread-local error message.  Not exported.
#define AWQ_HIDDEN __attribute__((visibility("hidden")))

AWQ_HIDDEN awq_status awq_internal_fail(awq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

AWQ_HIDDEN awq_status awq_internal_ok() { return ok(); }

AWQ_HIDDEN awq_status awq_internal_check_cfg(const awq_qconfig* cfg) { return check_cfg(cfg); }

AWQ_HIDDEN bool awq_internal_k_fits(int64_t K, const awq_qconfig* cfg) { return k_fits(K, cfg); }

AWQ_HIDDEN cudaError_t awq_internal_pool_alloc(void** p, size_t bytes, cudaStream_t st) {
  return pool_alloc(p, bytes, st);
}

AWQ_HIDDEN awq_status awq_internal_check_dev(const void* p, const char* name, uintptr_t align) {
  return check_dev(p, name, align);
}

AWQ_HIDDEN awq_status awq_internal_cuda_fail(cudaError_t e, const char* what) {
  return cuda_fail(e, what);
}
