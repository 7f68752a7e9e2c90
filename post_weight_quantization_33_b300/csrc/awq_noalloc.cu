// awq_stats_noalloc: the channel statistic without any device allocation.
//
// awq_stats takes its 64-bit accumulator (8 bytes per input channel) from the
// library's stream-ordered pool.  Some callers cannot let a library allocate
// device memory: a serving process that hands all of HBM to its own
// allocator at start-up and forbids later allocations, a latency-critical
// loop where cudaMalloc/cudaFree would synchronise the device, or code that
// runs inside another allocator's callback and must not re-enter it.  This
// variant uses a fixed scratch array that lives in the library's own device
// image instead, so it allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kNoAllocMaxK * 8 bytes of it until the process exits.  Host
// code must not use the array's name as a device address; its address is
// looked up with cudaGetSymbolAddress once per CUDA context (once per device,
// and again in a context created after a device reset).
#include <map>
#include <mutex>

#include "awq.h"
#include "awq_internal.h"

namespace {

constexpr int64_t kNoAllocMaxK = AWQ_STATS_NOALLOC_MAX_K;

// Per-channel 64-bit sums of |x| in units of 2^-24 (see awq_stats.cu); the
// word after a call's K sums holds the status of its bounded waits.
static __device__ __align__(256) unsigned long long g_stats_scratch[kNoAllocMaxK + 1];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_setup_mu;
// Address of g_stats_scratch per CUDA context, keyed by the context's
// process-unique id: a context created after a device reset (or a
// non-primary context) loads the library's device code again at another
// address, and gets its own entry.
std::map<unsigned long long, unsigned long long*> g_scratch_addr;

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// Address of g_stats_scratch in the current context.  The first call in a
// context (normally the first call on a device) looks it up with
// cudaGetSymbolAddress, with that device current, and caches it.
cudaError_t scratch_for_current_context(unsigned long long** out) {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (get_current == nullptr || get_id == nullptr) return cudaErrorNotSupported;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  CUcontext ctx = nullptr;
  void* looked_up = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
    // No context bound to this thread yet: the runtime binds the current
    // device's primary context while it looks the symbol up.
    const cudaError_t e = cudaGetSymbolAddress(&looked_up, g_stats_scratch);
    if (e != cudaSuccess) return e;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  auto it = g_scratch_addr.find(id);
  if (it == g_scratch_addr.end()) {
    if (looked_up == nullptr) {
      const cudaError_t e = cudaGetSymbolAddress(&looked_up, g_stats_scratch);
      if (e != cudaSuccess) return e;
    }
    it = g_scratch_addr.emplace(id, static_cast<unsigned long long*>(looked_up)).first;
  }
  *out = it->second;
  return cudaSuccess;
}

}  // namespace

// Status helpers shared with awq_api.cu (same thread-local error message).
awq_status awq_internal_fail(awq_status st, const char* fmt, ...);
awq_status awq_internal_ok();
awq_status awq_internal_check_dev(const void* p, const char* name, uintptr_t align);
awq_status awq_internal_cuda_fail(cudaError_t e, const char* what);

extern "C" __attribute__((visibility("default"))) awq_status awq_stats_noalloc(
    const void* X, int64_t T, int64_t K, double* sX, void* stream) {
  awq::NvtxScope nvtx("awq_stats_noalloc");
  if (T < 1)
    return awq_internal_fail(AWQ_ERR_INVALID, "T=%lld (must be >= 1)", static_cast<long long>(T));
  if (T > awq::kMaxStatTokens)
    return awq_internal_fail(AWQ_ERR_INVALID,
                             "T=%lld exceeds AWQ_MAX_STAT_TOKENS=%lld (the exact 64-bit "
                             "channel sums)",
                             static_cast<long long>(T),
                             static_cast<long long>(awq::kMaxStatTokens));
  if (K < 8 || K % 8)
    return awq_internal_fail(AWQ_ERR_INVALID, "K=%lld (must be a positive multiple of 8)",
                             static_cast<long long>(K));
  if (K > kNoAllocMaxK)
    return awq_internal_fail(AWQ_ERR_INVALID,
                             "K=%lld exceeds the fixed scratch of awq_stats_noalloc "
                             "(at most %lld channels); use awq_stats",
                             static_cast<long long>(K), static_cast<long long>(kNoAllocMaxK));
  awq_status st;
  if ((st = awq_internal_check_dev(X, "X", 16)) != AWQ_OK) return st;
  if ((st = awq_internal_check_dev(sX, "sX", 8)) != AWQ_OK) return st;
  unsigned long long* acc = nullptr;
  cudaError_t e = scratch_for_current_context(&acc);
  if (e != cudaSuccess) return awq_internal_cuda_fail(e, "scratch address lookup");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The status word of this call follows its K sums.  The array keeps the
  // last call's contents: launch_stats_accumulate clears acc[0..K] (sums and
  // status) on the stream before accumulating.
  int* status = reinterpret_cast<int*>(acc + K);
  e = awq::launch_stats_accumulate(static_cast<const __half*>(X), T, K, acc, status, s);
  if (e != cudaSuccess) return awq_internal_cuda_fail(e, "stats kernel");
  e = awq::launch_stats_finalize(acc, T, K, sX, status, s);
  if (e != cudaSuccess) return awq_internal_cuda_fail(e, "stats finalize kernel");
  return awq_internal_ok();
}
