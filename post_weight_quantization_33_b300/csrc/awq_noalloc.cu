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
// looked up once per device with cudaGetSymbolAddress.
#include <mutex>

#include "awq.h"
#include "awq_internal.h"

namespace {

constexpr int64_t kNoAllocMaxK = AWQ_STATS_NOALLOC_MAX_K;

// Per-channel 64-bit sums of |x| in units of 2^-24 (see awq_stats.cu).
static __device__ __align__(256) unsigned long long g_stats_scratch[kNoAllocMaxK];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
unsigned long long* g_scratch_addr[kMaxDevices] = {};

// Address of g_stats_scratch on the current device, looked up on the first
// call for that device (with the device current) and cached.
cudaError_t scratch_for_current_device(unsigned long long** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_stats_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<unsigned long long*>(p);
  }
  *out = g_scratch_addr[dev];
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
  if (T < 1)
    return awq_internal_fail(AWQ_ERR_INVALID, "T=%lld (must be >= 1)", static_cast<long long>(T));
  if (K < 8 || K % 8)
    return awq_internal_fail(AWQ_ERR_INVALID, "K=%lld (must be a positive multiple of 8)",
                             static_cast<long long>(K));
  if (K > kNoAllocMaxK)
    return awq_internal_fail(AWQ_ERR_INVALID,
                             "K=%lld exceeds the fixed scratch of awq_stats_noalloc "
                             "(at most %lld channels); use awq_stats",
                             static_cast<long long>(K), static_cast<long long>(kNoAllocMaxK));
  if (T > (int64_t(1) << 31))
    return awq_internal_fail(AWQ_ERR_INVALID, "T too large");
  awq_status st;
  if ((st = awq_internal_check_dev(X, "X", 16)) != AWQ_OK) return st;
  if ((st = awq_internal_check_dev(sX, "sX", 8)) != AWQ_OK) return st;
  unsigned long long* acc = nullptr;
  cudaError_t e = scratch_for_current_device(&acc);
  if (e != cudaSuccess) return awq_internal_cuda_fail(e, "scratch address lookup");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // launch_stats_accumulate clears acc[0..K) on the stream before summing.
  e = awq::launch_stats_accumulate(static_cast<const __half*>(X), T, K, acc, s);
  if (e != cudaSuccess) return awq_internal_cuda_fail(e, "stats kernel");
  e = awq::launch_stats_finalize(acc, T, K, sX, s);
  if (e != cudaSuccess) return awq_internal_cuda_fail(e, "stats finalize kernel");
  return awq_internal_ok();
}
