// Launch facts cached per device: SM count, resident blocks per SM and the
// pair GEMM's co-resident clusters.  Looking these up (and raising a kernel's
// dynamic shared memory limit) costs host time on every launch otherwise,
// while the kernels of a small search run for microseconds.
#include <map>
#include <mutex>
#include <tuple>

#include "awq_internal.h"

namespace awq {
namespace {

std::mutex g_mu;
std::map<std::tuple<int, const void*, int, int>, LaunchFacts> g_facts;   // dev, fn, threads, smem
std::map<std::pair<int, const void*>, int> g_smem_limit;                   // dev, fn -> bytes set
std::map<std::tuple<int, const void*, int>, int> g_clusters;              // dev, fn, smem
std::map<int, int> g_sms;                                                  // dev -> SMs

int sms_locked(int dev) {
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 148;
  }
  g_sms[dev] = n;
  return n;
}

// Raises the kernel's dynamic shared memory limit to `smem` (never lowers it).
cudaError_t smem_limit_locked(int dev, const void* fn, int smem) {
  int& cur = g_smem_limit[{dev, fn}];
  if (smem <= cur) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) cur = smem;
  return e;
}

}  // namespace

int device_sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(g_mu);
  return sms_locked(dev);
}

cudaError_t launch_facts(const void* fn, int threads, int smem, LaunchFacts* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  const auto key = std::make_tuple(dev, fn, threads, smem);
  auto it = g_facts.find(key);
  if (it != g_facts.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  if ((e = smem_limit_locked(dev, fn, smem)) != cudaSuccess) return e;
  LaunchFacts f{sms_locked(dev), 1};
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&f.per_sm, fn, threads, smem) != cudaSuccess ||
      f.per_sm < 1) {
    cudaGetLastError();
    f.per_sm = 1;
  }
  g_facts[key] = f;
  *out = f;
  return cudaSuccess;
}

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

cudaError_t cluster_facts(const void* fn, int threads, int smem, int* max_clusters) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  const auto key = std::make_tuple(dev, fn, smem);
  auto it = g_clusters.find(key);
  if (it != g_clusters.end()) {
    *max_clusters = it->second;
    return cudaSuccess;
  }
  if ((e = smem_limit_locked(dev, fn, smem)) != cudaSuccess) return e;
  const int sms = sms_locked(dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = sms / 2;   // one 2-CTA cluster per SM pair
  }
  g_clusters[key] = n;
  *max_clusters = n;
  return cudaSuccess;
}

}  // namespace awq
