// The bounds-checked build (compiled with -DAWQ_CHECK_BOUNDS into
// libawq_checked.so), in place of a memory sanitizer: every checked global
// access compares its element index with the extent of the buffer it
// touches (the statistic, scales, quantizers, decode product, losses and
// fold; the GEMMs read their operands by TMA, whose bounds the hardware
// applies, and are not instrumented).  A violation is counted, the first one's (site, index, extent) is
// recorded in a device word of its translation unit, and the access is
// skipped; nothing traps.  awq_bounds_report reads and clears the records of
// every translation unit.  In the normal build in_bounds() is a constant true
// and the checks compile away.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace awq {

// Check sites (the `site` of a record).
enum BoundsSite : int {
  kSiteSelfTest = 0,        // awq_bounds_selftest: a synthetic index, no access
  kSiteStatsAcc = 1,        // statistic: 64-bit channel sums
  kSiteStatsOut = 2,        // statistic: sX
  kSiteScalesOut = 3,       // scales: s and 1/s per grid point
  kSiteResidualW = 4,       // residual pass: W row segment read
  kSiteResidualS = 5,       // residual pass: s and 1/s read
  kSiteResidualOut = 6,     // residual pass: residual store
  kSiteResidualRowmm = 7,   // residual pass: per-row min / max read
  kSiteFinalW = 8,          // final quantizer: W row segment read
  kSiteFinalCodes = 9,      // final quantizer: packed codes store
  kSiteFinalParams = 10,    // final quantizer: scale and zero store
  kSiteDecodeY = 11,        // decode product: y
  kSiteDecodeParams = 12,   // decode product: group zero / scale read
  kSiteDecodeX = 13,        // decode product: x read
  kSiteLosses = 16,         // losses: row and grid-point outputs
  kSiteFold = 17,           // fold: folded vector store
  kSiteDecodeCodes = 18,    // decode product: code words read (register-prefetch kernel)
};

struct BoundsRecord {
  unsigned long long count;   // violations since the last reset
  long long site, index, extent;
};

#ifdef AWQ_CHECK_BOUNDS
// One record per translation unit (each .cu file is its own device module).
static __device__ BoundsRecord g_bounds_record;

__device__ __forceinline__ bool in_bounds(int site, int64_t index, int64_t extent) {
  if (index >= 0 && index < extent) return true;
  if (atomicAdd(&g_bounds_record.count, 1ull) == 0ull) {
    g_bounds_record.site = site;
    g_bounds_record.index = index;
    g_bounds_record.extent = extent;
  }
  return false;
}

// Defines the host function that reads (and, with reset, clears) this
// translation unit's record.
#define AWQ_BOUNDS_READER(fn)                                                          \
  cudaError_t fn(BoundsRecord* out, bool reset) {                                     \
    cudaError_t e = cudaMemcpyFromSymbol(out, g_bounds_record, sizeof(BoundsRecord)); \
    if (e != cudaSuccess || !reset) return e;                                          \
    const BoundsRecord zero{};                                                         \
    return cudaMemcpyToSymbol(g_bounds_record, &zero, sizeof(BoundsRecord));           \
  }
#else
__device__ __forceinline__ constexpr bool in_bounds(int, int64_t, int64_t) { return true; }

#define AWQ_BOUNDS_READER(fn)                  \
  cudaError_t fn(BoundsRecord* out, bool) {    \
    *out = BoundsRecord{};                      \
    return cudaSuccess;                         \
  }
#endif

// Readers, one per translation unit with checked kernels.
cudaError_t bounds_api(BoundsRecord* out, bool reset);
cudaError_t bounds_stats(BoundsRecord* out, bool reset);
cudaError_t bounds_quant(BoundsRecord* out, bool reset);
cudaError_t bounds_matvec(BoundsRecord* out, bool reset);
cudaError_t bounds_reduce(BoundsRecord* out, bool reset);
cudaError_t bounds_fold(BoundsRecord* out, bool reset);

}  // namespace awq
