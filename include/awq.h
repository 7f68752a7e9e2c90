/*
 * awq.h -- C ABI of libawq: the activation-aware weight quantization (AWQ)
 * per-layer scale search on one NVIDIA B300 (sm_103a).
 *
 * What the library computes (passages by page title and section):
 *  - "AWQ explained" (hungho77.github.io), "Scaling instead of mixed
 *    precision": for a linear layer Y = W X, W' = W diag(s) and
 *    X' = diag(s)^-1 X leave the product unchanged before quantization;
 *    s = sX^alpha with sX the average activation magnitude per input channel;
 *    alpha is grid-searched in [0, 1] to minimise the layer-output error
 *    after quantization, with no backpropagation.
 *  - "AWQ Explained: Protecting the Weights That Matter Most" (multigrid.ai),
 *    "Scaling instead of mixed precision": the grid step is the group's range
 *    divided by the number of levels; "How the scale is chosen":
 *    alpha* = argmin over the grid of || W x - Q(W diag(s)) diag(s)^-1 x ||,
 *    and the knobs bits (4), group_size (128), zero_point (true).
 *  - "activation-aware weight quantization (AWQ)" (realpython.com): codes
 *    packed at 3 or 4 bits in groups, commonly 128.
 *  - "AWQ" (ai360xpert.com), "How It Works", step 4: round-to-nearest.
 *
 * Conventions for every call:
 *  - Pointers documented "device" must be device (or managed) memory of the
 *    current CUDA device; the library checks this and returns
 *    AWQ_ERR_INVALID otherwise, before launching anything.
 *  - fp16 matrices are row-major IEEE binary16, 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is
 *    enqueued on it; calls return before the GPU finishes.  Outputs are valid
 *    once the caller has synchronised the stream.
 *  - No exception crosses the ABI.  On failure a call returns a non-zero
 *    awq_status and awq_last_error() (per thread) describes it; argument
 *    errors are detected before any launch.
 *  - Device-side waits inside the tensor-core kernels are bounded (2 s); an
 *    expired wait is reported as AWQ_ERR_TIMEOUT through a status word
 *    (never a trap), see awq_result_check and awq_reference_output.
 *  - Calls may come from several host threads at once: the library's caches
 *    (memory pool, pinned result mirrors, launch facts) are locked and the
 *    error message is per thread.  Each call's work is ordered only on its
 *    own stream; awq_stats_noalloc is the one call whose concurrent use must
 *    be ordered by the caller (it shares one fixed array).
 *
 * Quantizer (fp32, every operation correctly rounded, none fused), per group
 * of `group_size` consecutive input channels of one output row (group_size
 * -1: the whole row is one group):
 *   w' = w * s_k;
 *   asymmetric (zero_point 1): step = max(max w' - min w', 1e-5) / (2^b - 1),
 *     zero = clamp(rne(-min w' * rcp), 0, 2^b - 1);
 *   symmetric (zero_point 0): step = max(max |w'|, 1e-5) / (2^(b-1) - 1),
 *     zero = 2^(b-1);
 *   scale = fp16_rne(step);  rcp = 1 / float(scale);
 *   code = clamp(rne(w' * rcp) + zero, 0, 2^b - 1);   rne = half to even.
 * Dequantization is (code - zero) * scale in both forms.
 * Scale vector: u_k = max(sX_k, 1e-4)^alpha (fp64),
 *   s_k = fp32(u_k / sqrt(max_k u * min_k u)),  alpha_i = i / n_grid.
 * Loss: ||W X^T - deq(Q(W diag(s))) diag(s)^-1 X^T||_F^2 / (N T), summed over
 *   the weights of one call; alpha* = first index of the minimum.
 * Packed codes: INT4 row n, word j = sum_m code[n][8j+m] << 4m;
 *   INT3 row n = little-endian bit stream, code k in bits [3k, 3k+3),
 *   32 codes per 3 words.
 */
#ifndef AWQ_H
#define AWQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AWQ_ABI_VERSION 1
#define AWQ_MAX_GRID 64
#define AWQ_MAX_WEIGHTS 16
/* Largest T of the channel statistic (awq_stats, awq_stats_noalloc, and
 * awq_search_layer* when they compute sX): its exact 64-bit channel sums stay
 * below 2^62 units of 2^-24, and the top two bits mark channels that held an
 * infinity or a NaN.  Larger T: AWQ_ERR_INVALID. */
#define AWQ_MAX_STAT_TOKENS 4194304

/* Stages of awq_search_layer, in order (for awq_result_stage_ms). */
#define AWQ_STAGE_STATS 0       /* channel statistic (skipped when sX is given) */
#define AWQ_STAGE_SCALES 1      /* s and 1/s for every grid point */
#define AWQ_STAGE_RESIDUAL 2    /* quantizer residual for every weight and grid point */
#define AWQ_STAGE_ERROR_GEMM 3  /* tcgen05 GEMM + squared-error epilogue */
#define AWQ_STAGE_LOSS 4        /* per-row and per-grid-point losses, argmin */
#define AWQ_STAGE_FINAL 5       /* quantize + pack at the chosen grid point */
#define AWQ_NUM_STAGES 6

typedef enum awq_status {
  AWQ_OK = 0,
  AWQ_ERR_INVALID = 1,     /* bad argument (null, misaligned, host pointer, bad size) */
  AWQ_ERR_UNSUPPORTED = 2, /* well-formed configuration this library does not implement */
  AWQ_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  AWQ_ERR_OOM = 4,         /* device memory exhausted */
  AWQ_ERR_TIMEOUT = 5      /* a bounded device-side wait expired */
} awq_status;

/* Quantizer configuration ("AWQ Explained", multigrid.ai, "How the scale is
 * chosen": bits, group_size, zero_point).  Supported: bits 3 or 4,
 * group_size 64, 128 or -1 (one group per output row; K must then be a
 * multiple of 64), zero_point 1 (asymmetric) or 0 (symmetric), n_grid
 * 1..AWQ_MAX_GRID (20 is the default grid alpha = 0, 0.05, ..., 0.95). */
typedef struct awq_qconfig {
  int bits;
  int group_size;
  int zero_point;
  int n_grid;
} awq_qconfig;

/* One weight matrix of a search call: device fp16 [N][K] row-major
 * (the nn.Linear.weight layout), N >= 1. */
typedef struct awq_weight {
  const void* W;
  int64_t N;
} awq_weight;

/* Opaque search result, owned by the library until awq_free. */
typedef struct awq_result awq_result;

/* ABI version of the loaded library (AWQ_ABI_VERSION). */
int awq_abi_version(void);

/* Message of the last failed call on this thread ("" if none).  Owned by
 * the library, valid until the next call on the same thread. */
const char* awq_last_error(void);

/* Constant name of a status code. */
const char* awq_status_string(int status);

/* uint32 words of N packed rows of K codes at `bits` (3 or 4); -1 if the
 * shape is invalid (K % 8 for INT4, K % 32 for INT3).  Host-only. */
int64_t awq_packed_words(int64_t N, int64_t K, int bits);

/* Channel statistic sX_k = (1/T) sum_t |X[t][k]| ("AWQ explained",
 * "Scaling instead of mixed precision": average activation magnitude per
 * input channel).
 *   X  : device fp16 [T][K], 1 <= T <= AWQ_MAX_STAT_TOKENS, K >= 8 and
 *        K % 8 == 0.
 *   sX : device fp64 [K], written.  The channel sums are exact (64-bit
 *        integer accumulation of |x| in units of 2^-24); the mean is one
 *        correctly rounded fp64 division.  A channel that holds an infinity
 *        gets +inf, one that holds a NaN gets NaN (what an IEEE fp64 sum
 *        gives).  If a bounded device wait expired, every sX is NaN.
 * Allocates K*8 + 8 bytes of stream-ordered scratch from the library's pool. */
awq_status awq_stats(const void* X, int64_t T, int64_t K, double* sX, void* stream);

/* Scale vectors for every grid point ("AWQ explained": s = sX^alpha).
 *   sX : device fp64 [K], K >= 1.
 *   s  : device fp32 [n_grid][K], written; row i uses alpha = i / n_grid.
 * x^alpha is formed in fp64 from one log and one exp per channel (relative
 * error below 2^-47 before the fp32 rounding).  Allocates 16 bytes of
 * stream-ordered scratch. */
awq_status awq_scales(const double* sX, int64_t K, int n_grid, float* s, void* stream);

/* Scale, group-quantize and pack one weight ("AWQ Explained", multigrid.ai,
 * "Scaling instead of mixed precision"; realpython glossary: 3/4-bit codes in
 * groups).  One pass over W; allocates nothing, except N*8 bytes of
 * stream-ordered scratch for group_size -1 (a row min / max pre-pass).
 *   W      : device fp16 [N][K]; N >= 0 (N = 0 is a no-op), K % group == 0.
 *   s      : device fp32 [K] (the per-input-channel scale).
 *   codes  : device uint32 [awq_packed_words(N, K, bits)], written.
 *   scales : device fp16 [N][K/group] ([N][1] for group_size -1), written.
 *   zeros  : device uint8 [N][K/group] ([N][1] for group_size -1), written. */
awq_status awq_quantize_pack(const void* W, int64_t N, int64_t K, const float* s,
                             const awq_qconfig* cfg, uint32_t* codes, void* scales,
                             uint8_t* zeros, void* stream);

/* Inverse of the packing: q[n][k] = code k of row n.
 *   codes : device uint32 [awq_packed_words(N, K, bits)];  q : device uint8 [N][K]. */
awq_status awq_unpack_codes(const uint32_t* codes, int64_t N, int64_t K, int bits, uint8_t* q,
                            void* stream);

/* Deploy step: fold diag(s)^-1 into the operation that produces the
 * layer's input ("AWQ Explained", multigrid.ai, "Scaling instead of mixed
 * precision": the inverse scale folds offline into the preceding LayerNorm /
 * RMSNorm weight or preceding linear layer, so what ships is the quantized
 * matrix and a modified norm).
 *   V    : device fp16 [rows][cols] row-major, 2-byte aligned.  rows = K of
 *          the quantized layer; cols = 1 for a vector (a norm weight or a
 *          bias), or the preceding linear layer's input width (its weight is
 *          [K][cols]: output row k feeds input channel k).
 *   s    : device fp32 [rows] (the scale the search chose, awq_result_s).
 *   out  : device fp16 [rows][cols], written:
 *          out[i][j] = fp16_rne(fp32(V[i][j]) / s[i]) (correctly rounded fp32
 *          division).  May be V itself (in place).
 * rows, cols >= 1.  One HBM pass; allocates nothing. */
awq_status awq_fold_scale(const void* V, int64_t rows, int64_t cols, const float* s, void* out,
                          void* stream);

/* Decode product with a packed layer, W4A16 or W3A16 ("AWQ explained",
 * "Why weight-only quantization fits decoding": at small batch each token
 * reads every weight once, so 3- or 4-bit weights with 16-bit activations cut
 * the dominant traffic four times or more).
 *   codes  : device uint32 packed codes as written by the search or
 *            awq_quantize_pack (INT4 [N][K/8] or INT3 [N][3K/32]), 16-byte
 *            aligned.
 *   scales : device fp16 [N][K/group] ([N][1] for group_size -1).
 *   zeros  : device uint8, same shape (integers in [0, 2^bits - 1], as the
 *            search and awq_quantize_pack write them).
 *   cfg    : the configuration the codes were made with (bits 3 or 4,
 *            group_size; zero_point and n_grid are not used).
 *   x      : device fp16 [M][K], 1 <= M <= 16, 16-byte aligned: activations
 *            with diag(s)^-1 already folded into their producer
 *            (awq_fold_scale).
 *   y      : device fp32 [M][N], written:
 *            y[m][n] = sum_g scale[n][g] * sum_{k in g} (code - zero) * x[m][k];
 *            (code - zero) * x is exact, the sums are fp32 on the tensor cores
 *            (mma.sync, fp16 operands), and each group's sum is scaled in fp32.
 *            Deterministic: run-to-run identical.
 * K % 64 == 0 and K % group == 0.  Allocates nothing: y is zeroed on the
 * stream by a small kernel, then accumulated; both kernels are launched with
 * programmatic dependent launch behind the stream's previous kernel and wait
 * for it before touching y or reading x, so inputs written by the kernel
 * just before the call are seen.  K % 128 == 0 streams the codes through TMA
 * (a device wait bounded at 2 s: if one expires, the outputs of the rows
 * concerned read NaN); other K read them with plain loads. */
awq_status awq_w4a16_matvec(const uint32_t* codes, const void* scales, const uint8_t* zeros,
                            int64_t N, int64_t K, const awq_qconfig* cfg, const void* x, int M,
                            float* y, void* stream);

/* Layer output before quantization, Y = W X^T ("AWQ Explained", multigrid.ai,
 * "How the scale is chosen": the W x term), on tcgen05 tensor cores.
 *   W : device fp16 [N][K];  X : device fp16 [T][K];  K % 64 == 0.
 *   Y : device fp32 [N][T], written.
 *   status_dev : optional device int (caller zeroes it); receives a non-zero
 *                code if a bounded device wait expired.  May be NULL. */
awq_status awq_reference_output(const void* W, int64_t N, const void* X, int64_t T, int64_t K,
                                float* Y, int* status_dev, void* stream);

/* The whole per-layer scale search ("AWQ explained", "Scaling instead of
 * mixed precision"; "AWQ Explained", multigrid.ai, "How the scale is chosen").
 *   X   : device fp16 [T][K] calibration activations, T >= 1, K % group == 0.
 *   sX  : optional device fp64 [K]; NULL computes it with awq_stats.
 *   Ws  : host array of n_w (1..AWQ_MAX_WEIGHTS) weights sharing X (one s,
 *         one alpha; the loss is the sum of their losses).
 *   cfg : quantizer configuration.
 *   out : receives a library-owned result (free with awq_free).
 * Inputs must be finite: if X or W holds an infinity or a NaN, a grid
 * point's loss is not finite, and awq_result_check reports AWQ_ERR_INVALID
 * (the outputs are then undefined).  With sX NULL, T <= AWQ_MAX_STAT_TOKENS.
 * Steps, all stream-ordered on the device: sX; s for every grid point; for
 * every weight and grid point the fp16 quantization residual
 * W - deq(Q(W diag(s))) diag(s)^-1 (the same quantizer as awq_quantize_pack);
 * one tcgen05 GEMM of all residuals with X whose epilogue sums the squared
 * layer-output errors per row; losses and argmin; the final quantization at
 * the chosen alpha (read on the device, no host round trip).  Scratch is
 * n_grid * sum_i(round_up(N_i, 128)) * K * 2 bytes of residuals plus small
 * buffers.  Device memory for the result and the scratch comes from a
 * library-owned stream-ordered pool;
 * the scratch is released in stream order before the call returns. */
awq_status awq_search_layer(const void* X, int64_t T, int64_t K, const double* sX,
                            const awq_weight* Ws, int n_w, const awq_qconfig* cfg, void* stream,
                            awq_result** out);

/* The same search with the loss evaluated in its Gram form: for output row n
 * with residual d_n, sum_t (d_n . x_t)^2 = d_n^T G d_n with G = X^T X ("AWQ
 * Explained", multigrid.ai, "How the scale is chosen": the layer-output error
 * over the calibration batch; the identity is plain linear algebra).  G is
 * formed once (T K^2 flops, fp32 on the tensor cores) and stored as fp16
 * G * c / T with a power of two c chosen from max |G|; each grid point then
 * costs N K^2 flops instead of N K T, so the variant pays off when T > K.
 * Arguments, outputs, ownership and errors as awq_search_layer; losses agree
 * with it within the fp16 rounding of G (about 1e-5 relative on the
 * workloads tested, bar 1e-3).  Extra scratch: 2*K*Tp + 6*K*K bytes
 * (Tp = T rounded up to 64). */
awq_status awq_search_layer_gram(const void* X, int64_t T, int64_t K, const double* sX,
                                 const awq_weight* Ws, int n_w, const awq_qconfig* cfg,
                                 void* stream, awq_result** out);

/* One layer of awq_search_host_layers: inputs and outputs in host memory
 * (pinned memory lets the copies overlap the searches; pageable memory works
 * but serialises them).  Output buffers are owned by the caller. */
typedef struct awq_host_layer {
  const void* X;             /* host fp16 [T][K] calibration activations */
  int64_t T;                 /* 1 <= T <= AWQ_MAX_STAT_TOKENS */
  int64_t K;                 /* as awq_search_layer: K % group == 0, K % 32 for INT3 */
  const awq_weight* Ws;      /* host array of n_w weights; each W is host fp16 [N][K] */
  int n_w;                   /* 1..AWQ_MAX_WEIGHTS, sharing X (one s, one alpha) */
  uint32_t* const* codes;    /* n_w host buffers, uint32 [awq_packed_words(N_i, K, bits)] */
  void* const* scales;       /* n_w host buffers, fp16 [N_i][K/group] ([N_i][1] for -1) */
  uint8_t* const* zeros;     /* n_w host buffers, uint8, same shape as scales */
  float* s;                  /* host fp32 [K]: s at alpha* */
  double* losses;            /* host fp64 [n_grid]: the loss of every grid point */
  int* best;                 /* host int: index of alpha* (alpha* = best / n_grid) */
} awq_host_layer;

/* The search of awq_search_layer for a sequence of layers whose inputs and
 * outputs are in host memory (the end-to-end use: calibration data and
 * weights on the host, quantized layers back to the host).  Each layer's
 * search runs on `stream`; two library-owned streams copy layer i+1's inputs
 * in and layer i-1's outputs out while layer i is searched.  Device inputs
 * are double-buffered in two slots sized for the largest layer (from the
 * library's pool); each layer's device result is freed after its copy-out.
 * Every layer is checked on the host before anything is copied.  Returns
 * when every output is in the caller's buffers (synchronous).  On failure
 * (a layer the search refuses, a CUDA error, AWQ_ERR_OOM, or a non-finite
 * loss / expired wait reported by awq_result_check) the work already enqueued
 * is completed, every device buffer of the call is released, and the status
 * of the first failure is returned; the outputs are then incomplete.
 * n_layers 0 is a no-op. */
awq_status awq_search_host_layers(const awq_host_layer* layers, int n_layers,
                                  const awq_qconfig* cfg, void* stream);

/* After the search's stream is synchronised: AWQ_OK; AWQ_ERR_INVALID if a
 * grid point's loss is not finite (X or W held an infinity or a NaN); or
 * AWQ_ERR_TIMEOUT if a bounded device wait expired during the search. */
awq_status awq_result_check(const awq_result* r);

/* Result accessors.  Host values (alpha, best index, losses) are valid once
 * the stream is synchronised.  Device pointers stay valid until awq_free. */
int awq_result_n_grid(const awq_result* r);
int awq_result_n_weights(const awq_result* r);
int awq_result_best_index(const awq_result* r);        /* host */
double awq_result_alpha(const awq_result* r);          /* host: best / n_grid */
const double* awq_result_losses(const awq_result* r);  /* host fp64 [n_grid] */
const float* awq_result_s(const awq_result* r);        /* device fp32 [K], s at alpha* */
const float* awq_result_s_grid(const awq_result* r);   /* device fp32 [n_grid][K] */
const double* awq_result_row_losses(const awq_result* r); /* device fp64 [n_grid][sum N_i]:
                                                              sum_t error^2 per output row,
                                                              weights concatenated in order */
const uint32_t* awq_result_codes(const awq_result* r, int i);  /* device packed codes of W_i */
const void* awq_result_scales(const awq_result* r, int i);     /* device fp16 [N_i][K/group],
                                                                  [N_i][1] for group -1 */
const uint8_t* awq_result_zeros(const awq_result* r, int i);   /* device uint8, same shape */

/* Number of kernels the search enqueued (host value, valid on return). */
int awq_result_kernel_launches(const awq_result* r);

/* Turn per-stage timing of later awq_search_layer calls on (1) or off (0),
 * process-wide.  When on, each search records CUDA events on its stream at
 * the stage boundaries (a few microseconds of overhead). */
void awq_set_stage_timing(int enable);

/* Milliseconds the GPU spent in `stage` (AWQ_STAGE_*) of a search that ran
 * with stage timing on; valid once the stream is synchronised. */
awq_status awq_result_stage_ms(const awq_result* r, int stage, float* ms);

/* Release a result.  Its device memory returns to the library's pool in the
 * order of the stream the search ran on, so call this before destroying that
 * stream.  NULL is ignored. */
void awq_free(awq_result* r);

/* Return the library pool's cached, unused device memory on the current
 * device to the driver (synchronises the device). */
awq_status awq_release_cached_memory(void);

/* The channel statistic of awq_stats, computed without allocating any device
 * memory (no counterpart on the AWQ pages: this is an operational variant).
 * For callers that cannot let a library allocate: processes that give all
 * device memory to their own allocator at start-up and forbid later
 * allocations, latency-critical loops in which cudaMalloc/cudaFree would
 * synchronise the device, or code running inside another allocator's
 * callback.  The 64-bit accumulator lives in a fixed array inside the
 * library (AWQ_STATS_NOALLOC_MAX_K * 8 + 8 bytes, about 512 KiB, held on
 * every device that loads the library until the process exits).
 *   X, T, K, sX, stream : as awq_stats; K <= AWQ_STATS_NOALLOC_MAX_K, else
 *                         AWQ_ERR_INVALID (use awq_stats for wider layers).
 * The first call in each CUDA context (normally the first call on each
 * device; again after a device reset) looks the array's device address up,
 * with that device current; make that first call before any stream capture.
 * Every call on a device shares the one array, which keeps the last call's
 * sums; each call clears the K entries it uses, on its stream, before
 * accumulating.  Calls whose work overlaps on the GPU (different streams, or
 * different host threads without ordering) race on the array and give wrong
 * results: order them. */
#define AWQ_STATS_NOALLOC_MAX_K 65536
awq_status awq_stats_noalloc(const void* X, int64_t T, int64_t K, double* sX, void* stream);

/* Test hook of the out-of-memory path: after the next `skip` device
 * allocations from the library's pool, the following `count` fail as if the
 * device memory were exhausted, without reaching the allocator (the calls
 * that make them return AWQ_ERR_OOM and release what they held).  count 0
 * disarms it.  Process-wide; for tests of callers' error handling. */
void awq_inject_allocation_failures(int skip, int count);

/* Bytes of the library pool on the current device: handed out to results or
 * in-flight scratch (used), and held from the driver (reserved, >= used;
 * freed blocks stay cached until awq_release_cached_memory). */
awq_status awq_pool_usage(int64_t* used_bytes, int64_t* reserved_bytes);

/* Self-test of the bounded device wait: launches one CTA that waits on a
 * barrier nothing arrives at, with a limit of limit_ns nanoseconds
 * (1e3..5e9), synchronises, and returns AWQ_ERR_TIMEOUT when the wait expired
 * and was reported as it should (AWQ_OK would mean the wait did not expire).
 * Exists for testing the failure path without faulting the GPU. */
awq_status awq_selftest_bounded_wait(int64_t limit_ns);

/* The bounds-checked build: libawq_checked.so has the same interface and
 * results, and in it the kernels of the statistic, scales, quantizers,
 * decode product, losses and fold compare each computed global index with the
 * extent of its buffer before the access; an out-of-range access is skipped
 * and recorded (no trap).  A stand-in for a memory sanitizer, which is not
 * available on every GPU host.
 *   awq_bounds_checked : 1 in libawq_checked.so, 0 in libawq.so.
 *   awq_bounds_report  : synchronises the current device and returns the
 *     number of out-of-range accesses since the last reset (count) and the
 *     first recorded one's check site, element index and buffer extent (-1
 *     when count is 0); reset != 0 clears the records.  In libawq.so count is
 *     always 0.  Any output pointer may be NULL. */
int awq_bounds_checked(void);
/* Bounds-checked build only: records one synthetic out-of-range index (site
 * 0, index -1, extent 0) without touching memory, so that a test can see the
 * record path work; AWQ_ERR_UNSUPPORTED in libawq.so. */
awq_status awq_bounds_selftest(void);
awq_status awq_bounds_report(int64_t* count, int* site, int64_t* index, int64_t* extent,
                             int reset);

#ifdef __cplusplus
}
#endif

#endif /* AWQ_H */
