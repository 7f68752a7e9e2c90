/*
 * A plain C99 client of include/awq.h (no C++, no Python): the boundary is
 * usable as a C library.
 *
 *   awq_client cpu
 *     calls that need no GPU: ABI version, packed sizes, status strings,
 *     argument checks (NULL and misaligned pointers, bad configurations),
 *     awq_free(NULL); takes the address of every declared call so that the
 *     link resolves each of them.
 *   awq_client gpu T K N X.bin W.bin losses.bin codes.bin
 *     one search (INT4, group 128, 20 grid points) of W [N][K] fp16 with
 *     X [T][K] fp16 read from the files; writes the 20 fp64 losses and the
 *     packed codes, prints alpha.
 *   awq_client host T K N X.bin W.bin losses.bin codes.bin
 *     the same layer searched three times in one awq_search_host_layers call
 *     from plain host buffers (malloc, not pinned); checks that the three
 *     results agree, writes the first.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "awq.h"

#define CHECK(cond)                                                   \
  do {                                                                \
    if (!(cond)) {                                                    \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      return 1;                                                       \
    }                                                                 \
  } while (0)

static int cpu_checks(void) {
  typedef void (*fn_t)(void);   /* conversions between function pointer types are ISO C */
  const fn_t calls[] = {
      (fn_t)awq_abi_version, (fn_t)awq_last_error,
      (fn_t)awq_status_string, (fn_t)awq_packed_words,
      (fn_t)awq_stats, (fn_t)awq_scales, (fn_t)awq_quantize_pack,
      (fn_t)awq_unpack_codes, (fn_t)awq_fold_scale,
      (fn_t)awq_w4a16_matvec, (fn_t)awq_reference_output,
      (fn_t)awq_search_layer, (fn_t)awq_search_layer_gram,
      (fn_t)awq_result_check, (fn_t)awq_result_n_grid,
      (fn_t)awq_result_n_weights, (fn_t)awq_result_best_index,
      (fn_t)awq_result_alpha, (fn_t)awq_result_losses,
      (fn_t)awq_result_s, (fn_t)awq_result_s_grid,
      (fn_t)awq_result_row_losses, (fn_t)awq_result_codes,
      (fn_t)awq_result_scales, (fn_t)awq_result_zeros,
      (fn_t)awq_result_kernel_launches, (fn_t)awq_set_stage_timing,
      (fn_t)awq_result_stage_ms, (fn_t)awq_free,
      (fn_t)awq_release_cached_memory, (fn_t)awq_stats_noalloc,
      (fn_t)awq_selftest_bounded_wait, (fn_t)awq_search_host_layers,
      (fn_t)awq_inject_allocation_failures, (fn_t)awq_pool_usage};
  for (size_t i = 0; i < sizeof(calls) / sizeof(calls[0]); ++i) CHECK(calls[i] != NULL);

  CHECK(awq_abi_version() == AWQ_ABI_VERSION);
  CHECK(awq_packed_words(4096, 4096, 4) == 4096 * 4096 / 8);
  CHECK(awq_packed_words(3, 64, 3) == 3 * 3 * 64 / 32);
  CHECK(awq_packed_words(1, 64, 5) == -1);
  for (int st = AWQ_OK; st <= AWQ_ERR_TIMEOUT; ++st) {
    const char* s = awq_status_string(st);
    CHECK(s != NULL && s[0] != '\0');
  }

  awq_qconfig cfg = {4, 128, 1, 20};
  awq_weight w = {NULL, 64};
  awq_result* r = (awq_result*)0x1;
  CHECK(awq_search_layer(NULL, 16, 256, NULL, &w, 1, &cfg, NULL, &r) == AWQ_ERR_INVALID);
  CHECK(r == NULL);   /* cleared before any check that can fail */
  CHECK(strlen(awq_last_error()) > 0);
  CHECK(awq_search_layer(NULL, 16, 256, NULL, &w, 1, &cfg, NULL, NULL) == AWQ_ERR_INVALID);
  awq_qconfig bad = {5, 128, 1, 20};
  CHECK(awq_quantize_pack(NULL, 4, 256, NULL, &bad, NULL, NULL, NULL, NULL) ==
        AWQ_ERR_UNSUPPORTED);
  CHECK(awq_stats(NULL, 0, 64, NULL, NULL) == AWQ_ERR_INVALID);
  /* a 4-byte aligned codes pointer: the W4A16 product reads 16 bytes at a time */
  CHECK(awq_w4a16_matvec((const uint32_t*)(uintptr_t)0x1004, NULL, NULL, 4, 256, &cfg, NULL, 1,
                         NULL, NULL) == AWQ_ERR_INVALID);
  CHECK(strstr(awq_last_error(), "16-byte") != NULL);
  CHECK(awq_result_check(NULL) == AWQ_ERR_INVALID);
  /* the host pipeline: nothing to do, and layers it refuses before any copy */
  CHECK(awq_search_host_layers(NULL, 0, &cfg, NULL) == AWQ_OK);
  CHECK(awq_search_host_layers(NULL, 1, &cfg, NULL) == AWQ_ERR_INVALID);
  CHECK(awq_search_host_layers(NULL, -1, &cfg, NULL) == AWQ_ERR_INVALID);
  {
    static uint16_t x[16 * 256], wbuf[64 * 256];
    static uint32_t codes[64 * 32];
    static uint16_t scales[64 * 2];
    static uint8_t zeros[64 * 2];
    static float s[256];
    static double losses[20];
    static int best;
    uint32_t* c[1] = {codes};
    void* sc[1] = {scales};
    uint8_t* z[1] = {zeros};
    awq_weight hw = {wbuf, 64};
    awq_host_layer L = {x, 16, 250, &hw, 1, c, sc, z, s, losses, &best};   /* K not a multiple of 128 */
    CHECK(awq_search_host_layers(&L, 1, &cfg, NULL) == AWQ_ERR_INVALID);
    CHECK(strstr(awq_last_error(), "K=250") != NULL);
    L.K = 256;
    L.losses = NULL;
    CHECK(awq_search_host_layers(&L, 1, &cfg, NULL) == AWQ_ERR_INVALID);
    CHECK(awq_search_host_layers(&L, 1, &bad, NULL) == AWQ_ERR_UNSUPPORTED);
  }
  awq_free(NULL);
  printf("c client ok (cpu)\n");
  return 0;
}

static void* read_file(const char* path, size_t bytes) {
  FILE* f = fopen(path, "rb");
  if (f == NULL) return NULL;
  void* p = malloc(bytes);
  if (p != NULL && fread(p, 1, bytes, f) != bytes) {
    free(p);
    p = NULL;
  }
  fclose(f);
  return p;
}

static int write_file(const char* path, const void* p, size_t bytes) {
  FILE* f = fopen(path, "wb");
  if (f == NULL) return 0;
  const int ok = fwrite(p, 1, bytes, f) == bytes;
  fclose(f);
  return ok;
}

static int gpu_search(int argc, char** argv) {
  CHECK(argc == 9);
  const int64_t T = atoll(argv[2]), K = atoll(argv[3]), N = atoll(argv[4]);
  const size_t xb = (size_t)(T * K * 2), wb = (size_t)(N * K * 2);
  void* xh = read_file(argv[5], xb);
  void* wh = read_file(argv[6], wb);
  CHECK(xh != NULL && wh != NULL);
  void *xd = NULL, *wd = NULL;
  CHECK(cudaMalloc(&xd, xb) == cudaSuccess && cudaMalloc(&wd, wb) == cudaSuccess);
  CHECK(cudaMemcpy(xd, xh, xb, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemcpy(wd, wh, wb, cudaMemcpyHostToDevice) == cudaSuccess);

  awq_qconfig cfg = {4, 128, 1, 20};
  awq_weight w = {wd, N};
  awq_result* r = NULL;
  const awq_status st = awq_search_layer(xd, T, K, NULL, &w, 1, &cfg, NULL, &r);
  if (st != AWQ_OK) {
    fprintf(stderr, "search failed: %s (%s)\n", awq_status_string(st), awq_last_error());
    return 1;
  }
  CHECK(cudaDeviceSynchronize() == cudaSuccess);
  CHECK(awq_result_check(r) == AWQ_OK);
  CHECK(awq_result_n_grid(r) == 20 && awq_result_n_weights(r) == 1);
  const int64_t words = awq_packed_words(N, K, 4);
  uint32_t* codes = (uint32_t*)malloc((size_t)words * 4);
  CHECK(codes != NULL);
  CHECK(cudaMemcpy(codes, awq_result_codes(r, 0), (size_t)words * 4, cudaMemcpyDeviceToHost) ==
        cudaSuccess);
  CHECK(write_file(argv[7], awq_result_losses(r), 20 * sizeof(double)));
  CHECK(write_file(argv[8], codes, (size_t)words * 4));
  printf("alpha %.2f best %d\n", awq_result_alpha(r), awq_result_best_index(r));
  awq_free(r);
  free(codes);
  free(xh);
  free(wh);
  cudaFree(xd);
  cudaFree(wd);
  return 0;
}

static int host_search(int argc, char** argv) {
  CHECK(argc == 9);
  const int64_t T = atoll(argv[2]), K = atoll(argv[3]), N = atoll(argv[4]);
  const size_t xb = (size_t)(T * K * 2), wb = (size_t)(N * K * 2);
  void* xh = read_file(argv[5], xb);
  void* wh = read_file(argv[6], wb);
  CHECK(xh != NULL && wh != NULL);
  enum { LAYERS = 3 };
  const int64_t words = awq_packed_words(N, K, 4), groups = N * (K / 128);
  awq_qconfig cfg = {4, 128, 1, 20};
  awq_weight hw = {wh, N};
  awq_host_layer L[LAYERS];
  uint32_t* codes[LAYERS];
  void* scales[LAYERS];
  uint8_t* zeros[LAYERS];
  float* s[LAYERS];
  double losses[LAYERS][20];
  int best[LAYERS];
  for (int i = 0; i < LAYERS; ++i) {
    codes[i] = (uint32_t*)malloc((size_t)words * 4);
    scales[i] = malloc((size_t)groups * 2);
    zeros[i] = (uint8_t*)malloc((size_t)groups);
    s[i] = (float*)malloc((size_t)K * 4);
    CHECK(codes[i] && scales[i] && zeros[i] && s[i]);
    L[i].X = xh;
    L[i].T = T;
    L[i].K = K;
    L[i].Ws = &hw;
    L[i].n_w = 1;
    L[i].codes = &codes[i];
    L[i].scales = &scales[i];
    L[i].zeros = &zeros[i];
    L[i].s = s[i];
    L[i].losses = losses[i];
    L[i].best = &best[i];
  }
  const awq_status st = awq_search_host_layers(L, LAYERS, &cfg, NULL);
  if (st != AWQ_OK) {
    fprintf(stderr, "host search failed: %s (%s)\n", awq_status_string(st), awq_last_error());
    return 1;
  }
  for (int i = 1; i < LAYERS; ++i) {
    CHECK(best[i] == best[0]);
    CHECK(memcmp(losses[i], losses[0], sizeof(losses[0])) == 0);
    CHECK(memcmp(codes[i], codes[0], (size_t)words * 4) == 0);
    CHECK(memcmp(scales[i], scales[0], (size_t)groups * 2) == 0);
    CHECK(memcmp(zeros[i], zeros[0], (size_t)groups) == 0);
    CHECK(memcmp(s[i], s[0], (size_t)K * 4) == 0);
  }
  CHECK(write_file(argv[7], losses[0], 20 * sizeof(double)));
  CHECK(write_file(argv[8], codes[0], (size_t)words * 4));
  printf("alpha %.2f best %d\n", best[0] / 20.0, best[0]);
  for (int i = 0; i < LAYERS; ++i) {
    free(codes[i]);
    free(scales[i]);
    free(zeros[i]);
    free(s[i]);
  }
  free(xh);
  free(wh);
  return 0;
}

int main(int argc, char** argv) {
  if (argc >= 2 && strcmp(argv[1], "cpu") == 0) return cpu_checks();
  if (argc >= 2 && strcmp(argv[1], "gpu") == 0) return gpu_search(argc, argv);
  if (argc >= 2 && strcmp(argv[1], "host") == 0) return host_search(argc, argv);
  fprintf(stderr, "usage: awq_client cpu | gpu|host T K N X.bin W.bin losses.bin codes.bin\n");
  return 2;
}
