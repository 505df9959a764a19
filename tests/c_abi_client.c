/*
 * A plain C client of libar_gb300.so: it uses only include/ar.h and the CUDA
 * runtime's C API, so it shows that the boundary needs neither Python nor
 * C++.  Every expected value is an exact-integer closed form computed here:
 * rank s holds x_s[i] = (s + 1) + (i mod 5), small integers that bf16
 * represents exactly, so the rank-order fp32 sum is exact and
 *   sum_s x_s[i] = R(R+1)/2 + R (i mod 5)   (at most 68 for R = 8).
 *
 *   c_abi_client --host-only   argument checks that return before any CUDA
 *                              call (runs without a GPU)
 *   c_abi_client               every variant of ar_allreduce, ar_reduce_scatter,
 *                              ar_all_gather and ar_allreduce_host on a GPU
 * Exit status 0 when every check passes.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ar.h"

#define R 8
#define COUNT 100003

static int failures = 0;
static long checks = 0;

#define CHECK(cond, ...)                    \
  do {                                      \
    ++checks;                               \
    if (!(cond)) {                          \
      ++failures;                           \
      fprintf(stderr, "FAIL: " __VA_ARGS__); \
      fprintf(stderr, "\n");                \
    }                                       \
  } while (0)

#define CUDA(call)                                                                    \
  do {                                                                                \
    cudaError_t e_ = (call);                                                          \
    if (e_ != cudaSuccess) {                                                          \
      fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, \
              __LINE__);                                                              \
      exit(2);                                                                        \
    }                                                                                 \
  } while (0)

/* bf16 bits of a small integer (exact: the low 16 bits of its fp32 form are 0). */
static uint16_t bf16_of_int(int v) {
  const float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

static int input_value(int s, size_t i) { return (s + 1) + (int)(i % 5); }
static int sum_value(size_t i) { return R * (R + 1) / 2 + R * (int)(i % 5); }

static int host_only(void) {
  ar_handle_t h = (ar_handle_t)1;
  for (int s = 0; s <= 5; ++s) CHECK(ar_status_string(s) != NULL, "status string %d", s);
  CHECK(strcmp(ar_status_string(99), "unknown status") == 0, "unknown status string");
  CHECK(strcmp(ar_variant_name(AR_FUSED_LL8), "fused_ll8") == 0, "variant name");
  CHECK(strcmp(ar_variant_name(42), "?") == 0, "unknown variant name");
  CHECK(ar_create(0, 16, AR_BF16, &h) == AR_ERR_INVALID_ARG && h == NULL, "R = 0 rejected");
  CHECK(ar_create(AR_MAX_RANKS + 1, 16, AR_BF16, &h) == AR_ERR_INVALID_ARG, "R too large");
  CHECK(ar_create(R, 0, AR_BF16, &h) == AR_ERR_INVALID_ARG, "max_count = 0 rejected");
  CHECK(ar_create(R, 16, 7, &h) == AR_ERR_UNSUPPORTED, "unknown dtype rejected");
  CHECK(ar_create(R, 16, AR_BF16, NULL) == AR_ERR_INVALID_ARG, "NULL out rejected");
  CHECK(ar_allreduce(NULL, (const void* const*)8, (void* const*)8, 1, NULL) == AR_ERR_INVALID_ARG,
        "NULL handle rejected");
  CHECK(ar_destroy(NULL) == AR_OK, "destroy NULL");
  return failures;
}

/* Copy R device buffers of n bf16 back and compare with want(r, i). */
static void check_outputs(uint16_t* const* d_out, size_t n, int (*want)(int, size_t),
                          const char* what) {
  uint16_t* host = (uint16_t*)malloc(n * sizeof(uint16_t));
  for (int r = 0; r < R; ++r) {
    CUDA(cudaMemcpy(host, d_out[r], n * sizeof(uint16_t), cudaMemcpyDeviceToHost));
    size_t bad = 0, first = 0;
    for (size_t i = 0; i < n; ++i)
      if (host[i] != bf16_of_int(want(r, i)) && bad++ == 0) first = i;
    CHECK(bad == 0, "%s rank %d: %zu of %zu differ, first at %zu (0x%04x, want 0x%04x)", what,
          r, bad, n, first, bad ? host[first] : 0, bad ? bf16_of_int(want(r, first)) : 0);
  }
  free(host);
}

static size_t g_block;
static int want_allreduce(int r, size_t i) { (void)r; return sum_value(i); }
static int want_reduce_scatter(int r, size_t j) { return sum_value((size_t)r * g_block + j); }
static int want_all_gather(int r, size_t k) {
  (void)r;
  return input_value((int)(k / g_block), k % g_block);
}

static int gpu(void) {
  uint16_t* host_in[R];
  uint16_t* host_out[R];
  uint16_t* d_in[R];
  uint16_t* d_out[R];
  for (int s = 0; s < R; ++s) {
    host_in[s] = (uint16_t*)malloc(COUNT * sizeof(uint16_t));
    host_out[s] = (uint16_t*)malloc(COUNT * sizeof(uint16_t));
    for (size_t i = 0; i < COUNT; ++i) host_in[s][i] = bf16_of_int(input_value(s, i));
    CUDA(cudaMalloc((void**)&d_in[s], COUNT * sizeof(uint16_t)));
    CUDA(cudaMalloc((void**)&d_out[s], COUNT * sizeof(uint16_t)));
    CUDA(cudaMemcpy(d_in[s], host_in[s], COUNT * sizeof(uint16_t), cudaMemcpyHostToDevice));
  }
  /* the two device-resident pointer tables */
  void** d_in_tbl;
  void** d_out_tbl;
  CUDA(cudaMalloc((void**)&d_in_tbl, R * sizeof(void*)));
  CUDA(cudaMalloc((void**)&d_out_tbl, R * sizeof(void*)));
  CUDA(cudaMemcpy(d_in_tbl, d_in, R * sizeof(void*), cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_out_tbl, d_out, R * sizeof(void*), cudaMemcpyHostToDevice));

  ar_handle_t h = NULL;
  CHECK(ar_create(R, COUNT, AR_BF16, &h) == AR_OK && h != NULL, "ar_create");
  if (!h) return failures;
  for (int v = 0; v < AR_NUM_VARIANTS; ++v) {
    for (int r = 0; r < R; ++r) CUDA(cudaMemset(d_out[r], 0xFF, COUNT * sizeof(uint16_t)));
    CHECK(ar_set_variant(h, v) == AR_OK, "set variant %d", v);
    CHECK(ar_allreduce(h, (const void* const*)d_in_tbl, (void* const*)d_out_tbl, COUNT, NULL) ==
              AR_OK,
          "ar_allreduce %s", ar_variant_name(v));
    CUDA(cudaDeviceSynchronize());
    CHECK(ar_get_device_status(h, NULL) == AR_OK, "device status after %s", ar_variant_name(v));
    check_outputs(d_out, COUNT, want_allreduce, ar_variant_name(v));
  }

  g_block = COUNT / R;
  CHECK(ar_reduce_scatter(h, (const void* const*)d_in_tbl, (void* const*)d_out_tbl, g_block,
                          NULL) == AR_OK,
        "ar_reduce_scatter");
  CUDA(cudaDeviceSynchronize());
  check_outputs(d_out, g_block, want_reduce_scatter, "reduce_scatter");
  CHECK(ar_all_gather(h, (const void* const*)d_in_tbl, (void* const*)d_out_tbl, g_block, NULL) ==
            AR_OK,
        "ar_all_gather");
  CUDA(cudaDeviceSynchronize());
  check_outputs(d_out, (size_t)R * g_block, want_all_gather, "all_gather");

  /* host buffers (pageable: the staging path) */
  CHECK(ar_set_variant(h, AR_AUTO) == AR_OK, "auto");
  CHECK(ar_reserve_host_staging(h) == AR_OK, "reserve staging");
  CHECK(ar_allreduce_host(h, (const void* const*)host_in, (void* const*)host_out, COUNT, NULL) ==
            AR_OK,
        "ar_allreduce_host");
  CUDA(cudaDeviceSynchronize());
  for (int r = 0; r < R; ++r) {
    size_t bad = 0;
    for (size_t i = 0; i < COUNT; ++i) bad += host_out[r][i] != bf16_of_int(sum_value(i));
    CHECK(bad == 0, "host path rank %d: %zu differ", r, bad);
  }
  CHECK(ar_destroy(h) == AR_OK, "ar_destroy");

  for (int s = 0; s < R; ++s) {
    CUDA(cudaFree(d_in[s]));
    CUDA(cudaFree(d_out[s]));
    free(host_in[s]);
    free(host_out[s]);
  }
  CUDA(cudaFree(d_in_tbl));
  CUDA(cudaFree(d_out_tbl));
  return failures;
}

int main(int argc, char** argv) {
  const int host = argc > 1 && strcmp(argv[1], "--host-only") == 0;
  const int f = host ? host_only() : gpu();
  printf("c_abi_client%s: %ld checks, %d failed\n", host ? " (host only)" : "", checks, f);
  return f == 0 ? 0 : 1;
}
