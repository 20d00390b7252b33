/*
 * The C ABI of libarx used from plain C: no Python, no torch.  Device memory
 * comes from the CUDA runtime, inputs from a counter hash of the index (finite
 * bf16 bit patterns), and every output is compared bit for bit with the CPU
 * oracle (oracle_reduce from the oracle's C library, test infrastructure).
 * Exit status 0 when everything matches.
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "arx.h"

int oracle_reduce(const uint16_t* const* slots, int W, uint16_t* out, size_t n);

static int failures = 0;

#define CHECK_CUDA(x)                                                     \
  do {                                                                    \
    cudaError_t e_ = (x);                                                 \
    if (e_ != cudaSuccess) {                                              \
      fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #x,           \
              cudaGetErrorString(e_));                                    \
      exit(2);                                                            \
    }                                                                     \
  } while (0)

#define CHECK_ARX(x)                                                      \
  do {                                                                    \
    arx_status s_ = (x);                                                  \
    if (s_ != ARX_OK) {                                                   \
      fprintf(stderr, "%s:%d %s: %s (%s)\n", __FILE__, __LINE__, #x,      \
              arx_status_string(s_), arx_last_error());                   \
      exit(3);                                                            \
    }                                                                     \
  } while (0)

/* A finite bf16 pattern from (seed, index): a 32-bit mix of the two, with the
 * all-ones exponent (inf / NaN) avoided. */
static uint16_t pattern(uint32_t seed, uint32_t i) {
  uint32_t h = seed * 0x9E3779B9u ^ (i + 0x7F4A7C15u);
  h ^= h >> 16;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  h *= 0xC2B2AE35u;
  h ^= h >> 16;
  uint16_t b = (uint16_t)(h & 0xFFFFu);
  if ((b & 0x7F80u) == 0x7F80u) b &= 0xBFFFu; /* clear one exponent bit */
  return b;
}

static void compare(const char* what, int W, size_t n, const uint16_t* got, const uint16_t* want) {
  for (size_t i = 0; i < n; ++i) {
    if (got[i] != want[i]) {
      fprintf(stderr, "%s W=%d n=%zu: element %zu gpu 0x%04x oracle 0x%04x\n", what, W, n, i,
              got[i], want[i]);
      ++failures;
      return;
    }
  }
}

static void reduce_case(int W, size_t n, int in_place) {
  uint16_t* host[ARX_MAX_W];
  void* dev[ARX_MAX_W];
  const uint16_t* hs[ARX_MAX_W];
  uint16_t* want = (uint16_t*)malloc((n ? n : 1) * 2);
  uint16_t* got = (uint16_t*)malloc((n ? n : 1) * 2);
  void* out = NULL;
  for (int r = 0; r < W; ++r) {
    host[r] = (uint16_t*)malloc((n ? n : 1) * 2);
    for (size_t i = 0; i < n; ++i) host[r][i] = pattern((uint32_t)(W * 131 + r), (uint32_t)i);
    hs[r] = host[r];
    CHECK_CUDA(cudaMalloc(&dev[r], n * 2 + 16));
    CHECK_CUDA(cudaMemcpy(dev[r], host[r], n * 2, cudaMemcpyHostToDevice));
  }
  oracle_reduce(hs, W, want, n);
  if (in_place) {
    out = dev[0];
  } else {
    CHECK_CUDA(cudaMalloc(&out, n * 2 + 16));
  }
  CHECK_ARX(arx_reduce((const void* const*)dev, W, out, n, NULL));
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(got, out, n * 2, cudaMemcpyDeviceToHost));
  compare(in_place ? "arx_reduce in place" : "arx_reduce", W, n, got, want);
  if (!in_place) CHECK_CUDA(cudaFree(out));
  for (int r = 0; r < W; ++r) {
    CHECK_CUDA(cudaFree(dev[r]));
    free(host[r]);
  }
  free(want);
  free(got);
}

/* Three protocol steps on one context (every barrier variant in turn), then
 * the allocation-free step, each checked against the oracle. */
static void step_cases(int W, size_t n) {
  void* dev[ARX_MAX_W];
  uint16_t* host[ARX_MAX_W];
  const uint16_t* hs[ARX_MAX_W];
  uint16_t* want = (uint16_t*)malloc(n * 2);
  uint16_t* got = (uint16_t*)malloc(n * 2);
  void* out = NULL;
  CHECK_CUDA(cudaMalloc(&out, n * 2));
  for (int r = 0; r < W; ++r) {
    host[r] = (uint16_t*)malloc(n * 2);
    hs[r] = host[r];
    CHECK_CUDA(cudaMalloc(&dev[r], n * 2));
  }
  const size_t ws_bytes = arx_ctx_workspace_bytes(W, n, 0);
  void* ws = NULL;
  CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
  CHECK_CUDA(cudaMemset(ws, 0, ws_bytes));
  arx_ctx ctx;
  CHECK_ARX(arx_ctx_init(&ctx, ws, ws_bytes, W, n, 0));
  const int modes[5] = {ARX_SYNC_SEMAPHORE, ARX_SYNC_PAD, ARX_SYNC_PAD_FENCED, ARX_SYNC_CLUSTER,
                        ARX_SYNC_SEMAPHORE_GLOBAL};
  for (int step = 0; step < 6; ++step) {
    for (int r = 0; r < W; ++r) {
      for (size_t i = 0; i < n; ++i) host[r][i] = pattern((uint32_t)(1000 + step * 17 + r), (uint32_t)i);
      CHECK_CUDA(cudaMemcpy(dev[r], host[r], n * 2, cudaMemcpyHostToDevice));
    }
    oracle_reduce(hs, W, want, n);
    if (step < 5) {
      CHECK_ARX(arx_ctx_set_sync(&ctx, modes[step]));
      CHECK_ARX(arx_step(&ctx, (const void* const*)dev, out, n, NULL));
      uint32_t seq = 0, err = 0;
      CHECK_ARX(arx_ctx_query(&ctx, &seq, &err, NULL));
      if (seq != (uint32_t)(step + 1) || err != 0) {
        fprintf(stderr, "arx_step W=%d: seq %u err 0x%08x after step %d\n", W, seq, err, step + 1);
        ++failures;
      }
    } else if (n <= ARX_NOALLOC_MAX_N) {
      CHECK_ARX(arx_step_noalloc((const void* const*)dev, W, out, n, NULL, NULL));
    } else {
      continue;
    }
    CHECK_CUDA(cudaDeviceSynchronize());
    CHECK_CUDA(cudaMemcpy(got, out, n * 2, cudaMemcpyDeviceToHost));
    compare(step < 5 ? "arx_step" : "arx_step_noalloc", W, n, got, want);
  }
  CHECK_CUDA(cudaFree(ws));
  CHECK_CUDA(cudaFree(out));
  for (int r = 0; r < W; ++r) {
    CHECK_CUDA(cudaFree(dev[r]));
    free(host[r]);
  }
  free(want);
  free(got);
}

/* Host partials in page-locked memory: the kernel reads and writes them directly. */
static void host_case(int W, size_t n) {
  void* host[ARX_MAX_W];
  uint16_t* want = (uint16_t*)malloc(n * 2);
  void* hout = NULL;
  for (int r = 0; r < W; ++r) {
    CHECK_CUDA(cudaHostAlloc(&host[r], n * 2, cudaHostAllocDefault));
    for (size_t i = 0; i < n; ++i) ((uint16_t*)host[r])[i] = pattern((uint32_t)(7000 + r), (uint32_t)i);
  }
  CHECK_CUDA(cudaHostAlloc(&hout, n * 2, cudaHostAllocDefault));
  oracle_reduce((const uint16_t* const*)host, W, want, n);
  CHECK_ARX(arx_reduce_host((const void* const*)host, W, hout, n, NULL, 0, NULL));
  CHECK_CUDA(cudaDeviceSynchronize());
  compare("arx_reduce_host (page-locked)", W, n, (const uint16_t*)hout, want);
  for (int r = 0; r < W; ++r) CHECK_CUDA(cudaFreeHost(host[r]));
  CHECK_CUDA(cudaFreeHost(hout));
  free(want);
}

/* External-writer form: this thread is the producer (posts steps 1 and 2,
 * the two banks, before the GPU runs), then the GPU consumes both steps. */
static void ext_case(int W, size_t n) {
  const size_t rb = arx_ext_region_bytes(W, n);
  void* region = NULL;
  void* words = NULL;
  void* out = NULL;
  CHECK_CUDA(cudaHostAlloc(&region, rb, cudaHostAllocDefault));
  memset(region, 0, rb);
  CHECK_CUDA(cudaMalloc(&words, arx_ext_words_bytes()));
  CHECK_CUDA(cudaMemset(words, 0, arx_ext_words_bytes()));
  CHECK_CUDA(cudaMalloc(&out, 2 * n * 2));
  arx_ext x;
  CHECK_ARX(arx_ext_init(&x, words, arx_ext_words_bytes(), region, rb, W, n, 0));
  uint16_t* part[ARX_MAX_W];
  uint16_t* want[2];
  uint16_t* got = (uint16_t*)malloc(n * 2);
  for (int s = 0; s < 2; ++s) {
    want[s] = (uint16_t*)malloc(n * 2);
    for (int r = 0; r < W; ++r) {
      part[r] = (uint16_t*)malloc(n * 2);
      for (size_t i = 0; i < n; ++i) part[r][i] = pattern((uint32_t)(9000 + 31 * s + r), (uint32_t)i);
      CHECK_ARX(arx_ext_post(&x, r, (uint32_t)(s + 1), part[r], n, 1000000000ull));
    }
    oracle_reduce((const uint16_t* const*)part, W, want[s], n);
    for (int r = 0; r < W; ++r) free(part[r]);
  }
  CHECK_ARX(arx_ext_step(&x, out, n, NULL));
  CHECK_ARX(arx_ext_step(&x, (uint16_t*)out + n, n, NULL));
  uint32_t seq = 0, err = 0;
  CHECK_ARX(arx_ext_query(&x, &seq, &err, NULL));
  if (seq != 2 || err != 0) {
    fprintf(stderr, "arx_ext_step W=%d: seq %u err 0x%08x\n", W, seq, err);
    ++failures;
  }
  for (int s = 0; s < 2; ++s) {
    CHECK_CUDA(cudaMemcpy(got, (uint16_t*)out + (size_t)s * n, n * 2, cudaMemcpyDeviceToHost));
    compare("arx_ext_step", W, n, got, want[s]);
    free(want[s]);
  }
  free(got);
  CHECK_CUDA(cudaFree(out));
  CHECK_CUDA(cudaFree(words));
  CHECK_CUDA(cudaFreeHost(region));
}

int main(void) {
  const size_t sizes[4] = {1, 13, 4099, 131072 + 5};
  for (int W = 1; W <= ARX_MAX_W; ++W)
    for (int k = 0; k < 4; ++k) {
      reduce_case(W, sizes[k], 0);
      reduce_case(W, sizes[k], 1);
    }
  step_cases(8, 131072);
  step_cases(3, 5003);
  host_case(8, 131072);
  ext_case(8, 131072);
  ext_case(3, 4099);
  /* Argument errors come back as status codes. */
  if (arx_reduce(NULL, 2, (void*)16, 8, NULL) != ARX_EINVAL) {
    fprintf(stderr, "null slot array not rejected\n");
    ++failures;
  }
  if (failures) {
    fprintf(stderr, "%d failure(s)\n", failures);
    return 1;
  }
  printf("c abi ok\n");
  return 0;
}
