/*
 * A plain C99 program that uses the library through include/ra.h alone: no
 * C++, no Python.  It shows that the boundary is a C ABI.
 *
 *   ra_consumer cpu   status strings, argument validation and workspace
 *                     sizes: no CUDA call is reached (runs without a GPU).
 *   ra_consumer gpu   a bf16 ring forward (B = 1, H = 2, N = 512, d = 128,
 *                     P = 4, "Ring Attention: the math", section "The ring
 *                     schedule: passing K/V around") on device buffers, checked
 *                     against the fp64 oracle's ring (C entry point ora_ring).
 *
 * Prints "ok" and exits 0 on success.  Build lines are in
 * tests/test_c_consumer.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ra.h"

#define CHECK(cond, ...)                      \
  do {                                        \
    if (!(cond)) {                            \
      fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
      fprintf(stderr, __VA_ARGS__);           \
      fprintf(stderr, "\n");                  \
      exit(1);                                \
    }                                         \
  } while (0)

static int cpu_checks(void) {
  /* 16-byte aligned stand-ins, never dereferenced.  Every call below breaks
     one rule and also passes a backstop that the library checks later, still
     before any device work: a misaligned lse (or, where the broken rule is
     an alignment, a NULL out).  A validation that failed to reject its case
     would then return that later error, not launch anything. */
  static unsigned char raw[1024];
  void* buf = (void*)(((uintptr_t)raw + 15u) & ~(uintptr_t)15u);
  const void* p = buf;
  float* lse_bad = (float*)((char*)buf + 2);
  int code;
  for (code = RA_OK; code <= RA_ERR_TIMEOUT; ++code) {
    const char* s = ra_status_string((ra_status)code);
    CHECK(s && s[0], "status string %d", code);
  }
  CHECK(ra_forward(NULL, p, p, buf, lse_bad, 1, 1, 256, 128, 2, RA_BF16, NULL) ==
            RA_ERR_INVALID_ARG, "null q");
  CHECK(ra_forward(p, p, p, buf, lse_bad, -1, 1, 256, 128, 2, RA_BF16, NULL) ==
            RA_ERR_INVALID_ARG, "negative B");
  CHECK(ra_forward(p, p, p, buf, lse_bad, 1, 1, 256, 128, 0, RA_BF16, NULL) ==
            RA_ERR_INVALID_ARG, "P = 0");
  CHECK(ra_forward(p, p, p, buf, lse_bad, 1, 1, 256, 128, 2, (ra_dtype)7, NULL) ==
            RA_ERR_INVALID_ARG, "bad dtype");
  CHECK(ra_forward(p, p, p, buf, lse_bad, 1, 1, 300, 128, 7, RA_BF16, NULL) ==
            RA_ERR_UNSUPPORTED, "P does not divide N");
  CHECK(ra_forward(p, p, p, buf, lse_bad, 1, 1, 256, 96, 2, RA_BF16, NULL) ==
            RA_ERR_UNSUPPORTED, "bf16 d = 96");
  CHECK(ra_forward(p, p, p, buf, lse_bad, 1, 1, 256, 300, 2, RA_F32, NULL) ==
            RA_ERR_UNSUPPORTED, "f32 d > 256");
  CHECK(ra_forward((const char*)p + 4, p, p, NULL, (float*)buf, 1, 1, 256, 128, 2, RA_BF16,
                   NULL) == RA_ERR_MISALIGNED, "misaligned q");
  CHECK(ra_forward_causal(p, p, p, buf, lse_bad, 1, 1, 256, 128, 2, (ra_layout)9, RA_BF16,
                          NULL) == RA_ERR_INVALID_ARG, "bad layout");
  CHECK(ra_forward(p, p, p, buf, lse_bad, 1, 1, 256, 128, 2, RA_BF16, NULL) ==
            RA_ERR_MISALIGNED, "the backstop itself");
  /* zero rows: nothing to do, and no device needed */
  CHECK(ra_forward(NULL, NULL, NULL, NULL, NULL, 0, 4, 256, 128, 2, RA_BF16, NULL) == RA_OK,
        "empty call");
  /* G partial states of rows x d fp32, each section rounded up to 256 bytes */
  {
    const int64_t rows = 1 * 8 * 4096, d = 64, G = 4;
    const int64_t want = G * (2 * ((rows * 4 + 255) / 256 * 256) + (rows * d * 4 + 255) / 256 * 256);
    CHECK(ra_forward_split_workspace_bytes(1, 8, 4096, 64, 4) == want, "split workspace");
    CHECK(ra_forward_split_workspace_bytes(1, 8, 4096, 64, 0) < 0, "G = 0");
  }
  return 0;
}

#ifdef RA_CONSUMER_GPU
#include <cuda_runtime.h>

int ora_ring(const void* q, const void* k, const void* v, int dtype, int64_t BH, int64_t N,
             int d, int64_t P, const int64_t* order, int64_t t0, int64_t t1, int64_t tile,
             int causal, int layout, const int64_t* rows, int64_t R, double* out, double* lse,
             double* m_out, double* l_out, double* o_out, int threads);

static uint64_t splitmix64(uint64_t* s) {
  uint64_t z = (*s += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* roughly N(0, 1): the sum of four uniforms, centred and scaled (Irwin-Hall) */
static float draw(uint64_t* s) {
  double u = 0.0;
  int x;
  for (x = 0; x < 4; ++x) u += (double)(splitmix64(s) >> 11) * (1.0 / 9007199254740992.0);
  return (float)((u - 2.0) * sqrt(3.0));
}

/* float -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t to_bf16(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  b += 0x7FFFu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

static float from_bf16(uint16_t h) {
  uint32_t b = (uint32_t)h << 16;
  float f;
  memcpy(&f, &b, 4);
  return f;
}

static int gpu_check(void) {
  const int B = 1, H = 2, d = 128, P = 4;
  const int64_t N = 512, rows = (int64_t)B * H * N, n = rows * d;
  uint16_t *hq = malloc(n * 2), *hk = malloc(n * 2), *hv = malloc(n * 2), *ho = malloc(n * 2);
  float* hl = malloc(rows * 4);
  double *wo = malloc(n * 8), *wl = malloc(rows * 8);
  void *dq, *dk, *dv, *dout;
  float* dlse;
  uint64_t seed = 20261203u;
  int64_t x;
  double e_out = 0.0, e_lse = 0.0, ref_max = 0.0;
  for (x = 0; x < n; ++x) hq[x] = to_bf16(draw(&seed));
  for (x = 0; x < n; ++x) hk[x] = to_bf16(draw(&seed));
  for (x = 0; x < n; ++x) hv[x] = to_bf16(draw(&seed));
  CHECK(cudaMalloc(&dq, n * 2) == cudaSuccess && cudaMalloc(&dk, n * 2) == cudaSuccess &&
            cudaMalloc(&dv, n * 2) == cudaSuccess && cudaMalloc(&dout, n * 2) == cudaSuccess &&
            cudaMalloc((void**)&dlse, rows * 4) == cudaSuccess, "cudaMalloc");
  cudaMemcpy(dq, hq, n * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dk, hk, n * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dv, hv, n * 2, cudaMemcpyHostToDevice);
  CHECK(ra_forward(dq, dk, dv, dout, dlse, B, H, N, d, P, RA_BF16, NULL) == RA_OK, "ra_forward");
  CHECK(ra_last_device_status(NULL) == RA_OK, "device status");
  CHECK(cudaMemcpy(ho, dout, n * 2, cudaMemcpyDeviceToHost) == cudaSuccess &&
            cudaMemcpy(hl, dlse, rows * 4, cudaMemcpyDeviceToHost) == cudaSuccess, "copy back");
  CHECK(ora_ring(hq, hk, hv, 2, (int64_t)B * H, N, d, P, NULL, 0, P, 0, 0, 0, NULL, rows, wo, wl,
                 NULL, NULL, NULL, 4) == 0, "ora_ring");
  for (x = 0; x < n; ++x) {
    const double e = fabs((double)from_bf16(ho[x]) - wo[x]);
    if (e > e_out) e_out = e;
    if (fabs(wo[x]) > ref_max) ref_max = fabs(wo[x]);
  }
  for (x = 0; x < rows; ++x) {
    const double e = fabs((double)hl[x] - wl[x]);
    if (e > e_lse) e_lse = e;
  }
  printf("max-abs out %.3e (max|ref| %.3e), max-abs lse %.3e\n", e_out, ref_max, e_lse);
  CHECK(e_out <= 2e-2 && e_out <= ref_max / 64.0, "out error %.3e", e_out);
  CHECK(e_lse <= 1e-3, "lse error %.3e", e_lse);
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(dout);
  cudaFree(dlse);
  free(hq); free(hk); free(hv); free(ho); free(hl); free(wo); free(wl);
  return 0;
}
#endif

int main(int argc, char** argv) {
  const char* mode = argc > 1 ? argv[1] : "cpu";
  cpu_checks();
  if (strcmp(mode, "gpu") == 0) {
#ifdef RA_CONSUMER_GPU
    gpu_check();
#else
    fprintf(stderr, "built without RA_CONSUMER_GPU\n");
    return 2;
#endif
  }
  printf("ok\n");
  return 0;
}
