/*
 * abi_smoke.c — uses libloco through include/loco.h only, as a C caller would.
 *
 *   abi_smoke cpu   sizes, status strings and host-side argument errors (no GPU needed)
 *   abi_smoke gpu   the caller allocates device buffers with cudaMalloc and runs the
 *                   hand-derived worked example of "LoCo: Low-Bit Communication Adaptor
 *                   for Large-scale Model Training" §3.1-3.2 (4-bit, block 64, beta 1/2,
 *                   two steps) and the two-rank average of §3.3, checking exact values.
 *
 * Exit status 0 on success; the first failed check is printed.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "loco.h"

#define CHECK(cond, ...)                      \
  do {                                        \
    if (!(cond)) {                            \
      fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
      fprintf(stderr, __VA_ARGS__);           \
      fprintf(stderr, "\n");                  \
      return 1;                               \
    }                                         \
  } while (0)

static int cpu_checks(void) {
  loco_config cfg = {4, 256, LOCO_SCALE_ABSMAX, 0.0f, 0.9f, 4.0f, 0};
  CHECK(loco_num_blocks(257, 256) == 2, "num_blocks");
  CHECK(loco_code_bytes(6738415616LL, 4, 256) == 3369207808LL, "code_bytes 7B");
  CHECK(strcmp(loco_status_string(LOCO_ERR_MISALIGNED), "LOCO_ERR_MISALIGNED") == 0, "status string");
  /* argument errors are reported before any CUDA call */
  loco_config bad = cfg;
  bad.bits = 5;
  CHECK(loco_compress(&bad, (void*)0x1000, LOCO_F32, (float*)0x2000, 100, 1, (uint8_t*)0x3000, (float*)0x4000, NULL) ==
            LOCO_ERR_UNSUPPORTED, "bits 5");
  CHECK(loco_compress(&cfg, (void*)0x1001, LOCO_F32, (float*)0x2000, 100, 1, (uint8_t*)0x3000, (float*)0x4000, NULL) ==
            LOCO_ERR_MISALIGNED, "misaligned grad");
  CHECK(loco_compress(&cfg, NULL, LOCO_F32, (float*)0x2000, 100, 1, (uint8_t*)0x3000, (float*)0x4000, NULL) ==
            LOCO_ERR_INVALID_ARG, "null grad");
  CHECK(strlen(loco_last_error()) > 0, "last error text");
  CHECK(loco_compress(&cfg, NULL, LOCO_F32, NULL, 0, 1, NULL, NULL, NULL) == LOCO_OK, "empty call");
  const uint8_t* codes[17] = {0};
  const float* scales[17] = {0};
  CHECK(loco_decode_reduce(&cfg, codes, scales, 17, 10, (float*)0x1000, NULL) == LOCO_ERR_UNSUPPORTED, "W 17");
  CHECK(loco_decode_reduce(&cfg, codes, scales, 0, 10, (float*)0x1000, NULL) == LOCO_ERR_INVALID_ARG, "W 0");
  return 0;
}

/* Minimal CUDA runtime declarations (the caller links libcudart). */
typedef int cudaError_t;
extern cudaError_t cudaMalloc(void** p, size_t n);
extern cudaError_t cudaFree(void* p);
extern cudaError_t cudaMemcpy(void* dst, const void* src, size_t n, int kind);
extern cudaError_t cudaMemset(void* p, int v, size_t n);
extern cudaError_t cudaDeviceSynchronize(void);
enum { H2D = 1, D2H = 2 };

static int gpu_checks(void) {
  const float u = 1.0f / 1024.0f; /* 2^-10 */
  const float head[8] = {7, -3.5f, 2.5f, 1.5f, 0.5f, -0.5f, -2.5f, 3.25f};
  _Alignas(16) float g[64] = {0};
  for (int j = 0; j < 8; ++j) g[j] = head[j] * u;
  loco_config cfg = {4, 64, LOCO_SCALE_ABSMAX, 0.0f, 0.5f, 4.0f, 0};
  void *dg, *de, *dc0, *dc1, *ds0, *ds1, *dm;
  CHECK(cudaMalloc(&dg, 256) == 0 && cudaMalloc(&de, 256) == 0 && cudaMalloc(&dc0, 32) == 0 &&
            cudaMalloc(&dc1, 32) == 0 && cudaMalloc(&ds0, 4) == 0 && cudaMalloc(&ds1, 4) == 0 &&
            cudaMalloc(&dm, 256) == 0, "cudaMalloc");
  CHECK(cudaMemcpy(dg, g, sizeof g, H2D) == 0 && cudaMemset(de, 0, 256) == 0, "upload");
  /* step 1 and step 2 of worked example A */
  CHECK(loco_compress(&cfg, dg, LOCO_F32, (float*)de, 64, 1, (uint8_t*)dc0, (float*)ds0, NULL) == LOCO_OK, "%s",
        loco_last_error());
  CHECK(loco_compress(&cfg, dg, LOCO_F32, (float*)de, 64, 2, (uint8_t*)dc1, (float*)ds1, NULL) == LOCO_OK, "%s",
        loco_last_error());
  uint8_t c0[32], c1[32];
  float e[64], s0, s1;
  CHECK(cudaMemcpy(c0, dc0, 32, D2H) == 0 && cudaMemcpy(c1, dc1, 32, D2H) == 0 && cudaMemcpy(e, de, 256, D2H) == 0 &&
            cudaMemcpy(&s0, ds0, 4, D2H) == 0 && cudaMemcpy(&s1, ds1, 4, D2H) == 0, "download");
  const uint8_t want0[4] = {0xc7, 0x22, 0x00, 0x3e}, want1[4] = {0xd7, 0x13, 0xf1, 0x3d};
  CHECK(memcmp(c0, want0, 4) == 0, "step 1 codes %02x %02x %02x %02x", c0[0], c0[1], c0[2], c0[3]);
  CHECK(memcmp(c1, want1, 4) == 0, "step 2 codes %02x %02x %02x %02x", c1[0], c1[1], c1[2], c1[3]);
  for (int j = 4; j < 32; ++j) CHECK(c0[j] == 0 && c1[j] == 0, "zero codes");
  CHECK(s0 == u && s1 == u, "scales");
  for (int j = 0; j < 64; ++j) CHECK(e[j] == (j == 7 ? 0.25f * u : 0.0f), "error %d = %g", j, e[j]);
  /* average of the two packed buckets (§3.3): [7,-3.5,2.5,1.5,0.5,-0.5,-2.5,3] u */
  const uint8_t* cc[2] = {(const uint8_t*)dc0, (const uint8_t*)dc1};
  const float* ss[2] = {(const float*)ds0, (const float*)ds1};
  CHECK(loco_decode_reduce(&cfg, cc, ss, 2, 64, (float*)dm, NULL) == LOCO_OK, "%s", loco_last_error());
  float mean[64];
  CHECK(cudaMemcpy(mean, dm, 256, D2H) == 0, "download mean");
  const float wm[8] = {7, -3.5f, 2.5f, 1.5f, 0.5f, -0.5f, -2.5f, 3};
  for (int j = 0; j < 64; ++j) CHECK(mean[j] == (j < 8 ? wm[j] * u : 0.0f), "mean %d = %g", j, mean[j]);
  /* a (16-byte aligned) host pointer is refused, not dereferenced */
  loco_status hs = loco_compress(&cfg, g, LOCO_F32, (float*)de, 64, 3, (uint8_t*)dc0, (float*)ds0, NULL);
  CHECK(hs == LOCO_ERR_INVALID_ARG, "host pointer: status %s (%s)", loco_status_string(hs), loco_last_error());
  CHECK(cudaDeviceSynchronize() == 0, "sync");
  cudaFree(dg); cudaFree(de); cudaFree(dc0); cudaFree(dc1); cudaFree(ds0); cudaFree(ds1); cudaFree(dm);
  return 0;
}

int main(int argc, char** argv) {
  if (argc > 1 && strcmp(argv[1], "gpu") == 0) {
    int rc = cpu_checks();
    if (rc == 0) rc = gpu_checks();
    if (rc == 0) printf("abi_smoke gpu: ok\n");
    return rc;
  }
  int rc = cpu_checks();
  if (rc == 0) printf("abi_smoke cpu: ok\n");
  return rc;
}
