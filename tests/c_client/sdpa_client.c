/*
 * A plain C caller of libsdpa (no Python, no torch): it allocates device and
 * page-locked host memory with the CUDA runtime, runs the bf16 attention of
 * "Attention Is All You Need" (section 3.2.1, Eq. (1), causal and key
 * padding masks of section 3.2.3) through sdpa_forward on device buffers and
 * through sdpa_forward_host on host buffers, and compares both with the C
 * oracle (test infrastructure, linked only here) row by row.
 *
 * Inputs come from a fixed linear congruential sequence rounded to bf16; the
 * same arrays go to the library and to the oracle.  Prints "c client ok" and
 * returns 0 when every output row is within 2e-2 of its own scale.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "sdpa.h"

/* the oracle's entry point (oracle/oracle.c) */
int oracle_sdpa(const float* q, const float* k, const float* v, double* out, int b, int h, int n_q,
                int n_k, int d_k, int d_v, int mask_kind, const int32_t* kv_lengths, double scale,
                const int64_t* rows, int64_t n_rows, int n_threads);

static uint64_t g_state = 12345u;

/* uniform in (-1, 1), then rounded to bf16 (nearest even); returns the bits */
static uint16_t next_bf16(float* as_float) {
  g_state = g_state * 6364136223846793005ull + 1442695040888963407ull;
  const float x = (float)((double)(g_state >> 11) / 9007199254740992.0) * 2.0f - 1.0f;
  uint32_t bits;
  memcpy(&bits, &x, 4);
  bits = (bits + 0x7fffu + ((bits >> 16) & 1u)) & 0xffff0000u;
  memcpy(as_float, &bits, 4);
  return (uint16_t)(bits >> 16);
}

static float bf16_to_float(uint16_t u) {
  const uint32_t bits = (uint32_t)u << 16;
  float f;
  memcpy(&f, &bits, 4);
  return f;
}

#define CHECK_CUDA(x)                                                         \
  do {                                                                        \
    cudaError_t e_ = (x);                                                     \
    if (e_ != cudaSuccess) {                                                  \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                \
      return 2;                                                               \
    }                                                                         \
  } while (0)

#define CHECK_SDPA(x)                                                         \
  do {                                                                        \
    sdpa_status s_ = (x);                                                     \
    if (s_ != SDPA_OK) {                                                      \
      fprintf(stderr, "%s: %s\n", #x, sdpa_status_string(s_));                \
      return 3;                                                               \
    }                                                                         \
  } while (0)

/* largest per-row error: max_c |got - ref| / max_c |ref| (absolute for a zero row) */
static double row_error(const uint16_t* got, const double* ref, long rows, int cols) {
  double worst = 0.0;
  for (long r = 0; r < rows; ++r) {
    double scale = 0.0, err = 0.0;
    for (int c = 0; c < cols; ++c) {
      const double g = bf16_to_float(got[r * cols + c]), x = ref[r * cols + c];
      if (fabs(x) > scale) scale = fabs(x);
      if (fabs(g - x) > err) err = fabs(g - x);
    }
    const double e = scale > 0.0 ? err / scale : err;
    if (e > worst) worst = e;
  }
  return worst;
}

int main(void) {
  const int b = 2, h = 3, n = 300, d = 64;
  const int mask = SDPA_MASK_CAUSAL | SDPA_MASK_PADDING;
  const long elems = (long)b * h * n * d;
  const size_t bytes = (size_t)elems * 2;
  const int32_t lens[2] = {300, 171};

  uint16_t *qh, *kh, *vh, *oh;
  CHECK_CUDA(cudaMallocHost((void**)&qh, bytes));
  CHECK_CUDA(cudaMallocHost((void**)&kh, bytes));
  CHECK_CUDA(cudaMallocHost((void**)&vh, bytes));
  CHECK_CUDA(cudaMallocHost((void**)&oh, bytes));
  float* qf = (float*)malloc(elems * 4);
  float* kf = (float*)malloc(elems * 4);
  float* vf = (float*)malloc(elems * 4);
  double* ref = (double*)malloc(elems * 8);
  uint16_t* od_host = (uint16_t*)malloc(bytes);
  for (long i = 0; i < elems; ++i) qh[i] = next_bf16(&qf[i]);
  for (long i = 0; i < elems; ++i) kh[i] = next_bf16(&kf[i]);
  for (long i = 0; i < elems; ++i) vh[i] = next_bf16(&vf[i]);

  if (oracle_sdpa(qf, kf, vf, ref, b, h, n, n, d, d, mask, lens, 0.0, NULL, 0, 4) != 0) {
    fprintf(stderr, "oracle rejected the arguments\n");
    return 4;
  }

  void *qd, *kd, *vd, *od;
  int32_t* lens_d;
  CHECK_CUDA(cudaMalloc(&qd, bytes));
  CHECK_CUDA(cudaMalloc(&kd, bytes));
  CHECK_CUDA(cudaMalloc(&vd, bytes));
  CHECK_CUDA(cudaMalloc(&od, bytes));
  CHECK_CUDA(cudaMalloc((void**)&lens_d, sizeof(lens)));
  CHECK_CUDA(cudaMemcpy(lens_d, lens, sizeof(lens), cudaMemcpyHostToDevice));

  /* 1. device buffers */
  CHECK_CUDA(cudaMemcpy(qd, qh, bytes, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(kd, kh, bytes, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(vd, vh, bytes, cudaMemcpyHostToDevice));
  CHECK_SDPA(sdpa_forward(qd, kd, vd, od, b, h, n, n, d, d, mask, lens_d, 0.0f, NULL));
  CHECK_SDPA(sdpa_device_check());
  CHECK_CUDA(cudaMemcpy(od_host, od, bytes, cudaMemcpyDeviceToHost));
  const double e1 = row_error(od_host, ref, (long)b * h * n, d);

  /* 2. host buffers, pipelined inside the library, two heads per chunk */
  CHECK_CUDA(cudaMemset(od, 0, bytes));
  CHECK_SDPA(sdpa_forward_host(qh, kh, vh, oh, qd, kd, vd, od, b, h, n, n, d, d, mask, lens_d,
                               0.0f, 2, NULL));
  CHECK_CUDA(cudaStreamSynchronize(NULL));
  CHECK_SDPA(sdpa_device_check());
  const double e2 = row_error(oh, ref, (long)b * h * n, d);
  const int same = memcmp(oh, od_host, bytes) == 0;

  /* 3. a bad argument is refused on the host, by name */
  const sdpa_status bad = sdpa_forward(NULL, kd, vd, od, b, h, n, n, d, d, mask, lens_d, 0.0f, NULL);

  printf("row error: device buffers %.3g, host buffers %.3g; identical %d; null q -> %s\n", e1, e2,
         same, sdpa_status_string(bad));
  if (e1 > 2e-2 || e2 > 2e-2 || !same || bad != SDPA_ERR_INVALID_ARG) return 1;
  printf("c client ok\n");
  return 0;
}
