/*
 * c_abi_check.c -- calls libfp8attn.so from plain C through include/fp8attn.h,
 * with no Python or PyTorch: device buffers from the CUDA runtime, a stream,
 * one Lean-P call, one BF16 call and one rejected call.  Built and run by
 * tests/test_gpu_c_abi.py.
 *
 * Checks (exact, so no reference computation is needed):
 *   - V = e4m3 1.0 everywhere with descale_v = 1: every output is bf16 1.0,
 *     because the rounded row sum makes the weights sum to one exactly
 *     ("Per-block scaling and a rounded row sum").
 *   - The same for the BF16 path with V = bf16 1.0 (the probabilities are
 *     rounded to bf16 but the row sum is not, so the output is only close to
 *     1; it must be within 2^-7).
 *   - A NULL q pointer returns ATTN_ERR_INVALID_ARG before any launch.
 * Exit status 0 on success; the failing check is printed otherwise.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fp8attn.h"

#define CHECK_CUDA(x)                                                              \
  do {                                                                             \
    cudaError_t e_ = (x);                                                          \
    if (e_ != cudaSuccess) {                                                       \
      fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));              \
      return 2;                                                                    \
    }                                                                              \
  } while (0)

static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Deterministic pseudo-random bytes (xorshift32) turned into e4m3 codes of
 * magnitude below 2 (exponent field 0..7) so that every code is finite. */
static uint32_t rng_state = 12345u;
static uint8_t next_code(void) {
  rng_state ^= rng_state << 13;
  rng_state ^= rng_state >> 17;
  rng_state ^= rng_state << 5;
  return (uint8_t)(rng_state & 0xBFu); /* clear bit 6: exponent < 8 */
}

int main(void) {
  const int B = 1, Hq = 4, Hkv = 2, S = 300, D = 128;
  const size_t nq = (size_t)B * S * Hq * D, nk = (size_t)B * S * Hkv * D;
  printf("fp8attn API version %d\n", attn_api_version());
  if (attn_api_version() != FP8ATTN_API_VERSION) {
    fprintf(stderr, "library and header versions differ\n");
    return 1;
  }
  /* the split schedule, from the host alone: 4 heads at 8K keys on 152 SMs
   * split their last 13 query blocks in two */
  {
    int qb = -1, ns = -1;
    size_t nb = 0;
    if (attn_split_plan(ATTN_VARIANT_LEANP, 1, 4, 4, 8192, 128, 128, 1, 0, 152, &qb, &ns, &nb) !=
            ATTN_OK ||
        qb != 19 || ns != 2 || nb == 0) {
      fprintf(stderr, "attn_split_plan: %d %d %zu\n", qb, ns, nb);
      return 1;
    }
  }

  uint8_t *hq = malloc(nq), *hk = malloc(nk), *hv = malloc(nk);
  uint16_t* hout = malloc(nq * 2);
  for (size_t i = 0; i < nq; ++i) hq[i] = next_code();
  for (size_t i = 0; i < nk; ++i) hk[i] = next_code();
  memset(hv, 0x38, nk); /* e4m3 1.0 */
  const float desc[3] = {0.05f, 0.05f, 1.0f};

  void *q, *k, *v, *out;
  float* d;
  cudaStream_t st;
  CHECK_CUDA(cudaMalloc(&q, nq));
  CHECK_CUDA(cudaMalloc(&k, nk));
  CHECK_CUDA(cudaMalloc(&v, nk));
  CHECK_CUDA(cudaMalloc(&out, nq * 2));
  CHECK_CUDA(cudaMalloc((void**)&d, 3 * sizeof(float)));
  CHECK_CUDA(cudaStreamCreate(&st));
  CHECK_CUDA(cudaMemcpy(q, hq, nq, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(k, hk, nk, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(v, hv, nk, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(d, desc, sizeof desc, cudaMemcpyHostToDevice));

  int rc = attn_fwd_fp8(q, k, v, d, d + 1, d + 2, out, B, Hq, Hkv, S, D, D, 1, st);
  if (rc != ATTN_OK) {
    fprintf(stderr, "attn_fwd_fp8: %s\n", attn_status_string(rc));
    return 1;
  }
  CHECK_CUDA(cudaStreamSynchronize(st));
  CHECK_CUDA(cudaMemcpy(hout, out, nq * 2, cudaMemcpyDeviceToHost));
  for (size_t i = 0; i < nq; ++i)
    if (hout[i] != 0x3F80u) { /* bf16 1.0 */
      fprintf(stderr, "Lean-P with V = 1: element %zu is %g\n", i, bf16_to_float(hout[i]));
      return 1;
    }

  /* BF16: q, k, v as bf16 bit patterns (q, k small integers / 16; v = 1.0) */
  uint16_t *bq = malloc(nq * 2), *bk = malloc(nk * 2), *bv = malloc(nk * 2);
  for (size_t i = 0; i < nq; ++i) bq[i] = (uint16_t)(0x3D80u + (next_code() & 0x3Fu));
  for (size_t i = 0; i < nk; ++i) bk[i] = (uint16_t)(0x3D80u + (next_code() & 0x3Fu));
  for (size_t i = 0; i < nk; ++i) bv[i] = 0x3F80u;
  void *q2, *k2, *v2;
  CHECK_CUDA(cudaMalloc(&q2, nq * 2));
  CHECK_CUDA(cudaMalloc(&k2, nk * 2));
  CHECK_CUDA(cudaMalloc(&v2, nk * 2));
  CHECK_CUDA(cudaMemcpy(q2, bq, nq * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(k2, bk, nk * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(v2, bv, nk * 2, cudaMemcpyHostToDevice));
  rc = attn_fwd_bf16(q2, k2, v2, out, B, Hq, Hkv, S, D, D, 1, st);
  if (rc != ATTN_OK) {
    fprintf(stderr, "attn_fwd_bf16: %s\n", attn_status_string(rc));
    return 1;
  }
  CHECK_CUDA(cudaStreamSynchronize(st));
  CHECK_CUDA(cudaMemcpy(hout, out, nq * 2, cudaMemcpyDeviceToHost));
  for (size_t i = 0; i < nq; ++i)
    if (fabsf(bf16_to_float(hout[i]) - 1.0f) > 0.0078125f) {
      fprintf(stderr, "BF16 with V = 1: element %zu is %g\n", i, bf16_to_float(hout[i]));
      return 1;
    }

  rc = attn_fwd_fp8(NULL, k, v, d, d + 1, d + 2, out, B, Hq, Hkv, S, D, D, 1, st);
  if (rc != ATTN_ERR_INVALID_ARG) {
    fprintf(stderr, "NULL q returned %d\n", rc);
    return 1;
  }
  printf("C ABI check ok: Lean-P and BF16 calls from C, V = 1 gives 1, NULL q rejected (%s)\n",
         attn_status_string(rc));
  cudaFree(q), cudaFree(k), cudaFree(v), cudaFree(out), cudaFree(d);
  cudaFree(q2), cudaFree(k2), cudaFree(v2);
  cudaStreamDestroy(st);
  free(hq), free(hk), free(hv), free(hout), free(bq), free(bk), free(bv);
  return 0;
}
