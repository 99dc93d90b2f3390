/* The C ABI used from plain C: device buffers from the CUDA runtime, one call
 * of attn_res on padded rows and a padded bank, and the same inputs through
 * the CPU oracle (attn_res_ref).  Checks: the updated prefix and every bank
 * element bit-exact, out within max(2 bf16 ulp, 1e-2) of the oracle, padding
 * untouched, and the argument errors returned before any launch.  Prints
 * "ok" and exits 0 on success.  Test infrastructure: built and run by
 * tests/test_abi_from_c_gpu.py. */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "attn_res.h"

/* the oracle (oracle/attn_res_ref.c) */
int attn_res_ref(uint16_t* prefix, const uint16_t* delta, uint16_t* blocks, int num_blocks,
                 int block_write_idx, int blocks_capacity, const uint16_t* res_w,
                 const uint16_t* rms_w, const uint16_t* out_norm_w, float eps, float out_eps,
                 uint16_t* out, int64_t T, int64_t H, int64_t prefix_row, int64_t delta_row,
                 int64_t blocks_token, int64_t blocks_slot, int64_t out_row,
                 int64_t blocks_group, double* weights_out, double* logits_out, int n_threads);

#define H ATTN_RES_HIDDEN
#define T 33
#define S 5
#define CAP 9
#define WIDX 8
#define ROW (H + 64)           /* prefix / delta / out row stride */
#define SLOT (H + 64)          /* bank slot stride */
#define TOK (CAP * SLOT + 128) /* bank token stride */
#define PAD_BITS 0x7FA1u       /* a NaN pattern in the padding */

#define CK(x)                                                         \
  do {                                                                \
    cudaError_t e_ = (x);                                             \
    if (e_ != cudaSuccess) {                                          \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));        \
      return 1;                                                       \
    }                                                                 \
  } while (0)

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static double uniform(void) { /* xorshift64*, in [0, 1) */
  rng_state ^= rng_state >> 12;
  rng_state ^= rng_state << 25;
  rng_state ^= rng_state >> 27;
  return (double)((rng_state * 0x2545F4914F6CDD1Dull) >> 11) * (1.0 / 9007199254740992.0);
}
static uint16_t to_bf16(float f) { /* round to nearest even (finite inputs) */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}
static double from_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static void fill(uint16_t* a, size_t n, double lo, double hi) {
  for (size_t i = 0; i < n; ++i) a[i] = to_bf16((float)(lo + (hi - lo) * uniform()));
}

int main(void) {
  const size_t n_row = (size_t)T * ROW, n_bank = (size_t)T * TOK;
  uint16_t* prefix = malloc(n_row * 2);
  uint16_t* delta = malloc(n_row * 2);
  uint16_t* bank = malloc(n_bank * 2);
  uint16_t *res = malloc(H * 2), *rms = malloc(H * 2), *onw = malloc(H * 2);
  uint16_t* out_gpu = malloc(n_row * 2);
  uint16_t *prefix_gpu = malloc(n_row * 2), *bank_gpu = malloc(n_bank * 2);
  uint16_t* out_ref = malloc(n_row * 2);
  if (!prefix || !delta || !bank || !res || !rms || !onw || !out_gpu || !prefix_gpu ||
      !bank_gpu || !out_ref)
    return 1;
  for (size_t i = 0; i < n_row; ++i) prefix[i] = delta[i] = (uint16_t)PAD_BITS;
  for (size_t i = 0; i < n_bank; ++i) bank[i] = (uint16_t)PAD_BITS;
  for (int t = 0; t < T; ++t) {
    fill(prefix + (size_t)t * ROW, H, -2.0, 2.0);
    fill(delta + (size_t)t * ROW, H, -0.5, 0.5);
    for (int i = 0; i < CAP; ++i)
      fill(bank + (size_t)t * TOK + (size_t)i * SLOT, H, -1.0 - i, 1.0 + i);
  }
  fill(res, H, 0.5, 1.5);
  fill(rms, H, 0.5, 1.5);
  fill(onw, H, 0.5, 1.5);

  /* the GPU call */
  void *d_prefix, *d_delta, *d_bank, *d_res, *d_rms, *d_onw, *d_out;
  CK(cudaMalloc(&d_prefix, n_row * 2));
  CK(cudaMalloc(&d_delta, n_row * 2));
  CK(cudaMalloc(&d_bank, n_bank * 2));
  CK(cudaMalloc(&d_res, H * 2));
  CK(cudaMalloc(&d_rms, H * 2));
  CK(cudaMalloc(&d_onw, H * 2));
  CK(cudaMalloc(&d_out, n_row * 2));
  CK(cudaMemcpy(d_prefix, prefix, n_row * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_delta, delta, n_row * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_bank, bank, n_bank * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_res, res, H * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_rms, rms, H * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_onw, onw, H * 2, cudaMemcpyHostToDevice));
  {
    uint16_t* pad = malloc(n_row * 2);
    for (size_t i = 0; i < n_row; ++i) pad[i] = (uint16_t)PAD_BITS;
    CK(cudaMemcpy(d_out, pad, n_row * 2, cudaMemcpyHostToDevice));
    free(pad);
  }
  attn_res_layout_t lay;
  memset(&lay, 0, sizeof lay);
  lay.prefix_row = ROW;
  lay.delta_row = ROW;
  lay.blocks_token = TOK;
  lay.blocks_slot = SLOT;
  lay.out_row = ROW;
  lay.blocks_capacity = CAP;
  lay.flags = 0;
  lay.blocks_group = 1;
  int st = attn_res(d_prefix, d_delta, d_bank, S, WIDX, d_res, d_rms, d_onw, 1e-6f, 1e-6f, d_out, T,
                    &lay, NULL);
  if (st != ATTN_RES_OK) {
    fprintf(stderr, "attn_res: %s\n", attn_res_status_string(st));
    return 1;
  }
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(out_gpu, d_out, n_row * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(prefix_gpu, d_prefix, n_row * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(bank_gpu, d_bank, n_bank * 2, cudaMemcpyDeviceToHost));

  /* the oracle on the host copies (in place, like the call) */
  for (size_t i = 0; i < n_row; ++i) out_ref[i] = (uint16_t)PAD_BITS;
  if (attn_res_ref(prefix, delta, bank, S, WIDX, CAP, res, rms, onw, 1e-6f, 1e-6f, out_ref, T, H,
                   ROW, ROW, TOK, SLOT, ROW, 1, NULL, NULL, 1) != 0) {
    fprintf(stderr, "attn_res_ref failed\n");
    return 1;
  }
  int bad = 0;
  for (size_t i = 0; i < n_row; ++i) {
    const size_t col = i % ROW;
    if (col >= H) {
      bad += out_gpu[i] != PAD_BITS || prefix_gpu[i] != PAD_BITS;
      continue;
    }
    bad += prefix_gpu[i] != prefix[i];
    const double g = from_bf16(out_gpu[i]), r = from_bf16(out_ref[i]);
    const double ulp = ldexp(1.0, (r == 0.0 ? -133 : ilogb(r)) - 7);
    const double tol = fmax(2.0 * ulp, 1e-2);
    bad += !(fabs(g - r) <= tol);
  }
  for (size_t i = 0; i < n_bank; ++i) bad += bank_gpu[i] != bank[i];
  if (bad) {
    fprintf(stderr, "%d elements differ from the oracle\n", bad);
    return 1;
  }

  /* argument errors, returned before any launch */
  if (attn_res(d_prefix, d_delta, d_bank, 9, -1, d_res, d_rms, d_onw, 1e-6f, 1e-6f, d_out, T, &lay,
               NULL) != ATTN_RES_EINVAL)
    return 1;
  if (attn_res((void*)((char*)d_prefix + 2), d_delta, d_bank, S, -1, d_res, d_rms, d_onw, 1e-6f, 1e-6f,
               d_out, T, &lay, NULL) != ATTN_RES_EALIGN)
    return 1;
  if (attn_res(d_prefix, d_delta, d_bank, S, -1, d_res, d_rms, d_onw, 1e-6f, 1e-6f, d_prefix, T,
               &lay, NULL) != ATTN_RES_EALIAS)
    return 1;
  if (attn_res_status_string(ATTN_RES_EINVAL) == NULL || attn_res_hidden_size() != H) return 1;
  unsigned bits = 1;
  if (attn_res_device_status(&bits, 0) != ATTN_RES_OK || bits != 0) return 1;
  printf("ok\n");
  return 0;
}
