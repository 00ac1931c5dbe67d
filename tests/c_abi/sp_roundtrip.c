/*
 * A plain C consumer of the boundary's C ABI (include/sp_boundary.h): no
 * C++, no Python, no PyTorch -- device memory from the CUDA runtime API
 * (whose header needs C11; sp_boundary.h alone is plain C89),
 * one forward (sp_rs_norm_fwd) and the backward that reads its saved Z,
 * mask and statistics (sp_norm_bwd), on the legacy default stream.
 *
 * usage: sp_roundtrip IN OUT t b s h norm p seed offset eps [bits]
 *
 * With the last argument "bits" the pair is sp_rs_norm_fwd_bitmask /
 * sp_norm_bwd_bitmask and the masks are (b, s_k, h / 8) bit-packed bytes.
 *
 * IN holds, as raw little-endian arrays in this order: the t partials
 * (b, s, h) bf16; the t residual shards (b, s_k, h) bf16; bias, gamma,
 * beta (h) bf16; the t dY shards (b, s_k, h) bf16.  Shard k is tokens
 * [o_k, o_{k+1}) of every batch row, o_k = floor(k * s / t).
 * OUT receives: the t Z shards (bf16), the t masks (u8, bytes or bits), the
 * t mean rows (f32, LayerNorm only), the t rstd rows (f32), one gathered copy of O
 * (b, s, h) bf16, the t dResidual shards (bf16), one dYpre copy (b, s, h)
 * bf16, dgamma, dbeta (LayerNorm only), dbias (h) f32, and the int32
 * device status word.  Exit status 0 on success, 1 on any error (with the
 * library's or the runtime's message on stderr).
 */
#include <inttypes.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "sp_boundary.h"

#define MAXT SP_MAX_RANKS

static int cuda_ok(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return 1;
  fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
  return 0;
}

static int sp_ok(sp_status_t st, const char* what) {
  if (st == SP_OK) return 1;
  fprintf(stderr, "%s: status %d: %s\n", what, (int)st, sp_last_error());
  return 0;
}

/* A device buffer of `bytes` (at least 16, so empty shards still get a pointer). */
static void* dev_alloc(size_t bytes) {
  void* p = NULL;
  if (!cuda_ok(cudaMalloc(&p, bytes < 16 ? 16 : bytes), "cudaMalloc")) return NULL;
  return p;
}

/* Reads `bytes` from f into a new device buffer. */
static void* read_to_device(FILE* f, size_t bytes) {
  void* d = dev_alloc(bytes);
  void* h = malloc(bytes < 16 ? 16 : bytes);
  if (d == NULL || h == NULL) return NULL;
  if (bytes > 0 && fread(h, 1, bytes, f) != bytes) {
    fprintf(stderr, "short input file\n");
    return NULL;
  }
  if (!cuda_ok(cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice), "copy in")) return NULL;
  free(h);
  return d;
}

/* Appends `bytes` of device buffer d to f. */
static int write_from_device(FILE* f, const void* d, size_t bytes) {
  void* h = malloc(bytes < 16 ? 16 : bytes);
  if (h == NULL) return 0;
  if (!cuda_ok(cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost), "copy out")) return 0;
  const int ok = fwrite(h, 1, bytes, f) == bytes;
  free(h);
  return ok;
}

int main(int argc, char** argv) {
  if (argc != 12 && argc != 13) {
    fprintf(stderr, "usage: %s IN OUT t b s h norm p seed offset eps [bits]\n", argv[0]);
    return 1;
  }
  const int bits = argc == 13 && strcmp(argv[12], "bits") == 0;
  const int32_t t = (int32_t)atoi(argv[3]);
  const int64_t b = strtoll(argv[4], NULL, 10), s = strtoll(argv[5], NULL, 10);
  const int64_t h = strtoll(argv[6], NULL, 10);
  const sp_norm_t norm = strcmp(argv[7], "rmsnorm") == 0 ? SP_NORM_RMSNORM : SP_NORM_LAYERNORM;
  const double p = strtod(argv[8], NULL);
  const uint64_t seed = strtoull(argv[9], NULL, 10), offset = strtoull(argv[10], NULL, 10);
  const float eps = (float)strtod(argv[11], NULL);
  const int ln = norm == SP_NORM_LAYERNORM;
  if (t < 1 || t > MAXT || b < 1 || s < 1 || h < 8) {
    fprintf(stderr, "bad sizes\n");
    return 1;
  }
  if (sp_abi_version() < 1) return 1;

  size_t rows_k[MAXT];
  for (int k = 0; k < t; ++k)
    rows_k[k] = (size_t)(b * (((int64_t)(k + 1) * s) / t - ((int64_t)k * s) / t));
  const size_t full = (size_t)(b * s * h);

  FILE* in = fopen(argv[1], "rb");
  if (in == NULL) {
    perror(argv[1]);
    return 1;
  }
  const void* partials[MAXT];
  const void* residual[MAXT];
  const void* dy[MAXT];
  for (int r = 0; r < t; ++r)
    if ((partials[r] = read_to_device(in, full * 2)) == NULL) return 1;
  for (int k = 0; k < t; ++k)
    if ((residual[k] = read_to_device(in, rows_k[k] * h * 2)) == NULL) return 1;
  const void* bias = read_to_device(in, (size_t)h * 2);
  const void* gamma = read_to_device(in, (size_t)h * 2);
  const void* beta = read_to_device(in, (size_t)h * 2);
  if (bias == NULL || gamma == NULL || beta == NULL) return 1;
  for (int k = 0; k < t; ++k)
    if ((dy[k] = read_to_device(in, rows_k[k] * h * 2)) == NULL) return 1;
  fclose(in);

  void* z[MAXT];
  uint8_t* mask[MAXT];
  float* mean[MAXT];
  float* rstd[MAXT];
  void* dres[MAXT];
  const size_t mask_row = bits ? (size_t)h / 8 : (size_t)h;   /* mask bytes per token */
  for (int k = 0; k < t; ++k) {
    z[k] = dev_alloc(rows_k[k] * h * 2);
    mask[k] = (uint8_t*)dev_alloc(rows_k[k] * mask_row);
    mean[k] = (float*)dev_alloc(rows_k[k] * 4);
    rstd[k] = (float*)dev_alloc(rows_k[k] * 4);
    dres[k] = dev_alloc(rows_k[k] * h * 2);
    if (!z[k] || !mask[k] || !mean[k] || !rstd[k] || !dres[k]) return 1;
  }
  void* gathered = dev_alloc(full * 2);
  void* dgat = dev_alloc(full * 2);
  float* dgamma = (float*)dev_alloc((size_t)h * 4);
  float* dbeta = (float*)dev_alloc((size_t)h * 4);
  float* dbias = (float*)dev_alloc((size_t)h * 4);
  int32_t* status = (int32_t*)dev_alloc(4);
  const size_t ws_bytes = sp_norm_bwd_workspace_bytes(b, s, h, t, norm);
  void* ws = dev_alloc(ws_bytes);
  if (!gathered || !dgat || !dgamma || !dbeta || !dbias || !status || !ws) return 1;
  if (!cuda_ok(cudaMemset(status, 0, 4), "cudaMemset")) return 1;

  sp_status_t st = (bits ? sp_rs_norm_fwd_bitmask : sp_rs_norm_fwd)(
      partials, residual, bias, gamma, ln ? beta : NULL, b, s, h, t, eps, p, seed, offset, NULL,
      0, norm, (void* const*)z, (uint8_t* const*)mask, ln ? (float* const*)mean : NULL,
      (float* const*)rstd, (void* const*)&gathered, 1, status, NULL);
  if (!sp_ok(st, "forward")) return 1;
  st = (bits ? sp_norm_bwd_bitmask : sp_norm_bwd)(
      dy, (const void* const*)z, (const uint8_t* const*)mask,
      ln ? (const float* const*)mean : NULL, (const float* const*)rstd, gamma, NULL, b, s, h, t,
      p, NULL, 0, norm, (void* const*)dres, (void* const*)&dgat, 1, dgamma, ln ? dbeta : NULL,
      dbias, ws, ws_bytes, status, NULL);
  if (!sp_ok(st, "backward")) return 1;
  if (!cuda_ok(cudaDeviceSynchronize(), "cudaDeviceSynchronize")) return 1;

  FILE* out = fopen(argv[2], "wb");
  if (out == NULL) {
    perror(argv[2]);
    return 1;
  }
  int ok = 1;
  for (int k = 0; k < t; ++k) ok = ok && write_from_device(out, z[k], rows_k[k] * h * 2);
  for (int k = 0; k < t; ++k) ok = ok && write_from_device(out, mask[k], rows_k[k] * mask_row);
  if (ln)
    for (int k = 0; k < t; ++k) ok = ok && write_from_device(out, mean[k], rows_k[k] * 4);
  for (int k = 0; k < t; ++k) ok = ok && write_from_device(out, rstd[k], rows_k[k] * 4);
  ok = ok && write_from_device(out, gathered, full * 2);
  for (int k = 0; k < t; ++k) ok = ok && write_from_device(out, dres[k], rows_k[k] * h * 2);
  ok = ok && write_from_device(out, dgat, full * 2);
  ok = ok && write_from_device(out, dgamma, (size_t)h * 4);
  if (ln) ok = ok && write_from_device(out, dbeta, (size_t)h * 4);
  ok = ok && write_from_device(out, dbias, (size_t)h * 4);
  ok = ok && write_from_device(out, status, 4);
  ok = (fclose(out) == 0) && ok;
  if (!ok) {
    fprintf(stderr, "writing %s failed\n", argv[2]);
    return 1;
  }
  printf("ok t=%" PRId32 " b=%" PRId64 " s=%" PRId64 " h=%" PRId64 "\n", t, b, s, h);
  return 0;
}
