/*
 * A plain C (C11) caller of libpoetx: one fp32 POET-X layer step (block build of
 * both factors, forward with v saved, backward) through poetx.h, on device
 * memory from the CUDA runtime, checked against stored float64-oracle
 * results.  Usage: layer_step <case.bin>; exit status 0 when y, dx,
 * dtheta_P and dtheta_R are within 1e-4 relative Frobenius error.
 * The case file layout is described in tests/golden/make_c_abi_case.py.
 */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "poetx.h"

enum { N_ARRAYS = 9 };

static float* read_floats(FILE* f, size_t n) {
  float* p = (float*)malloc(n * sizeof(float) + 1);
  if (p == NULL || fread(p, sizeof(float), n, f) != n) {
    free(p);
    return NULL;
  }
  return p;
}

static void* dev_copy(const float* h, size_t n) {
  void* d = NULL;
  if (cudaMalloc(&d, n * sizeof(float) + 16) != cudaSuccess) return NULL;
  if (h != NULL && cudaMemcpy(d, h, n * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess)
    return NULL;
  return d;
}

static double rel_fro(const float* got, const float* want, size_t n) {
  double num = 0.0, den = 0.0;
  size_t i;
  for (i = 0; i < n; ++i) {
    const double e = (double)got[i] - (double)want[i];
    num += e * e;
    den += (double)want[i] * (double)want[i];
  }
  return sqrt(num) / (den > 0.0 ? sqrt(den) : 1.0);
}

#define CHECK(call)                                                          \
  do {                                                                       \
    poetx_status st_ = (call);                                               \
    if (st_ != POETX_OK) {                                                   \
      fprintf(stderr, "%s: %s\n", #call, poetx_status_string(st_));         \
      return 2;                                                              \
    }                                                                        \
  } while (0)

int main(int argc, char** argv) {
  FILE* f;
  char magic[8];
  int hdr[5];
  int d_in, d_out, b, k, T, i;
  size_t n[N_ARRAYS];
  float* h[N_ARRAYS];
  size_t ws_bytes, w;
  void *d_theta, *d_W0, *d_x, *d_dy, *d_blocks, *d_y, *d_v, *d_dx, *d_dtheta, *d_ws;
  float *got_y, *got_dx, *got_dtheta;
  size_t mP, mR;
  double err[4];
  const char* names[4] = {"y", "dx", "dtheta_P", "dtheta_R"};
  int bad = 0;

  if (argc != 2 || (f = fopen(argv[1], "rb")) == NULL) {
    fprintf(stderr, "usage: %s case.bin\n", argv[0]);
    return 2;
  }
  if (fread(magic, 1, 8, f) != 8 || memcmp(magic, "POETXC1", 8) != 0 ||
      fread(hdr, sizeof(int), 5, f) != 5) {
    fprintf(stderr, "bad case file\n");
    return 2;
  }
  d_in = hdr[0];
  d_out = hdr[1];
  b = hdr[2];
  k = hdr[3];
  T = hdr[4];
  mP = poetx_packed_size(d_in, b);
  mR = poetx_packed_size(d_out, b);
  n[0] = mP;
  n[1] = mR;
  n[2] = (size_t)d_out * d_in;
  n[3] = (size_t)T * d_in;
  n[4] = (size_t)T * d_out;
  n[5] = (size_t)T * d_out;
  n[6] = (size_t)T * d_in;
  n[7] = mP;
  n[8] = mR;
  for (i = 0; i < N_ARRAYS; ++i)
    if ((h[i] = read_floats(f, n[i])) == NULL) {
      fprintf(stderr, "short case file (array %d)\n", i);
      return 2;
    }
  fclose(f);

  /* theta_P and theta_R back to back: both factors in one build call */
  d_theta = dev_copy(NULL, mP + mR);
  d_W0 = dev_copy(h[2], n[2]);
  d_x = dev_copy(h[3], n[3]);
  d_dy = dev_copy(h[4], n[4]);
  d_blocks = dev_copy(NULL, (size_t)(d_in + d_out) * b);
  d_y = dev_copy(NULL, n[5]);
  d_v = dev_copy(NULL, n[5]);
  d_dx = dev_copy(NULL, n[6]);
  d_dtheta = dev_copy(NULL, mP + mR);
  if (!d_theta || !d_W0 || !d_x || !d_dy || !d_blocks || !d_y || !d_v || !d_dx || !d_dtheta) {
    fprintf(stderr, "cudaMalloc failed\n");
    return 2;
  }
  if (cudaMemcpy(d_theta, h[0], mP * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy((float*)d_theta + mP, h[1], mR * sizeof(float), cudaMemcpyHostToDevice) !=
          cudaSuccess)
    return 2;

  ws_bytes = poetx_build_workspace_size(d_in + d_out, b, k, POETX_F32);
  w = poetx_forward_workspace_size(d_in, d_out, b, T, POETX_F32);
  if (w > ws_bytes) ws_bytes = w;
  w = poetx_backward_workspace_size(d_in, d_out, b, k, T, POETX_F32, 0);
  if (w > ws_bytes) ws_bytes = w;
  if (ws_bytes == 0 || cudaMalloc(&d_ws, ws_bytes) != cudaSuccess) {
    fprintf(stderr, "workspace\n");
    return 2;
  }

  CHECK(poetx_build_blocks((const float*)d_theta, d_in + d_out, b, k, POETX_F32, d_blocks, d_ws,
                           ws_bytes, NULL));
  CHECK(poetx_forward(d_x, d_W0, d_blocks, (float*)d_blocks + (size_t)d_in * b, d_y, d_v, d_in,
                      d_out, b, T, POETX_F32, d_ws, ws_bytes, NULL));
  CHECK(poetx_backward(d_dy, d_x, d_W0, (const float*)d_theta, (const float*)d_theta + mP,
                       d_blocks, (float*)d_blocks + (size_t)d_in * b, d_v, d_dx,
                       (float*)d_dtheta, (float*)d_dtheta + mP, d_in, d_out, b, k, T, POETX_F32,
                       d_ws, ws_bytes, NULL));
  CHECK(poetx_device_status());

  got_y = (float*)malloc(n[5] * sizeof(float));
  got_dx = (float*)malloc(n[6] * sizeof(float));
  got_dtheta = (float*)malloc((mP + mR) * sizeof(float));
  if (!got_y || !got_dx || !got_dtheta ||
      cudaMemcpy(got_y, d_y, n[5] * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(got_dx, d_dx, n[6] * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(got_dtheta, d_dtheta, (mP + mR) * sizeof(float), cudaMemcpyDeviceToHost) !=
          cudaSuccess) {
    fprintf(stderr, "copy back failed\n");
    return 2;
  }
  err[0] = rel_fro(got_y, h[5], n[5]);
  err[1] = rel_fro(got_dx, h[6], n[6]);
  err[2] = rel_fro(got_dtheta, h[7], mP);
  err[3] = rel_fro(got_dtheta + mP, h[8], mR);
  for (i = 0; i < 4; ++i) {
    printf("%s rel_fro %.3e\n", names[i], err[i]);
    if (!(err[i] <= 1e-4)) bad = 1;
  }
  printf(bad ? "FAIL\n" : "OK\n");
  return bad;
}
