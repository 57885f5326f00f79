/* A plain-C consumer of libflce.so: no Python, no torch. It reads one
 * problem's inputs from a file, runs flce_forward and flce_backward on device
 * buffers it allocates itself, and writes the outputs to another file, which
 * the calling test compares with the fp64 oracle.
 *
 * Input file (little-endian):  int64 n, h, v; int64 ignore_index;
 *   hidden bf16 [n*h]; weight bf16 [v*h]; targets int64 [n]
 * Output file: float loss; int32 n_valid; float metrics[2]; float lse[n];
 *   grad_hidden bf16 [n*h]; grad_weight bf16 [v*h]
 *
 *   roundtrip <in> <out>   exit status 0 on success */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "flce.h"

#define CHECK_CUDA(x)                                                         \
  do {                                                                        \
    cudaError_t e_ = (x);                                                     \
    if (e_ != cudaSuccess) {                                                  \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                \
      return 1;                                                               \
    }                                                                         \
  } while (0)

#define CHECK_FLCE(x)                                                         \
  do {                                                                        \
    flce_status s_ = (x);                                                     \
    if (s_ != FLCE_OK) {                                                      \
      fprintf(stderr, "%s: %s: %s\n", #x, flce_status_string(s_),             \
              flce_last_error());                                             \
      return 1;                                                               \
    }                                                                         \
  } while (0)

static void* read_all(FILE* f, size_t bytes) {
  void* p = malloc(bytes ? bytes : 1);
  if (p && bytes && fread(p, 1, bytes, f) != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static void* to_device(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 1) != cudaSuccess) return NULL;
  if (bytes && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s <in> <out>\n", argv[0]);
    return 2;
  }
  FILE* fi = fopen(argv[1], "rb");
  if (!fi) return 1;
  int64_t hdr[4];
  if (fread(hdr, sizeof(int64_t), 4, fi) != 4) return 1;
  const int64_t n = hdr[0], h = hdr[1], v = hdr[2];
  const size_t hb = (size_t)(n * h) * 2, wb = (size_t)(v * h) * 2, tb = (size_t)n * 8;
  void* hidden = read_all(fi, hb);
  void* weight = read_all(fi, wb);
  void* targets = read_all(fi, tb);
  fclose(fi);
  if (!hidden || !weight || !targets) return 1;
  if (!flce_device_supported()) {
    fprintf(stderr, "device not supported\n");
    return 1;
  }

  flce_problem p = {0};
  p.n = n;
  p.h = h;
  p.v = v;
  p.dtype = FLCE_BF16;
  p.has_bias = 0;
  p.ignore_index = hdr[3];
  p.logit_scale = 1.0f;
  p.softcap = 0.0f;
  p.reduction = FLCE_RED_MEAN;
  p.grad_weight_dtype = FLCE_BF16;
  p.flags = FLCE_SKIP_IGNORED_ROWS;

  void *d_h = to_device(hidden, hb), *d_w = to_device(weight, wb), *d_t = to_device(targets, tb);
  float *d_loss_rows, *d_lse, *d_loss, *d_metrics, *d_go;
  int32_t *d_nv, *d_err;
  void *d_gh, *d_gw, *d_ws;
  if (!d_h || !d_w || !d_t) return 1;
  CHECK_CUDA(cudaMalloc((void**)&d_loss_rows, n * 4 + 4));
  CHECK_CUDA(cudaMalloc((void**)&d_lse, n * 4 + 4));
  CHECK_CUDA(cudaMalloc((void**)&d_loss, 4));
  CHECK_CUDA(cudaMalloc((void**)&d_metrics, 8));
  CHECK_CUDA(cudaMalloc((void**)&d_go, 4));
  CHECK_CUDA(cudaMalloc((void**)&d_nv, 4));
  CHECK_CUDA(cudaMalloc((void**)&d_err, 4));
  CHECK_CUDA(cudaMemset(d_err, 0, 4));
  CHECK_CUDA(cudaMalloc(&d_gh, hb + 2));
  CHECK_CUDA(cudaMalloc(&d_gw, wb + 2));
  const float one = 1.0f;
  CHECK_CUDA(cudaMemcpy(d_go, &one, 4, cudaMemcpyHostToDevice));
  size_t ws_f = flce_forward_workspace_size(&p), ws_b = flce_backward_workspace_size(&p);
  size_t ws = ws_f > ws_b ? ws_f : ws_b;
  CHECK_CUDA(cudaMalloc(&d_ws, ws ? ws : 1)); /* cudaMalloc returns 256-byte aligned memory */

  CHECK_FLCE(flce_forward(&p, d_h, d_w, NULL, (const int64_t*)d_t, d_loss_rows, d_lse, NULL, NULL,
                          d_loss, d_metrics, d_nv, d_err, d_ws, ws, NULL));
  CHECK_FLCE(flce_backward(&p, d_h, d_w, NULL, (const int64_t*)d_t, d_lse, d_nv, d_go, d_gh, d_gw,
                           NULL, d_err, d_ws, ws, NULL));
  CHECK_CUDA(cudaDeviceSynchronize());

  int32_t err = 0, nv = 0;
  float loss = 0.0f, metrics[2];
  CHECK_CUDA(cudaMemcpy(&err, d_err, 4, cudaMemcpyDeviceToHost));
  if (err != 0) {
    fprintf(stderr, "device error word %d\n", (int)err);
    return 1;
  }
  float* lse = (float*)malloc((size_t)n * 4 + 4);
  void* gh = malloc(hb + 2);
  void* gw = malloc(wb + 2);
  if (!lse || !gh || !gw) return 1;
  CHECK_CUDA(cudaMemcpy(&loss, d_loss, 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(&nv, d_nv, 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(metrics, d_metrics, 8, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(lse, d_lse, (size_t)n * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(gh, d_gh, hb, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(gw, d_gw, wb, cudaMemcpyDeviceToHost));

  FILE* fo = fopen(argv[2], "wb");
  if (!fo) return 1;
  fwrite(&loss, 4, 1, fo);
  fwrite(&nv, 4, 1, fo);
  fwrite(metrics, 4, 2, fo);
  fwrite(lse, 4, (size_t)n, fo);
  fwrite(gh, 1, hb, fo);
  fwrite(gw, 1, wb, fo);
  fclose(fo);
  printf("roundtrip ok: n=%lld loss=%.6f n_valid=%d\n", (long long)n, loss, (int)nv);
  return 0;
}
