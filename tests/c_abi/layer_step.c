/* One forward + backward step of the layer through the C ABI alone (no Python, no PyTorch):
 * reads the step's inputs from raw little-endian files in a directory, runs mm_forward and
 * mm_backward on the default stream with a workspace of mm_workspace_size bytes, and writes
 * y, dx, d_topk_weights, d_up_proj_weight and d_down_proj_weight back as raw files.
 *
 *     layer_step DIR T H I E K
 *
 * Inputs in DIR: x.bin (bf16 [T,H]), ids.bin (int32 [T,K]), tw.bin (fp32 [T,K]),
 * wu.bin (bf16 [E,H,2I]), wd.bin (bf16 [E,I,H]), dy.bin (bf16 [T,H]).
 * Exit status 0 on success; otherwise the failing step is printed. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "mm.h"

static void* load(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* host = malloc(bytes ? bytes : 1);
  const size_t got = host ? fread(host, 1, bytes, f) : 0;
  fclose(f);
  if (got != bytes) {
    free(host);
    return NULL;
  }
  void* dev = NULL;
  if (cudaMalloc(&dev, bytes ? bytes : 1) != cudaSuccess ||
      cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
    free(host);
    return NULL;
  }
  free(host);
  return dev;
}

static int save(const char* dir, const char* name, const void* dev, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  void* host = malloc(bytes ? bytes : 1);
  if (!host || cudaMemcpy(host, dev, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  const size_t put = fwrite(host, 1, bytes, f);
  fclose(f);
  free(host);
  return put != bytes;
}

static void* zeros(size_t bytes) {
  void* dev = NULL;
  if (cudaMalloc(&dev, bytes ? bytes : 1) != cudaSuccess) return NULL;
  return dev;
}

int main(int argc, char** argv) {
  if (argc != 7) {
    fprintf(stderr, "usage: %s DIR T H I E K\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  mm_dims d;
  d.T = atoll(argv[2]);
  d.H = atoll(argv[3]);
  d.I = atoll(argv[4]);
  d.E = atoll(argv[5]);
  d.K = atoll(argv[6]);
  const size_t TH = (size_t)(d.T * d.H), TK = (size_t)(d.T * d.K);
  const size_t wu_n = (size_t)(d.E * d.H * 2 * d.I), wd_n = (size_t)(d.E * d.I * d.H);
  void* x = load(dir, "x.bin", TH * 2);
  int32_t* ids = (int32_t*)load(dir, "ids.bin", TK * 4);
  float* tw = (float*)load(dir, "tw.bin", TK * 4);
  void* wu = load(dir, "wu.bin", wu_n * 2);
  void* wd = load(dir, "wd.bin", wd_n * 2);
  void* dy = load(dir, "dy.bin", TH * 2);
  if (!x || !ids || !tw || !wu || !wd || !dy) {
    fprintf(stderr, "could not load the inputs from %s\n", dir);
    return 1;
  }
  const size_t ws_bytes = mm_workspace_size(d, 0);
  if (ws_bytes == 0) {
    fprintf(stderr, "unsupported sizes\n");
    return 1;
  }
  void* ws = zeros(ws_bytes);
  void* y = zeros(TH * 2);
  void* dx = zeros(TH * 2);
  float* dtk = (float*)zeros(TK * 4);
  void* du = zeros(wu_n * 2);
  void* dd = zeros(wd_n * 2);
  if (!ws || !y || !dx || !dtk || !du || !dd) {
    fprintf(stderr, "device allocation failed\n");
    return 1;
  }
  mm_status s = mm_forward(d, x, ids, tw, wu, wd, y, ws, ws_bytes, NULL, 0);
  if (s != MM_OK) {
    fprintf(stderr, "mm_forward: %s (%s)\n", mm_status_string(s), mm_last_error_detail());
    return 1;
  }
  s = mm_backward(d, dy, x, ids, tw, wu, wd, ws, ws_bytes, dx, dtk, du, dd, NULL, 0);
  if (s != MM_OK) {
    fprintf(stderr, "mm_backward: %s (%s)\n", mm_status_string(s), mm_last_error_detail());
    return 1;
  }
  s = mm_get_status(ws, NULL);
  if (s != MM_OK) {
    fprintf(stderr, "device status: %s\n", mm_status_string(s));
    return 1;
  }
  if (save(dir, "y.bin", y, TH * 2) || save(dir, "dx.bin", dx, TH * 2) ||
      save(dir, "dtk.bin", dtk, TK * 4) || save(dir, "du.bin", du, wu_n * 2) ||
      save(dir, "dd.bin", dd, wd_n * 2)) {
    fprintf(stderr, "could not write the outputs\n");
    return 1;
  }
  printf("layer_step: T=%lld H=%lld I=%lld E=%lld K=%lld ok\n", (long long)d.T, (long long)d.H,
         (long long)d.I, (long long)d.E, (long long)d.K);
  return 0;
}
