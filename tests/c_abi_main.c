/*
 * A plain C caller of the library: no Python, no torch.  Reads bf16 inputs
 * from files, runs the forward (fa_fwd) and the backward (fa_bwd) through
 * the C ABI on buffers it allocates with the CUDA runtime, checks the device
 * status word, and writes the outputs back to files.
 *
 *   c_abi_main <dir> B H N D causal scale
 *
 * <dir> holds q.bin, k.bin, v.bin, do.bin (bf16 [B, H, N, D], raw
 * little-endian); the program writes o.bin (bf16), lse.bin (f32 [B, H, N]),
 * dq.bin, dk.bin, dv.bin (bf16).  Exit status 0 on success.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fa_gb300.h"

static int read_file(const char* dir, const char* name, void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return -1;
  const size_t got = fread(buf, 1, bytes, f);
  fclose(f);
  return got == bytes ? 0 : -1;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return -1;
  const size_t put = fwrite(buf, 1, bytes, f);
  fclose(f);
  return put == bytes ? 0 : -1;
}

#define CHECK_CUDA(x)                                                        \
  do {                                                                       \
    cudaError_t e_ = (x);                                                    \
    if (e_ != cudaSuccess) {                                                 \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));              \
      return 2;                                                              \
    }                                                                        \
  } while (0)

#define CHECK_FA(x)                                                          \
  do {                                                                       \
    int rc_ = (x);                                                           \
    if (rc_ != FA_OK) {                                                      \
      fprintf(stderr, "%s: %s (%d)\n", #x, fa_status_string(rc_), rc_);     \
      return 3;                                                              \
    }                                                                        \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 8) {
    fprintf(stderr, "usage: %s dir B H N D causal scale\n", argv[0]);
    return 1;
  }
  const char* dir = argv[1];
  const int B = atoi(argv[2]), H = atoi(argv[3]), N = atoi(argv[4]), D = atoi(argv[5]);
  const int causal = atoi(argv[6]);
  const float scale = (float)atof(argv[7]);
  const size_t elems = (size_t)B * H * N * D;
  const size_t rows = (size_t)B * H * N;
  const size_t tb = elems * sizeof(uint16_t);

  const char* in_names[4] = {"q.bin", "k.bin", "v.bin", "do.bin"};
  void* host[4];
  void* dev[4];
  for (int i = 0; i < 4; ++i) {
    host[i] = malloc(tb);
    if (!host[i] || read_file(dir, in_names[i], host[i], tb) != 0) {
      fprintf(stderr, "cannot read %s\n", in_names[i]);
      return 1;
    }
    CHECK_CUDA(cudaMalloc(&dev[i], tb));
    CHECK_CUDA(cudaMemcpy(dev[i], host[i], tb, cudaMemcpyHostToDevice));
  }
  void *o, *dq, *dk, *dv;
  float *lse, *ws;
  CHECK_CUDA(cudaMalloc(&o, tb));
  CHECK_CUDA(cudaMalloc(&dq, tb));
  CHECK_CUDA(cudaMalloc(&dk, tb));
  CHECK_CUDA(cudaMalloc(&dv, tb));
  CHECK_CUDA(cudaMalloc((void**)&lse, rows * sizeof(float)));
  const size_t wsb = fa_bwd_workspace_bytes(B, H, N);
  CHECK_CUDA(cudaMalloc((void**)&ws, wsb > 0 ? wsb : 4));
  cudaStream_t stream;
  CHECK_CUDA(cudaStreamCreate(&stream));

  CHECK_FA(fa_fwd(dev[0], dev[1], dev[2], o, lse, B, H, N, D, scale, causal, stream));
  CHECK_FA(fa_bwd(dev[0], dev[1], dev[2], o, dev[3], lse, dq, dk, dv, ws, B, H, N, D, scale,
                  causal, stream));
  CHECK_FA(fa_check_device_status(stream));

  void* out = malloc(tb);
  float* lse_h = (float*)malloc(rows * sizeof(float));
  if (!out || !lse_h) return 1;
  const char* out_names[4] = {"o.bin", "dq.bin", "dk.bin", "dv.bin"};
  void* outs[4] = {o, dq, dk, dv};
  for (int i = 0; i < 4; ++i) {
    CHECK_CUDA(cudaMemcpy(out, outs[i], tb, cudaMemcpyDeviceToHost));
    if (write_file(dir, out_names[i], out, tb) != 0) return 1;
  }
  CHECK_CUDA(cudaMemcpy(lse_h, lse, rows * sizeof(float), cudaMemcpyDeviceToHost));
  if (write_file(dir, "lse.bin", lse_h, rows * sizeof(float)) != 0) return 1;

  /* argument checks answer without touching the device */
  if (fa_fwd(dev[0], dev[1], dev[2], o, lse, B, H, N, 96, scale, causal, stream) !=
      FA_ERR_INVALID_ARG)
    return 4;

  for (int i = 0; i < 4; ++i) {
    cudaFree(dev[i]);
    free(host[i]);
  }
  cudaFree(o);
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(lse);
  cudaFree(ws);
  cudaStreamDestroy(stream);
  free(out);
  free(lse_h);
  printf("c abi ok\n");
  return 0;
}
