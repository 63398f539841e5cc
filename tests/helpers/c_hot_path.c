/* A plain C11 program that runs the hot path on the GPU through include/mx.h, the
 * way a C user of the library would: it allocates device buffers itself, copies
 * host inputs in, quantizes the weights (mx_quantize, and mx_quantize_stacked for a
 * stacked [W_g; W_u]), runs mx_mlp and mx_gated_mlp, and copies the results back.
 *
 *   c_hot_path <dir> <M> <d> <ff> <ffg>
 *
 * Reads raw little-endian BF16 files from <dir>: x [M][d], w1 [ff][d], b1 [ff],
 * w2 [d][ff], b2 [d], wg and wu [ffg][d], bgu [2 ffg], w2g [d][ffg]. Writes y.bin
 * ([M][d] BF16, mx_mlp), yg.bin ([M][d] BF16, mx_gated_mlp), and the stacked
 * weight's codes and scales (wgu_codes.bin, wgu_scales.bin). Exits non-zero with a
 * message on the first failing call. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "mx.h"

static const char* g_dir;

static void* read_file(const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", g_dir, name);
  FILE* f = fopen(path, "rb");
  if (f == NULL) {
    fprintf(stderr, "cannot open %s\n", path);
    exit(2);
  }
  void* buf = malloc(bytes);
  if (buf == NULL || fread(buf, 1, bytes, f) != bytes) {
    fprintf(stderr, "short read of %s\n", path);
    exit(2);
  }
  fclose(f);
  return buf;
}

static void write_file(const char* name, const void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", g_dir, name);
  FILE* f = fopen(path, "wb");
  if (f == NULL || fwrite(buf, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot write %s\n", path);
    exit(2);
  }
  fclose(f);
}

#define CUDA_OK(call)                                                             \
  do {                                                                            \
    cudaError_t e_ = (call);                                                      \
    if (e_ != cudaSuccess) {                                                      \
      fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));          \
      exit(3);                                                                    \
    }                                                                             \
  } while (0)

#define MX_OK_(call)                                                              \
  do {                                                                            \
    mx_status s_ = (call);                                                        \
    if (s_ != MX_OK) {                                                            \
      fprintf(stderr, "%s failed: %s\n", #call, mx_status_string(s_));            \
      exit(4);                                                                    \
    }                                                                             \
  } while (0)

/* Device copy of a host file of `bytes` bytes. */
static void* upload(const char* name, size_t bytes) {
  void* h = read_file(name, bytes);
  void* d = NULL;
  CUDA_OK(cudaMalloc(&d, bytes));
  CUDA_OK(cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice));
  free(h);
  return d;
}

typedef struct {
  void* codes;
  void* scales;
} mx_buf;

static mx_buf mx_alloc(int64_t rows, int64_t k) {
  mx_buf b;
  CUDA_OK(cudaMalloc(&b.codes, mx_codes_bytes(rows, k)));
  CUDA_OK(cudaMalloc(&b.scales, mx_scales_bytes(rows, k)));
  return b;
}

int main(int argc, char** argv) {
  if (argc != 6) {
    fprintf(stderr, "usage: %s <dir> <M> <d> <ff> <ffg>\n", argv[0]);
    return 1;
  }
  g_dir = argv[1];
  const int64_t M = atoll(argv[2]), d = atoll(argv[3]), ff = atoll(argv[4]), ffg = atoll(argv[5]);
  const size_t bf = 2;
  cudaStream_t stream;
  CUDA_OK(cudaStreamCreate(&stream));

  void* x = upload("x.bin", (size_t)(M * d) * bf);
  void* w1 = upload("w1.bin", (size_t)(ff * d) * bf);
  void* b1 = upload("b1.bin", (size_t)ff * bf);
  void* w2 = upload("w2.bin", (size_t)(d * ff) * bf);
  void* b2 = upload("b2.bin", (size_t)d * bf);
  void* wg = upload("wg.bin", (size_t)(ffg * d) * bf);
  void* wu = upload("wu.bin", (size_t)(ffg * d) * bf);
  void* bgu = upload("bgu.bin", (size_t)(2 * ffg) * bf);
  void* w2g = upload("w2g.bin", (size_t)(d * ffg) * bf);

  /* weights: quantized once */
  mx_buf w1q = mx_alloc(ff, d), w2q = mx_alloc(d, ff), wguq = mx_alloc(2 * ffg, d), w2gq = mx_alloc(d, ffg);
  MX_OK_(mx_quantize(w1, ff, d, d, w1q.codes, w1q.scales, stream));
  MX_OK_(mx_quantize(w2, d, ff, ff, w2q.codes, w2q.scales, stream));
  const void* parts[2] = {wg, wu};
  const int64_t part_rows[2] = {ffg, ffg};
  MX_OK_(mx_quantize_stacked(parts, part_rows, NULL, 2, d, wguq.codes, wguq.scales, stream));
  MX_OK_(mx_quantize(w2g, d, ffg, ffg, w2gq.codes, w2gq.scales, stream));

  /* one workspace for both MLPs (the larger of the two sizes) */
  size_t ws_bytes = mx_mlp_workspace_bytes(M, d, ff);
  const size_t ws_g = mx_mlp_workspace_bytes(M, d, ffg);
  if (ws_g > ws_bytes) ws_bytes = ws_g;
  void* ws = NULL;
  CUDA_OK(cudaMalloc(&ws, ws_bytes));
  void* y = NULL;
  void* yg = NULL;
  CUDA_OK(cudaMalloc(&y, (size_t)(M * d) * bf));
  CUDA_OK(cudaMalloc(&yg, (size_t)(M * d) * bf));
  MX_OK_(mx_mlp(x, M, d, ff, w1q.codes, w1q.scales, b1, w2q.codes, w2q.scales, b2, y, ws, ws_bytes, stream));
  MX_OK_(mx_gated_mlp(x, M, d, ffg, wguq.codes, wguq.scales, bgu, w2gq.codes, w2gq.scales, b2, yg, ws, ws_bytes,
                      stream));
  CUDA_OK(cudaStreamSynchronize(stream));
  unsigned flags = 0;
  MX_OK_(mx_device_error(&flags, 0));
  if (flags != 0) {
    fprintf(stderr, "device error word %u\n", flags);
    return 5;
  }

  const size_t ybytes = (size_t)(M * d) * bf;
  void* h = malloc(ybytes);
  CUDA_OK(cudaMemcpy(h, y, ybytes, cudaMemcpyDeviceToHost));
  write_file("y.bin", h, ybytes);
  CUDA_OK(cudaMemcpy(h, yg, ybytes, cudaMemcpyDeviceToHost));
  write_file("yg.bin", h, ybytes);
  free(h);
  const size_t cb = mx_codes_bytes(2 * ffg, d), sb = mx_scales_bytes(2 * ffg, d);
  void* hc = malloc(cb);
  void* hs = malloc(sb);
  CUDA_OK(cudaMemcpy(hc, wguq.codes, cb, cudaMemcpyDeviceToHost));
  CUDA_OK(cudaMemcpy(hs, wguq.scales, sb, cudaMemcpyDeviceToHost));
  write_file("wgu_codes.bin", hc, cb);
  write_file("wgu_scales.bin", hs, sb);
  free(hc);
  free(hs);

  void* bufs[] = {x, w1, b1, w2, b2, wg, wu, bgu, w2g, w1q.codes, w1q.scales, w2q.codes, w2q.scales,
                  wguq.codes, wguq.scales, w2gq.codes, w2gq.scales, ws, y, yg};
  for (size_t i = 0; i < sizeof(bufs) / sizeof(bufs[0]); ++i) CUDA_OK(cudaFree(bufs[i]));
  CUDA_OK(cudaStreamDestroy(stream));
  printf("ok\n");
  return 0;
}
