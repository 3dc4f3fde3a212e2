/* Plain-C (C11) user of the libzero ABI on the GPU, without any Python framework:
 * reads N gradient buffers and the fp32 master weights (float32, native byte
 * order) from argv[1], allocates device buffers with the CUDA runtime, runs
 * `steps` fused zero_step calls (the same gradients each step) and writes the
 * master weights, m, v and the bf16 gathered parameters to argv[2].
 * Input layout: int32 N, int32 steps, int64 psi_pad, int32 T, T x int64
 * numels, then N x psi_pad gradients and psi_pad master weights. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "zero.h"

#define CHECK_CUDA(x)                                                           \
  do {                                                                          \
    cudaError_t e_ = (x);                                                       \
    if (e_ != cudaSuccess) {                                                    \
      fprintf(stderr, "CUDA error %d at line %d\n", (int)e_, __LINE__);         \
      return 2;                                                                 \
    }                                                                           \
  } while (0)
#define CHECK_ZERO(x)                                                           \
  do {                                                                          \
    int s_ = (x);                                                               \
    if (s_ != ZERO_OK) {                                                        \
      fprintf(stderr, "libzero: %s at line %d\n", zero_strerror(s_), __LINE__); \
      return 3;                                                                 \
    }                                                                           \
  } while (0)

static int read_all(FILE* f, void* p, size_t bytes) { return fread(p, 1, bytes, f) == bytes; }

int main(int argc, char** argv) {
  int32_t n = 0, steps = 0, t_count = 0, r, t;
  int64_t psi_pad = 0;
  int64_t* numels;
  float *h_grads, *h_master, *h_m, *h_v;
  uint16_t* h_out;
  void* d_grads[ZERO_MAX_RANKS];
  float *d_master, *d_m, *d_v;
  void* d_out;
  zero_plan_t* plan = NULL;
  zero_plan_info_t info;
  FILE *in, *out;
  size_t vec;
  if (argc != 3 || !(in = fopen(argv[1], "rb"))) return 1;
  if (!read_all(in, &n, 4) || !read_all(in, &steps, 4) || !read_all(in, &psi_pad, 8) ||
      !read_all(in, &t_count, 4) || n < 1 || n > ZERO_MAX_RANKS || t_count < 1)
    return 1;
  numels = (int64_t*)malloc(sizeof(int64_t) * (size_t)t_count);
  vec = sizeof(float) * (size_t)psi_pad;
  h_grads = (float*)malloc(vec * (size_t)n);
  h_master = (float*)malloc(vec);
  h_m = (float*)malloc(vec);
  h_v = (float*)malloc(vec);
  h_out = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)psi_pad);
  if (!numels || !h_grads || !h_master || !h_m || !h_v || !h_out) return 1;
  if (!read_all(in, numels, sizeof(int64_t) * (size_t)t_count) ||
      !read_all(in, h_grads, vec * (size_t)n) || !read_all(in, h_master, vec))
    return 1;
  fclose(in);

  CHECK_ZERO(zero_plan(numels, t_count, n, 16, NULL, &plan));
  CHECK_ZERO(zero_plan_info(plan, &info));
  if (info.psi_pad != psi_pad) return 4;
  for (r = 0; r < n; ++r) {
    CHECK_CUDA(cudaMalloc(&d_grads[r], vec));
    CHECK_CUDA(cudaMemcpy(d_grads[r], h_grads + (size_t)r * (size_t)psi_pad, vec,
                          cudaMemcpyHostToDevice));
  }
  CHECK_CUDA(cudaMalloc((void**)&d_master, vec));
  CHECK_CUDA(cudaMalloc((void**)&d_m, vec));
  CHECK_CUDA(cudaMalloc((void**)&d_v, vec));
  CHECK_CUDA(cudaMalloc(&d_out, sizeof(uint16_t) * (size_t)psi_pad));
  CHECK_CUDA(cudaMemcpy(d_master, h_master, vec, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemset(d_m, 0, vec));
  CHECK_CUDA(cudaMemset(d_v, 0, vec));
  for (t = 1; t <= steps; ++t) {
    zero_adam_t hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.0f, 1.0f / (float)n, t, NULL};
    CHECK_ZERO(zero_step(plan, 0, (const void* const*)d_grads, ZERO_F32, d_master, d_m, d_v, &hp,
                         NULL, d_out, ZERO_BF16, NULL));
  }
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(h_master, d_master, vec, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_m, d_m, vec, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_v, d_v, vec, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_out, d_out, sizeof(uint16_t) * (size_t)psi_pad,
                        cudaMemcpyDeviceToHost));
  if (!(out = fopen(argv[2], "wb"))) return 1;
  fwrite(h_master, 1, vec, out);
  fwrite(h_m, 1, vec, out);
  fwrite(h_v, 1, vec, out);
  fwrite(h_out, sizeof(uint16_t), (size_t)psi_pad, out);
  fclose(out);
  for (r = 0; r < n; ++r) cudaFree(d_grads[r]);
  cudaFree(d_master);
  cudaFree(d_m);
  cudaFree(d_v);
  cudaFree(d_out);
  zero_plan_destroy(plan);
  printf("ok %d steps\n", steps);
  return 0;
}
