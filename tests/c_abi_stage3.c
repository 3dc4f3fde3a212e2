/* Plain-C (C11) user of the libzero ABI for stage 3, without any Python
 * framework: plans a tensor list in layer groups, runs one stage-3 step (per
 * group, in reverse order, the fused step writing each owner's bf16 shard)
 * on buffers it allocates with the CUDA runtime, then gathers every layer
 * twice -- directly (zero_gather_layer) and by the two-stream prefetch pass
 * (zero_stage3_gather_pass, which also checksums each layer) -- and writes
 * the results to argv[2].
 *
 * Input (argv[1], native byte order): int32 N, int32 T, T x int64 numels,
 * T x int32 group of each tensor, then for each group g in order its N
 * rank gradients (N x psi_pad(g) float32), then the fp32 master weights
 * (psi_pad float32, all groups).
 * Output: master (psi_pad float32), then every group's directly gathered
 * layer (psi_pad(g) bf16 bits each, in group order), then the pass's 2G
 * checksums (uint64) for the order 0..G-1, G-1..0. */
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
  int32_t n = 0, t_count = 0;
  int64_t* numels;
  int32_t* groups;
  zero_plan_t* plan = NULL;
  zero_plan_info_t info;
  zero_group_info_t g;
  FILE *in, *out;
  int r, gi, j;
  if (argc != 3 || !(in = fopen(argv[1], "rb"))) return 1;
  if (!read_all(in, &n, 4) || !read_all(in, &t_count, 4) || n < 1 || n > ZERO_MAX_RANKS ||
      t_count < 1)
    return 1;
  numels = (int64_t*)malloc(sizeof(int64_t) * (size_t)t_count);
  groups = (int32_t*)malloc(sizeof(int32_t) * (size_t)t_count);
  if (!numels || !groups || !read_all(in, numels, sizeof(int64_t) * (size_t)t_count) ||
      !read_all(in, groups, sizeof(int32_t) * (size_t)t_count))
    return 1;
  CHECK_ZERO(zero_plan(numels, t_count, n, 16, groups, &plan));
  CHECK_ZERO(zero_plan_info(plan, &info));
  const int32_t G = info.n_groups;
  const size_t flat = sizeof(float) * (size_t)info.psi_pad;
  const size_t shard_bytes = sizeof(uint16_t) * (size_t)info.shard_total;

  /* each group's N gradient buffers, the flat state, the shard buffers */
  void** d_grads = (void**)calloc((size_t)G * (size_t)n, sizeof(void*));
  int64_t gmax = 0;
  if (!d_grads) return 1;
  for (gi = 0; gi < G; ++gi) {
    CHECK_ZERO(zero_plan_group(plan, gi, &g));
    if (g.psi_pad > gmax) gmax = g.psi_pad;
    const size_t bytes = sizeof(float) * (size_t)g.psi_pad;
    float* h = (float*)malloc(bytes > 0 ? bytes : 1);
    if (!h) return 1;
    for (r = 0; r < n; ++r) {
      if (!read_all(in, h, bytes)) return 1;
      CHECK_CUDA(cudaMalloc(&d_grads[(size_t)gi * n + r], bytes > 0 ? bytes : 16));
      if (bytes > 0)
        CHECK_CUDA(cudaMemcpy(d_grads[(size_t)gi * n + r], h, bytes, cudaMemcpyHostToDevice));
    }
    free(h);
  }
  float* h_master = (float*)malloc(flat);
  if (!h_master || !read_all(in, h_master, flat)) return 1;
  fclose(in);
  float *d_master, *d_m, *d_v;
  CHECK_CUDA(cudaMalloc((void**)&d_master, flat));
  CHECK_CUDA(cudaMalloc((void**)&d_m, flat));
  CHECK_CUDA(cudaMalloc((void**)&d_v, flat));
  CHECK_CUDA(cudaMemcpy(d_master, h_master, flat, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemset(d_m, 0, flat));
  CHECK_CUDA(cudaMemset(d_v, 0, flat));
  void* d_shards[ZERO_MAX_RANKS];
  for (r = 0; r < n; ++r) {
    CHECK_CUDA(cudaMalloc(&d_shards[r], shard_bytes));
    CHECK_CUDA(cudaMemset(d_shards[r], 0, shard_bytes));
  }

  /* the step: per group, in reverse order */
  zero_adam_t hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.0f, 1.0f / (float)n, 1, NULL};
  for (gi = G - 1; gi >= 0; --gi)
    CHECK_ZERO(zero_step_group(plan, gi, (const void* const*)&d_grads[(size_t)gi * n],
                               ZERO_F32, d_master, d_m, d_v, &hp, NULL, d_shards, NULL));

  /* every layer gathered directly ... */
  if (!(out = fopen(argv[2], "wb"))) return 1;
  uint16_t* h_layer = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(gmax > 0 ? gmax : 1));
  void* d_layer;
  if (!h_layer) return 1;
  CHECK_CUDA(cudaMalloc(&d_layer, sizeof(uint16_t) * (size_t)(gmax > 0 ? gmax : 8)));
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(h_master, d_master, flat, cudaMemcpyDeviceToHost));
  fwrite(h_master, 1, flat, out);
  for (gi = 0; gi < G; ++gi) {
    CHECK_ZERO(zero_plan_group(plan, gi, &g));
    CHECK_ZERO(zero_gather_layer(plan, gi, (const void* const*)d_shards, ZERO_BF16, d_layer,
                                 NULL));
    CHECK_CUDA(cudaMemcpy(h_layer, d_layer, sizeof(uint16_t) * (size_t)g.psi_pad,
                          cudaMemcpyDeviceToHost));
    fwrite(h_layer, sizeof(uint16_t), (size_t)g.psi_pad, out);
  }

  /* ... and by the two-stream prefetch pass, forward then backward */
  int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)(2 * G));
  uint64_t* h_sums = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(2 * G));
  void* d_bufs[2];
  uint64_t* d_sums;
  cudaStream_t sa, sb;
  if (!order || !h_sums) return 1;
  for (j = 0; j < G; ++j) {
    order[j] = j;
    order[2 * G - 1 - j] = j;
  }
  for (j = 0; j < 2; ++j)
    CHECK_CUDA(cudaMalloc(&d_bufs[j], sizeof(uint16_t) * (size_t)(gmax > 0 ? gmax : 8)));
  CHECK_CUDA(cudaMalloc((void**)&d_sums, sizeof(uint64_t) * (size_t)(2 * G)));
  CHECK_CUDA(cudaStreamCreate(&sa));
  CHECK_CUDA(cudaStreamCreate(&sb));
  CHECK_ZERO(zero_stage3_gather_pass(plan, order, 2 * G, (const void* const*)d_shards, d_bufs,
                                     gmax, d_sums, 1, sa, sb));
  CHECK_CUDA(cudaStreamSynchronize(sa));
  CHECK_CUDA(cudaMemcpy(h_sums, d_sums, sizeof(uint64_t) * (size_t)(2 * G),
                        cudaMemcpyDeviceToHost));
  fwrite(h_sums, sizeof(uint64_t), (size_t)(2 * G), out);
  fclose(out);
  int64_t timeouts = 0;
  CHECK_ZERO(zero_async_status(&timeouts, 0));
  if (timeouts != 0) return 5;

  cudaStreamDestroy(sa);
  cudaStreamDestroy(sb);
  for (j = 0; j < 2; ++j) cudaFree(d_bufs[j]);
  cudaFree(d_sums);
  cudaFree(d_layer);
  for (r = 0; r < n; ++r) cudaFree(d_shards[r]);
  for (j = 0; j < G * n; ++j) cudaFree(d_grads[j]);
  cudaFree(d_master);
  cudaFree(d_m);
  cudaFree(d_v);
  zero_plan_destroy(plan);
  printf("ok %d groups\n", (int)G);
  return 0;
}
