// Seeded synthetic inputs on the device: the CUDA twin of synth/__init__.py.
//
// Element i of a stream keyed K takes outputs 2i+1 and 2i+2 of the SplitMix64
// stream (Steele, Lea and Flood, OOPSLA 2014) seeded with K, sums their eight
// 16-bit slices (Irwin-Hall, 8 terms), centres and scales that to unit variance
// in fp32, multiplies by sigma, applies the optional x100 heavy tail and rounds
// to the storage dtype.  Elements at or beyond `valid` are zero.  Test and
// benchmark infrastructure only: this library holds none of the method's
// arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t fmix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float value_at(uint64_t i, uint64_t k, uint64_t kt, int heavy,
                                          float c, float sigma) {
  uint64_t w0 = fmix(k + (2 * i + 1) * kGolden);
  uint64_t w1 = fmix(k + (2 * i + 2) * kGolden);
  int64_t s = 0;
#pragma unroll
  for (int sh = 0; sh < 64; sh += 16) {
    s += (int64_t)((w0 >> sh) & 0xFFFFull);
    s += (int64_t)((w1 >> sh) & 0xFFFFull);
  }
  float z = __fmul_rn((float)(s - 262140), c);
  float v = __fmul_rn(z, sigma);
  if (heavy) {
    uint64_t h = fmix(kt + (i + 1) * kGolden) >> 32;
    if (h < 42949672ull) v = __fmul_rn(v, 100.0f);
  }
  return v;
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  uint32_t u = __float_as_uint(v);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

__global__ void synth_fill_kernel(void* out, int dtype, int64_t begin, int64_t count,
                                  int64_t valid, uint64_t k, uint64_t kt, int heavy,
                                  float c, float sigma) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride) {
    int64_t i = begin + j;
    float v = (i < valid) ? value_at((uint64_t)i, k, kt, heavy, c, sigma) : 0.0f;
    if (dtype == 0) {
      static_cast<float*>(out)[j] = v;
    } else {
      static_cast<uint16_t*>(out)[j] = bf16_bits(v);
    }
  }
}

}  // namespace

extern "C" int synth_fill(void* out, int dtype, int64_t begin, int64_t count, int64_t valid,
                          uint64_t k, uint64_t kt, int heavy, float c, float sigma,
                          void* stream) {
  if (count <= 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (count + 255) / 256;
  int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  synth_fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      out, dtype, begin, count, valid, k, kt, heavy, c, sigma);
  return (int)cudaGetLastError();
}
