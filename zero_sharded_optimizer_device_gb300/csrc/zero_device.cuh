// Device helpers: streaming 16-byte loads and stores, bf16 packing, the ring
// summation order and the per-element Adam update.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zero_internal.h"

namespace zk {

constexpr int kThreads = 256;

// Resident 256-thread blocks per SM of each kernel family (the grid is one
// wave: SMs x this cap, or less where the occupancy limit is lower).  The
// defaults and the measurements behind them are in zero_rs.cu; callers may
// override them with zero_set_occupancy().
int occupancy_cap(int kind);

// 16-byte load of data read exactly once (read-only path, no L1 allocation).
__device__ __forceinline__ uint4 ld_once(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16-byte load of optimizer state (read once, then overwritten by this thread).
__device__ __forceinline__ float4 ld_state(const float* p) {
  float4 r;
  asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

// 16-byte streaming store (the data is not read again by this kernel).
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_stream(float* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two bf16 (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint16_t to_bf16(float a) {
  __nv_bfloat16 h = __float2bfloat16_rn(a);
  return *reinterpret_cast<uint16_t*>(&h);
}

// ------------------------------------------------------------------------
// Gradient vectors of 8 elements: bf16 (one 16-byte load) or fp32 (two).
// ------------------------------------------------------------------------
template <typename GT>
struct GradVec;

template <>
struct GradVec<uint16_t> {
  uint4 a;
  __device__ __forceinline__ void load(const void* base, int64_t i) {
    a = ld_once(static_cast<const uint16_t*>(base) + i);
  }
  __device__ __forceinline__ void get(float f[8]) const {
    f[0] = bf16_lo(a.x); f[1] = bf16_hi(a.x);
    f[2] = bf16_lo(a.y); f[3] = bf16_hi(a.y);
    f[4] = bf16_lo(a.z); f[5] = bf16_hi(a.z);
    f[6] = bf16_lo(a.w); f[7] = bf16_hi(a.w);
  }
  __device__ __forceinline__ static float load1(const void* base, int64_t i) {
    uint16_t b = static_cast<const uint16_t*>(base)[i];
    return __uint_as_float((uint32_t)b << 16);
  }
};

template <>
struct GradVec<float> {
  uint4 a, b;
  __device__ __forceinline__ void load(const void* base, int64_t i) {
    const float* p = static_cast<const float*>(base) + i;
    a = ld_once(p);
    b = ld_once(p + 4);
  }
  __device__ __forceinline__ void get(float f[8]) const {
    f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
    f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
    f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
    f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
  }
  __device__ __forceinline__ static float load1(const void* base, int64_t i) {
    return static_cast<const float*>(base)[i];
  }
};

// fp32 gradients whose buffers are 32-byte aligned: the 8 values of a thread
// in one 32-byte load, so that a warp's load covers 1 KiB without gaps (two
// 16-byte loads per thread leave every other 16 bytes to the second load,
// which host memory read over the link serves at half rate).
struct F32x8 {};

template <>
struct GradVec<F32x8> {
  float r[8];
  __device__ __forceinline__ void load(const void* base, int64_t i) {
    const float* p = static_cast<const float*>(base) + i;
    asm volatile("ld.global.nc.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]),
                   "=f"(r[6]), "=f"(r[7])
                 : "l"(p));
  }
  __device__ __forceinline__ void get(float f[8]) const {
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = r[e];
  }
  __device__ __forceinline__ static float load1(const void* base, int64_t i) {
    return static_cast<const float*>(base)[i];
  }
};

// Owner rank of group-local element i: floor(i / S), found from an fp32
// estimate and corrected with exact integer compares.  The estimate converts
// i/256 as a 32-bit integer (i < 2^40): a 64-bit integer conversion would run
// on the FP64 pipe, which is narrow on this GPU.
__device__ __forceinline__ int owner_of(int64_t i, const GroupK& g) {
  int k = __float2int_rz(__uint2float_rz((uint32_t)(i >> 8)) * g.invS256);
  k = k < 0 ? 0 : (k > g.n - 1 ? g.n - 1 : k);
  while (k > 0 && (int64_t)k * g.S > i) --k;
  while (k < g.n - 1 && (int64_t)(k + 1) * g.S <= i) ++k;
  return k;
}

// ------------------------------------------------------------------------
// Ring summation order ["Why DeepSpeed ZeRO paper says reduce-scatter (or
// all-gather) has data movement of Psi elements?"]: the partial sum of owner
// k's chunk starts at rank k+1 and every rank on the ring adds its own copy,
// the owner last: ((g[k+1] + g[k+2]) + ...) + g[k], indices mod N, each add
// rounded to fp32.
// ------------------------------------------------------------------------

// 8 consecutive elements starting at i (i % 8 == 0), all owned by k.
// NT = N known at compile time (batches of up to 16 sources in flight), or
// NT = 0 for any N (batches of 8).
template <int NT, typename GT>
__device__ __forceinline__ void ring_sum8(const RankPtrs& src, int n, int k, int64_t i,
                                          float acc[8]) {
  if constexpr (NT > 0) {
    constexpr int B = NT < 16 ? NT : 16;
    {
      GradVec<GT> g[B];
#pragma unroll
      for (int j = 0; j < B; ++j) {
        int r = k + 1 + j;
        r -= (r >= NT) ? NT : 0;
        g[j].load(src.p[r], i);
      }
      float f[8];
      g[0].get(acc);
#pragma unroll
      for (int j = 1; j < B; ++j) {
        g[j].get(f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
      }
    }
#pragma unroll 1
    for (int jb = B; jb < NT; jb += B) {
      GradVec<GT> g[B];
#pragma unroll
      for (int j = 0; j < B; ++j) {
        int r = k + 1 + jb + j;
        r -= (r >= NT) ? NT : 0;
        g[j].load(src.p[r], i);
      }
#pragma unroll
      for (int j = 0; j < B; ++j) {
        float f[8];
        g[j].get(f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
      }
    }
  } else {
    constexpr int B = 8;
#pragma unroll 1
    for (int jb = 0; jb < n; jb += B) {
      GradVec<GT> g[B];
      const int cnt = (n - jb) < B ? (n - jb) : B;
#pragma unroll
      for (int j = 0; j < B; ++j) {
        if (j < cnt) {
          int r = k + 1 + jb + j;
          r -= (r >= n) ? n : 0;
          g[j].load(src.p[r], i);
        }
      }
#pragma unroll
      for (int j = 0; j < B; ++j) {
        if (j < cnt) {
          float f[8];
          g[j].get(f);
          if (jb == 0 && j == 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = f[e];
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
          }
        }
      }
    }
  }
}

// One element, same order (used for window edges and shard boundaries that
// cut a vector).
template <typename GT>
__device__ __forceinline__ float ring_sum1(const RankPtrs& src, int n, int k, int64_t i) {
  int r = k + 1;
  r -= (r >= n) ? n : 0;
  float acc = GradVec<GT>::load1(src.p[r], i);
  for (int j = 2; j <= n; ++j) {
    r = k + j;
    r -= (r >= n) ? n : 0;
    acc = __fadd_rn(acc, GradVec<GT>::load1(src.p[r], i));
  }
  return acc;
}

// ------------------------------------------------------------------------
// Adam on one element [Kingma and Ba 2015, Algorithm 1], fp32, one IEEE
// rounding per operation, no contraction into FMA:
//   p -= (lr*wd)*p (wd != 0); m = b1*m + (1-b1)*g; v = b2*v + (1-b2)*(g*g);
//   p -= (lr*(m/bc1)) / (sqrt(v/bc2) + eps)
// ------------------------------------------------------------------------
__device__ __forceinline__ void adam1(float& p, float& m, float& v, float g, const AdamK& h) {
  if (h.has_wd) p = __fsub_rn(p, __fmul_rn(h.lrwd, p));
  m = __fadd_rn(__fmul_rn(h.b1, m), __fmul_rn(h.omb1, g));
  v = __fadd_rn(__fmul_rn(h.b2, v), __fmul_rn(h.omb2, __fmul_rn(g, g)));
  const float mh = __fdiv_rn(m, h.bc1);
  const float vh = __fdiv_rn(v, h.bc2);
  const float den = __fadd_rn(__fsqrt_rn(vh), h.eps);
  p = __fsub_rn(p, __fdiv_rn(__fmul_rn(h.lr, mh), den));
}

// Gradient handed to Adam: reduced * scale * coef (coef = 1 without clip;
// multiplying by 1.0f is exact).
__device__ __forceinline__ float scaled(float red, const AdamK& h, float coef) {
  return __fmul_rn(__fmul_rn(red, h.scale), coef);
}

// ------------------------------------------------------------------------
// Checked build (-DZERO_CHECKED): every global access is first tested
// against the extent the C ABI gives its buffer, and one outside is skipped
// and recorded in this translation unit's g_bounds (the first in detail), so
// an indexing mistake shows as a count the host reads rather than as a memory
// fault.  The release build compiles every test to `true`.
// ------------------------------------------------------------------------
#ifdef ZERO_CHECKED
static __device__ BoundsRec g_bounds;
#endif

// True when the access [a, b) lies inside the extent [lo, hi).
__device__ __forceinline__ bool in_extent(int64_t a, int64_t b, int64_t lo, int64_t hi,
                                          int site) {
#ifdef ZERO_CHECKED
  if (a <= b && a >= lo && b <= hi) return true;
  if (atomicAdd(&g_bounds.count, 1ull) == 0ull) {
    g_bounds.site = site;
    g_bounds.index = a;
    g_bounds.lo = lo;
    g_bounds.hi = hi;
  }
  return false;
#else
  (void)a, (void)b, (void)lo, (void)hi, (void)site;
  return true;
#endif
}

// Host side of the record, one copy per translation unit that includes this
// header (zeros, and no CUDA call, in the release build).
static inline cudaError_t bounds_record(BoundsRec* out, bool reset) {
#ifdef ZERO_CHECKED
  cudaError_t e = cudaMemcpyFromSymbol(out, g_bounds, sizeof(BoundsRec));
  if (e == cudaSuccess && reset) {
    const BoundsRec zero{};
    e = cudaMemcpyToSymbol(g_bounds, &zero, sizeof(BoundsRec));
  }
  return e;
#else
  *out = BoundsRec{};
  (void)reset;
  return cudaSuccess;
#endif
}

// Grid-stride loop helper.
__device__ __forceinline__ int64_t gtid() {
  return (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
}
__device__ __forceinline__ int64_t gstride() { return (int64_t)gridDim.x * blockDim.x; }

}  // namespace zk
