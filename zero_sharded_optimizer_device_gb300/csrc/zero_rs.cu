// Reduce-scatter over N emulated ranks, and the fused reduce-scatter + scale
// + Adam + all-gather step.
//
// ["[REQUEST] Direct Correspondence between Gradient and Optimizer States to
// Reduce Communication?", "Problem"]: reduce-scatter the gradients to the
// owners of the optimizer state, update, all-gather the parameters.  All N
// ranks live on this GPU as N gradient buffers, so the reduce-scatter is an
// on-chip N-source reduction in the ring order (zero_device.cuh) and the
// all-gather is the write of the updated parameters into the one full flat
// parameter buffer (or, stage 3, into each owner's shard buffer).
//
// Both kernels stream: every thread owns 8 consecutive elements per
// iteration, loads them from the N sources with 16-byte loads, and the grid
// strides over the window with one resident wave of blocks.
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "zero_device.cuh"

namespace zk {

namespace {

template <typename K>
int resident_blocks(K kernel, int threads) {
  return occupancy_of(reinterpret_cast<const void*>(kernel), threads);
}

int64_t grid_for(int64_t items, int threads, int per_sm) {
  int64_t want = (items + threads - 1) / threads;
  int64_t cap = (int64_t)sm_count() * per_sm;
  if (want > cap) want = cap;
  return want < 1 ? 1 : want;
}

}  // namespace

// Occupancy caps (resident 256-thread blocks per SM) of the kernel families.
// Measured on GB300 with the benchmark's workloads: HBM throughput of these
// streaming kernels often peaks below full occupancy, because fewer
// concurrent request streams per SM keep DRAM accesses more local (the sweep
// below).  zero_set_occupancy() overrides them.
namespace {
// Best caps of a sweep on GB300 with the workloads' random data (GB/s):
// fused N=8 step 3 (6699; 6326 at 2, 6097 at 4), fused N=16 3 (7069), Adam
// 2 (6418; 5775 at 4), reduce-scatter with norm partials 8 (6550-6732;
// 5780 at 3), all-gather cast 4 (6494).  The stage-3 gather's bulk-copy form
// (one issuing thread per CTA, 4 x 8 KiB ring) over the 68 Llama-7B gathers:
// 2 CTAs per SM 6619-6758 (5234 at 1, 6201 at 3, 6294 at 4; the retired
// 16-byte vector form peaked at 6125 with 8 blocks per SM).  Two-stream
// gather pass (ms, 68 gathers + consumers; prefetch CTAs x consumer blocks
// per SM): the two kernels must fit on an SM together to overlap at all;
// 2 x 7 gave 12.28 (one-round consumer) and 28.12 (64 rounds), 4 x 4 11.89
// and 30.55, 3 x 6 12.23 and 29.11, 2 x 5 12.30 and 28.68: the default
// favours the arithmetic-bound consumer, whose time prefetch exists to hide.
constexpr int kOccDefault[ZERO_OCC_KINDS] = {
    3,   // ZERO_OCC_FUSED
    8,   // ZERO_OCC_RS
    2,   // ZERO_OCC_ADAM
    2,   // ZERO_OCC_GATHER
    4,   // ZERO_OCC_STREAM
    7,   // ZERO_OCC_CONSUMER
    2,   // ZERO_OCC_PREFETCH
};
std::atomic<int> g_occ[ZERO_OCC_KINDS] = {{0}, {0}, {0}, {0}, {0}, {0}, {0}};
}  // namespace

int occupancy_cap(int kind) {
  const int v = g_occ[kind].load(std::memory_order_relaxed);
  return v > 0 ? v : kOccDefault[kind];
}

namespace {
std::mutex g_dev_mu;
std::map<int, int> g_sms;                                // device -> SM count
std::map<std::pair<int, const void*>, int> g_resident;   // (device, kernel) -> blocks/SM
}  // namespace

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) return it->second;
  int s = 0;
  if (cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || s < 1)
    s = 1;
  g_sms[dev] = s;
  return s;
}

int occupancy_of(const void* kernel, int threads) {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  auto key = std::make_pair(dev, kernel);
  auto it = g_resident.find(key);
  if (it != g_resident.end()) return it->second;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, 0) != cudaSuccess ||
      nb < 1)
    nb = 1;
  g_resident[key] = nb;
  return nb;
}

// ---------------------------------------------------------------------------
// Reduce-scatter: reduced[flat_off + i] = ring sum, i in [begin, end);
// optional fp64 per-block partial sums of (reduced*scale)^2.
// ---------------------------------------------------------------------------
template <int NT, typename GT>
__global__ void __launch_bounds__(kThreads)
    rs_kernel(RankPtrs src, GroupK g, int64_t begin, int64_t end, float* __restrict__ reduced,
              float scale, double* __restrict__ partials, int mode) {
  const int n = NT > 0 ? NT : g.n;
  const int64_t q0 = begin >> 3, q1 = (end + 7) >> 3;
  const bool flat_vec_ok = (g.flat_off & 7) == 0;  // 16-byte vectors in flat arrays
  double ss = 0.0;
  for (int64_t q = q0 + gtid(); q < q1; q += gstride()) {
    const int64_t i = q << 3;
    const int k = owner_of(i, g);
    float* out = reduced + g.flat_off + i;  // not dereferenced in RS_NORM_ONLY
    if (flat_vec_ok && i >= begin && i + 8 <= end && i + 7 < (int64_t)(k + 1) * g.S) {
      if (!in_extent(i, i + 8, (int64_t)k * g.S, (int64_t)(k + 1) * g.S, ZERO_SITE_RS_OWNER) ||
          !in_extent(i, i + 8, 0, (int64_t)n * g.S, ZERO_SITE_RS_GRAD) ||
          !in_extent(i, i + 8, begin, end, ZERO_SITE_RS_FLAT))
        continue;
      float acc[8];
      ring_sum8<NT, GT>(src, n, k, i, acc);
      if (mode == RS_ACCUMULATE) {  // previous micro-batches first, then this one
        const float4 a = ld_state(out), b = ld_state(out + 4);
        const float prev[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(prev[e], acc[e]);
      }
      if (mode != RS_NORM_ONLY) {
        st_stream(out, make_float4(acc[0], acc[1], acc[2], acc[3]));
        st_stream(out + 4, make_float4(acc[4], acc[5], acc[6], acc[7]));
      }
      if (partials) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = __fmul_rn(acc[e], scale);
          s = __fadd_rn(s, __fmul_rn(x, x));
        }
        ss += (double)s;
      }
    } else {
      float s = 0.f;
      for (int e = 0; e < 8; ++e) {
        const int64_t j = i + e;
        if (j < begin || j >= end) continue;
        const int kj = owner_of(j, g);
        if (!in_extent(j, j + 1, (int64_t)kj * g.S, (int64_t)(kj + 1) * g.S,
                       ZERO_SITE_RS_OWNER) ||
            !in_extent(j, j + 1, 0, (int64_t)n * g.S, ZERO_SITE_RS_GRAD) ||
            !in_extent(j, j + 1, begin, end, ZERO_SITE_RS_FLAT))
          continue;
        float r = ring_sum1<GT>(src, n, kj, j);
        if (mode == RS_ACCUMULATE) r = __fadd_rn(out[e], r);
        if (mode != RS_NORM_ONLY) out[e] = r;
        const float x = __fmul_rn(r, scale);
        s = __fadd_rn(s, __fmul_rn(x, x));
      }
      ss += (double)s;
    }
  }
  if (!partials) return;
  // fixed-order block reduction: warp shuffle tree, then warp 0
  __shared__ double red[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_down_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    double t = threadIdx.x < kThreads / 32 ? red[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_down_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) partials[blockIdx.x] = t;
  }
}

// ---------------------------------------------------------------------------
// Fused step: ring sum -> scale (-> clip) -> Adam -> cast, one pass.
// ---------------------------------------------------------------------------
template <int NT, typename GT>
__global__ void __launch_bounds__(kThreads)
    fused_kernel(RankPtrs src, GroupK g, int64_t begin, int64_t end, float* __restrict__ master,
                 float* __restrict__ mom, float* __restrict__ var, AdamK h,
                 const float* __restrict__ coef_ptr, const float* __restrict__ prev,
                 int out_mode, void* __restrict__ out_full, OutPtrs shards) {
  const int n = NT > 0 ? NT : g.n;
  const float coef = coef_ptr ? *coef_ptr : 1.0f;
  if (h.bcp) {  // bias corrections kept on the device (graph-replayable steps)
    h.bc1 = h.bcp[0];
    h.bc2 = h.bcp[1];
  }
  const int64_t q0 = begin >> 3, q1 = (end + 7) >> 3;
  const bool shard_vec_ok = ((g.rank_off | g.S) & 7) == 0;
  const bool flat_vec_ok = (g.flat_off & 7) == 0;  // 16-byte vectors in flat arrays
  for (int64_t q = q0 + gtid(); q < q1; q += gstride()) {
    const int64_t i = q << 3;
    const int64_t f = g.flat_off + i;
    const int k = owner_of(i, g);
    if (flat_vec_ok && i >= begin && i + 8 <= end && i + 7 < (int64_t)(k + 1) * g.S) {
      if (!in_extent(i, i + 8, (int64_t)k * g.S, (int64_t)(k + 1) * g.S,
                     ZERO_SITE_STEP_OWNER) ||
          !in_extent(i, i + 8, 0, (int64_t)n * g.S, ZERO_SITE_STEP_GRAD) ||
          !in_extent(f, f + 8, g.flat_off + begin, g.flat_off + end, ZERO_SITE_STEP_FLAT))
        continue;
      const float4 p0 = ld_state(master + f), p1 = ld_state(master + f + 4);
      const float4 m0 = ld_state(mom + f), m1 = ld_state(mom + f + 4);
      const float4 v0 = ld_state(var + f), v1 = ld_state(var + f + 4);
      float acc[8];
      ring_sum8<NT, GT>(src, n, k, i, acc);
      if (prev) {  // gradient accumulation: earlier micro-batches first, then this one
        const uint4 a = ld_once(prev + f), b = ld_once(prev + f + 4);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(__uint_as_float(w[e]), acc[e]);
      }
      float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) adam1(p[e], m[e], v[e], scaled(acc[e], h, coef), h);
      st_stream(master + f, make_float4(p[0], p[1], p[2], p[3]));
      st_stream(master + f + 4, make_float4(p[4], p[5], p[6], p[7]));
      st_stream(mom + f, make_float4(m[0], m[1], m[2], m[3]));
      st_stream(mom + f + 4, make_float4(m[4], m[5], m[6], m[7]));
      st_stream(var + f, make_float4(v[0], v[1], v[2], v[3]));
      st_stream(var + f + 4, make_float4(v[4], v[5], v[6], v[7]));
      if (out_mode == OUT_FULL_BF16) {
        st_stream(static_cast<uint16_t*>(out_full) + f,
                  make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                             pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7])));
      } else if (out_mode == OUT_FULL_F32) {
        float* o = static_cast<float*>(out_full) + f;
        st_stream(o, make_float4(p[0], p[1], p[2], p[3]));
        st_stream(o + 4, make_float4(p[4], p[5], p[6], p[7]));
      } else if (out_mode == OUT_SHARDS_BF16) {
        const int64_t so = g.rank_off + (i - (int64_t)k * g.S);
        if (!in_extent(so, so + 8, g.rank_off, g.rank_off + g.S, ZERO_SITE_STEP_SHARD)) continue;
        uint16_t* o = static_cast<uint16_t*>(shards.p[k]) + so;
        if (shard_vec_ok) {
          st_stream(o, make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                                  pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7])));
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = to_bf16(p[e]);
        }
      }
    } else {
      for (int e = 0; e < 8; ++e) {
        const int64_t j = i + e;
        if (j < begin || j >= end) continue;
        const int kj = owner_of(j, g);
        const int64_t so = g.rank_off + (j - (int64_t)kj * g.S);
        if (!in_extent(j, j + 1, (int64_t)kj * g.S, (int64_t)(kj + 1) * g.S,
                       ZERO_SITE_STEP_OWNER) ||
            !in_extent(j, j + 1, 0, (int64_t)n * g.S, ZERO_SITE_STEP_GRAD) ||
            !in_extent(f + e, f + e + 1, g.flat_off + begin, g.flat_off + end,
                       ZERO_SITE_STEP_FLAT) ||
            (out_mode == OUT_SHARDS_BF16 &&
             !in_extent(so, so + 1, g.rank_off, g.rank_off + g.S, ZERO_SITE_STEP_SHARD)))
          continue;
        float r = ring_sum1<GT>(src, n, kj, j);
        if (prev) r = __fadd_rn(prev[f + e], r);
        float p = master[f + e], m = mom[f + e], v = var[f + e];
        adam1(p, m, v, scaled(r, h, coef), h);
        master[f + e] = p;
        mom[f + e] = m;
        var[f + e] = v;
        if (out_mode == OUT_FULL_BF16) {
          static_cast<uint16_t*>(out_full)[f + e] = to_bf16(p);
        } else if (out_mode == OUT_FULL_F32) {
          static_cast<float*>(out_full)[f + e] = p;
        } else if (out_mode == OUT_SHARDS_BF16) {
          static_cast<uint16_t*>(shards.p[kj])[so] = to_bf16(p);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Dispatch on N (compile-time specialisations for common N) and dtype.
// ---------------------------------------------------------------------------
namespace {

template <template <int, typename> class Launch, typename... A>
cudaError_t dispatch(int n, int gdtype, A&&... a) {
  if (gdtype == ZERO_BF16) {
    switch (n) {
      case 2: return Launch<2, uint16_t>::run(a...);
      case 4: return Launch<4, uint16_t>::run(a...);
      case 8: return Launch<8, uint16_t>::run(a...);
      case 16: return Launch<16, uint16_t>::run(a...);
      case 32: return Launch<32, uint16_t>::run(a...);
      case 64: return Launch<64, uint16_t>::run(a...);
      default: return Launch<0, uint16_t>::run(a...);
    }
  }
  switch (n) {
    case 2: return Launch<2, float>::run(a...);
    case 4: return Launch<4, float>::run(a...);
    case 8: return Launch<8, float>::run(a...);
    case 16: return Launch<16, float>::run(a...);
    case 32: return Launch<32, float>::run(a...);
    case 64: return Launch<64, float>::run(a...);
    default: return Launch<0, float>::run(a...);
  }
}

// The fused step only: fp32 sources that are all 32-byte aligned.
template <template <int, typename> class Launch, typename... A>
cudaError_t dispatch_f32_wide(int n, A&&... a) {
  switch (n) {
    case 2: return Launch<2, F32x8>::run(a...);
    case 4: return Launch<4, F32x8>::run(a...);
    case 8: return Launch<8, F32x8>::run(a...);
    case 16: return Launch<16, F32x8>::run(a...);
    case 32: return Launch<32, F32x8>::run(a...);
    case 64: return Launch<64, F32x8>::run(a...);
    default: return Launch<0, F32x8>::run(a...);
  }
}

template <int NT, typename GT>
struct RsLaunch {
  // One grid for a window of n elements: one block per 256 vectors, at most
  // one resident wave.  The partial count a caller reserves is this grid.
  static int64_t grid(int64_t n_elements) {
    const int64_t vecs = (n_elements + 7) / 8 + 1;
    const int nb = resident_blocks(rs_kernel<NT, GT>, kThreads);
    const int cap = occupancy_cap(ZERO_OCC_RS);
    return grid_for(vecs, kThreads, nb < cap ? nb : cap);
  }
  static cudaError_t run(const RankPtrs& src, const GroupK& g, int64_t begin, int64_t end,
                         float* reduced, float scale, double* partials, int mode,
                         cudaStream_t st, int64_t fixed) {
    const int64_t blocks = fixed > 0 ? fixed : grid(end - begin);
    rs_kernel<NT, GT><<<(unsigned)blocks, kThreads, 0, st>>>(
        src, g, begin, end, reduced, scale, partials, mode);
    return cudaGetLastError();
  }
};

template <int NT, typename GT>
struct RsGrid {
  static cudaError_t run(int64_t n_elements, int64_t* out) {
    *out = RsLaunch<NT, GT>::grid(n_elements);
    return cudaSuccess;
  }
};

template <int NT, typename GT>
struct FusedLaunch {
  static cudaError_t run(const RankPtrs& src, const GroupK& g, int64_t begin, int64_t end,
                         float* master, float* m, float* v, const AdamK& h, const float* coef,
                         const float* prev, int out_mode, void* out_full, const OutPtrs& shards,
                         cudaStream_t st) {
    auto kern = fused_kernel<NT, GT>;
    const int64_t vecs = ((end + 7) >> 3) - (begin >> 3);
    const int nb = resident_blocks(kern, kThreads);
    const int cap = occupancy_cap(ZERO_OCC_FUSED);
    const int64_t grid = grid_for(vecs, kThreads, nb < cap ? nb : cap);
    kern<<<(unsigned)grid, kThreads, 0, st>>>(src, g, begin, end, master, m, v, h, coef, prev,
                                               out_mode, out_full, shards);
    return cudaGetLastError();
  }
};

}  // namespace

// Partials written by one reduce-scatter call over n elements with N ranks.
int64_t rs_partials_for(int n, int gdtype, int64_t n_elements) {
  int64_t out = 0;
  dispatch<RsGrid>(n, gdtype, n_elements, &out);
  return out;
}

cudaError_t launch_reduce_scatter(const RankPtrs& src, int gdtype, const GroupK& g,
                                  float* reduced, int64_t begin, int64_t end, float scale,
                                  double* partials, int mode, cudaStream_t st, int64_t grid) {
  if (end <= begin) return cudaSuccess;
  return dispatch<RsLaunch>(g.n, gdtype, src, g, begin, end, reduced, scale, partials, mode,
                            st, grid);
}

cudaError_t launch_fused(const RankPtrs& src, int gdtype, const GroupK& g, int64_t begin,
                         int64_t end, float* master, float* m, float* v, const AdamK& h,
                         const float* coef, const float* prev, int out_mode, void* out_full,
                         const OutPtrs& shards, cudaStream_t st) {
  if (end <= begin) return cudaSuccess;
  if (gdtype == kF32Aligned32)
    return dispatch_f32_wide<FusedLaunch>(g.n, src, g, begin, end, master, m, v, h, coef, prev,
                                          out_mode, out_full, shards, st);
  return dispatch<FusedLaunch>(g.n, gdtype, src, g, begin, end, master, m, v, h, coef, prev,
                               out_mode, out_full, shards, st);
}

cudaError_t bounds_rs(BoundsRec* out, bool reset) { return bounds_record(out, reset); }

}  // namespace zk

extern "C" int zero_set_occupancy(int32_t kind, int32_t blocks_per_sm, int32_t* previous) {
  if (kind < 0 || kind >= ZERO_OCC_KINDS || blocks_per_sm < 0 || blocks_per_sm > 32)
    return ZERO_EINVAL;
  if (previous) *previous = zk::occupancy_cap(kind);
  zk::g_occ[kind].store(blocks_per_sm, std::memory_order_relaxed);
  return ZERO_OK;
}
