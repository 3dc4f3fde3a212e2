// Unfused pieces of the step and the stage-3 gather:
//   adam_kernel     Adam over a window of the materialised reduced gradient
//   cast_kernel     all-gather of the updated parameters into the full buffer
//   norm_kernel     global gradient norm and clip coefficient
//   gather_bulk_kernel / gather_kernel  stage-3 per-layer gather of N rank shards
//   checksum_kernel consumer of a gathered layer (stands in for its computation)
//   copy_kernel     16-byte device copy (achievable HBM bandwidth)
#include <atomic>

#include "zero_device.cuh"

namespace zk {

namespace {

template <typename K>
int64_t wave_grid(K kernel, int64_t items, int kind) {
  const int cap = occupancy_cap(kind);
  int nb = occupancy_of(reinterpret_cast<const void*>(kernel), kThreads);
  if (nb > cap) nb = cap;
  int64_t want = (items + kThreads - 1) / kThreads;
  const int64_t wave = (int64_t)sm_count() * nb;
  if (want > wave) want = wave;
  return want < 1 ? 1 : want;
}

}  // namespace

// ---------------------------------------------------------------------------
// Adam on [begin, end) of a group from the fp32 reduced gradient.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
    adam_kernel(GroupK g, int64_t begin, int64_t end, float* __restrict__ master,
                float* __restrict__ mom, float* __restrict__ var,
                const float* __restrict__ reduced, AdamK h, const float* __restrict__ coef_ptr,
                int out_mode, void* __restrict__ out) {
  const float coef = coef_ptr ? *coef_ptr : 1.0f;
  if (h.bcp) {  // bias corrections kept on the device (graph-replayable steps)
    h.bc1 = h.bcp[0];
    h.bc2 = h.bcp[1];
  }
  const int64_t q0 = begin >> 3, q1 = (end + 7) >> 3;
  const bool flat_vec_ok = (g.flat_off & 7) == 0;
  for (int64_t q = q0 + gtid(); q < q1; q += gstride()) {
    const int64_t i = q << 3;
    const int64_t f = g.flat_off + i;
    if (flat_vec_ok && i >= begin && i + 8 <= end) {
      if (!in_extent(f, f + 8, g.flat_off + begin, g.flat_off + end, ZERO_SITE_ADAM_FLAT))
        continue;
      const uint4 r0 = ld_once(reduced + f), r1 = ld_once(reduced + f + 4);
      const float4 p0 = ld_state(master + f), p1 = ld_state(master + f + 4);
      const float4 m0 = ld_state(mom + f), m1 = ld_state(mom + f + 4);
      const float4 v0 = ld_state(var + f), v1 = ld_state(var + f + 4);
      float r[8] = {__uint_as_float(r0.x), __uint_as_float(r0.y), __uint_as_float(r0.z),
                    __uint_as_float(r0.w), __uint_as_float(r1.x), __uint_as_float(r1.y),
                    __uint_as_float(r1.z), __uint_as_float(r1.w)};
      float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) adam1(p[e], m[e], v[e], scaled(r[e], h, coef), h);
      st_stream(master + f, make_float4(p[0], p[1], p[2], p[3]));
      st_stream(master + f + 4, make_float4(p[4], p[5], p[6], p[7]));
      st_stream(mom + f, make_float4(m[0], m[1], m[2], m[3]));
      st_stream(mom + f + 4, make_float4(m[4], m[5], m[6], m[7]));
      st_stream(var + f, make_float4(v[0], v[1], v[2], v[3]));
      st_stream(var + f + 4, make_float4(v[4], v[5], v[6], v[7]));
      if (out_mode == OUT_FULL_BF16) {
        st_stream(static_cast<uint16_t*>(out) + f,
                  make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                             pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7])));
      } else if (out_mode == OUT_FULL_F32) {
        float* o = static_cast<float*>(out) + f;
        st_stream(o, make_float4(p[0], p[1], p[2], p[3]));
        st_stream(o + 4, make_float4(p[4], p[5], p[6], p[7]));
      }
    } else {
      for (int e = 0; e < 8; ++e) {
        const int64_t j = i + e;
        if (j < begin || j >= end) continue;
        if (!in_extent(f + e, f + e + 1, g.flat_off + begin, g.flat_off + end,
                       ZERO_SITE_ADAM_FLAT))
          continue;
        float p = master[f + e], m = mom[f + e], v = var[f + e];
        adam1(p, m, v, scaled(reduced[f + e], h, coef), h);
        master[f + e] = p;
        mom[f + e] = m;
        var[f + e] = v;
        if (out_mode == OUT_FULL_BF16) static_cast<uint16_t*>(out)[f + e] = to_bf16(p);
        else if (out_mode == OUT_FULL_F32) static_cast<float*>(out)[f + e] = p;
      }
    }
  }
}

cudaError_t launch_adam(const GroupK& g, int64_t begin, int64_t end, float* master, float* m,
                        float* v, const float* reduced, const AdamK& h, const float* coef,
                        int out_mode, void* out, cudaStream_t st) {
  if (end <= begin) return cudaSuccess;
  const int64_t vecs = ((end + 7) >> 3) - (begin >> 3);
  adam_kernel<<<(unsigned)wave_grid(adam_kernel, vecs, ZERO_OCC_ADAM), kThreads, 0, st>>>(
      g, begin, end, master, m, v, reduced, h, coef, out_mode, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// All-gather: dst[i] = cast(src[i]) for i in [a, b) (flat indices).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
    cast_kernel(const float* __restrict__ src, int64_t a, int64_t b, int out_dtype,
                void* __restrict__ dst) {
  const int64_t q0 = a >> 3, q1 = (b + 7) >> 3;
  for (int64_t q = q0 + gtid(); q < q1; q += gstride()) {
    const int64_t i = q << 3;
    if (i >= a && i + 8 <= b) {
      if (!in_extent(i, i + 8, a, b, ZERO_SITE_CAST_FLAT)) continue;
      const uint4 x0 = ld_once(src + i), x1 = ld_once(src + i + 4);
      if (out_dtype == ZERO_BF16) {
        st_stream(static_cast<uint16_t*>(dst) + i,
                  make_uint4(pack_bf16x2(__uint_as_float(x0.x), __uint_as_float(x0.y)),
                             pack_bf16x2(__uint_as_float(x0.z), __uint_as_float(x0.w)),
                             pack_bf16x2(__uint_as_float(x1.x), __uint_as_float(x1.y)),
                             pack_bf16x2(__uint_as_float(x1.z), __uint_as_float(x1.w))));
      } else {
        float* o = static_cast<float*>(dst) + i;
        st_stream((void*)o, x0);
        st_stream((void*)(o + 4), x1);
      }
    } else {
      for (int e = 0; e < 8; ++e) {
        const int64_t j = i + e;
        if (j < a || j >= b) continue;
        if (!in_extent(j, j + 1, a, b, ZERO_SITE_CAST_FLAT)) continue;
        if (out_dtype == ZERO_BF16) static_cast<uint16_t*>(dst)[j] = to_bf16(src[j]);
        else static_cast<float*>(dst)[j] = src[j];
      }
    }
  }
}

cudaError_t launch_cast(const float* src, int64_t a, int64_t b, int out_dtype, void* dst,
                        cudaStream_t st) {
  if (b <= a) return cudaSuccess;
  const int64_t vecs = ((b + 7) >> 3) - (a >> 3);
  cast_kernel<<<(unsigned)wave_grid(cast_kernel, vecs, ZERO_OCC_STREAM), kThreads, 0, st>>>(src, a, b, out_dtype,
                                                                           dst);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Global norm: one block sums the fp64 partials in a fixed order.
// ---------------------------------------------------------------------------
constexpr int kNormThreads = 1024;

__global__ void __launch_bounds__(kNormThreads)
    norm_kernel(const double* __restrict__ partials, int64_t n, float max_norm,
                float* __restrict__ d_norm, float* __restrict__ d_coef) {
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += kNormThreads)
    if (in_extent(i, i + 1, 0, n, ZERO_SITE_NORM)) s += partials[i];
  __shared__ double red[kNormThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    double t = red[threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_down_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) {
      const double norm = sqrt(t);
      double coef = (double)max_norm / (norm + 1e-6);
      if (coef > 1.0) coef = 1.0;
      if (d_norm) *d_norm = (float)norm;
      if (d_coef) *d_coef = (float)coef;
    }
  }
}

cudaError_t launch_norm(const double* partials, int64_t n, float max_norm, float* d_norm,
                        float* d_coef, cudaStream_t st) {
  norm_kernel<<<1, kNormThreads, 0, st>>>(partials, n, max_norm, d_norm, d_coef);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Stage-3 gather, element by element: out[j] = shards[j / S][rank_off + j % S]
// for j < psi_pad.  Only for shards whose start or length breaks the 16-byte
// rule of the bulk-copy form below (align < 8 bf16 elements).
// ---------------------------------------------------------------------------
template <int ES>
__global__ void __launch_bounds__(kThreads)
    gather_kernel(RankPtrs shards, GroupK g, int64_t psi_pad, void* __restrict__ out) {
  for (int64_t j = gtid(); j < psi_pad; j += gstride()) {
    const int k = owner_of(j, g);
    const int64_t src = g.rank_off + (j - (int64_t)k * g.S);
    if (!in_extent(src, src + 1, g.rank_off, g.rank_off + g.S, ZERO_SITE_GATHER_SHARD) ||
        !in_extent(j, j + 1, 0, psi_pad, ZERO_SITE_GATHER_OUT))
      continue;
    if (ES == 2)
      static_cast<uint16_t*>(out)[j] = static_cast<const uint16_t*>(shards.p[k])[src];
    else
      static_cast<uint32_t*>(out)[j] = static_cast<const uint32_t*>(shards.p[k])[src];
  }
}

// ---------------------------------------------------------------------------
// Stage-3 gather with 1-D bulk copies (TMA).  The layer is N contiguous
// segments (owner k's S elements land at k*S), cut into pieces of up to
// kBulkChunk bytes.  One thread per CTA moves its pieces global -> shared ->
// global through a ring of STAGES buffers: a piece's load completes on its
// stage's mbarrier (expect_tx), its store is a bulk-group copy, and a stage is
// refilled once the store that read it has finished reading.  Every mbarrier
// wait gives up after ~2 s: the timeout is counted in g_async_timeouts
// (zero_async_status), the CTA lets the loads it issued land (again bounded)
// and returns.  Used when every segment start and length is a multiple of 16
// bytes; gather_kernel otherwise.
//
// Ring depth and launch, measured over the 68 Llama-7B gathers (GB/s at 1 /
// 2 / 3 / 4 CTAs per SM): 8 KiB x 4 stages 5234 / 6619 / 6201 / 6294, x 6
// stages 6158 / 6237 / 6175 / 6136; 16 KiB x 4 6437 / 6287 / 6135 / 6256;
// 32 KiB x 3 6614 / 6299 / 6369 / 6416 -- about 48-64 KiB of loads in flight
// per SM is best, more is slower.  Inside the two-stream pass, beside the
// consumer, the deeper ring is better (pass 12.3 ms at 6 stages against 13.0
// at 4, 2 CTAs per SM beside 7 consumer blocks).  Standalone gathers also use
// programmatic dependent launch (PDL): the CTAs become resident while the
// kernel before them finishes and start copying once it has
// (griddepcontrol.wait), which removes the gap between back-to-back gathers
// (68 gathers +1.4 %, the 16 launches of a broadcast -11 % time); inside the
// pass the gathers wait on events anyway, and PDL there measured 1.6 % slower.
// ---------------------------------------------------------------------------
constexpr int kBulkChunk = 8192;
constexpr int kBulkStagesAlone = 4;     // zero_gather_layer, zero_gather_groups, broadcast
constexpr int kBulkStagesPrefetch = 6;  // inside zero_stage3_gather_pass
constexpr int kBulkThreads = 32;       // one warp per CTA; lane 0 issues
constexpr int kGatherElemBlocks = 8;   // resident blocks per SM of the element fallback
constexpr unsigned long long kWaitNs = 2000000000ull;

static __device__ unsigned long long g_async_timeouts;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait until the mbarrier's phase of this parity has completed; false after
// kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (true) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}

// The pieces of one launch are numbered owner by owner: owner k's pieces of
// all the launch's groups come before owner k+1's, so the CTAs stream one
// rank's shard buffer at a time, as for a single group.  Within owner k,
// group i's segment is pieces [first[i], first[i+1]).  CTA b takes pieces
// b, b + G, b + 2G, ... (G CTAs); it walks them with a cursor (owner k, piece
// co inside the owner, group gi holding co) instead of dividing per piece:
// one 32-bit division where the cursor passes an owner's end, a short forward
// scan of the group boundaries otherwise.  Piece counts stay below 2^31 (the
// host refuses larger launches).  Each stage remembers the destination and
// size of the piece it holds, so the store does not recompute them.
template <int STAGES, bool PDL>
__global__ void __launch_bounds__(kBulkThreads)
    gather_bulk_kernel(RankPtrs shards, BulkGroups bg) {
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[STAGES];
  __shared__ char* stage_dst[STAGES];
  __shared__ uint32_t stage_bytes[STAGES];
  if (threadIdx.x != 0) return;
  if constexpr (PDL) {
    // let the next kernel on the stream become resident now; copy only once
    // the kernel before this one has finished and its writes are visible
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
  }
  const uint32_t bar0 = smem_addr(full), buf0 = smem_addr(ring);
  for (int s = 0; s < STAGES; ++s)
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8 * s));
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const uint32_t G = gridDim.x, b = blockIdx.x;
  const uint32_t per_owner = (uint32_t)bg.first[bg.ng];
  const uint32_t nchunks = per_owner * (uint32_t)bg.n;
  const uint32_t niter = b < nchunks ? (nchunks - b + G - 1) / G : 0;
  const int es = bg.es, ng = bg.ng;
  // cursor at this CTA's first piece
  uint32_t k = b / per_owner, co = b - k * per_owner;
  int gi = 0;
  while (gi + 1 < ng && (uint32_t)bg.first[gi + 1] <= co) ++gi;

  // issue the load of the cursor's piece into stage s, then advance
  auto load = [&](int s) {
    const int64_t S = bg.S[gi], ro = bg.rank_off[gi];
    const int64_t off = (int64_t)(co - (uint32_t)bg.first[gi]) * kBulkChunk;  // bytes
    const int64_t rem = S * es - off;
    const uint32_t bytes = (uint32_t)(rem < kBulkChunk ? rem : kBulkChunk);
    const char* src = static_cast<const char*>(shards.p[k]) + ro * es + off;
    char* dst = bg.out[gi] + (int64_t)k * S * es + off;
    // element ranges of the checked build (compiled out of the release build)
    const int64_t so = ro + off / es, j = (int64_t)k * S + off / es, len = bytes / es;
    const bool ok =
        in_extent(co, co + 1, bg.first[gi], bg.first[gi + 1], ZERO_SITE_GATHER_OUT) &&
        in_extent(k, k + 1, 0, bg.n, ZERO_SITE_GATHER_SHARD) &&
        in_extent(so, so + len, ro, ro + S, ZERO_SITE_GATHER_SHARD) &&
        in_extent(j, j + len, 0, (int64_t)bg.n * S, ZERO_SITE_GATHER_OUT);
    const uint32_t bar = bar0 + 8 * (uint32_t)s;
    stage_dst[s] = ok ? dst : nullptr;
    stage_bytes[s] = bytes;
    if (ok) {
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                   "r"(bytes)
                   : "memory");
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
          "[%3];" ::"r"(buf0 + (uint32_t)s * kBulkChunk),
          "l"(src), "r"(bytes), "r"(bar)
          : "memory");
    } else {  // skipped piece: complete the phase with no bytes
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
    }
    co += G;
    if (co >= per_owner) {
      const uint32_t q = co / per_owner;
      k += q;
      co -= q * per_owner;
      gi = 0;
    }
    while (gi + 1 < ng && (uint32_t)bg.first[gi + 1] <= co) ++gi;
  };

  const uint32_t pro = niter < STAGES - 1 ? niter : STAGES - 1;
  for (uint32_t i = 0; i < pro; ++i) load((int)i);
  uint32_t loaded = pro, i = 0;
  int s = 0;          // stage of piece i
  uint32_t ph = 0;    // its mbarrier phase parity
  for (; i < niter; ++i) {
    if (!mbar_wait(bar0 + 8 * s, ph)) {
      atomicAdd(&g_async_timeouts, 1ull);
      break;
    }
    if (stage_dst[s])
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                       stage_dst[s]),
                   "r"(buf0 + (uint32_t)s * kBulkChunk), "r"(stage_bytes[s])
                   : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    // refill the stage of piece i - 1 once its store has read it
    if (loaded < niter) {
      asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
      load(s == 0 ? STAGES - 1 : s - 1);
      ++loaded;
    }
    if (++s == STAGES) {
      s = 0;
      ph ^= 1u;
    }
  }
  // after a timeout: the loads still in flight land before the CTA exits
  for (uint32_t j = i; j < loaded; ++j) {
    if (!mbar_wait(bar0 + 8 * s, ph)) atomicAdd(&g_async_timeouts, 1ull);
    if (++s == STAGES) {
      s = 0;
      ph ^= 1u;
    }
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

bool bulk_eligible(int64_t S, int64_t rank_off, int elem_bytes) {
  return (S * elem_bytes) % 16 == 0 && (rank_off * elem_bytes) % 16 == 0;
}

void bulk_add(BulkGroups& bg, int64_t S, int64_t rank_off, void* out) {
  const int i = bg.ng++;
  const int64_t cps = S > 0 ? (S * bg.es + kBulkChunk - 1) / kBulkChunk : 0;
  bg.S[i] = S;
  bg.rank_off[i] = rank_off;
  bg.out[i] = static_cast<char*>(out);
  bg.first[i + 1] = bg.first[i] + cps;
}

// The ring plus the kernel's static shared memory may pass the default 48 KiB
// per CTA, so the kernel's dynamic limit is raised once per device.
template <int STAGES, bool PDL>
static cudaError_t bulk_ring_attr() {
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load() & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(gather_bulk_kernel<STAGES, PDL>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, STAGES * kBulkChunk);
  if (e == cudaSuccess) done.fetch_or(bit);
  return e;
}

template <int STAGES, bool PDL>
static cudaError_t launch_bulk(const RankPtrs& shards, const BulkGroups& bg, int64_t grid,
                               cudaStream_t st) {
  cudaError_t e = bulk_ring_attr<STAGES, PDL>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kBulkThreads);
  cfg.dynamicSmemBytes = STAGES * kBulkChunk;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PDL ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gather_bulk_kernel<STAGES, PDL>, shards, bg);
}

cudaError_t launch_gather_bulk(const RankPtrs& shards, const BulkGroups& bg, int occ_kind,
                               cudaStream_t st) {
  const int64_t nchunks = bg.first[bg.ng] * bg.n;
  if (nchunks <= 0) return cudaSuccess;
  if (nchunks >= (1ll << 31)) return cudaErrorInvalidValue;  // the kernel counts in 32 bits
  int64_t grid = (int64_t)sm_count() * occupancy_cap(occ_kind);
  if (grid > nchunks) grid = nchunks;
  if (occ_kind == ZERO_OCC_PREFETCH)
    return launch_bulk<kBulkStagesPrefetch, false>(shards, bg, grid, st);
  return launch_bulk<kBulkStagesAlone, true>(shards, bg, grid, st);
}

cudaError_t launch_gather(const RankPtrs& shards, int elem_bytes, const GroupK& g,
                          int64_t psi_pad, void* out, int occ_kind, cudaStream_t st) {
  if (psi_pad <= 0) return cudaSuccess;
  if (bulk_eligible(g.S, g.rank_off, elem_bytes)) {
    BulkGroups bg{};
    bg.es = elem_bytes;
    bg.n = g.n;
    bulk_add(bg, g.S, g.rank_off, out);
    return launch_gather_bulk(shards, bg, occ_kind, st);
  }
  const int64_t wave = (int64_t)sm_count() * kGatherElemBlocks;
  const int64_t want = psi_pad / kThreads + 1;
  const unsigned grid = (unsigned)(want < wave ? want : wave);
  if (elem_bytes == 2)
    gather_kernel<2><<<grid, kThreads, 0, st>>>(shards, g, psi_pad, out);
  else
    gather_kernel<4><<<grid, kThreads, 0, st>>>(shards, g, psi_pad, out);
  return cudaGetLastError();
}

cudaError_t launch_broadcast(const RankPtrs& shards, int elem_bytes, const GroupK& g, void* out,
                             int occ_kind, cudaStream_t st) {
  if (g.S <= 0) return cudaSuccess;
  GroupK one = g;  // a group of one rank: owner k's shard alone
  one.n = 1;
  one.invS256 = 0.0f;
  for (int k = 0; k < g.n; ++k) {
    RankPtrs root{};
    root.p[0] = shards.p[k];
    void* dst = static_cast<char*>(out) + (int64_t)k * g.S * elem_bytes;
    const cudaError_t e = launch_gather(root, elem_bytes, one, g.S, dst, occ_kind, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t async_timeouts(unsigned long long* out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_async_timeouts, sizeof(unsigned long long));
  if (e == cudaSuccess && reset) {
    const unsigned long long zero = 0;
    e = cudaMemcpyToSymbol(g_async_timeouts, &zero, sizeof(zero));
  }
  return e;
}

// ---------------------------------------------------------------------------
// Layer consumer (stands in for the layer's computation): for each 8-element
// vector, c = sum of bits[j] * (1 + (j mod 65536)); its term is c after
// rounds - 1 dependent multiply-adds t = t*K + c, i.e. c * (1 + K + ... +
// K^(rounds-1)) mod 2^64.  The on-chip work grows with rounds while the
// memory traffic stays one read of the layer.
// ---------------------------------------------------------------------------
constexpr unsigned long long kConsumeK = 6364136223846793005ull;  // Knuth's MMIX LCG multiplier

__device__ __forceinline__ unsigned long long consume_term(unsigned long long c, int rounds) {
  unsigned long long t = c;
  for (int r = 1; r < rounds; ++r) t = t * kConsumeK + c;
  return t;
}

// c of the 8-element vector q.  (8q mod 65536) + e never wraps for e < 8, so
// with b = 1 + (8q mod 65536), c = b * sum_e bits_e + sum_e e * bits_e: two
// 32-bit sums (below 2^20 and 2^21) and one widening multiply.
__device__ __forceinline__ unsigned long long vec_weighted(uint4 x, int64_t q) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t s0 = 0, s1 = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t lo = w[e] & 0xFFFFu, hi = w[e] >> 16;
    s0 += lo + hi;
    s1 += (uint32_t)(2 * e) * lo + (uint32_t)(2 * e + 1) * hi;
  }
  const uint32_t b = 1u + (((uint32_t)q & 0x1FFFu) << 3);
  return (unsigned long long)b * s0 + s1;
}

// Vectors each thread loads before it computes: the consumer reads the layer
// once, so bytes in flight, not arithmetic, decide its speed at one round.
constexpr int kConsumeUnroll = 4;

__global__ void __launch_bounds__(kThreads)
    checksum_kernel(const uint16_t* __restrict__ bits, int64_t n, int rounds,
                    unsigned long long* __restrict__ out) {
  unsigned long long s = 0;
  const int64_t nv = n >> 3, stride = gstride();
  for (int64_t q0 = gtid(); q0 < nv; q0 += kConsumeUnroll * stride) {
    uint4 x[kConsumeUnroll];
    bool ok[kConsumeUnroll];
#pragma unroll
    for (int u = 0; u < kConsumeUnroll; ++u) {
      const int64_t q = q0 + u * stride;
      ok[u] = q < nv && in_extent(q * 8, q * 8 + 8, 0, n, ZERO_SITE_CHECKSUM);
      if (ok[u]) x[u] = ld_once(bits + q * 8);
    }
#pragma unroll
    for (int u = 0; u < kConsumeUnroll; ++u)
      if (ok[u]) s += consume_term(vec_weighted(x[u], q0 + u * stride), rounds);
  }
  for (int64_t j = (nv << 3) + gtid(); j < n; j += stride)
    if (in_extent(j, j + 1, 0, n, ZERO_SITE_CHECKSUM))
      s += consume_term((unsigned long long)bits[j] * (1ull + (unsigned long long)(j & 0xFFFF)),
                        rounds);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0 && s != 0) atomicAdd(out, s);
}

cudaError_t launch_checksum(const void* layer, int64_t n, int rounds, uint64_t* out,
                            cudaStream_t st, bool clear) {
  if (clear) {
    const cudaError_t e = cudaMemsetAsync(out, 0, sizeof(uint64_t), st);
    if (e != cudaSuccess) return e;
  }
  if (n <= 0) return cudaSuccess;
  const int64_t items = (n / 8) / kConsumeUnroll + 1;
  checksum_kernel<<<(unsigned)wave_grid(checksum_kernel, items, ZERO_OCC_CONSUMER), kThreads, 0,
                    st>>>(static_cast<const uint16_t*>(layer), n, rounds,
                          reinterpret_cast<unsigned long long*>(out));
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Copy (bytes a multiple of 16).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
    copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int64_t nv) {
  for (int64_t q = gtid(); q < nv; q += gstride())
    if (in_extent(q, q + 1, 0, nv, ZERO_SITE_COPY)) st_stream(dst + q, ld_once(src + q));
}

cudaError_t launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t st) {
  const int64_t nv = bytes / 16;
  if (nv <= 0) return cudaSuccess;
  copy_kernel<<<(unsigned)wave_grid(copy_kernel, nv, ZERO_OCC_STREAM), kThreads, 0, st>>>(
      static_cast<uint4*>(dst), static_cast<const uint4*>(src), nv);
  return cudaGetLastError();
}

}  // namespace zk

namespace zk {

// ---------------------------------------------------------------------------
// Bounded wait on a flag (failure detection): poll *flag until it equals
// `expected` or max_polls polls about 1 us apart have passed; never hangs.
// ---------------------------------------------------------------------------
__global__ void wait_flag_kernel(const volatile uint32_t* flag, uint32_t expected,
                                 int64_t max_polls, int32_t* status) {
  int32_t st = ZERO_ETIMEOUT;
  for (int64_t i = 0; i < max_polls; ++i) {
    if (*flag == expected) {
      st = ZERO_OK;
      break;
    }
    __nanosleep(1000);
  }
  *status = st;
}

cudaError_t launch_wait_flag(const uint32_t* flag, uint32_t expected, int64_t max_polls,
                             int32_t* status, cudaStream_t st) {
  wait_flag_kernel<<<1, 1, 0, st>>>(flag, expected, max_polls, status);
  return cudaGetLastError();
}

}  // namespace zk

namespace zk {

// ---------------------------------------------------------------------------
// Device-resident Adam step: st <- init (when given), then one step on.
// The same fp64 products and early stop as the host's computation.
// ---------------------------------------------------------------------------
__global__ void adam_state_kernel(AdamState* st, AdamState init, int has_init, double b1,
                                  double b2) {
  AdamState s = has_init ? init : *st;
  if (!has_init) {
    const double tiny = 8.673617379884035e-19;  // 2^-60
    if (s.pow1 >= tiny) s.pow1 = __dmul_rn(s.pow1, b1);
    if (s.pow2 >= tiny) s.pow2 = __dmul_rn(s.pow2, b2);
    s.step += 1;
    s.bc1 = __double2float_rn(__dsub_rn(1.0, s.pow1));
    s.bc2 = __double2float_rn(__dsub_rn(1.0, s.pow2));
  }
  *st = s;
}

cudaError_t launch_adam_state(AdamState* st, const AdamState* init, double b1, double b2,
                              cudaStream_t s) {
  AdamState z{};
  adam_state_kernel<<<1, 1, 0, s>>>(st, init ? *init : z, init ? 1 : 0, b1, b2);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Checked build: this unit's out-of-extent record, and a probe kernel that
// records one (index 1 outside [0, 1)) without making any memory access.
// ---------------------------------------------------------------------------
cudaError_t bounds_kernels(BoundsRec* out, bool reset) { return bounds_record(out, reset); }

#ifdef ZERO_CHECKED
__global__ void bounds_probe_kernel() { (void)in_extent(1, 2, 0, 1, ZERO_SITE_PROBE); }
#endif

cudaError_t launch_bounds_probe(cudaStream_t st) {
#ifdef ZERO_CHECKED
  bounds_probe_kernel<<<1, 1, 0, st>>>();
  return cudaGetLastError();
#else
  (void)st;
  return cudaSuccess;
#endif
}

}  // namespace zk
