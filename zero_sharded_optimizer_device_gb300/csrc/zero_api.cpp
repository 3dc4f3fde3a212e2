// C-ABI layer of libzero: argument checks, error codes, and the hand-off of
// plan geometry and Adam constants to the kernels.  No call here allocates
// device memory.
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "zero_internal.h"

namespace {

// An NVTX range around each device entry point, so that timeline profilers
// show which C-ABI call launched which kernel (a no-op without a tool).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

thread_local int g_last_cuda = 0;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return ZERO_OK;
  g_last_cuda = (int)e;
  return ZERO_ECUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool dtype_ok(int d) { return d == ZERO_F32 || d == ZERO_BF16; }

int check_group(const zero_plan_t* p, int32_t group) {
  if (!p) return ZERO_EINVAL;
  if (group < 0 || group >= (int32_t)p->groups.size()) return ZERO_ERANGE;
  return ZERO_OK;
}

int check_window(const zero_plan_t* p, int32_t group, int64_t begin, int64_t end) {
  const zero_group_info_t& g = p->groups[group];
  if (begin < 0 || end < begin || end > g.psi_pad) return ZERO_ERANGE;
  return ZERO_OK;
}

// A host array of N device pointers, each non-null and 16-byte aligned.
template <typename P>
int check_rank_ptrs(const zero_plan_t* p, P const* ptrs) {
  if (!ptrs) return ZERO_EINVAL;
  for (int r = 0; r < p->n_ranks; ++r) {
    if (!ptrs[r]) return ZERO_EINVAL;
    if (!aligned16(ptrs[r])) return ZERO_EALIGN;
  }
  return ZERO_OK;
}

int check_buf(const void* q) {
  if (!q) return ZERO_EINVAL;
  return aligned16(q) ? ZERO_OK : ZERO_EALIGN;
}

int check_opt_buf(const void* q) { return (!q || aligned16(q)) ? ZERO_OK : ZERO_EALIGN; }

// fp32 scalars (norm, clip coefficient) are read and written singly.
int check_opt_f32(const void* q) { return (!q || ((uintptr_t)q & 3u) == 0) ? ZERO_OK : ZERO_EALIGN; }

// fp64 partial sums are read and written one value at a time.
int check_opt_f64(const void* q) { return (!q || ((uintptr_t)q & 7u) == 0) ? ZERO_OK : ZERO_EALIGN; }

zk::GroupK group_k(const zero_plan_t* p, int32_t group) {
  const zero_group_info_t& g = p->groups[group];
  zk::GroupK k;
  k.S = g.shard;
  k.flat_off = g.flat_off;
  k.rank_off = g.rank_off;
  k.invS256 = g.shard > 0 ? 256.0f / (float)g.shard : 0.0f;
  k.n = p->n_ranks;
  return k;
}

// fp32 gradients with every buffer 32-byte aligned take the fused kernel's
// one-load-per-thread variant.
int fused_gdtype(const zero_plan_t* p, int gdtype, const void* const* grads) {
  if (gdtype != ZERO_F32) return gdtype;
  for (int r = 0; r < p->n_ranks; ++r)
    if ((uintptr_t)grads[r] & 31u) return gdtype;
  return zk::kF32Aligned32;
}

zk::RankPtrs rank_ptrs(const zero_plan_t* p, const void* const* ptrs) {
  zk::RankPtrs r{};
  for (int i = 0; i < p->n_ranks; ++i) r.p[i] = ptrs[i];
  return r;
}

// beta^t for both moments: the fp32 beta raised to t by t successive fp64
// multiplications, each factor stopping once below 2^-60 (where 1 - beta^t
// is exactly 1 in fp64).  The bias corrections are 1 - beta^t in fp64,
// rounded once to fp32; (1 - beta) and lr*wd are fp32 operations.
//
// Training calls this with step numbers that grow by one, and the product
// takes up to ~41 500 factors (0.999^t reaches 2^-60 only then), so each host
// thread remembers where its last call ended for that pair of betas and
// continues the same product from there when the step has not gone back: the
// same multiplications in the same order, hence the same result.
struct BetaPows {
  float beta1 = -1.0f, beta2 = -1.0f;
  int64_t step = 0;
  double a = 1.0, b = 1.0;
};
thread_local BetaPows g_pows;

void beta_pows(float beta1, float beta2, int64_t step, double* p1, double* p2) {
  double a = 1.0, b = 1.0;
  int64_t t = 0;
  BetaPows& c = g_pows;
  if (c.beta1 == beta1 && c.beta2 == beta2 && c.step <= step) {
    t = c.step;
    a = c.a;
    b = c.b;
  }
  const double b1 = (double)beta1, b2 = (double)beta2;
  const double tiny = 8.673617379884035e-19;  // 2^-60
  for (; t < step && (a >= tiny || b >= tiny); ++t) {
    if (a >= tiny) a *= b1;
    if (b >= tiny) b *= b2;
  }
  c.beta1 = beta1;
  c.beta2 = beta2;
  c.step = step;
  c.a = a;
  c.b = b;
  *p1 = a;
  *p2 = b;
}

int check_hp(const zero_adam_t* hp) {
  if (!hp) return ZERO_EINVAL;
  if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
    return ZERO_EINVAL;
  if (!isfinite(hp->lr) || !isfinite(hp->eps) || !isfinite(hp->weight_decay) ||
      !isfinite(hp->grad_scale))
    return ZERO_EINVAL;
  if (hp->d_state && ((uintptr_t)hp->d_state & 7u) != 0) return ZERO_EALIGN;
  return ZERO_OK;
}

int adam_k(const zero_adam_t* hp, zk::AdamK* out) {
  int s = check_hp(hp);
  if (s != ZERO_OK) return s;
  if (!hp->d_state && hp->step < 1) return ZERO_EINVAL;
  double p1 = 1.0, p2 = 1.0;
  if (!hp->d_state) beta_pows(hp->beta1, hp->beta2, hp->step, &p1, &p2);
  zk::AdamK k;
  k.lr = hp->lr;
  k.b1 = hp->beta1;
  k.b2 = hp->beta2;
  k.omb1 = 1.0f - hp->beta1;
  k.omb2 = 1.0f - hp->beta2;
  k.eps = hp->eps;
  k.bc1 = (float)(1.0 - p1);
  k.bc2 = (float)(1.0 - p2);
  k.lrwd = hp->lr * hp->weight_decay;
  k.has_wd = hp->weight_decay != 0.0f;
  k.scale = hp->grad_scale;
  k.bcp = hp->d_state ? reinterpret_cast<const float*>(static_cast<const char*>(hp->d_state) +
                                                       offsetof(zk::AdamState, bc1))
                      : nullptr;
  *out = k;
  return ZERO_OK;
}

#define ZERO_TRY(x)              \
  do {                           \
    int _s = (x);                \
    if (_s != ZERO_OK) return _s; \
  } while (0)

}  // namespace

extern "C" int zero_version(void) { return 10000; }

extern "C" const char* zero_strerror(int status) {
  switch (status) {
    case ZERO_OK: return "ok";
    case ZERO_EINVAL: return "invalid argument";
    case ZERO_EALIGN: return "device pointer not 16-byte aligned";
    case ZERO_ERANGE: return "group, rank, tensor or window outside the plan";
    case ZERO_EDTYPE: return "unsupported dtype";
    case ZERO_ENOMEM: return "host allocation failed";
    case ZERO_ECUDA: return "CUDA runtime error";
    case ZERO_ETIMEOUT: return "bounded device wait timed out";
    default: return "unknown status";
  }
}

extern "C" int zero_last_cuda_error(void) { return g_last_cuda; }

void zk::record_cuda_error(int err) { g_last_cuda = err; }

extern "C" int zero_rs_partials(const zero_plan_t* plan, zero_dtype_t gdtype, int64_t n_elements,
                                int64_t* n_partials) {
  if (!plan || !n_partials || n_elements < 0) return ZERO_EINVAL;
  if (!dtype_ok(gdtype)) return ZERO_EDTYPE;
  *n_partials = zk::rs_partials_for(plan->n_ranks, gdtype, n_elements);
  return ZERO_OK;
}

int zk::reduce_scatter_entry(const zero_plan_t* plan, int32_t group, const void* const* grads,
                             zero_dtype_t gdtype, float* reduced, int64_t begin, int64_t end,
                             float grad_scale, double* sumsq_partials, int64_t grid,
                             cudaStream_t stream) {
  ZERO_TRY(check_group(plan, group));
  if (!dtype_ok(gdtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_window(plan, group, begin, end));
  ZERO_TRY(check_rank_ptrs(plan, grads));
  if (!reduced && !sumsq_partials) return ZERO_EINVAL;  // nothing to produce
  ZERO_TRY(check_opt_buf(reduced));
  ZERO_TRY(check_opt_f64(sumsq_partials));
  return cuda_status(zk::launch_reduce_scatter(
      rank_ptrs(plan, grads), gdtype, group_k(plan, group), reduced, begin, end, grad_scale,
      sumsq_partials, reduced ? zk::RS_STORE : zk::RS_NORM_ONLY, stream, grid));
}

extern "C" int zero_reduce_scatter(const zero_plan_t* plan, int32_t group,
                                   const void* const* grads, zero_dtype_t gdtype, float* reduced,
                                   int64_t begin, int64_t end, float grad_scale,
                                   double* sumsq_partials, zero_stream_t stream) {
  NvtxRange nvtx("zero_reduce_scatter");
  return zk::reduce_scatter_entry(plan, group, grads, gdtype, reduced, begin, end, grad_scale,
                                  sumsq_partials, 0, (cudaStream_t)stream);
}

extern "C" int zero_reduce_scatter_acc(const zero_plan_t* plan, int32_t group,
                                       const void* const* grads, zero_dtype_t gdtype,
                                       float* reduced, int64_t begin, int64_t end,
                                       float grad_scale, double* sumsq_partials,
                                       zero_stream_t stream) {
  NvtxRange nvtx("zero_reduce_scatter_acc");
  ZERO_TRY(check_group(plan, group));
  if (!dtype_ok(gdtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_window(plan, group, begin, end));
  ZERO_TRY(check_rank_ptrs(plan, grads));
  ZERO_TRY(check_buf(reduced));
  ZERO_TRY(check_opt_f64(sumsq_partials));
  return cuda_status(zk::launch_reduce_scatter(
      rank_ptrs(plan, grads), gdtype, group_k(plan, group), reduced, begin, end, grad_scale,
      sumsq_partials, zk::RS_ACCUMULATE, (cudaStream_t)stream));
}

extern "C" int zero_grad_norm(const double* partials, int64_t n, float max_norm, float* d_norm,
                              float* d_coef, zero_stream_t stream) {
  NvtxRange nvtx("zero_grad_norm");
  if (n < 0 || (n > 0 && !partials) || !isfinite(max_norm) || max_norm <= 0.0f)
    return ZERO_EINVAL;
  ZERO_TRY(check_opt_f64(partials));
  ZERO_TRY(check_opt_f32(d_norm));
  ZERO_TRY(check_opt_f32(d_coef));
  return cuda_status(zk::launch_norm(partials, n, max_norm, d_norm, d_coef, (cudaStream_t)stream));
}

extern "C" int zero_adam_shard(const zero_plan_t* plan, int32_t group, float* master, float* m,
                               float* v, const float* reduced, const zero_adam_t* hp,
                               const float* d_coef, int64_t begin, int64_t end, void* out,
                               zero_dtype_t out_dtype, zero_stream_t stream) {
  NvtxRange nvtx("zero_adam_shard");
  ZERO_TRY(check_group(plan, group));
  ZERO_TRY(check_window(plan, group, begin, end));
  ZERO_TRY(check_buf(master));
  ZERO_TRY(check_buf(m));
  ZERO_TRY(check_buf(v));
  ZERO_TRY(check_buf(reduced));
  ZERO_TRY(check_opt_buf(out));
  if (out && !dtype_ok(out_dtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_opt_f32(d_coef));
  zk::AdamK k;
  ZERO_TRY(adam_k(hp, &k));
  const int mode = !out ? zk::OUT_NONE
                        : (out_dtype == ZERO_BF16 ? zk::OUT_FULL_BF16 : zk::OUT_FULL_F32);
  return cuda_status(zk::launch_adam(group_k(plan, group), begin, end, master, m, v, reduced, k,
                                     d_coef, mode, out, (cudaStream_t)stream));
}

// The clipped step's reduce-scatter windows: every window but the last has
// `bucket` elements, so two grids describe them all.  The grids are fixed
// once per call and each window is launched with its stored grid, so the
// partial count written equals the count checked even if another host thread
// changes the occupancy setting meanwhile.
struct ClippedGrids {
  int64_t windows = 0, full = 0, last = 0;
  int64_t total() const { return windows > 0 ? (windows - 1) * full + last : 0; }
};
static ClippedGrids clipped_grids(const zero_plan_t* plan, int32_t group, int gdtype,
                                  int64_t bucket) {
  const int64_t P = plan->groups[group].psi_pad;
  ClippedGrids c;
  if (P <= 0) return c;
  c.windows = (P + bucket - 1) / bucket;
  c.full = zk::rs_partials_for(plan->n_ranks, gdtype, bucket < P ? bucket : P);
  c.last = zk::rs_partials_for(plan->n_ranks, gdtype, P - (c.windows - 1) * bucket);
  return c;
}
static int64_t clipped_partials(const zero_plan_t* plan, int32_t group, int gdtype,
                                int64_t bucket) {
  return clipped_grids(plan, group, gdtype, bucket).total();
}

extern "C" int zero_step_clipped_partials(const zero_plan_t* plan, int32_t group,
                                          zero_dtype_t gdtype, int64_t bucket,
                                          int64_t* n_partials) {
  ZERO_TRY(check_group(plan, group));
  if (!dtype_ok(gdtype)) return ZERO_EDTYPE;
  if (bucket < 1 || !n_partials) return ZERO_EINVAL;
  *n_partials = clipped_partials(plan, group, gdtype, bucket);
  return ZERO_OK;
}

extern "C" int zero_step_clipped(const zero_plan_t* plan, int32_t group, const void* const* grads,
                                 zero_dtype_t gdtype, float* reduced, float* master, float* m,
                                 float* v, const zero_adam_t* hp, float max_norm, int64_t bucket,
                                 int64_t chunk, double* partials, int64_t n_partials,
                                 float* d_norm, float* d_coef, void* full_out,
                                 zero_dtype_t out_dtype, zero_stream_t stream) {
  NvtxRange nvtx("zero_step_clipped");
  ZERO_TRY(check_group(plan, group));
  if (!dtype_ok(gdtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_rank_ptrs(plan, grads));
  ZERO_TRY(check_buf(reduced));
  ZERO_TRY(check_buf(master));
  ZERO_TRY(check_buf(m));
  ZERO_TRY(check_buf(v));
  ZERO_TRY(check_opt_buf(full_out));
  if (full_out && !dtype_ok(out_dtype)) return ZERO_EDTYPE;
  if (!partials || !d_coef || bucket < 1 || chunk < 1) return ZERO_EINVAL;
  if (!isfinite(max_norm) || max_norm <= 0.0f) return ZERO_EINVAL;
  ZERO_TRY(check_opt_f64(partials));
  ZERO_TRY(check_opt_f32(d_norm));
  ZERO_TRY(check_opt_f32(d_coef));
  zk::AdamK k;
  ZERO_TRY(adam_k(hp, &k));
  const ClippedGrids grids = clipped_grids(plan, group, gdtype, bucket);
  if (n_partials < grids.total()) return ZERO_ERANGE;
  const cudaStream_t st = (cudaStream_t)stream;
  const zk::RankPtrs src = rank_ptrs(plan, grads);
  const zk::GroupK g = group_k(plan, group);
  const int64_t P = plan->groups[group].psi_pad;
  // 1. reduce-scatter window by window, each writing its slice of partials
  //    with the grid fixed above
  cudaError_t e = cudaSuccess;
  int64_t off = 0;
  for (int64_t a = 0; a < P && e == cudaSuccess; a += bucket) {
    const int64_t b = P - a < bucket ? P : a + bucket;
    const int64_t grid = b == P ? grids.last : grids.full;
    e = zk::launch_reduce_scatter(src, gdtype, g, reduced, a, b, hp->grad_scale, partials + off,
                                  zk::RS_STORE, st, grid);
    off += grid;
  }
  // 2. global norm and clip coefficient on the device
  if (e == cudaSuccess) e = zk::launch_norm(partials, off, max_norm, d_norm, d_coef, st);
  // 3. Adam chunk by chunk with the coefficient, writing the gathered output
  const int mode = !full_out ? zk::OUT_NONE
                             : (out_dtype == ZERO_BF16 ? zk::OUT_FULL_BF16 : zk::OUT_FULL_F32);
  for (int64_t a = 0; a < P && e == cudaSuccess; a += chunk) {
    const int64_t b = P - a < chunk ? P : a + chunk;
    e = zk::launch_adam(g, a, b, master, m, v, reduced, k, d_coef, mode, full_out, st);
  }
  return cuda_status(e);
}

extern "C" int zero_all_gather(const zero_plan_t* plan, int32_t group, const float* master,
                               void* full_out, zero_dtype_t out_dtype, zero_stream_t stream) {
  NvtxRange nvtx("zero_all_gather");
  if (!plan) return ZERO_EINVAL;
  if (group != -1) ZERO_TRY(check_group(plan, group));
  if (!dtype_ok(out_dtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_buf(master));
  ZERO_TRY(check_buf(full_out));
  int64_t a = 0, b = plan->psi_pad;
  if (group >= 0) {
    a = plan->groups[group].flat_off;
    b = a + plan->groups[group].psi_pad;
  }
  return cuda_status(zk::launch_cast(master, a, b, out_dtype, full_out, (cudaStream_t)stream));
}

static int fused_step(const zero_plan_t* plan, int32_t group, const void* const* grads,
                      zero_dtype_t gdtype, const float* prev, float* master, float* m, float* v,
                      const zero_adam_t* hp, const float* d_coef, void* full_out,
                      zero_dtype_t out_dtype, zero_stream_t stream) {
  ZERO_TRY(check_group(plan, group));
  if (!dtype_ok(gdtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_rank_ptrs(plan, grads));
  ZERO_TRY(check_buf(master));
  ZERO_TRY(check_buf(m));
  ZERO_TRY(check_buf(v));
  ZERO_TRY(check_opt_buf(full_out));
  if (full_out && !dtype_ok(out_dtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_opt_f32(d_coef));
  zk::AdamK k;
  ZERO_TRY(adam_k(hp, &k));
  const int mode = !full_out ? zk::OUT_NONE
                             : (out_dtype == ZERO_BF16 ? zk::OUT_FULL_BF16 : zk::OUT_FULL_F32);
  zk::OutPtrs none{};
  return cuda_status(zk::launch_fused(rank_ptrs(plan, grads), fused_gdtype(plan, gdtype, grads),
                                      group_k(plan, group), 0, plan->groups[group].psi_pad,
                                      master, m, v, k, d_coef, prev, mode, full_out, none,
                                      (cudaStream_t)stream));
}

extern "C" int zero_step(const zero_plan_t* plan, int32_t group, const void* const* grads,
                         zero_dtype_t gdtype, float* master, float* m, float* v,
                         const zero_adam_t* hp, const float* d_coef, void* full_out,
                         zero_dtype_t out_dtype, zero_stream_t stream) {
  NvtxRange nvtx("zero_step");
  return fused_step(plan, group, grads, gdtype, nullptr, master, m, v, hp, d_coef, full_out,
                    out_dtype, stream);
}

extern "C" int zero_step_acc(const zero_plan_t* plan, int32_t group, const void* const* grads,
                             zero_dtype_t gdtype, const float* accumulated, float* master,
                             float* m, float* v, const zero_adam_t* hp, const float* d_coef,
                             void* full_out, zero_dtype_t out_dtype, zero_stream_t stream) {
  NvtxRange nvtx("zero_step_acc");
  ZERO_TRY(check_buf(accumulated));
  // the kernel reads `accumulated` through a restrict pointer while it writes
  // the state and the output: the same buffer in two roles is refused
  const void* acc = accumulated;
  if (acc == master || acc == m || acc == v || acc == full_out) return ZERO_EINVAL;
  return fused_step(plan, group, grads, gdtype, accumulated, master, m, v, hp, d_coef, full_out,
                    out_dtype, stream);
}

// The stage-3 fused step: owner k writes its updated bf16 parameters into its
// own shard buffer; prev (may be NULL) is the accumulated reduced gradient of
// earlier micro-batches.
static int group_step(const zero_plan_t* plan, int32_t group, const void* const* grads,
                      zero_dtype_t gdtype, const float* prev, float* master, float* m, float* v,
                      const zero_adam_t* hp, const float* d_coef, void* const* shards,
                      zero_stream_t stream) {
  ZERO_TRY(check_group(plan, group));
  if (!dtype_ok(gdtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_rank_ptrs(plan, grads));
  ZERO_TRY(check_rank_ptrs(plan, shards));
  ZERO_TRY(check_buf(master));
  ZERO_TRY(check_buf(m));
  ZERO_TRY(check_buf(v));
  ZERO_TRY(check_opt_f32(d_coef));
  zk::AdamK k;
  ZERO_TRY(adam_k(hp, &k));
  zk::OutPtrs out{};
  for (int r = 0; r < plan->n_ranks; ++r) out.p[r] = shards[r];
  return cuda_status(zk::launch_fused(rank_ptrs(plan, grads), fused_gdtype(plan, gdtype, grads),
                                      group_k(plan, group), 0, plan->groups[group].psi_pad,
                                      master, m, v, k, d_coef, prev, zk::OUT_SHARDS_BF16,
                                      nullptr, out, (cudaStream_t)stream));
}

extern "C" int zero_step_group(const zero_plan_t* plan, int32_t group, const void* const* grads,
                               zero_dtype_t gdtype, float* master, float* m, float* v,
                               const zero_adam_t* hp, const float* d_coef, void* const* shards,
                               zero_stream_t stream) {
  NvtxRange nvtx("zero_step_group");
  return group_step(plan, group, grads, gdtype, nullptr, master, m, v, hp, d_coef, shards,
                    stream);
}

extern "C" int zero_step_group_acc(const zero_plan_t* plan, int32_t group,
                                   const void* const* grads, zero_dtype_t gdtype,
                                   const float* accumulated, float* master, float* m, float* v,
                                   const zero_adam_t* hp, const float* d_coef,
                                   void* const* shards, zero_stream_t stream) {
  NvtxRange nvtx("zero_step_group_acc");
  ZERO_TRY(check_buf(accumulated));
  // read through a restrict pointer while the state is written: one buffer in
  // two roles is refused
  const void* acc = accumulated;
  if (acc == master || acc == m || acc == v) return ZERO_EINVAL;
  return group_step(plan, group, grads, gdtype, accumulated, master, m, v, hp, d_coef, shards,
                    stream);
}

extern "C" int zero_gather_layer(const zero_plan_t* plan, int32_t group, const void* const* shards,
                                 zero_dtype_t dtype, void* layer_out, zero_stream_t stream) {
  NvtxRange nvtx("zero_gather_layer");
  ZERO_TRY(check_group(plan, group));
  if (!dtype_ok(dtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_rank_ptrs(plan, shards));
  ZERO_TRY(check_buf(layer_out));
  return cuda_status(zk::launch_gather(rank_ptrs(plan, shards), dtype == ZERO_BF16 ? 2 : 4,
                                       group_k(plan, group), plan->groups[group].psi_pad,
                                       layer_out, ZERO_OCC_GATHER, (cudaStream_t)stream));
}

extern "C" int zero_broadcast_layer(const zero_plan_t* plan, int32_t group,
                                    const void* const* shards, zero_dtype_t dtype,
                                    void* layer_out, zero_stream_t stream) {
  NvtxRange nvtx("zero_broadcast_layer");
  ZERO_TRY(check_group(plan, group));
  if (!dtype_ok(dtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_rank_ptrs(plan, shards));
  ZERO_TRY(check_buf(layer_out));
  return cuda_status(zk::launch_broadcast(rank_ptrs(plan, shards), dtype == ZERO_BF16 ? 2 : 4,
                                          group_k(plan, group), layer_out, ZERO_OCC_GATHER,
                                          (cudaStream_t)stream));
}

extern "C" int zero_gather_groups(const zero_plan_t* plan, const int32_t* groups, int32_t k,
                                  const void* const* shards, zero_dtype_t dtype,
                                  void* const* layer_outs, zero_stream_t stream) {
  NvtxRange nvtx("zero_gather_groups");
  if (!plan || !groups || !layer_outs || k < 1 || k > ZERO_MAX_COALESCE) return ZERO_EINVAL;
  if (!dtype_ok(dtype)) return ZERO_EDTYPE;
  ZERO_TRY(check_rank_ptrs(plan, shards));
  for (int32_t i = 0; i < k; ++i) {
    ZERO_TRY(check_group(plan, groups[i]));
    ZERO_TRY(check_buf(layer_outs[i]));
  }
  const int es = dtype == ZERO_BF16 ? 2 : 4;
  const zk::RankPtrs src = rank_ptrs(plan, shards);
  zk::BulkGroups bg{};
  bg.es = es;
  bg.n = plan->n_ranks;
  cudaError_t e = cudaSuccess;
  for (int32_t i = 0; i < k && e == cudaSuccess; ++i) {
    const zero_group_info_t& g = plan->groups[groups[i]];
    if (zk::bulk_eligible(g.shard, g.rank_off, es))
      zk::bulk_add(bg, g.shard, g.rank_off, layer_outs[i]);
    else
      e = zk::launch_gather(src, es, group_k(plan, groups[i]), g.psi_pad, layer_outs[i],
                            ZERO_OCC_GATHER, (cudaStream_t)stream);
  }
  if (e == cudaSuccess && bg.ng > 0)
    e = zk::launch_gather_bulk(src, bg, ZERO_OCC_GATHER, (cudaStream_t)stream);
  return cuda_status(e);
}

extern "C" int zero_layer_checksum(const void* layer, int64_t n, int32_t rounds,
                                   uint64_t* d_out, zero_stream_t stream) {
  NvtxRange nvtx("zero_layer_checksum");
  if (n < 0 || !d_out || (n > 0 && !layer)) return ZERO_EINVAL;
  if (rounds < 1 || rounds > ZERO_MAX_CONSUMER_ROUNDS) return ZERO_EINVAL;
  ZERO_TRY(check_opt_buf(layer));
  if (((uintptr_t)d_out & 7u) != 0) return ZERO_EALIGN;
  return cuda_status(zk::launch_checksum(layer, n, rounds, d_out, (cudaStream_t)stream));
}

extern "C" int zero_copy(void* dst, const void* src, int64_t bytes, zero_stream_t stream) {
  NvtxRange nvtx("zero_copy");
  if (bytes < 0 || (bytes % 16) != 0) return ZERO_EINVAL;
  if (bytes == 0) return ZERO_OK;
  ZERO_TRY(check_buf(dst));
  ZERO_TRY(check_buf(src));
  return cuda_status(zk::launch_copy(dst, src, bytes, (cudaStream_t)stream));
}

extern "C" int zero_wait_flag(const uint32_t* flag, uint32_t expected, int64_t max_polls,
                              int32_t* d_status, zero_stream_t stream) {
  NvtxRange nvtx("zero_wait_flag");
  if (!flag || !d_status || max_polls < 0 || max_polls > ZERO_MAX_POLLS) return ZERO_EINVAL;
  if (((uintptr_t)flag & 3u) != 0 || ((uintptr_t)d_status & 3u) != 0) return ZERO_EALIGN;
  return cuda_status(zk::launch_wait_flag(flag, expected, max_polls, d_status,
                                          (cudaStream_t)stream));
}

extern "C" int zero_adam_bias_corrections(const zero_adam_t* hp, float* bc1, float* bc2) {
  if (!bc1 || !bc2) return ZERO_EINVAL;
  ZERO_TRY(check_hp(hp));
  if (hp->step < 1) return ZERO_EINVAL;
  double p1 = 1.0, p2 = 1.0;
  beta_pows(hp->beta1, hp->beta2, hp->step, &p1, &p2);
  *bc1 = (float)(1.0 - p1);
  *bc2 = (float)(1.0 - p2);
  return ZERO_OK;
}

extern "C" int zero_adam_state_init(const zero_adam_t* hp, void* d_state, zero_stream_t stream) {
  NvtxRange nvtx("zero_adam_state_init");
  int s = check_hp(hp);
  if (s != ZERO_OK) return s;
  if (!d_state || hp->step < 1) return ZERO_EINVAL;
  if (((uintptr_t)d_state & 7u) != 0) return ZERO_EALIGN;
  zk::AdamState init{};
  init.step = hp->step - 1;
  beta_pows(hp->beta1, hp->beta2, init.step, &init.pow1, &init.pow2);
  init.bc1 = (float)(1.0 - init.pow1);
  init.bc2 = (float)(1.0 - init.pow2);
  return cuda_status(zk::launch_adam_state(static_cast<zk::AdamState*>(d_state), &init,
                                           (double)hp->beta1, (double)hp->beta2,
                                           (cudaStream_t)stream));
}

extern "C" int zero_adam_state_advance(const zero_adam_t* hp, void* d_state,
                                       zero_stream_t stream) {
  NvtxRange nvtx("zero_adam_state_advance");
  int s = check_hp(hp);
  if (s != ZERO_OK) return s;
  if (!d_state) return ZERO_EINVAL;
  if (((uintptr_t)d_state & 7u) != 0) return ZERO_EALIGN;
  return cuda_status(zk::launch_adam_state(static_cast<zk::AdamState*>(d_state), nullptr,
                                           (double)hp->beta1, (double)hp->beta2,
                                           (cudaStream_t)stream));
}

extern "C" int zero_bounds_report(zero_bounds_t* out, int32_t reset) {
  if (!out) return ZERO_EINVAL;
  *out = zero_bounds_t{};
#ifdef ZERO_CHECKED
  out->checked = 1;
  zk::BoundsRec rec[2] = {};
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = zk::bounds_rs(&rec[0], reset != 0);
  if (e == cudaSuccess) e = zk::bounds_kernels(&rec[1], reset != 0);
  if (e != cudaSuccess) return cuda_status(e);
  for (const zk::BoundsRec& r : rec) {
    if (r.count && !out->count) {  // the first unit with a record gives the details
      out->site = (int32_t)r.site;
      out->index = r.index;
      out->lo = r.lo;
      out->hi = r.hi;
    }
    out->count += (int64_t)r.count;
  }
#else
  (void)reset;
#endif
  return ZERO_OK;
}

extern "C" int zero_bounds_probe(zero_stream_t stream) {
  return cuda_status(zk::launch_bounds_probe((cudaStream_t)stream));
}

extern "C" int zero_async_status(int64_t* timeouts, int32_t reset) {
  if (!timeouts) return ZERO_EINVAL;
  unsigned long long n = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = zk::async_timeouts(&n, reset != 0);
  if (e != cudaSuccess) return cuda_status(e);
  *timeouts = (int64_t)n;
  return ZERO_OK;
}
