// Private declarations shared by the planner, the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "zero.h"

// Opaque plan (see zero_plan in zero.h).
struct zero_plan {
  int32_t n_ranks = 0;
  int32_t align = 0;
  std::vector<int64_t> numels;
  std::vector<int32_t> tensor_group;
  std::vector<int64_t> tensor_group_off;  // offset of the tensor inside its group
  std::vector<zero_group_info_t> groups;
  int64_t psi = 0, psi_pad = 0, shard_total = 0;
};

namespace zk {

constexpr int kMaxRanks = ZERO_MAX_RANKS;

// N rank pointers, passed to kernels by value (kernel parameter space).
struct RankPtrs {
  const void* p[kMaxRanks];
};
struct OutPtrs {
  void* p[kMaxRanks];
};

// One group's geometry as the kernels see it.
struct GroupK {
  int64_t S;         // shard size
  int64_t flat_off;  // group start in flat arrays
  int64_t rank_off;  // group start in per-rank shard buffers
  float invS256;     // ~256/S, for the owner estimate (refined with integer checks)
  int n;             // ranks
};

// Adam constants prepared on the host (fp32 values; bc from fp64).
struct AdamK {
  float lr, b1, b2, omb1, omb2, eps, bc1, bc2, lrwd, scale;
  int has_wd;
  const float* bcp;  // device {bc1, bc2} replacing bc1/bc2 when not null
};

// Device-resident Adam step state (ZERO_ADAM_STATE_BYTES).
struct AdamState {
  double pow1, pow2;  // beta1^t, beta2^t
  int64_t step;       // t
  float bc1, bc2;     // 1 - beta^t, rounded to fp32
};
static_assert(sizeof(AdamState) == ZERO_ADAM_STATE_BYTES, "device Adam state layout");

cudaError_t launch_adam_state(AdamState* st, const AdamState* init, double b1, double b2,
                              cudaStream_t s);

// launch_fused only: fp32 gradients whose N buffers are all 32-byte aligned.
constexpr int kF32Aligned32 = 2;

enum OutMode : int { OUT_NONE = 0, OUT_FULL_BF16 = 1, OUT_FULL_F32 = 2, OUT_SHARDS_BF16 = 3 };

// What the reduce-scatter does with the ring sum of each element.
enum RsMode : int {
  RS_STORE = 0,       // reduced = sum
  RS_NORM_ONLY = 1,   // only the sum-of-squares partials (reduced untouched)
  RS_ACCUMULATE = 2,  // reduced = reduced + sum (gradient accumulation)
};

// Launchers (zero_kernels.cu, zero_rs.cu).  Each returns the launch status.
// grid > 0 fixes the launch's block count (and so the number of partials it
// writes); 0 takes the default one-wave grid of rs_partials_for().
cudaError_t launch_reduce_scatter(const RankPtrs& src, int gdtype, const GroupK& g,
                                  float* reduced, int64_t begin, int64_t end, float scale,
                                  double* partials, int mode, cudaStream_t st,
                                  int64_t grid = 0);
int64_t rs_partials_for(int n, int gdtype, int64_t n_elements);

// zero_reduce_scatter's checks and launch with the grid fixed by the caller
// (see launch_reduce_scatter).
int reduce_scatter_entry(const zero_plan_t* plan, int32_t group, const void* const* grads,
                         zero_dtype_t gdtype, float* reduced, int64_t begin, int64_t end,
                         float grad_scale, double* sumsq_partials, int64_t grid,
                         cudaStream_t stream);

// prev (may be NULL): the fp32 reduced gradient accumulated over earlier
// micro-batches, added before this one's ring sum (flat indices).
cudaError_t launch_fused(const RankPtrs& src, int gdtype, const GroupK& g, int64_t begin,
                         int64_t end, float* master, float* m, float* v, const AdamK& h,
                         const float* coef, const float* prev, int out_mode, void* out_full,
                         const OutPtrs& shards, cudaStream_t st);

cudaError_t launch_adam(const GroupK& g, int64_t begin, int64_t end, float* master, float* m,
                        float* v, const float* reduced, const AdamK& h, const float* coef,
                        int out_mode, void* out, cudaStream_t st);

// dst[i] = cast(src[i]) for flat indices i in [a, b).
cudaError_t launch_cast(const float* src, int64_t a, int64_t b, int out_dtype, void* dst,
                        cudaStream_t st);

cudaError_t launch_norm(const double* partials, int64_t n, float max_norm, float* d_norm,
                        float* d_coef, cudaStream_t st);

// occ_kind: the occupancy cap to launch with (ZERO_OCC_GATHER standalone,
// ZERO_OCC_PREFETCH inside the two-stream gather pass).
cudaError_t launch_gather(const RankPtrs& shards, int elem_bytes, const GroupK& g,
                          int64_t psi_pad, void* out, int occ_kind, cudaStream_t st);

// Broadcast form of the same gather: N launches, launch k copying owner k's
// shard of the group to out[k*S, (k+1)*S) (one launch per broadcast root).
cudaError_t launch_broadcast(const RankPtrs& shards, int elem_bytes, const GroupK& g, void* out,
                             int occ_kind, cudaStream_t st);

// Groups gathered by one bulk-copy launch (kernel parameter, by value).
struct BulkGroups {
  int ng;  // groups in use
  int es;  // element bytes
  int n;   // ranks
  int64_t first[ZERO_MAX_COALESCE + 1];  // within one owner: first piece of each group
  int64_t S[ZERO_MAX_COALESCE], rank_off[ZERO_MAX_COALESCE];
  char* out[ZERO_MAX_COALESCE];
};
// Shard start and length both multiples of 16 bytes (the bulk copies' rule).
bool bulk_eligible(int64_t S, int64_t rank_off, int elem_bytes);
// Append a group (bg.es and bg.n set, bg.ng < ZERO_MAX_COALESCE).
void bulk_add(BulkGroups& bg, int64_t S, int64_t rank_off, void* out);
cudaError_t launch_gather_bulk(const RankPtrs& shards, const BulkGroups& bg, int occ_kind,
                               cudaStream_t st);

// clear: zero *out first (false: the caller has zeroed it, e.g. once for all
// the consumers of a gather pass).
cudaError_t launch_checksum(const void* layer, int64_t n, int rounds, uint64_t* out,
                            cudaStream_t st, bool clear = true);

cudaError_t launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t st);

cudaError_t launch_wait_flag(const uint32_t* flag, uint32_t expected, int64_t max_polls,
                             int32_t* status, cudaStream_t st);

// Number of SMs of the current device (cached per device).
int sm_count();

// Resident blocks per SM of `kernel` at `threads` per block on the current
// device (the occupancy limit; cached per device and kernel).
int occupancy_of(const void* kernel, int threads);

// Records a CUDA error for zero_last_cuda_error() on this host thread.
void record_cuda_error(int err);

// Checked build: the out-of-extent record of one translation unit's kernels
// (device memory of that unit; see in_extent in zero_device.cuh).
struct BoundsRec {
  unsigned long long count;
  long long site, index, lo, hi;
};
// Copy the record of zero_rs.cu / zero_kernels.cu to *out, then clear it if
// `reset`; the release build writes zeros and makes no CUDA call.
cudaError_t bounds_rs(BoundsRec* out, bool reset);
cudaError_t bounds_kernels(BoundsRec* out, bool reset);
cudaError_t launch_bounds_probe(cudaStream_t st);

// Bounded device waits that gave up (zero_async_status), current device.
cudaError_t async_timeouts(unsigned long long* out, bool reset);

}  // namespace zk
