// Stage-3 gather schedule on two streams.
//
// ["ZeRO Optimizer", "Implementation Strategy"]: stage 3 gathers a layer's
// parameters just before they are used and discards them afterwards, in the
// forward and again in the backward pass; "Communication Optimization":
// parameter gathering is hidden behind computation by prefetching the next
// layer.  Here the gather of the next group runs on stream B into the free
// one of two layer buffers while stream A consumes the current one.  The two
// kernels can only run at the same time if their blocks fit on an SM
// together, so the gathers launch with their own occupancy cap
// (ZERO_OCC_PREFETCH, default 2 one-warp bulk-copy CTAs per SM, each with a
// 6-stage ring) beside the consumer's (ZERO_OCC_CONSUMER, default 7
// 256-thread blocks, of which the consumer's register use lets 6 be
// resident).
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <vector>

#include "zero_internal.h"

namespace {

struct Events {
  cudaEvent_t e[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  cudaError_t create() {
    for (auto& x : e) {
      cudaError_t r = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  }
  ~Events() {
    // destroying an event that is still pending is allowed: its resources
    // are released once it completes
    for (auto& x : e)
      if (x) cudaEventDestroy(x);
  }
};

}  // namespace

// Step j of a pass gathers groups groups[first[j]] .. groups[first[j+1]-1]
// into layer buffer j % 2, one after another (each at the running element
// offset), and the consumer then reads the step's elements as one layer.
static int gather_pass(const zero_plan_t* plan, const int32_t* first, const int32_t* groups,
                       int32_t n, const void* const* shards, void* const* layer_bufs,
                       int64_t buf_elems, uint64_t* d_sums, int32_t consumer_rounds,
                       zero_stream_t stream_a, zero_stream_t stream_b, const char* name) {
  if (!plan || n < 0 || (n > 0 && (!first || !groups || !layer_bufs || !d_sums)) || !shards)
    return ZERO_EINVAL;
  if (consumer_rounds < 1 || consumer_rounds > ZERO_MAX_CONSUMER_ROUNDS) return ZERO_EINVAL;
  if (n == 0) return ZERO_OK;
  if (stream_a == stream_b) return ZERO_EINVAL;
  for (int r = 0; r < plan->n_ranks; ++r) {
    if (!shards[r]) return ZERO_EINVAL;
    if ((uintptr_t)shards[r] & 15u) return ZERO_EALIGN;
  }
  for (int b = 0; b < 2; ++b) {
    if (!layer_bufs[b]) return ZERO_EINVAL;
    if ((uintptr_t)layer_bufs[b] & 15u) return ZERO_EALIGN;
  }
  if ((uintptr_t)d_sums & 7u) return ZERO_EALIGN;
  if (first[0] != 0) return ZERO_EINVAL;
  std::vector<int64_t> step_elems(n);
  for (int32_t j = 0; j < n; ++j) {
    const int32_t k = first[j + 1] - first[j];
    if (k < 1 || k > ZERO_MAX_COALESCE) return ZERO_EINVAL;
    int64_t total = 0;
    for (int32_t i = first[j]; i < first[j + 1]; ++i) {
      if (groups[i] < 0 || groups[i] >= (int32_t)plan->groups.size()) return ZERO_ERANGE;
      const int64_t p = plan->groups[groups[i]].psi_pad;
      if (k > 1 && (p * 2) % 16 != 0) return ZERO_EALIGN;  // packed outputs stay 16-byte aligned
      total += p;
    }
    if (total > buf_elems) return ZERO_ERANGE;
    step_elems[j] = total;
  }
  nvtxRangePushA(name);
  cudaStream_t sa = (cudaStream_t)stream_a, sb = (cudaStream_t)stream_b;
  zk::RankPtrs src{};
  for (int r = 0; r < plan->n_ranks; ++r) src.p[r] = shards[r];
  Events ev;  // 0: start; 1, 2: gather j ready (slot j%2); 3, 4: consumer j done
  cudaError_t e = ev.create();
  auto gk = [&](int32_t g) {
    const zero_group_info_t& gi = plan->groups[g];
    zk::GroupK k;
    k.S = gi.shard;
    k.flat_off = gi.flat_off;
    k.rank_off = gi.rank_off;
    k.invS256 = gi.shard > 0 ? 256.0f / (float)gi.shard : 0.0f;
    k.n = plan->n_ranks;
    return k;
  };
  // the step's groups: those the bulk copies can take share one launch
  auto gather_step = [&](int32_t j) -> cudaError_t {
    char* base = static_cast<char*>(layer_bufs[j & 1]);
    zk::BulkGroups bg{};
    bg.es = 2;
    bg.n = plan->n_ranks;
    cudaError_t r = cudaSuccess;
    int64_t off = 0;
    for (int32_t i = first[j]; i < first[j + 1] && r == cudaSuccess; ++i) {
      const zero_group_info_t& g = plan->groups[groups[i]];
      if (zk::bulk_eligible(g.shard, g.rank_off, 2))
        zk::bulk_add(bg, g.shard, g.rank_off, base + off * 2);
      else
        r = zk::launch_gather(src, 2, gk(groups[i]), g.psi_pad, base + off * 2,
                              ZERO_OCC_PREFETCH, sb);
      off += g.psi_pad;
    }
    if (r == cudaSuccess && bg.ng > 0) r = zk::launch_gather_bulk(src, bg, ZERO_OCC_PREFETCH, sb);
    return r;
  };
  // gather step j into buffer j%2 on stream B, once the consumer of j-2 is done
  auto issue = [&](int32_t j) -> cudaError_t {
    cudaError_t r = cudaSuccess;
    if (j >= 2) r = cudaStreamWaitEvent(sb, ev.e[3 + (j & 1)], 0);
    if (r == cudaSuccess) r = gather_step(j);
    if (r == cudaSuccess) r = cudaEventRecord(ev.e[1 + (j & 1)], sb);
    return r;
  };
  // stream B starts after everything already queued on stream A (the step
  // that wrote the shards)
  if (e == cudaSuccess) e = cudaEventRecord(ev.e[0], sa);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sb, ev.e[0], 0);
  if (e == cudaSuccess) e = issue(0);
  // every consumer's sum zeroed at once, off the per-layer path
  if (e == cudaSuccess) e = cudaMemsetAsync(d_sums, 0, sizeof(uint64_t) * (size_t)n, sa);
  for (int32_t j = 0; j < n && e == cudaSuccess; ++j) {
    if (j + 1 < n) e = issue(j + 1);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sa, ev.e[1 + (j & 1)], 0);
    if (e == cudaSuccess)
      e = zk::launch_checksum(layer_bufs[j & 1], step_elems[j], consumer_rounds, d_sums + j, sa,
                              false);
    if (e == cudaSuccess) e = cudaEventRecord(ev.e[3 + (j & 1)], sa);
  }
  nvtxRangePop();
  if (e != cudaSuccess) {
    zk::record_cuda_error((int)e);
    return ZERO_ECUDA;
  }
  return ZERO_OK;
}

extern "C" int zero_stage3_gather_pass(const zero_plan_t* plan, const int32_t* order, int32_t n,
                                       const void* const* shards, void* const* layer_bufs,
                                       int64_t buf_elems, uint64_t* d_sums,
                                       int32_t consumer_rounds, zero_stream_t stream_a,
                                       zero_stream_t stream_b) {
  if (n < 0) return ZERO_EINVAL;
  try {
    std::vector<int32_t> first(n + 1);
    for (int32_t j = 0; j <= n; ++j) first[j] = j;
    return gather_pass(plan, first.data(), order, n, shards, layer_bufs, buf_elems, d_sums,
                       consumer_rounds, stream_a, stream_b, "zero_stage3_gather_pass");
  } catch (...) {  // host allocation failed: no exception crosses the C ABI
    return ZERO_ENOMEM;
  }
}

extern "C" int zero_stage3_gather_pass_steps(const zero_plan_t* plan, const int32_t* step_first,
                                             const int32_t* step_groups, int32_t n_steps,
                                             const void* const* shards, void* const* layer_bufs,
                                             int64_t buf_elems, uint64_t* d_sums,
                                             int32_t consumer_rounds, zero_stream_t stream_a,
                                             zero_stream_t stream_b) {
  try {
    return gather_pass(plan, step_first, step_groups, n_steps, shards, layer_bufs, buf_elems,
                       d_sums, consumer_rounds, stream_a, stream_b,
                       "zero_stage3_gather_pass_steps");
  } catch (...) {  // host allocation failed: no exception crosses the C ABI
    return ZERO_ENOMEM;
  }
}
