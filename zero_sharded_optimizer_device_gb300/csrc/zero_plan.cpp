// Host planner: flat contiguous buffer, N equal owner shards, tail padding.
//
// ["[REQUEST] Direct Correspondence between Gradient and Optimizer States to
// Reduce Communication?", "Problem"]: gradients are partitioned so each rank
// owns the gradients that match its optimizer state.  ["Why does not the
// stage 3 implementation use broadcast and reduce-scatter?"]: the
// reduce-scatter runs over one contiguous gradient buffer.  ["ZeRO Optimizer",
// "ZeRO Stages" and "Theoretical Reductions"]: what each stage shards and the
// per-device memory it leaves.
#include <stdlib.h>
#include <string.h>

#include <limits>
#include <new>

#include "zero_internal.h"

namespace {

bool fault_injected(const char* what) {
  // Host-side fault injection for tests: ZERO_FAULT_INJECT=<what> makes the
  // matching host allocation report failure.
  const char* env = getenv("ZERO_FAULT_INJECT");
  return env && strcmp(env, what) == 0;
}

bool add_ok(int64_t a, int64_t b) { return a <= std::numeric_limits<int64_t>::max() - b; }

}  // namespace

extern "C" int zero_plan(const int64_t* numels, int64_t n_tensors, int32_t n_ranks,
                         int32_t align, const int32_t* group_of_tensor, zero_plan_t** out) {
  if (!out || n_tensors < 0 || (n_tensors > 0 && !numels)) return ZERO_EINVAL;
  if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || align < 1) return ZERO_EINVAL;
  if (fault_injected("plan_alloc")) return ZERO_ENOMEM;
  for (int64_t t = 0; t < n_tensors; ++t)
    if (numels[t] < 0) return ZERO_EINVAL;
  int32_t n_groups = 1;
  if (group_of_tensor && n_tensors > 0) {
    if (group_of_tensor[0] != 0) return ZERO_EINVAL;
    for (int64_t t = 1; t < n_tensors; ++t) {
      int32_t d = group_of_tensor[t] - group_of_tensor[t - 1];
      if (d != 0 && d != 1) return ZERO_EINVAL;
    }
    n_groups = group_of_tensor[n_tensors - 1] + 1;
  }
  zero_plan_t* p = nullptr;
  try {
    p = new zero_plan_t();
    p->n_ranks = n_ranks;
    p->align = align;
    p->numels.assign(numels, numels + n_tensors);
    p->tensor_group.resize(n_tensors);
    p->tensor_group_off.resize(n_tensors);
    p->groups.resize(n_groups);
    const int64_t quantum = (int64_t)n_ranks * align;
    int64_t t = 0, flat = 0, rank_off = 0;
    for (int32_t g = 0; g < n_groups; ++g) {
      zero_group_info_t& gi = p->groups[g];
      gi.first_tensor = t;
      int64_t psi = 0;
      while (t < n_tensors && (group_of_tensor ? group_of_tensor[t] : 0) == g) {
        if (!add_ok(psi, numels[t])) { delete p; return ZERO_EINVAL; }
        p->tensor_group[t] = g;
        p->tensor_group_off[t] = psi;
        psi += numels[t];
        ++t;
      }
      gi.n_tensors = t - gi.first_tensor;
      int64_t blocks = psi / quantum + (psi % quantum ? 1 : 0);
      if (blocks > std::numeric_limits<int64_t>::max() / quantum) { delete p; return ZERO_EINVAL; }
      gi.psi = psi;
      gi.psi_pad = blocks * quantum;
      if (gi.psi_pad >= (int64_t(1) << 40)) { delete p; return ZERO_EINVAL; }  // kernel index range
      gi.shard = gi.psi_pad / n_ranks;
      gi.flat_off = flat;
      gi.rank_off = rank_off;
      if (!add_ok(flat, gi.psi_pad) || !add_ok(p->psi, psi)) { delete p; return ZERO_EINVAL; }
      flat += gi.psi_pad;
      rank_off += gi.shard;
      p->psi += psi;
    }
    p->psi_pad = flat;
    p->shard_total = rank_off;
    // bytes of the stage-0 memory report must stay representable
    if (p->psi_pad > std::numeric_limits<int64_t>::max() / 16) { delete p; return ZERO_EINVAL; }
  } catch (const std::bad_alloc&) {
    delete p;
    return ZERO_ENOMEM;
  }
  *out = p;
  return ZERO_OK;
}

extern "C" int zero_plan_destroy(zero_plan_t* plan) {
  delete plan;
  return ZERO_OK;
}

extern "C" int zero_plan_info(const zero_plan_t* p, zero_plan_info_t* out) {
  if (!p || !out) return ZERO_EINVAL;
  out->psi = p->psi;
  out->psi_pad = p->psi_pad;
  out->shard_total = p->shard_total;
  out->n_tensors = (int64_t)p->numels.size();
  out->n_ranks = p->n_ranks;
  out->align = p->align;
  out->n_groups = (int32_t)p->groups.size();
  out->reserved = 0;
  return ZERO_OK;
}

extern "C" int zero_plan_group(const zero_plan_t* p, int32_t group, zero_group_info_t* out) {
  if (!p || !out) return ZERO_EINVAL;
  if (group < 0 || group >= (int32_t)p->groups.size()) return ZERO_ERANGE;
  *out = p->groups[group];
  return ZERO_OK;
}

extern "C" int zero_plan_tensor(const zero_plan_t* p, int64_t t, int64_t* flat_off,
                                int32_t* first_owner, int32_t* last_owner) {
  if (!p) return ZERO_EINVAL;
  if (t < 0 || t >= (int64_t)p->numels.size()) return ZERO_ERANGE;
  const zero_group_info_t& g = p->groups[p->tensor_group[t]];
  const int64_t off = p->tensor_group_off[t];
  if (flat_off) *flat_off = g.flat_off + off;
  int32_t a = -1, b = -1;
  if (p->numels[t] > 0) {
    a = (int32_t)(off / g.shard);
    b = (int32_t)((off + p->numels[t] - 1) / g.shard);
  }
  if (first_owner) *first_owner = a;
  if (last_owner) *last_owner = b;
  return ZERO_OK;
}

extern "C" int zero_plan_shard(const zero_plan_t* p, int32_t group, int32_t rank,
                               int64_t* begin, int64_t* len, int64_t* valid_len) {
  if (!p) return ZERO_EINVAL;
  if (group < 0 || group >= (int32_t)p->groups.size() || rank < 0 || rank >= p->n_ranks)
    return ZERO_ERANGE;
  const zero_group_info_t& g = p->groups[group];
  int64_t lo = (int64_t)rank * g.shard;
  int64_t valid = g.psi - lo;
  if (valid < 0) valid = 0;
  if (valid > g.shard) valid = g.shard;
  if (begin) *begin = g.flat_off + lo;
  if (len) *len = g.shard;
  if (valid_len) *valid_len = valid;
  return ZERO_OK;
}

extern "C" int zero_plan_segments(const zero_plan_t* p, int32_t rank, zero_seg_t* out,
                                  int64_t cap, int64_t* n) {
  if (!p || !n || cap < 0 || (cap > 0 && !out)) return ZERO_EINVAL;
  if (rank < 0 || rank >= p->n_ranks) return ZERO_ERANGE;
  int64_t count = 0;
  for (const zero_group_info_t& g : p->groups) {
    const int64_t lo_r = (int64_t)rank * g.shard, hi_r = lo_r + g.shard;
    for (int64_t t = g.first_tensor; t < g.first_tensor + g.n_tensors; ++t) {
      const int64_t a = p->tensor_group_off[t], b = a + p->numels[t];
      const int64_t lo = a > lo_r ? a : lo_r, hi = b < hi_r ? b : hi_r;
      if (hi <= lo) continue;
      if (count < cap) out[count] = zero_seg_t{t, lo - a, g.flat_off + lo, hi - lo};
      ++count;
    }
  }
  *n = count;
  return ZERO_OK;
}

extern "C" int zero_plan_memory(const zero_plan_t* p, int32_t stage, zero_mem_t* out) {
  if (!p || !out) return ZERO_EINVAL;
  const int64_t P = p->psi_pad, S = p->shard_total;
  switch (stage) {
    case 0: out->values = 4 * P;         out->bytes = 16 * P;          break;
    case 1: out->values = 2 * P + 2 * S; out->bytes = 4 * P + 12 * S;  break;
    case 2: out->values = P + 3 * S;     out->bytes = 2 * P + 14 * S;  break;
    case 3: out->values = 4 * S;         out->bytes = 16 * S;          break;
    default: return ZERO_ERANGE;
  }
  return ZERO_OK;
}

extern "C" int zero_plan_volume(const zero_plan_t* p, int64_t* send, int64_t* recv) {
  if (!p) return ZERO_EINVAL;
  const int64_t v = (int64_t)(p->n_ranks - 1) * p->shard_total;
  if (send) *send = v;
  if (recv) *recv = v;
  return ZERO_OK;
}
