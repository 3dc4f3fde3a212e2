/*
 * zero.h -- C ABI of libzero, the data-parallel hot path of ZeRO stages 1-3
 * on one GPU, with the N data-parallel ranks emulated as N device buffers.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "[REQUEST] Direct Correspondence between Gradient and Optimizer
 *        States to Reduce Communication?" (DeepSpeed issue 4582), "Problem":
 *        gradients are partitioned, reduce-scattered to the owners of the
 *        optimizer state, the owners update their parameters, and the
 *        parameters are all-gathered.
 *   [P2] "Why does not the stage 3 implementation use broadcast and
 *        reduce-scatter?" (DeepSpeed issue 1173), answers: stage 3 gathers
 *        parameters with all-gather; the reduce-scatter runs over contiguous
 *        gradient buffers only.
 *   [P3] "Why DeepSpeed ZeRO paper says reduce-scatter (or all-gather) has
 *        data movement of Psi elements?" (DeepSpeed discussion 6594):
 *        all-reduce = reduce-scatter + all-gather; the ring schedule.
 *   [P4] "ZeRO Optimizer" (wiki page): "Memory Components", "ZeRO Stages",
 *        "Implementation Strategy", "Communication Optimization",
 *        "Theoretical Reductions".
 *   [KB] Kingma and Ba, "Adam" (2015), Algorithm 1 (the pages name m and v
 *        but not the update formula).
 *
 * Conventions
 *   - Every function returns an int status: ZERO_OK (0) or a negative
 *     ZERO_E* code.  No C++ exception crosses this boundary.
 *   - Plans are opaque host objects owned by the library; free them with
 *     zero_plan_destroy().  A plan is immutable, so one plan may be used
 *     from several host threads at once.
 *   - Every device buffer is allocated and owned by the caller.  No hot call
 *     allocates device or pinned memory.
 *   - Device calls are asynchronous on the caller's stream (a cudaStream_t
 *     passed as zero_stream_t; NULL = the legacy default stream).  They
 *     report argument errors and launch errors only; a later
 *     cudaStreamSynchronize reports execution errors.
 *   - Calls launch on the calling thread's current CUDA device.
 *   - "Device pointer" means any address that device can access: its memory,
 *     pinned host memory mapped into the device address space (cudaHostAlloc
 *     on a unified-addressing system), or -- where the device reports
 *     cudaDevAttrPageableMemoryAccess, as a GB300 behind NVLink-C2C does --
 *     any host memory.  The library does not check; the Python binding
 *     refuses CPU tensors the device cannot reach.  Given mapped host buffers for grads or
 *     the gathered output, the kernels read and write them over the host link
 *     directly, overlapping the transfer with the step.
 *   - Every device pointer must be 16-byte aligned (ZERO_EALIGN otherwise),
 *     except fp64 partial sums (8 bytes) and the checksum word (8 bytes).
 *     Element offsets that break 16-byte vectors (odd windows, align=1
 *     shards) are handled inside the kernels.
 *   - Flat arrays ("flat"): reduced gradient, fp32 master, m, v and the full
 *     gathered parameter buffer.  Each holds psi_pad elements of all groups,
 *     group g at flat_off(g); inside a group, owner rank r's shard is
 *     [r*S_g, (r+1)*S_g).  A single-group plan (stages 1 and 2) has
 *     flat_off = 0, so rank r's shard sits at r*S.
 *   - Per-rank gradient buffers ("grads"): a host array of N device
 *     pointers; grads[r] holds rank r's full gradient of ONE group,
 *     psi_pad(g) elements in group-local order (padding elements must be 0).
 *   - Per-rank parameter shard buffers ("shards", stage 3): a host array of
 *     N device pointers; shards[r] holds rank r's bf16 shards of all groups,
 *     shard_total elements, group g's shard at rank_off(g).
 *   - Windows [begin, end) are group-local element indices,
 *     0 <= begin <= end <= psi_pad(g).  Any begin/end is accepted.
 */
#ifndef ZERO_H_
#define ZERO_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZERO_OK 0
#define ZERO_EINVAL (-1)   /* null/negative/invalid argument */
#define ZERO_EALIGN (-2)   /* device pointer not 16-byte aligned */
#define ZERO_ERANGE (-3)   /* group, rank, tensor or window outside the plan */
#define ZERO_EDTYPE (-4)   /* dtype not supported by this call */
#define ZERO_ENOMEM (-5)   /* host allocation failed */
#define ZERO_ECUDA (-6)    /* CUDA runtime error; see zero_last_cuda_error() */
#define ZERO_ETIMEOUT (-7) /* a bounded device wait ran out */

#define ZERO_MAX_RANKS 64  /* largest N the kernels accept */

typedef enum { ZERO_F32 = 0, ZERO_BF16 = 1 } zero_dtype_t;

typedef struct zero_plan zero_plan_t;
typedef void* zero_stream_t; /* a cudaStream_t */

typedef struct {
  int64_t psi;          /* real parameters, all groups */
  int64_t psi_pad;      /* padded flat length, all groups */
  int64_t shard_total;  /* elements each rank owns, all groups (sum of S_g) */
  int64_t n_tensors;
  int32_t n_ranks;      /* N */
  int32_t align;        /* shard size and start quantum, in elements */
  int32_t n_groups;
  int32_t reserved;
} zero_plan_info_t;

typedef struct {
  int64_t psi, psi_pad, shard; /* S_g = psi_pad / N */
  int64_t flat_off;            /* group start in flat arrays */
  int64_t rank_off;            /* group start in each rank's shard buffer */
  int64_t first_tensor, n_tensors;
} zero_group_info_t;

typedef struct {
  int64_t tensor;      /* tensor index */
  int64_t tensor_off;  /* first element of the piece inside the tensor */
  int64_t flat_off;    /* its flat index */
  int64_t len;         /* elements */
} zero_seg_t;

typedef struct {
  int64_t values; /* [P4 "Theoretical Reductions"] values per device */
  int64_t bytes;  /* bf16 params and grads, fp32 master + m + v */
} zero_mem_t;

typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
  float grad_scale; /* multiplies the reduced sum; 1/N averages */
  int64_t step;     /* t >= 1: this update's step number (ignored with d_state) */
  /* NULL, or a ZERO_ADAM_STATE_BYTES device buffer set up by
   * zero_adam_state_init: the kernels then take the bias corrections from it
   * instead of from `step`, so one captured CUDA graph of a step stays valid
   * for every later step (advance it with zero_adam_state_advance). */
  void* d_state;
} zero_adam_t;

#define ZERO_ADAM_STATE_BYTES 32

/* ------------------------------------------------------------- library -- */
int zero_version(void);
/* Text for a status code; a static string, never NULL. */
const char* zero_strerror(int status);
/* The cudaError_t of the last ZERO_ECUDA returned on this host thread. */
int zero_last_cuda_error(void);

/* ----------------------------------------------------------------- plan --
 * zero_plan: partition a list of tensors into N owner shards [P1
 * "Problem"; P2: one contiguous gradient buffer; P4 "ZeRO Stages"].
 * The tensors are concatenated in list order with no per-tensor padding.
 * Each group is padded at its tail to psi_pad(g) = ceil(psi(g)/(N*align))
 * * N*align and cut into N equal shards S_g = psi_pad(g)/N; rank r owns
 * [r*S_g, (r+1)*S_g).  group_of_tensor (may be NULL = one group) gives each
 * tensor's layer group; it must start at 0 and be non-decreasing without
 * gaps (stage 3 plans every layer group on its own [P4 "Implementation
 * Strategy"]).  numels[t] >= 0; 1 <= N <= 64; align >= 1; every group's
 * psi_pad below 2^40 elements (the kernels' index range).
 * Errors: ZERO_EINVAL (bad arguments or group list, size overflow),
 * ZERO_ENOMEM.  *out is set only on success. */
int zero_plan(const int64_t* numels, int64_t n_tensors, int32_t n_ranks, int32_t align,
              const int32_t* group_of_tensor, zero_plan_t** out);
int zero_plan_destroy(zero_plan_t* plan);
int zero_plan_info(const zero_plan_t* plan, zero_plan_info_t* out);
int zero_plan_group(const zero_plan_t* plan, int32_t group, zero_group_info_t* out);
/* Flat offset of tensor t and the ranks owning its first and last element
 * (-1 for an empty tensor).  Errors: EINVAL (plan NULL), ERANGE (t outside
 * the plan). */
int zero_plan_tensor(const zero_plan_t* plan, int64_t t, int64_t* flat_off,
                     int32_t* first_owner, int32_t* last_owner);
/* Rank r's shard of group g: flat begin, length S_g, real (non-padding)
 * elements.  Errors: EINVAL (plan NULL), ERANGE (group or rank outside the
 * plan). */
int zero_plan_shard(const zero_plan_t* plan, int32_t group, int32_t rank, int64_t* begin,
                    int64_t* len, int64_t* valid_len);
/* Pieces of tensors rank r owns, in flat order.  Writes min(cap, count)
 * entries to out (out may be NULL when cap == 0); *n = count.  Errors:
 * EINVAL (plan or n NULL, cap < 0, out NULL with cap > 0), ERANGE (rank). */
int zero_plan_segments(const zero_plan_t* plan, int32_t rank, zero_seg_t* out, int64_t cap,
                       int64_t* n);
/* Per-device memory of stage 0 (plain data parallelism: 4P values [P4
 * "Memory Components"]), 1 (2P + 2P/N), 2 (P + 3P/N) or 3 (4P/N) [P4
 * "Theoretical Reductions"], with P = psi_pad and P/N = shard_total; bytes
 * count bf16 params and grads and 12 bytes of fp32 master + m + v.
 * Errors: EINVAL (plan or out NULL), ERANGE (stage not 0..3). */
int zero_plan_memory(const zero_plan_t* plan, int32_t stage, zero_mem_t* out);
/* Elements each rank sends and receives in one ring reduce-scatter (and in
 * one all-gather): (N-1) * shard_total [P3].  Errors: EINVAL (plan NULL). */
int zero_plan_volume(const zero_plan_t* plan, int64_t* send_per_rank, int64_t* recv_per_rank);

/* ------------------------------------------------------- device calls -- */

/* zero_reduce_scatter [P1 "Problem"; P3]: for every i in [begin, end) of
 * group g, reduced[flat_off(g) + i] = the fp32 sum of grads[r][i] over the
 * N ranks, in the ring order of owner k = i / S_g: k+1, k+2, ..., N-1, 0,
 * ..., k (the owner adds last).  gdtype: ZERO_F32 or ZERO_BF16.
 * If sumsq_partials is not NULL, also writes zero_rs_partials() fp64
 * partial sums of (reduced * grad_scale)^2 over the window, for
 * zero_grad_norm().  With reduced == NULL (and sumsq_partials given) only the
 * partials are produced: the first pass of a fused clip that re-reads the
 * gradients instead of storing the fp32 reduced gradient (worth it when
 * N * sizeof(grad) < 8 bytes, i.e. the re-read costs less than the 8-byte
 * store + load of the reduced value).
 * Errors: EINVAL (also when both outputs are NULL), EALIGN, ERANGE, EDTYPE,
 * ECUDA. */
int zero_reduce_scatter(const zero_plan_t* plan, int32_t group, const void* const* grads,
                        zero_dtype_t gdtype, float* reduced, int64_t begin, int64_t end,
                        float grad_scale, double* sumsq_partials, zero_stream_t stream);
/* zero_reduce_scatter_acc: gradient accumulation over micro-batches
 * ["ZeRO Optimizer", "Hybrid Approaches": gradient accumulation with
 * micro-batching]: reduced[f] = reduced[f] + (ring sum of this micro-batch),
 * in that order, fp32, for i in [begin, end).  The first micro-batch uses
 * zero_reduce_scatter; Adam then takes grad_scale = 1/(N * micro_batches).
 * sumsq_partials (may be NULL) sum (accumulated * grad_scale)^2, so the last
 * micro-batch's call yields the norm of the accumulated gradient.
 * Errors: EINVAL, EALIGN, ERANGE, EDTYPE, ECUDA (as zero_reduce_scatter;
 * reduced is required). */
int zero_reduce_scatter_acc(const zero_plan_t* plan, int32_t group, const void* const* grads,
                            zero_dtype_t gdtype, float* reduced, int64_t begin, int64_t end,
                            float grad_scale, double* sumsq_partials, zero_stream_t stream);

/* Number of fp64 partials zero_reduce_scatter writes for a window of
 * n_elements with this plan's N and gdtype on the current device (one per
 * block of its launch; blocks without work write 0).  Errors: EINVAL (plan
 * or n_partials NULL, n_elements < 0), EDTYPE. */
int zero_rs_partials(const zero_plan_t* plan, zero_dtype_t gdtype, int64_t n_elements,
                     int64_t* n_partials);

/* zero_grad_norm: norm = sqrt(sum of n fp64 partials), summed in a fixed
 * order; coef = min(1, max_norm / (norm + 1e-6)) rounded to fp32.  Writes
 * *d_norm (fp32) and *d_coef (fp32) on the device; either may be NULL.
 * The clip is not on the pages; it is the coefficient torch's
 * clip_grad_norm_ applies.  Errors: EINVAL (n < 0, partials NULL with n > 0,
 * max_norm not finite and positive), EALIGN (partials not 8-byte, outputs
 * not 4-byte aligned), ECUDA. */
int zero_grad_norm(const double* partials, int64_t n, float max_norm, float* d_norm,
                   float* d_coef, zero_stream_t stream);

/* zero_adam_bias_corrections [KB, Algorithm 1: the bias corrections
 * 1 - beta^t]: the two fp32 values the device calls use for hp->step, bc1 =
 * 1 - beta1^t and bc2 = 1 - beta2^t, with beta^t the product of t fp64
 * factors of the fp32 beta (each stopping once below 2^-60) rounded once to
 * fp32.  Host only; touches no device.  Each host thread continues the
 * product from its previous call when the step has not gone back (for
 * growing step numbers the cost is one factor per step, not t), with results
 * identical to the full product.  Errors: EINVAL (hp or an output NULL,
 * invalid betas, step < 1). */
int zero_adam_bias_corrections(const zero_adam_t* hp, float* bc1, float* bc2);

/* zero_adam_state_init / zero_adam_state_advance: Adam's step-dependent
 * constants kept in device memory (no counterpart on the pages; it lets a
 * whole step be captured once in a CUDA graph and replayed).  d_state is a
 * caller-owned, 8-byte aligned device buffer of ZERO_ADAM_STATE_BYTES.
 * init sets it to "before step hp->step"; each advance (a one-thread
 * kernel on `stream`, enqueue it before the step's kernels) moves to the next
 * step: beta^t is multiplied once more by each fp32 beta in fp64 (stopping
 * once below 2^-60, exactly as the host computation of zero_adam_t.step
 * does) and bc = 1 - beta^t is rounded to fp32, so results are bit-identical
 * to passing the step number.  Errors: EINVAL, EALIGN, ECUDA. */
int zero_adam_state_init(const zero_adam_t* hp, void* d_state, zero_stream_t stream);
int zero_adam_state_advance(const zero_adam_t* hp, void* d_state, zero_stream_t stream);

/* zero_adam_shard [P1 "Problem"; P4 "Memory Components"; KB]: for i in
 * [begin, end) of group g (flat index f = flat_off(g) + i):
 *   grad = reduced[f] * grad_scale (* *d_coef when d_coef != NULL)
 *   p -= (lr*wd)*p (when wd != 0);  m = b1*m + (1-b1)*grad;
 *   v = b2*v + (1-b2)*grad^2;  p -= (lr * (m/bc1)) / (sqrt(v/bc2) + eps)
 * in fp32, one rounding per operation, bc = 1 - beta^t computed in fp64 on
 * the host and rounded to fp32.  If out != NULL also writes out[f] =
 * cast(p) (out_dtype ZERO_BF16: round to nearest even; ZERO_F32: copy).
 * Errors: EINVAL, EALIGN, ERANGE, EDTYPE, ECUDA. */
int zero_adam_shard(const zero_plan_t* plan, int32_t group, float* master, float* m, float* v,
                    const float* reduced, const zero_adam_t* hp, const float* d_coef,
                    int64_t begin, int64_t end, void* out, zero_dtype_t out_dtype,
                    zero_stream_t stream);

/* zero_step_clipped [P1 "Problem"; P3; KB; the clip is not on the pages]:
 * the step with gradient clipping of group g in one call (the path of a run
 * that clips: the reduced gradient has to exist before its global norm
 * does).  The plain step zero_step cannot clip by the norm
 * of the step's own gradient, since it never materialises the reduced
 * gradient; this call strings the unfused calls together on `stream`, with
 * results identical, bit for bit, to making them one by one:
 *   zero_reduce_scatter over windows [a, a+bucket) of the group, writing
 *     `reduced` and each window's norm partials into consecutive slices of
 *     `partials` (scale hp->grad_scale);
 *   zero_grad_norm over all of them with max_norm -> *d_norm (may be NULL)
 *     and *d_coef (required);
 *   zero_adam_shard over chunks [a, a+chunk) with d_coef, writing full_out
 *     (may be NULL) in out_dtype.
 * partials: caller-owned fp64 scratch of n_partials >= the count
 * zero_step_clipped_partials reports (ERANGE otherwise).  bucket, chunk >= 1.
 * The call fixes its reduce-scatter grids before the first launch, so it
 * writes exactly the partials it checked, even if zero_set_occupancy runs
 * on another host thread meanwhile.
 * Errors: EINVAL, EALIGN, ERANGE, EDTYPE, ECUDA. */
int zero_step_clipped_partials(const zero_plan_t* plan, int32_t group, zero_dtype_t gdtype,
                               int64_t bucket, int64_t* n_partials);
int zero_step_clipped(const zero_plan_t* plan, int32_t group, const void* const* grads,
                      zero_dtype_t gdtype, float* reduced, float* master, float* m, float* v,
                      const zero_adam_t* hp, float max_norm, int64_t bucket, int64_t chunk,
                      double* partials, int64_t n_partials, float* d_norm, float* d_coef,
                      void* full_out, zero_dtype_t out_dtype, zero_stream_t stream);

/* zero_all_gather [P1 "Problem"; P3 all-gather]: full_out[f] = cast(
 * master[f]) for every element of group g (g = -1: all groups), i.e. every
 * owner's updated shard lands in the one full flat parameter buffer all
 * ranks share.  out_dtype: ZERO_BF16 (round to nearest even) or ZERO_F32.
 * Errors: EINVAL, EALIGN, ERANGE (group), EDTYPE, ECUDA. */
int zero_all_gather(const zero_plan_t* plan, int32_t group, const float* master,
                    void* full_out, zero_dtype_t out_dtype, zero_stream_t stream);

/* zero_step: the fused reduce-scatter + scale (+ clip by *d_coef) + Adam +
 * all-gather of group g in one pass; the reduced gradient never reaches
 * memory.  Same arithmetic, per element, as zero_reduce_scatter followed by
 * zero_adam_shard with out = full_out (bit-identical results).  full_out
 * may be NULL (no gather).  Errors: EINVAL (NULL or invalid arguments, Adam
 * hyperparameters), EALIGN, ERANGE (group), EDTYPE, ECUDA. */
int zero_step(const zero_plan_t* plan, int32_t group, const void* const* grads,
              zero_dtype_t gdtype, float* master, float* m, float* v, const zero_adam_t* hp,
              const float* d_coef, void* full_out, zero_dtype_t out_dtype,
              zero_stream_t stream);

/* zero_step_acc: the last micro-batch of gradient accumulation ["ZeRO
 * Optimizer", "Hybrid Approaches": gradient accumulation with
 * micro-batching], fused: as zero_step, with the reduced gradient taken as
 * accumulated[f] + (this micro-batch's ring sum), in that order, fp32 --
 * `accumulated` being the flat fp32 buffer zero_reduce_scatter and
 * zero_reduce_scatter_acc filled for the earlier micro-batches (read only).
 * Bit-identical to zero_reduce_scatter_acc into that buffer followed by
 * zero_adam_shard over the group, without storing and re-reading the reduced
 * gradient (8 bytes per parameter less).  hp->grad_scale is 1/(N * micro-batches).
 * `accumulated` must not overlap master, m, v or full_out (the kernel reads it
 * while writing those); the same pointer in two of these roles returns
 * ZERO_EINVAL.  Errors: as zero_step. */
int zero_step_acc(const zero_plan_t* plan, int32_t group, const void* const* grads,
                  zero_dtype_t gdtype, const float* accumulated, float* master, float* m,
                  float* v, const zero_adam_t* hp, const float* d_coef, void* full_out,
                  zero_dtype_t out_dtype, zero_stream_t stream);

/* zero_step_group (stage 3) [P4 "ZeRO Stages", stage 3]: as zero_step, but
 * each owner writes its updated bf16 parameters only into its own shard
 * buffer: shards[k][rank_off(g) + (i - k*S_g)] for owner k of element i.
 * Errors: EINVAL (NULL or invalid arguments, Adam hyperparameters), EALIGN,
 * ERANGE (group), EDTYPE, ECUDA. */
int zero_step_group(const zero_plan_t* plan, int32_t group, const void* const* grads,
                    zero_dtype_t gdtype, float* master, float* m, float* v,
                    const zero_adam_t* hp, const float* d_coef, void* const* shards,
                    zero_stream_t stream);

/* zero_step_group_acc (stage 3): the last micro-batch of gradient
 * accumulation ["ZeRO Optimizer", "Hybrid Approaches": gradient accumulation
 * with micro-batching] fused, as zero_step_acc is for stages 1 and 2: the
 * reduced gradient is taken as accumulated[f] + (this micro-batch's ring
 * sum), in that order, fp32, `accumulated` being the flat fp32 buffer that
 * zero_reduce_scatter and zero_reduce_scatter_acc filled for the group's
 * earlier micro-batches (read only); then scale, Adam and each owner's bf16
 * parameters into its shard buffer, as zero_step_group.  hp->grad_scale is
 * 1/(N * micro-batches).  `accumulated` must not overlap master, m or v; the
 * same pointer in two of these roles returns ZERO_EINVAL.  Errors: as
 * zero_step_group. */
int zero_step_group_acc(const zero_plan_t* plan, int32_t group, const void* const* grads,
                        zero_dtype_t gdtype, const float* accumulated, float* master, float* m,
                        float* v, const zero_adam_t* hp, const float* d_coef,
                        void* const* shards, zero_stream_t stream);

/* zero_gather_layer (stage 3) [P4 "Implementation Strategy": gather a
 * layer's parameters just before use; P2: by all-gather]: layer_out[j] =
 * shards[j / S_g][rank_off(g) + j % S_g] for j in [0, psi_pad(g)): the N
 * ranks' shards of group g concatenated into one contiguous layer buffer.
 * dtype: element type of the shard buffers (ZERO_BF16 or ZERO_F32).  When
 * S_g and rank_off(g) are multiples of 16 bytes the N segments move by 1-D
 * bulk copies (TMA) through shared memory, issued by one thread per CTA;
 * their waits are bounded (see zero_async_status).  Otherwise element by
 * element.  The bulk-copy kernel is launched with programmatic dependent
 * launch: its CTAs may become resident while the kernel before it on the
 * stream is still running, but they copy only after that kernel has finished
 * and its writes are visible, so stream order holds as for any launch (also
 * inside a captured CUDA graph).  Errors: EINVAL, EALIGN, ERANGE (group),
 * EDTYPE, ECUDA. */
int zero_gather_layer(const zero_plan_t* plan, int32_t group, const void* const* shards,
                      zero_dtype_t dtype, void* layer_out, zero_stream_t stream);

/* zero_broadcast_layer (stage 3) ["Why does not the stage 3 implementation
 * use broadcast and reduce-scatter?", first question and answer 1: the ZeRO
 * paper's stage 3 sends each owner's parameters by broadcast; DeepSpeed
 * gathers them with all-gather, at a similar communication volume]: the same
 * layer buffer as zero_gather_layer, layer_out[j] = shards[j / S_g][rank_off(g)
 * + j % S_g] for j in [0, psi_pad(g)), built the broadcast way: N broadcasts
 * in rank order, broadcast k sending owner k's shard to every rank, i.e.
 * writing layer_out[k*S_g, (k+1)*S_g).  Each broadcast is one kernel launch on
 * `stream` (N launches per call: the N collectives of the broadcast form,
 * each a separate step), by 1-D bulk copies when S_g and rank_off(g) are
 * multiples of 16 bytes, element by element otherwise.  The result is
 * bit-identical to zero_gather_layer's.  dtype: element type of the shard
 * buffers (ZERO_BF16 or ZERO_F32); layer_out: psi_pad(g) elements,
 * caller-owned.  Errors: EINVAL, EALIGN, ERANGE (group id), EDTYPE, ECUDA. */
int zero_broadcast_layer(const zero_plan_t* plan, int32_t group, const void* const* shards,
                         zero_dtype_t dtype, void* layer_out, zero_stream_t stream);

/* zero_gather_groups (stage 3): zero_gather_layer for k groups at once:
 * layer_outs[i] receives group groups[i] (1 <= k <= ZERO_MAX_COALESCE; a
 * group may repeat).  Groups whose shards meet the 16-byte rule share one
 * bulk-copy launch; the others are gathered element by element, one launch
 * each.  Made for per-parameter partitioning, where every tensor is its own
 * group and a module's tensors are needed together ("ZeRO Optimizer",
 * "Implementation Strategy": a layer's parameters are gathered before use):
 * one launch instead of one per tensor, each tensor still in its own buffer.
 * Errors: EINVAL, EALIGN, ERANGE (group id), EDTYPE, ECUDA. */
#define ZERO_MAX_COALESCE 64
int zero_gather_groups(const zero_plan_t* plan, const int32_t* groups, int32_t k,
                       const void* const* shards, zero_dtype_t dtype, void* const* layer_outs,
                       zero_stream_t stream);

/* zero_stage3_gather_pass (stage 3) ["ZeRO Optimizer", "Implementation
 * Strategy": gather a layer's parameters just before use, discard after, in
 * forward and backward; "Communication Optimization": hide the gathering
 * behind computation by prefetching the next layer]: for j = 0..n-1, gather
 * group order[j] (zero_gather_layer) into layer_bufs[j % 2] on stream_b and
 * consume it on stream_a (zero_layer_checksum with consumer_rounds into
 * d_sums[j], standing in for the layer's computation: 1 round is bound by
 * memory, many rounds by on-chip arithmetic, like a layer's matrix
 * products).  The gather of order[j+1] is queued before
 * the consumer of order[j], so the two overlap; a buffer is refilled only
 * after the consumer that last read it has finished.  Stream B first waits
 * for the work already queued on stream A; work queued on stream A after the
 * call runs after every gather and consumer.  layer_bufs: 2 device buffers
 * of buf_elems bf16 elements each (>= psi_pad of every group in order);
 * d_sums: n uint64.  1 <= consumer_rounds <= ZERO_MAX_CONSUMER_ROUNDS.
 * The two kernels overlap only if their blocks fit on an SM together: the
 * gathers launch at the ZERO_OCC_PREFETCH cap and the consumer at the
 * ZERO_OCC_CONSUMER cap (by default 2 one-warp bulk-copy CTAs with a 6-stage
 * ring beside the consumer's cap of 7 256-thread blocks, of which its
 * register use lets 6 be resident; see zero_set_occupancy).  The call zeroes
 * d_sums[0..n) on stream_a before the first consumer.
 * stream_a != stream_b.  Uses five CUDA events created
 * and released inside the call; allocates no device memory.  The call may be
 * captured in a CUDA graph: with stream_a capturing, stream_b joins the
 * capture through those events and rejoins stream_a before the call returns.
 * Errors: EINVAL, EALIGN, ERANGE (group id or buffer size), ECUDA. */
int zero_stage3_gather_pass(const zero_plan_t* plan, const int32_t* order, int32_t n,
                            const void* const* shards, void* const* layer_bufs,
                            int64_t buf_elems, uint64_t* d_sums, int32_t consumer_rounds,
                            zero_stream_t stream_a, zero_stream_t stream_b);

/* zero_stage3_gather_pass_steps: zero_stage3_gather_pass whose step j
 * fetches several groups at once, step_groups[step_first[j]] ..
 * step_groups[step_first[j+1] - 1] (1 to ZERO_MAX_COALESCE groups;
 * step_first[0] = 0, n_steps + 1 entries), as zero_gather_groups does: into
 * layer_bufs[j % 2] one after another, each at the running element offset,
 * and the consumer then reads the step's sum of psi_pad elements as one
 * layer.  Made for per-parameter partitioning, where a module's tensors are
 * separate groups fetched together.  In a step of more than one group every
 * group's psi_pad * 2 bytes must be a multiple of 16 (ZERO_EALIGN otherwise),
 * and each step's elements must fit buf_elems (ZERO_ERANGE).  Otherwise as
 * zero_stage3_gather_pass, errors included (EINVAL also for a step of 0 or
 * more than ZERO_MAX_COALESCE groups, or step_first[0] != 0). */
int zero_stage3_gather_pass_steps(const zero_plan_t* plan, const int32_t* step_first,
                                  const int32_t* step_groups, int32_t n_steps,
                                  const void* const* shards, void* const* layer_bufs,
                                  int64_t buf_elems, uint64_t* d_sums, int32_t consumer_rounds,
                                  zero_stream_t stream_a, zero_stream_t stream_b);

/* zero_layer_checksum: stands in for the layer computation that consumes a
 * gathered buffer of n bf16 bit patterns (no counterpart on the pages).  For
 * each 8-element vector v (and each element of a ragged tail on its own),
 * c_v = sum over its j of bits[j] * (1 + j mod 65536); its term is
 * t_v = c_v * (1 + K + K^2 + ... + K^(rounds-1)) mod 2^64, computed as
 * rounds - 1 dependent multiply-adds t = t*K + c_v with K =
 * 6364136223846793005; *d_out = sum of the terms mod 2^64.  rounds = 1 is
 * the plain checksum, bound by the one read of the layer; larger rounds add
 * on-chip work only.  1 <= rounds <= ZERO_MAX_CONSUMER_ROUNDS.  Errors:
 * EINVAL (n < 0, d_out NULL, layer NULL with n > 0, rounds outside
 * [1, ZERO_MAX_CONSUMER_ROUNDS]), EALIGN (layer not 16-byte, d_out not
 * 8-byte aligned), ECUDA. */
#define ZERO_MAX_CONSUMER_ROUNDS 4096
int zero_layer_checksum(const void* layer, int64_t n, int32_t rounds, uint64_t* d_out,
                        zero_stream_t stream);

/* zero_reduce_scatter_norm_static: the pages have no counterpart to this
 * entry point; it exists for callers that cannot allocate device memory
 * where they clip (code running under another framework's allocator or
 * memory budget, where a raw cudaMalloc can fail or fragment the pool, and
 * loops that must not take the device-wide synchronisation cudaMalloc and
 * cudaFree can carry).  It computes what zero_reduce_scatter (with
 * sumsq_partials) followed by zero_grad_norm computes for one window:
 * reduced[...] over [begin, end), *d_norm and *d_coef; the fp64 partial sums
 * live in a static array of ZERO_STATIC_PARTIALS (4096, 32 KiB) slots in
 * this library's device memory, which every GPU that loads the library keeps
 * until the process exits.  It allocates nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first
 *     call before any stream capture.
 *   - A window needs zero_rs_partials(plan, gdtype, end-begin) slots; if
 *     that exceeds ZERO_STATIC_PARTIALS the call returns ZERO_ERANGE and
 *     launches nothing.  (On a 152-SM GB300 any window needs at most a few
 *     hundred to 1216 slots.)
 *   - The call fixes its reduce-scatter grid once and reads exactly the
 *     slots that launch writes, so nothing needs clearing and a concurrent
 *     zero_set_occupancy cannot make it read a slot it did not write.  An
 *     empty window (begin == end) launches no reduce-scatter: norm 0,
 *     coefficient 1.
 *   - All calls share the slots: calls that overlap on the GPU race on them.
 * Errors: as zero_reduce_scatter and zero_grad_norm, plus ERANGE above. */
#define ZERO_STATIC_PARTIALS 4096
int zero_reduce_scatter_norm_static(const zero_plan_t* plan, int32_t group,
                                    const void* const* grads, zero_dtype_t gdtype,
                                    float* reduced, int64_t begin, int64_t end,
                                    float grad_scale, float max_norm, float* d_norm,
                                    float* d_coef, zero_stream_t stream);

/* zero_wait_flag: failure detection without a device fault (no counterpart
 * on the pages, which have no failure handling).  A one-thread kernel polls
 * *flag -- device memory, or pinned host memory mapped into the device
 * address space that the host may write while the kernel runs -- until it
 * equals `expected` or max_polls polls about 1 us apart have passed, then
 * writes ZERO_OK or ZERO_ETIMEOUT to *d_status.  The wait always ends, so a
 * peer that never signals turns into a status the host reads after the
 * stream synchronizes, and the context stays usable.  0 <= max_polls <=
 * ZERO_MAX_POLLS (about 10 s).  Never use it to wait for another kernel of
 * this process: launches are not guaranteed to run concurrently.  Errors:
 * EINVAL (NULL pointer, max_polls outside [0, ZERO_MAX_POLLS]), EALIGN (flag
 * or d_status not 4-byte aligned), ECUDA (launch). */
#define ZERO_MAX_POLLS 10000000
int zero_wait_flag(const uint32_t* flag, uint32_t expected, int64_t max_polls,
                   int32_t* d_status, zero_stream_t stream);

/* zero_set_occupancy: tuning knob (no counterpart on the pages).  Every
 * streaming kernel runs one wave of 256-thread blocks striding over its
 * window; this sets how many blocks per SM a kernel family keeps resident
 * (1..32; 0 restores the library default; the register limit still caps
 * it).  HBM throughput of these kernels often peaks below full occupancy,
 * and the best value depends on the kernel and the GPU.  *previous (may be
 * NULL) receives the value in effect before the call.  Process-wide; set it
 * between steps, not while a reduce-scatter's partials are still to be
 * read: zero_rs_partials() follows the setting in effect.  Errors: EINVAL
 * (kind or blocks_per_sm out of range). */
#define ZERO_OCC_FUSED 0  /* zero_step, zero_step_group */
#define ZERO_OCC_RS 1     /* zero_reduce_scatter, zero_reduce_scatter_acc */
#define ZERO_OCC_ADAM 2   /* zero_adam_shard */
#define ZERO_OCC_GATHER 3 /* zero_gather_layer (CTAs per SM of its bulk-copy form) */
#define ZERO_OCC_STREAM 4 /* zero_all_gather, zero_copy */
#define ZERO_OCC_CONSUMER 5 /* zero_layer_checksum (also inside the gather pass) */
#define ZERO_OCC_PREFETCH 6 /* the gathers inside zero_stage3_gather_pass (as GATHER) */
#define ZERO_OCC_KINDS 7
int zero_set_occupancy(int32_t kind, int32_t blocks_per_sm, int32_t* previous);

/* zero_copy: device-to-device copy of `bytes` (a multiple of 16) with
 * 16-byte loads and stores; measures the achievable HBM copy bandwidth.
 * bytes == 0 is a no-op.  Errors: EINVAL (bytes < 0 or not a multiple of 16,
 * NULL pointer), EALIGN, ECUDA. */
int zero_copy(void* dst, const void* src, int64_t bytes, zero_stream_t stream);

/* zero_async_status: number of bounded waits inside the library's kernels
 * that gave up (a bulk copy that had not landed after about 2 s) on the
 * current device since the last reset; nonzero means a result is incomplete.
 * The kernel that gave up still returns (the context stays usable).  No
 * counterpart on the pages.  Synchronizes the device; reset != 0 clears the
 * count afterwards.  Errors: EINVAL (timeouts NULL), ECUDA. */
int zero_async_status(int64_t* timeouts, int32_t reset);

/* ------------------------------------------------------ checked build --
 * No counterpart on the pages: a stand-in for a device memory checker.  The
 * library built with -DZERO_CHECKED (libzero_checked.so, same ABI) tests
 * every global access of its kernels against the extent this header gives
 * the buffer: a gradient buffer's [0, psi_pad(g)), the call's window of a
 * flat array, owner k's chunk [k*S_g, (k+1)*S_g) of a group, a shard
 * buffer's [rank_off(g), rank_off(g) + S_g), a layer buffer's [0, psi_pad(g)),
 * a partial-sum array's [0, n).  An access outside is skipped (never made)
 * and counted; the first one is recorded with its site and extent.  The
 * release library has no checks and reports checked = 0, count = 0. */
#define ZERO_SITE_PROBE 1        /* zero_bounds_probe */
#define ZERO_SITE_RS_GRAD 2      /* reduce-scatter: gradient buffers */
#define ZERO_SITE_RS_FLAT 3      /* reduce-scatter: reduced window */
#define ZERO_SITE_RS_OWNER 4     /* reduce-scatter: owner chunk */
#define ZERO_SITE_STEP_GRAD 5    /* fused step: gradient buffers */
#define ZERO_SITE_STEP_FLAT 6    /* fused step: master, m, v, full output window */
#define ZERO_SITE_STEP_OWNER 7   /* fused step: owner chunk */
#define ZERO_SITE_STEP_SHARD 8   /* fused step: owner's shard buffer */
#define ZERO_SITE_ADAM_FLAT 9    /* Adam: reduced, master, m, v, output window */
#define ZERO_SITE_CAST_FLAT 10   /* all-gather cast window */
#define ZERO_SITE_NORM 11        /* norm: partial sums */
#define ZERO_SITE_GATHER_SHARD 12 /* stage-3 gather: source shard */
#define ZERO_SITE_GATHER_OUT 13  /* stage-3 gather: layer buffer */
#define ZERO_SITE_CHECKSUM 14    /* layer checksum: layer buffer */
#define ZERO_SITE_COPY 15        /* zero_copy */

typedef struct {
  int32_t checked; /* 1 in the checked build */
  int32_t site;    /* ZERO_SITE_* of the first access outside its extent; 0 if none */
  int64_t count;   /* accesses outside their extent since the last reset */
  int64_t index;   /* first one: start of the accessed element range */
  int64_t lo, hi;  /* first one: the extent [lo, hi) it broke */
} zero_bounds_t;

/* zero_bounds_report: synchronizes the current device, then copies the
 * record of the kernels run on it to *out; reset != 0 clears the record
 * afterwards.  Release build: fills checked = 0 and zeros, touches no device.
 * Errors: EINVAL (out NULL), ECUDA. */
int zero_bounds_report(zero_bounds_t* out, int32_t reset);

/* zero_bounds_probe: checked build only (a no-op returning ZERO_OK in the
 * release build): a one-thread kernel that makes no memory access and
 * records one out-of-extent access at ZERO_SITE_PROBE (index 1, extent
 * [0, 1)), so a caller can confirm the record reaches the host.  Errors:
 * ECUDA (launch, checked build only). */
int zero_bounds_probe(zero_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_H_ */
