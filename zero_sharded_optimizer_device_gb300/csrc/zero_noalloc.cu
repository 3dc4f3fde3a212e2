// Reduce-scatter + global gradient norm for callers that cannot allocate.
//
// zero_reduce_scatter followed by zero_grad_norm needs a caller-allocated
// fp64 buffer for the per-block partial sums of squares.  Some callers cannot
// allocate device memory at the point where they clip: code that runs under
// another framework's allocator or memory budget (a caching allocator that
// has already reserved the device's memory, where a raw cudaMalloc can fail
// or fragment it), and latency-critical loops that must not take the
// implicit device-wide synchronisation cudaMalloc and cudaFree can carry.
// zero_reduce_scatter_norm_static gives them the same result with the
// partials held in a fixed array in this library's own device memory.
//
// The array: kStaticPartials fp64 slots (32 KiB) of static device memory,
// which every GPU that loads this library holds until the process exits.
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (with
// that device current) and caches it; that first call should come before
// any stream capture.  Every call reuses the same slots: a call fixes its
// reduce-scatter grid once, every block of that launch writes its own slot
// (blocks without work write 0), and the norm kernel then reads exactly those
// slots, so nothing has to be cleared between calls, and a zero_set_occupancy
// on another host thread cannot change the grid between the launch and the
// norm.  An empty window launches no reduce-scatter and reads no slot (norm
// 0, coefficient 1).  Two calls that overlap on the GPU (different streams,
// no ordering between them) race on the slots and may both return a wrong
// norm.
#include <math.h>
#include <nvtx3/nvToolsExt.h>

#include <mutex>

#include "zero_internal.h"

namespace {

constexpr int64_t kStaticPartials = ZERO_STATIC_PARTIALS;
static_assert(kStaticPartials == 4096, "ZERO_STATIC_PARTIALS changed: update the docs");

static __device__ __align__(256) double g_norm_partials[kStaticPartials];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
double* g_addr[kMaxDevices] = {nullptr};

// Device address of g_norm_partials on the current device (looked up once
// per device, with that device current).
int static_partials(double** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_norm_partials);
    if (e != cudaSuccess) return (int)e;
    g_addr[dev] = static_cast<double*>(p);
  }
  *out = g_addr[dev];
  return 0;
}

bool aligned4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

}  // namespace

extern "C" int zero_reduce_scatter_norm_static(const zero_plan_t* plan, int32_t group,
                                               const void* const* grads, zero_dtype_t gdtype,
                                               float* reduced, int64_t begin, int64_t end,
                                               float grad_scale, float max_norm, float* d_norm,
                                               float* d_coef, zero_stream_t stream) {
  struct Range {  // NVTX range around the call, as for every device entry point
    Range() { nvtxRangePushA("zero_reduce_scatter_norm_static"); }
    ~Range() { nvtxRangePop(); }
  } nvtx;
  // checks of the norm's own arguments first, so that a rejected call
  // launches nothing; zero_reduce_scatter checks the rest
  if (!plan || !isfinite(max_norm) || !(max_norm > 0.0f)) return ZERO_EINVAL;
  if ((d_norm && !aligned4(d_norm)) || (d_coef && !aligned4(d_coef))) return ZERO_EALIGN;
  if (!(gdtype == ZERO_F32 || gdtype == ZERO_BF16)) return ZERO_EDTYPE;
  if (begin < 0 || end < begin) return ZERO_ERANGE;
  // the grid, and with it the number of slots written and read, is fixed here
  const int64_t n = end > begin ? zk::rs_partials_for(plan->n_ranks, gdtype, end - begin) : 0;
  if (n > kStaticPartials) return ZERO_ERANGE;  // more partials than static slots
  double* partials = nullptr;
  const int ce = static_partials(&partials);
  if (ce != 0) {
    zk::record_cuda_error(ce);
    return ZERO_ECUDA;
  }
  int s = zk::reduce_scatter_entry(plan, group, grads, gdtype, reduced, begin, end, grad_scale,
                                   partials, n, (cudaStream_t)stream);
  if (s != ZERO_OK) return s;
  return zero_grad_norm(partials, n, max_norm, d_norm, d_coef, stream);
}
