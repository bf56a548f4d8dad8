// attn_run_paged_no_workspace: attn_run_paged with library-owned scratch.
//
// Some callers cannot allocate device memory at the point where they run
// attention: plugins that a host framework hands tensor pointers but no
// allocator (the framework owns every device byte through its own pool), and
// serving loops that forbid cudaMalloc on the hot path (it can synchronise the
// device and its latency is unbounded).  attn_run_paged needs a caller-provided
// workspace for split-KV partials; this entry point instead uses one
// fixed-size array in device global memory that belongs to the library.  The
// array is a file-scope __device__ variable: every GPU that loads the library
// holds ATTN_NO_WORKSPACE_MAX_BYTES of it until the process exits, and all
// calls share it.
#include <cuda_runtime.h>

#include <mutex>

#include "attn_paged.h"
#include "kernels.hpp"
#include "plan.hpp"

namespace {

static __device__ __align__(256) uint8_t g_scratch[ATTN_NO_WORKSPACE_MAX_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on `device`, looked up once per device with that
// device current (in host code the symbol itself is only a host-side handle).
// The address is cached for the life of the process; after cudaDeviceReset it
// is stale (as are plans built before the reset).
attn_status_t scratch_address(int device, void **addr) {
  if (device < 0 || device >= kMaxDevices) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[device]) {
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return ATTN_ERR_CUDA;
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    // put the caller's device back before anything else can fail
    const cudaError_t back = prev != device ? cudaSetDevice(prev) : cudaSuccess;
    if (e != cudaSuccess || !p || back != cudaSuccess) return ATTN_ERR_CUDA;
    g_scratch_addr[device] = p;
  }
  *addr = g_scratch_addr[device];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_run_paged_no_workspace(
    attn_plan_t plan, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *page_table, const int32_t *seq_lens, const int32_t *qo_indptr,
    const float *sinks, int32_t window, float softmax_scale, float k_scale, float v_scale,
    void *out, float *lse_out, void *stream) {
  if (!plan || plan->device < 0) return ATTN_ERR_INVALID_ARG;
  // the split partials must fit; a prefill plan's K/V staging scratch is not
  // used here (its prefill kernel then reads the paged caches itself)
  if (plan->host.partial_bytes > (size_t)ATTN_NO_WORKSPACE_MAX_BYTES) return ATTN_ERR_WORKSPACE;
  void *scratch = nullptr;
  const attn_status_t st = scratch_address(plan->device, &scratch);
  if (st != ATTN_OK) return st;
  // Nothing in the scratch has to start at zero: every partial the merge reads
  // is written earlier in the same call, so the previous call's leftovers are
  // never used.
  return akp::run_paged_unstaged(plan, q, k_cache, v_cache, page_table, seq_lens, qo_indptr, sinks,
                                 window, softmax_scale, k_scale, v_scale, out, lse_out, scratch,
                                 (size_t)ATTN_NO_WORKSPACE_MAX_BYTES, stream);
}
