// Kernel launch interfaces (internal).
#pragma once
#include <cuda_runtime.h>

#include "plan.hpp"

namespace akp {

struct RunArgs {
  const void *q;
  const void *k_cache;
  const void *v_cache;
  const int32_t *page_table;
  const float *sinks;
  float scale_log2;  // softmax_scale * k_scale * log2(e)
  float v_scale;     // applied to every output (1 for bf16 caches)
  void *out;
  float *lse_out;
  float *part_o;
  float *part_lse;
  const BlockDesc *blocks;
  const SegDesc *segs;
  const int32_t *cta_seg_begin;
  const MergeItem *merge_items;
  int32_t hq, hkv, group, page_size, pt_stride, num_pages, window;
  int32_t *err;
};

// Split-KV attention over the plan's segments (decode, verify and prefill).
cudaError_t launch_split_kv(const HostPlan &hp, const RunArgs &a, cudaStream_t stream);
// Log-sum-exp merge of multi-split blocks.
cudaError_t launch_merge(const HostPlan &hp, const RunArgs &a, cudaStream_t stream);
// One-time per-device kernel attributes (dynamic shared memory limits).
cudaError_t prepare_kernels(const HostPlan &hp);
// Tensor-core (tcgen05) kernel for 128-row blocks.
cudaError_t launch_prefill_tc(const HostPlan &hp, const RunArgs &a, cudaStream_t stream);
cudaError_t prepare_prefill_tc(const HostPlan &hp);

}  // namespace akp
