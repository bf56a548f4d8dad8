// Kernel launch interfaces (internal).
#pragma once
#include <cuda.h>
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
  const CtaHead *cta_heads;
  const MergeItem *merge_items;
  int32_t hq, hkv, group, page_size, pt_stride, num_pages, window;
  int32_t *err;
};

// Launch `kernel` as a programmatic dependent of the stream's previous kernel:
// its CTAs may be scheduled while that kernel finishes (the launch latency is
// hidden), and the kernel itself waits (griddepcontrol.wait) before it reads
// anything an earlier kernel of the stream writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Tensor maps of the K and V caches as 3D tensors [slots][Hkv][D] (TMA loads).
struct TmaMaps {
  CUtensorMap k, v;
};

// Staging pass of prefill plans (kv_stage.cu): the keys of every StageUnit
// gathered into 16-bit scratch rows (k_stage: dqk values a row, v_stage: kDv).
struct StageArgs {
  const StageUnit *units;
  const void *k_cache, *v_cache;
  const int32_t *page_table;
  uint16_t *k_stage, *v_stage;
  int32_t *err;
  int64_t tiles;             // all units' tiles
  int32_t num_units, dqk, hkv, page_size, pt_stride, num_pages;
  bool fp8;
};
cudaError_t launch_kv_stage(const StageArgs &a, cudaStream_t stream);

// Split-KV attention over the plan's segments (decode, verify and prefill) on
// the tcgen05 tensor-core path.  `maps` is read only when hp.use_tma.
cudaError_t launch_attn_tc(const HostPlan &hp, const RunArgs &a, const TmaMaps &maps,
                           cudaStream_t stream);
// One-time per-device kernel attributes (dynamic shared memory limits).
cudaError_t prepare_attn_tc(const HostPlan &hp);
// Prefill plans (hp.prefill: 256-row blocks, 128-key tiles): attn_prefill.cu.
// With `stage` (2D maps of the staged K and V rows, boxes of 64 columns x 128
// rows) the K/V tiles are TMA loads from the staging scratch; without it the
// kernel's load warps read the paged caches themselves.
cudaError_t launch_attn_prefill(const HostPlan &hp, const RunArgs &a, const TmaMaps *stage,
                                cudaStream_t stream);
cudaError_t prepare_attn_prefill(const HostPlan &hp);
// Whether K/V tiles of this page size can be loaded as TMA boxes.
bool tc_tma_page_size(int32_t page_size, int32_t num_pages);
// Device planner of replayable plans (replan.cu): rewrites the work list
// from the run's lengths; launched before the attention kernel.
struct ReplanArgs;
cudaError_t launch_replan(const ReplanArgs &r, cudaStream_t stream);
// attn_run_paged without a prefill plan's staging scratch: the workspace
// holds the split partials only (api.cu; used by the no-workspace entry).
attn_status_t run_paged_unstaged(attn_plan_t plan, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *page_table,
                                 const int32_t *seq_lens, const int32_t *qo_indptr,
                                 const float *sinks, int32_t window, float softmax_scale,
                                 float k_scale, float v_scale, void *out, float *lse_out,
                                 void *workspace, size_t workspace_bytes, void *stream);
// Log-sum-exp merge of multi-split blocks.
cudaError_t launch_merge(const HostPlan &hp, const RunArgs &a, cudaStream_t stream);

}  // namespace akp
