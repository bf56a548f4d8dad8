// C ABI of the paged-attention library (declared in include/attn_paged.h).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <algorithm>
#include <new>
#include <vector>

#include "attn_paged.h"
#include "kernels.hpp"
#include "plan.hpp"
#include "replan.hpp"

namespace {

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess) ok = true;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// cuTensorMapEncodeTiled from the driver, reached through the runtime so the
// library does not link libcuda directly.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// K (d = 192 or 128) or V (d = 128) cache as a 3D tensor [slots][Hkv][d]; boxes of
// `rows` consecutive slots of one head: 64 bf16 columns with 128-byte swizzle
// (the tensor-core operand layout), or whole raw E4M3 rows without swizzle.
bool make_cache_map(CUtensorMap *map, const void *base, bool fp8, int d, int hkv, int64_t slots,
                    int rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t es = fp8 ? 1 : 2;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hkv, (cuuint64_t)slots};
  const cuuint64_t strides[2] = {d * es, (cuuint64_t)hkv * d * es};
  const cuuint32_t box[3] = {fp8 ? (cuuint32_t)d : 64u, 1u, (cuuint32_t)rows};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                  // 128-byte promotion: a 256-byte one pulls in part of the neighbouring
                  // head's K row (rows are 384 bytes at offset g * 384), which measured
                  // 2% slower on the batched decode
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Staging scratch of prefill plans (K: d = 192, V: d = 128 16-bit values a
// row) as a 2D tensor [rows][d]: boxes of 64 columns x 128 rows (one key tile
// of one 64-column operand block) with 128-byte swizzle.
bool make_stage_map(CUtensorMap *map, const void *base, bool f16, int d, int64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)akp::kStageTile};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

void free_device(attn_plan_s *p) {
  if (p->dev.blocks) cudaFree(p->dev.blocks);
  p->dev = akp::DevicePlan{};
}

attn_status_t upload(attn_plan_s *p) {
  const akp::HostPlan &hp = p->host;
  const size_t nsegs = std::max<size_t>(hp.segs.size(), (size_t)hp.seg_capacity);
  const size_t b_bytes = align256(hp.blocks.size() * sizeof(akp::BlockDesc));
  const size_t s_bytes = align256(nsegs * sizeof(akp::SegDesc));
  const size_t c_bytes = align256(hp.cta_seg_begin.size() * sizeof(int32_t));
  const size_t h_bytes = align256(hp.cta_heads.size() * sizeof(akp::CtaHead));
  const size_t m_bytes = align256(hp.merge_items.size() * sizeof(akp::MergeItem));
  const size_t u_bytes = align256(hp.stage_units.size() * sizeof(akp::StageUnit));
  const size_t e_bytes = 256;
  // replayable plans: the length bounds and two scratch arrays of the planner
  const size_t r_bytes = hp.replayable ? align256(hp.seq_lens.size() * sizeof(int32_t)) +
                                             2 * align256((hp.blocks.size() + 1) * sizeof(int32_t))
                                       : 0;
  const size_t total = b_bytes + s_bytes + c_bytes + m_bytes + e_bytes + r_bytes + h_bytes + u_bytes;
  uint8_t *base = nullptr;
  if (cudaMalloc(&base, total) != cudaSuccess) return ATTN_ERR_CUDA;
  p->dev.blocks = reinterpret_cast<akp::BlockDesc *>(base);
  p->dev.segs = reinterpret_cast<akp::SegDesc *>(base + b_bytes);
  p->dev.cta_seg_begin = reinterpret_cast<int32_t *>(base + b_bytes + s_bytes);
  p->dev.merge_items = reinterpret_cast<akp::MergeItem *>(base + b_bytes + s_bytes + c_bytes);
  p->dev.err = reinterpret_cast<int32_t *>(base + b_bytes + s_bytes + c_bytes + m_bytes);
  p->dev.cta_heads =
      reinterpret_cast<akp::CtaHead *>(base + b_bytes + s_bytes + c_bytes + m_bytes + e_bytes + r_bytes);
  if (!hp.stage_units.empty())
    p->dev.stage_units = reinterpret_cast<akp::StageUnit *>(base + b_bytes + s_bytes + c_bytes +
                                                            m_bytes + e_bytes + r_bytes + h_bytes);
  if (hp.replayable) {
    uint8_t *r = base + b_bytes + s_bytes + c_bytes + m_bytes + e_bytes;
    p->dev.seq_bounds = reinterpret_cast<int32_t *>(r);
    r += align256(hp.seq_lens.size() * sizeof(int32_t));
    p->dev.tile_start = reinterpret_cast<int32_t *>(r);
    r += align256((hp.blocks.size() + 1) * sizeof(int32_t));
    p->dev.part_start = reinterpret_cast<int32_t *>(r);
  }
  cudaError_t e = cudaSuccess;
  if (!hp.blocks.empty())
    e = cudaMemcpy(p->dev.blocks, hp.blocks.data(), hp.blocks.size() * sizeof(akp::BlockDesc),
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !hp.segs.empty())
    e = cudaMemcpy(p->dev.segs, hp.segs.data(), hp.segs.size() * sizeof(akp::SegDesc),
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(p->dev.cta_seg_begin, hp.cta_seg_begin.data(),
                   hp.cta_seg_begin.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !hp.cta_heads.empty())
    e = cudaMemcpy(p->dev.cta_heads, hp.cta_heads.data(), hp.cta_heads.size() * sizeof(akp::CtaHead),
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !hp.merge_items.empty())
    e = cudaMemcpy(p->dev.merge_items, hp.merge_items.data(),
                   hp.merge_items.size() * sizeof(akp::MergeItem), cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !hp.stage_units.empty())
    e = cudaMemcpy(p->dev.stage_units, hp.stage_units.data(),
                   hp.stage_units.size() * sizeof(akp::StageUnit), cudaMemcpyHostToDevice);
  if (e == cudaSuccess && hp.replayable && !hp.seq_lens.empty())
    e = cudaMemcpy(p->dev.seq_bounds, hp.seq_lens.data(), hp.seq_lens.size() * sizeof(int32_t),
                   cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(p->dev.err, 0, e_bytes);
  if (e == cudaSuccess) e = hp.prefill ? akp::prepare_attn_prefill(hp) : akp::prepare_attn_tc(hp);
  if (e != cudaSuccess) {
    free_device(p);
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

}  // namespace

extern "C" {

static attn_status_t plan_host(const attn_problem_t *problem, int32_t num_sms, bool replayable,
                               attn_plan_t *plan) {
  if (!plan) return ATTN_ERR_INVALID_ARG;
  *plan = nullptr;
  if (!problem) return ATTN_ERR_INVALID_ARG;
  attn_plan_s *p = new (std::nothrow) attn_plan_s();
  if (!p) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = replayable ? akp::build_replayable_plan(problem, num_sms, &p->host)
                                : akp::build_host_plan(problem, num_sms, &p->host);
  if (st != ATTN_OK) {
    delete p;
    return st;
  }
  p->host.use_tma = akp::tc_tma_page_size(problem->page_size, problem->num_pages);
  *plan = p;
  return ATTN_OK;
}

static attn_status_t plan_device(const attn_problem_t *problem, int device, bool replayable,
                                 attn_plan_t *plan, size_t *workspace_bytes) {
  if (!plan) return ATTN_ERR_INVALID_ARG;
  *plan = nullptr;
  if (!problem || !workspace_bytes || device < 0) return ATTN_ERR_INVALID_ARG;
  DeviceGuard guard(device);
  if (!guard.ok) return ATTN_ERR_CUDA;
  int num_sms = 0;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return ATTN_ERR_CUDA;
  attn_plan_t p = nullptr;
  attn_status_t st = plan_host(problem, num_sms, replayable, &p);
  if (st != ATTN_OK) return st;
  p->device = device;
  st = upload(p);
  if (st != ATTN_OK) {
    delete p;
    return st;
  }
  *workspace_bytes = p->host.workspace_bytes;
  *plan = p;
  return ATTN_OK;
}

attn_status_t attn_plan_host(const attn_problem_t *problem, int32_t num_sms, attn_plan_t *plan) {
  return plan_host(problem, num_sms, false, plan);
}

attn_status_t attn_plan_replayable_host(const attn_problem_t *bounds, int32_t num_sms,
                                        attn_plan_t *plan) {
  return plan_host(bounds, num_sms, true, plan);
}

attn_status_t attn_plan(const attn_problem_t *problem, int device, attn_plan_t *plan,
                        size_t *workspace_bytes) {
  return plan_device(problem, device, false, plan, workspace_bytes);
}

attn_status_t attn_plan_replayable(const attn_problem_t *bounds, int device, attn_plan_t *plan,
                                   size_t *workspace_bytes) {
  return plan_device(bounds, device, true, plan, workspace_bytes);
}

attn_status_t attn_plan_destroy(attn_plan_t plan) {
  if (!plan) return ATTN_OK;
  if (plan->device >= 0) {
    DeviceGuard guard(plan->device);
    cudaDeviceSynchronize();
    free_device(plan);
  }
  delete plan;
  return ATTN_OK;
}

// allow_stage: a prefill plan's K/V staging scratch follows the partials in
// the workspace; without it (the library-owned scratch of the no-workspace
// entry point holds the partials only) the prefill kernel reads the caches.
static attn_status_t run_impl(attn_plan_t plan, int phases, bool allow_stage, const void *q,
                              const void *k_cache,
                              const void *v_cache, const int32_t *page_table,
                              const int32_t *seq_lens, const int32_t *qo_indptr,
                              const float *sinks, int32_t window, float softmax_scale,
                              float k_scale, float v_scale, void *out, float *lse_out,
                              void *workspace, size_t workspace_bytes, void *stream) {
  if (!plan || plan->device < 0) return ATTN_ERR_INVALID_ARG;
  const akp::HostPlan &hp = plan->host;
  const attn_problem_t &pr = hp.prob;
  const bool has_rows = hp.qo_indptr.back() > 0;
  if (has_rows && (!q || !k_cache || !v_cache || !page_table || !seq_lens || !qo_indptr || !out))
    return ATTN_ERR_INVALID_ARG;
  if (window != pr.window) return ATTN_ERR_INVALID_ARG;
  if ((sinks != nullptr) != (pr.has_sinks != 0)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return ATTN_ERR_INVALID_ARG;
  // the kernels take score maxima on unscaled dot products: the scale must be > 0
  if (!(softmax_scale > 0.f) || (pr.kv_dtype == ATTN_KV_FP8_E4M3 && !(k_scale > 0.f)))
    return ATTN_ERR_INVALID_ARG;
  const bool staged = allow_stage && hp.stage_rows > 0;
  const size_t need = staged ? hp.workspace_bytes : hp.partial_bytes;
  if (workspace_bytes < need || (need && !workspace)) return ATTN_ERR_WORKSPACE;
  if (!has_rows) return ATTN_OK;

  const bool fp8 = pr.kv_dtype == ATTN_KV_FP8_E4M3;
  akp::RunArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.page_table = page_table;
  a.sinks = sinks;
  a.scale_log2 = softmax_scale * (fp8 ? k_scale : 1.f) * 1.4426950408889634f;
  a.v_scale = fp8 ? v_scale : 1.f;
  a.out = out;
  a.lse_out = lse_out;
  a.part_o = static_cast<float *>(workspace);
  a.part_lse = hp.part_rows ? reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                                        akp::part_o_bytes(hp.part_rows))
                            : nullptr;
  a.blocks = plan->dev.blocks;
  a.segs = plan->dev.segs;
  a.cta_seg_begin = plan->dev.cta_seg_begin;
  a.cta_heads = plan->dev.cta_heads;
  a.merge_items = plan->dev.merge_items;
  a.hq = pr.num_q_heads;
  a.hkv = pr.num_kv_heads;
  a.group = hp.group;
  a.page_size = pr.page_size;
  a.pt_stride = pr.page_table_stride;
  a.num_pages = pr.num_pages;
  a.window = pr.window;
  a.err = plan->dev.err;

  akp::TmaMaps maps{};
  if ((phases & 1) && hp.use_tma && !hp.prefill) {
    if ((reinterpret_cast<uintptr_t>(k_cache) & 15) || (reinterpret_cast<uintptr_t>(v_cache) & 15))
      return ATTN_ERR_INVALID_ARG;
    const int64_t slots = (int64_t)pr.num_pages * pr.page_size;
    const int rows = pr.page_size >= akp::kKeyTile ? akp::kKeyTile : pr.page_size;
    if (!make_cache_map(&maps.k, k_cache, fp8, pr.head_dim_qk, pr.num_kv_heads, slots, rows) ||
        !make_cache_map(&maps.v, v_cache, fp8, akp::kDv, pr.num_kv_heads, slots, rows))
      return ATTN_ERR_CUDA;
  }
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return ATTN_ERR_CUDA;
  DeviceGuard guard(cur == plan->device ? cur : plan->device);
  if (!guard.ok) return ATTN_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((phases & 1) && hp.replayable) {
    akp::ReplanArgs r{};
    r.blocks = plan->dev.blocks;
    r.segs = plan->dev.segs;
    r.cta_seg_begin = plan->dev.cta_seg_begin;
    r.cta_heads = plan->dev.cta_heads;
    r.tile_start = plan->dev.tile_start;
    r.part_start = plan->dev.part_start;
    r.seq_lens = seq_lens;
    r.seq_bounds = plan->dev.seq_bounds;
    r.err = plan->dev.err;
    r.nb = (int32_t)hp.blocks.size();
    r.num_ctas = hp.num_ctas;
    r.group = hp.group;
    r.window = pr.window;
    r.key_tile = hp.key_tile;
    if (akp::launch_replan(r, st) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  akp::TmaMaps stage_maps{};
  if ((phases & 1) && staged) {
    uint8_t *ws = static_cast<uint8_t *>(workspace) + hp.partial_bytes;
    akp::StageArgs sa{};
    sa.units = plan->dev.stage_units;
    sa.k_cache = k_cache;
    sa.v_cache = v_cache;
    sa.page_table = page_table;
    sa.k_stage = reinterpret_cast<uint16_t *>(ws);
    sa.v_stage = reinterpret_cast<uint16_t *>(ws + akp::stage_k_bytes(hp.stage_rows, pr.head_dim_qk));
    sa.err = plan->dev.err;
    sa.tiles = hp.stage_tiles;
    sa.num_units = (int32_t)hp.stage_units.size();
    sa.dqk = pr.head_dim_qk;
    sa.hkv = pr.num_kv_heads;
    sa.page_size = pr.page_size;
    sa.pt_stride = pr.page_table_stride;
    sa.num_pages = pr.num_pages;
    sa.fp8 = fp8;
    if ((reinterpret_cast<uintptr_t>(ws) & 255) ||
        !make_stage_map(&stage_maps.k, sa.k_stage, fp8, pr.head_dim_qk, hp.stage_rows) ||
        !make_stage_map(&stage_maps.v, sa.v_stage, fp8, akp::kDv, hp.stage_rows))
      return ATTN_ERR_CUDA;
    if (akp::launch_kv_stage(sa, st) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (phases & 1) {
    const cudaError_t le = hp.prefill ? akp::launch_attn_prefill(hp, a, staged ? &stage_maps : nullptr, st)
                                      : akp::launch_attn_tc(hp, a, maps, st);
    if (le != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if ((phases & 2) && akp::launch_merge(hp, a, st) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status_t attn_run_paged(attn_plan_t plan, const void *q, const void *k_cache,
                             const void *v_cache, const int32_t *page_table,
                             const int32_t *seq_lens, const int32_t *qo_indptr,
                             const float *sinks, int32_t window, float softmax_scale,
                             float k_scale, float v_scale, void *out, float *lse_out,
                             void *workspace, size_t workspace_bytes, void *stream) {
  return run_impl(plan, 3, true, q, k_cache, v_cache, page_table, seq_lens, qo_indptr, sinks, window,
                  softmax_scale, k_scale, v_scale, out, lse_out, workspace, workspace_bytes,
                  stream);
}

attn_status_t attn_run_phase(attn_plan_t plan, int32_t phase, const void *q,
                             const void *k_cache, const void *v_cache,
                             const int32_t *page_table, const int32_t *seq_lens,
                             const int32_t *qo_indptr, const float *sinks, int32_t window,
                             float softmax_scale, float k_scale, float v_scale, void *out,
                             float *lse_out, void *workspace, size_t workspace_bytes,
                             void *stream) {
  if (phase != 0 && phase != 1) return ATTN_ERR_INVALID_ARG;
  return run_impl(plan, phase == 0 ? 1 : 2, true, q, k_cache, v_cache, page_table, seq_lens,
                  qo_indptr, sinks, window, softmax_scale, k_scale, v_scale, out, lse_out,
                  workspace, workspace_bytes, stream);
}

attn_status_t attn_get_device_error(attn_plan_t plan, void *workspace, int32_t *err) {
  (void)workspace;
  if (!plan || !err || plan->device < 0) return ATTN_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return ATTN_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, plan->dev.err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaMemset(plan->dev.err, 0, sizeof v) != cudaSuccess) return ATTN_ERR_CUDA;
  *err = v;
  return ATTN_OK;
}

const char *attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported problem";
    case ATTN_ERR_WORKSPACE: return "workspace too small";
    case ATTN_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

attn_status_t attn_plan_info(attn_plan_t plan, int32_t info[8]) {
  if (!plan || !info) return ATTN_ERR_INVALID_ARG;
  const akp::HostPlan &hp = plan->host;
  info[0] = (int32_t)hp.blocks.size();
  info[1] = (int32_t)hp.segs.size();
  info[2] = hp.num_ctas;
  info[3] = hp.block_rows;
  info[4] = hp.key_tile;
  info[5] = hp.multi_split_blocks;
  info[6] = (int32_t)(hp.workspace_bytes & 0x7FFFFFFF);
  info[7] = (int32_t)(hp.workspace_bytes >> 31);
  return ATTN_OK;
}

attn_status_t attn_plan_blocks(attn_plan_t plan, int32_t *blocks_host) {
  if (!plan || (!blocks_host && !plan->host.blocks.empty())) return ATTN_ERR_INVALID_ARG;
  int32_t *d = blocks_host;
  for (const akp::BlockDesc &b : plan->host.blocks) {
    const int32_t v[8] = {b.b, b.g, b.row0, b.nrows, b.klo, b.khi, b.num_splits, b.part_row_base};
    std::memcpy(d, v, sizeof v);
    d += 8;
  }
  return ATTN_OK;
}

attn_status_t attn_plan_replan_host(attn_plan_t plan, const int32_t *seq_lens_host,
                                   int32_t *err) {
  if (!plan || !plan->host.replayable || !err) return ATTN_ERR_INVALID_ARG;
  if (!seq_lens_host && !plan->host.seq_lens.empty()) return ATTN_ERR_INVALID_ARG;
  *err = akp::replan_host(&plan->host, seq_lens_host);
  return ATTN_OK;
}

attn_status_t attn_plan_fetch_device(attn_plan_t plan) {
  if (!plan || !plan->host.replayable || plan->device < 0) return ATTN_ERR_INVALID_ARG;
  akp::HostPlan &hp = plan->host;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return ATTN_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  std::vector<akp::BlockDesc> blocks(hp.blocks.size());
  std::vector<int32_t> begin(hp.cta_seg_begin.size());
  if (!blocks.empty() &&
      cudaMemcpy(blocks.data(), plan->dev.blocks, blocks.size() * sizeof(akp::BlockDesc),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaMemcpy(begin.data(), plan->dev.cta_seg_begin, begin.size() * sizeof(int32_t),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const int32_t nsegs = begin.back();
  if (nsegs < 0 || nsegs > hp.seg_capacity) return ATTN_ERR_CUDA;
  std::vector<akp::SegDesc> segs(nsegs);
  if (nsegs > 0 && cudaMemcpy(segs.data(), plan->dev.segs, segs.size() * sizeof(akp::SegDesc),
                              cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  std::vector<int32_t> seg_cta(nsegs);
  for (int32_t c = 0; c + 1 < (int32_t)begin.size(); ++c)
    for (int32_t s = begin[c]; s < begin[c + 1] && s < nsegs; ++s) seg_cta[s] = c;
  hp.multi_split_blocks = 0;
  for (const akp::BlockDesc &b : blocks) hp.multi_split_blocks += b.num_splits > 1;
  std::vector<akp::CtaHead> heads(hp.cta_heads.size());
  if (!heads.empty() &&
      cudaMemcpy(heads.data(), plan->dev.cta_heads, heads.size() * sizeof(akp::CtaHead),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  hp.blocks = std::move(blocks);
  hp.cta_heads = std::move(heads);
  hp.cta_seg_begin = std::move(begin);
  hp.segs = std::move(segs);
  hp.seg_cta = std::move(seg_cta);
  return ATTN_OK;
}

attn_status_t attn_plan_cta_heads(attn_plan_t plan, int32_t *heads_host) {
  if (!plan || (!heads_host && !plan->host.cta_heads.empty())) return ATTN_ERR_INVALID_ARG;
  if (!plan->host.cta_heads.empty())
    std::memcpy(heads_host, plan->host.cta_heads.data(),
                plan->host.cta_heads.size() * sizeof(akp::CtaHead));
  return ATTN_OK;
}

attn_status_t attn_plan_merge_ctas(attn_plan_t plan, int32_t *ctas) {
  if (!plan || !ctas) return ATTN_ERR_INVALID_ARG;
  *ctas = (int32_t)plan->host.merge_items.size();
  return ATTN_OK;
}

attn_status_t attn_plan_stage_units(attn_plan_t plan, int32_t *count, int32_t *units_host) {
  if (!plan || !count) return ATTN_ERR_INVALID_ARG;
  const std::vector<akp::StageUnit> &u = plan->host.stage_units;
  *count = (int32_t)u.size();
  if (units_host && !u.empty()) std::memcpy(units_host, u.data(), u.size() * sizeof(akp::StageUnit));
  return ATTN_OK;
}

attn_status_t attn_plan_segments(attn_plan_t plan, int32_t *segments_host) {
  if (!plan || (!segments_host && !plan->host.segs.empty())) return ATTN_ERR_INVALID_ARG;
  int32_t *d = segments_host;
  for (size_t i = 0; i < plan->host.segs.size(); ++i) {
    const akp::SegDesc &s = plan->host.segs[i];
    const int32_t v[5] = {plan->host.seg_cta[i], s.block, s.tile_begin, s.tile_end, s.split};
    std::memcpy(d, v, sizeof v);
    d += 5;
  }
  return ATTN_OK;
}

}  // extern "C"

namespace akp {
attn_status_t run_paged_unstaged(attn_plan_t plan, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *page_table,
                                 const int32_t *seq_lens, const int32_t *qo_indptr,
                                 const float *sinks, int32_t window, float softmax_scale,
                                 float k_scale, float v_scale, void *out, float *lse_out,
                                 void *workspace, size_t workspace_bytes, void *stream) {
  return run_impl(plan, 3, false, q, k_cache, v_cache, page_table, seq_lens, qo_indptr, sinks,
                  window, softmax_scale, k_scale, v_scale, out, lse_out, workspace,
                  workspace_bytes, stream);
}
}  // namespace akp
