// Log-sum-exp merge of split-KV partials.
//
// Each split s of a row left o_s (normalised by its own denominator, already
// multiplied by v_scale) and lse_s = m_s + log2(l_s) in base 2 (-inf when the
// split saw no key).  With the sink sigma (base-2 units) the row is
//   M = max(sigma, max_s lse_s),  w_s = 2^(lse_s - M),
//   Z = sum_s w_s + 2^(sigma - M),  out = sum_s w_s o_s / Z,
//   lse = (M + log2 Z) * ln 2.
// Split-KV for verify is the fix the MiMo-V2.6-Flash-RL model card describes
// ("What the kernels do"); the combine is the standard one for softmax partials.
// One warp per row, four value columns per lane.
#include <cuda_bf16.h>

#include <cmath>

#include "kernels.hpp"

namespace akp {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Launched as a programmatic dependent of the attention kernel: everything
// that kernel does not write (the item, the block, the sink) is read before
// griddepcontrol.wait, so that part overlaps the attention kernel's tail; the
// partials are read after it, all splits' loads issued before any is used.
__global__ void __launch_bounds__(32 * kMergeRowsPerCta) merge_kernel(const RunArgs a) {
  const MergeItem it = a.merge_items[blockIdx.x];
  const BlockDesc bd = a.blocks[it.block];
  if (bd.num_splits <= 1) return;   // a replayable plan's run left the block whole
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = it.row_begin + warp;
  const bool live = r < bd.nrows;
  const int flat = bd.row0 + (live ? r : 0);
  const int tok = bd.tok0 + flat / a.group;
  const int h = bd.g * a.group + flat % a.group;
  const float sig = (a.sinks && live) ? a.sinks[h] * kLog2e : -INFINITY;
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (!live) return;
  const int S = bd.num_splits;
  const int base = bd.part_row_base + r;
  float M = sig;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, __ldcg(a.part_lse + base + s * bd.nrows));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float Z = 0.f, lse = -INFINITY;
  if (M != -INFINITY) {
    Z = exp2f(sig - M);
    // four splits per step: their loads are independent and go out together
    for (int s0 = 0; s0 < S; s0 += 4) {
      float ls[4];
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int prow = base + min(s0 + u, S - 1) * bd.nrows;
        ls[u] = __ldcg(a.part_lse + prow);
        v[u] = __ldcg(reinterpret_cast<const float4 *>(a.part_o + (int64_t)prow * kDv) + lane);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (s0 + u >= S || ls[u] == -INFINITY) continue;
        const float w = exp2f(ls[u] - M);
        Z += w;
        acc.x += w * v[u].x;
        acc.y += w * v[u].y;
        acc.z += w * v[u].z;
        acc.w += w * v[u].w;
      }
    }
    const float inv = 1.f / Z;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    lse = (M + log2f(Z)) * kLn2;
  }
  __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(
      static_cast<uint16_t *>(a.out) + ((int64_t)tok * a.hq + h) * kDv + lane * 4);
  dst[0] = __floats2bfloat162_rn(acc.x, acc.y);
  dst[1] = __floats2bfloat162_rn(acc.z, acc.w);
  if (a.lse_out && lane == 0) a.lse_out[(int64_t)tok * a.hq + h] = lse;
}

}  // namespace

cudaError_t launch_merge(const HostPlan &hp, const RunArgs &a, cudaStream_t stream) {
  if (hp.merge_items.empty()) return cudaSuccess;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)hp.merge_items.size());
  cfg.blockDim = dim3(32 * kMergeRowsPerCta);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel, a);
}

}  // namespace akp
