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

// Fold splits [0, S) of one row into (M, Z, acc), kB splits per step (see
// merge_kernel).
template <int kB>
__device__ __forceinline__ void combine(const RunArgs &a, int base, int nrows, int S, int lane,
                                        float &M, float &Z, float4 &acc) {
  for (int s0 = 0; s0 < S; s0 += kB) {
    float ls[kB];
    float4 v[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      ls[u] = -INFINITY;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s0 + u < S) {      // no load at all for splits past the row's last
        const int prow = base + (s0 + u) * nrows;
        ls[u] = __ldcg(a.part_lse + prow);
        v[u] = __ldcg(reinterpret_cast<const float4 *>(a.part_o + (int64_t)prow * kDv) + lane);
      }
    }
    float Mn = M;
#pragma unroll
    for (int u = 0; u < kB; ++u) Mn = fmaxf(Mn, ls[u]);
    if (Mn == -INFINITY) continue;          // nothing seen yet
    if (M != -INFINITY) {
      const float c = exp2f(M - Mn);
      Z *= c;
      acc.x *= c;
      acc.y *= c;
      acc.z *= c;
      acc.w *= c;
    }
    M = Mn;
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      if (ls[u] == -INFINITY) continue;
      const float w = exp2f(ls[u] - M);
      Z += w;
      acc.x += w * v[u].x;
      acc.y += w * v[u].y;
      acc.z += w * v[u].z;
      acc.w += w * v[u].w;
    }
  }
}

// Launched as a programmatic dependent of the attention kernel: everything
// that kernel does not write (the item, the block, the sink) is read before
// griddepcontrol.wait, so that part overlaps the attention kernel's tail; the
// partials are read after it, all splits' loads issued before any is used.
__global__ void __launch_bounds__(32 * kMergeRowsPerCta, 3) merge_kernel(const RunArgs a) {
  const MergeItem it = a.merge_items[blockIdx.x];
  const BlockDesc bd = a.blocks[it.block];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = it.row_begin + warp;
  const bool live = r < bd.nrows;
  const int flat = bd.row0 + (live ? r : 0);
  const int tok = bd.tok0 + flat / a.group;
  const int h = bd.g * a.group + flat % a.group;
  const float sig = (a.sinks && live) ? a.sinks[h] * kLog2e : -INFINITY;
  // Every CTA waits, also those with nothing to do: this grid's completion
  // then implies the attention kernel's, for a dependent launched after it.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (bd.num_splits <= 1 || !live) return;   // a replayable plan's run may leave the block whole
  const int S = bd.num_splits;
  const int base = bd.part_row_base + r;
  // One pass over the splits against a running maximum M (base 2), kB splits
  // per step with all their loads issued before any is used: every step is
  // one round trip to L2 (the maximum is not taken in a pass of its own).  The
  // sink enters as a split with no value row.  Rows of at most 4 splits (the
  // usual case) take a 4-wide step, longer ones (verify blocks cut over many
  // CTAs) an 8-wide one; the register count stays low enough for three CTAs of
  // eight warps per SM.
  float M = sig, Z = sig == -INFINITY ? 0.f : 1.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (S <= 4)
    combine<4>(a, base, bd.nrows, S, lane, M, Z, acc);
  else
    combine<8>(a, base, bd.nrows, S, lane, M, Z, acc);
  float lse = -INFINITY;
  if (M != -INFINITY) {
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
