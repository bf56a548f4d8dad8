// Staging pass of prefill plans: the keys that a call's prefill blocks read
// are gathered from the paged caches once, into a scratch of 16-bit rows in
// the workspace, so that the prefill kernel loads each 128-key tile of K and
// V as whole TMA boxes instead of looking pages up and widening E4M3 codes in
// every one of the (up to hundreds of) row blocks that share a KV head.
//
// Unit u (one (request, KV head), see StageUnit) owns scratch rows
// [row_base, row_base + 128 * tiles) for keys [j0, j0 + 128 * tiles).  A key
// in [klo, khi) is read from its page (page_table[b][j / P], offset j % P;
// the paged layout of the MiMo-V2.6-Flash-RL model card, "What the kernels
// do"): BF16 rows are copied bit for bit, E4M3 codes are widened exactly to
// fp16 (every E4M3 value is an fp16 value; the scale stays outside, as in the
// attention kernels).  Keys outside [klo, khi) are written as zeros: the
// kernel masks them, and zeros keep P.V free of whatever the pool holds
// there.  A page id outside the pool is read as zeros and reported in bit 1
// of the plan's error word, as the attention kernels do.
//
// One CTA per 128-key tile (grid-stride): the tile's page lookups first (one
// thread per key, into shared memory), then one thread per 16-byte source
// chunk, consecutive threads on consecutive chunks of a row.  The pass reads
// every staged key once and writes its 16-bit row once (HBM/L2-bound; tens of
// microseconds for a 4096-token chunk over 26K cached keys).
#include <cuda_runtime.h>

#include <cstdint>

#include "e4m3.cuh"
#include "kernels.hpp"

namespace akp {
namespace {

constexpr int kStageThreads = 256;

template <bool FP8>
__global__ void __launch_bounds__(kStageThreads) stage_kernel(const StageArgs a) {
  // Launched as a programmatic dependent of the stream's previous kernel (a
  // KV append writes the caches read here): wait for it before reading them.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  // The prefill kernel may be scheduled now; it waits for this grid's
  // completion before it reads the scratch.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  __shared__ int64_t s_slot[kStageTile];
  __shared__ StageUnit s_unit;
  // 16-byte chunks of a source row: E4M3 rows hold 16 codes per chunk, BF16 8 values
  constexpr int kCodes = FP8 ? 16 : 8;
  const int kch = a.dqk / kCodes, vch = kDv / kCodes;
  const int chunks = kch + vch;
  const uint8_t *kc = static_cast<const uint8_t *>(a.k_cache);
  const uint8_t *vc = static_cast<const uint8_t *>(a.v_cache);
  constexpr int kEs = FP8 ? 1 : 2;
  for (int64_t t = blockIdx.x; t < a.tiles; t += gridDim.x) {
    if (threadIdx.x == 0) {
      // the unit of tile t: the last one with tile_off <= t
      int lo = 0, hi = a.num_units - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.units[mid].tile_off <= t) lo = mid; else hi = mid - 1;
      }
      s_unit = a.units[lo];
    }
    __syncthreads();
    const StageUnit u = s_unit;
    const int ti = (int)(t - u.tile_off);
    const int key0 = u.j0 + ti * kStageTile;
    const int64_t row0 = (int64_t)u.row_base + (int64_t)ti * kStageTile;
    if (threadIdx.x < kStageTile) {
      const int j = key0 + threadIdx.x;
      int64_t slot = -1;
      if (j >= u.klo && j < u.khi) {
        const int32_t page = __ldg(a.page_table + (int64_t)u.b * a.pt_stride + j / a.page_size);
        if (page >= 0 && page < a.num_pages)
          slot = (int64_t)page * a.page_size + j % a.page_size;
        else
          atomicOr(a.err, 1);
      }
      s_slot[threadIdx.x] = slot;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kStageTile * chunks; i += kStageThreads) {
      const int key = i / chunks, c = i % chunks;
      const bool is_k = c < kch;
      const int cc = is_k ? c : c - kch;
      const int d = is_k ? a.dqk : kDv;
      const int64_t slot = s_slot[key];
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (slot >= 0)
        raw = __ldg(reinterpret_cast<const uint4 *>((is_k ? kc : vc) +
                                                    (slot * a.hkv + u.g) * (int64_t)(d * kEs)) +
                    cc);
      uint4 *dst = reinterpret_cast<uint4 *>((is_k ? a.k_stage : a.v_stage) + (row0 + key) * d);
      if (FP8) {
        uint4 lo, hi;
        e4m3x16_to_f16(raw, lo, hi);
        dst[2 * cc] = lo;
        dst[2 * cc + 1] = hi;
      } else {
        dst[cc] = raw;
      }
    }
    __syncthreads();   // s_slot and s_unit are rewritten for the next tile
  }
}

}  // namespace

cudaError_t launch_kv_stage(const StageArgs &a, cudaStream_t stream) {
  if (a.tiles == 0) return cudaSuccess;
  const int64_t grid = a.tiles < 152 * 8 ? a.tiles : 152 * 8;
  if (a.fp8)
    return launch_dependent(stage_kernel<true>, dim3((unsigned)grid), dim3(kStageThreads), 0,
                            stream, a);
  return launch_dependent(stage_kernel<false>, dim3((unsigned)grid), dim3(kStageThreads), 0,
                          stream, a);
}

}  // namespace akp
