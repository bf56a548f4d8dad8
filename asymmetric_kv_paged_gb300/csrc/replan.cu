// Device planner of replayable plans: before each attention launch, one CTA
// reads the run's request lengths and rewrites the plan's work list (block
// key ranges, segments, CTA segment ranges, splits, partial-row offsets and
// the CTAs' head records)
// in place, so that a captured CUDA graph stays valid while requests grow.
// The arithmetic is in replan.hpp, shared with the host mirror.
#include <cuda_runtime.h>

#include "kernels.hpp"
#include "replan.hpp"

namespace akp {

namespace {

constexpr int kReplanThreads = 1024;   // 32 warps: the scan's second level is one warp

// Exclusive prefix sum of v[0, n) in place, with v[n] = the total; every
// thread of the CTA takes part.
__device__ void cta_exclusive_scan(int32_t *v, int32_t n) {
  __shared__ int32_t warp_sum[32];
  __shared__ int32_t carry;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int32_t base = 0; base < n; base += kReplanThreads) {
    const int32_t i = base + tid;
    const int32_t x = i < n ? v[i] : 0;
    int32_t s = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    if (lane == 31) warp_sum[warp] = s;
    __syncthreads();
    if (warp == 0) {
      int32_t t = warp_sum[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, t, off);
        if (lane >= off) t += y;
      }
      warp_sum[lane] = t;
    }
    __syncthreads();
    const int32_t before = carry + (warp > 0 ? warp_sum[warp - 1] : 0) + s - x;
    if (i < n) v[i] = before;
    __syncthreads();
    if (tid == kReplanThreads - 1) carry = before + x;
    __syncthreads();
  }
  if (tid == 0) v[n] = carry;
  __syncthreads();
}

__global__ void __launch_bounds__(kReplanThreads, 1) replan_kernel(const ReplanArgs r) {
  const int tid = threadIdx.x;
  // Launched as a programmatic dependent: the previous kernels of the stream
  // (the last run's attention and merge, or the KV append) have completed once
  // this wait returns, so the work list they read may be rewritten.  The
  // attention kernel that follows may be scheduled now; it waits for this
  // grid to complete.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  // lengths (clamped into [n_b, bound_b]) and key ranges of every block
  for (int32_t bi = tid; bi < r.nb; bi += kReplanThreads) {
    BlockDesc &bd = r.blocks[bi];
    const int32_t bound = r.seq_bounds[bd.b];
    int32_t L = r.seq_lens[bd.b];
    if (L < bd.n || L > bound) {
      atomicOr(r.err, 4);
      L = L < bd.n ? bd.n : bound;
    }
    int32_t klo, khi;
    block_keys(bd, L, r.group, r.window, &klo, &khi);
    bd.L = L;
    bd.klo = klo;
    bd.khi = khi;
    r.tile_start[bi] = block_tile_count(klo, khi, r.key_tile);
  }
  __syncthreads();
  cta_exclusive_scan(r.tile_start, r.nb);
  const int64_t T = r.tile_start[r.nb];
  const int64_t ctas = T < r.num_ctas ? T : r.num_ctas;
  const int32_t charge = switch_charge(T, ctas);
  const int64_t P = T + (int64_t)charge * r.nb;     // global positions

  // segments per CTA (blocks its share holds tiles of), then their offsets
  for (int32_t c = tid; c < r.num_ctas; c += kReplanThreads) {
    int32_t cnt = 0;
    if (c < ctas) {
      const int64_t a = share_begin(c, P, ctas), e = share_begin(c + 1, P, ctas);
      for (int32_t bi = block_at(r.tile_start, r.nb, a, charge); bi < r.nb; ++bi) {
        const int64_t gs = block_pos(r.tile_start, bi, charge);
        if (gs >= e) break;
        const SegDesc sd =
            share_segment(bi, r.blocks[bi], gs, block_pos(r.tile_start, bi + 1, charge), a, e, c,
                          P, ctas, r.key_tile, charge);
        cnt += sd.tile_end > sd.tile_begin;
      }
    }
    r.cta_seg_begin[c] = cnt;
  }
  __syncthreads();
  cta_exclusive_scan(r.cta_seg_begin, r.num_ctas);

  for (int32_t c = tid; c < ctas; c += kReplanThreads) {
    const int64_t a = share_begin(c, P, ctas), e = share_begin(c + 1, P, ctas);
    int32_t s = r.cta_seg_begin[c];
    for (int32_t bi = block_at(r.tile_start, r.nb, a, charge); bi < r.nb; ++bi) {
      const int64_t gs = block_pos(r.tile_start, bi, charge);
      if (gs >= e) break;
      const SegDesc sd =
          share_segment(bi, r.blocks[bi], gs, block_pos(r.tile_start, bi + 1, charge), a, e, c, P,
                        ctas, r.key_tile, charge);
      if (sd.tile_end > sd.tile_begin) r.segs[s++] = sd;
    }
  }

  // splits and partial-row offsets of every block
  for (int32_t bi = tid; bi < r.nb; bi += kReplanThreads) {
    const int32_t ns = share_splits(block_pos(r.tile_start, bi, charge),
                                    block_pos(r.tile_start, bi + 1, charge), P, ctas, charge);
    r.blocks[bi].num_splits = ns;
    r.part_start[bi] = ns > 1 ? ns * r.blocks[bi].nrows : 0;
  }
  __syncthreads();
  cta_exclusive_scan(r.part_start, r.nb);
  for (int32_t bi = tid; bi < r.nb; bi += kReplanThreads)
    r.blocks[bi].part_row_base = r.blocks[bi].num_splits > 1 ? r.part_start[bi] : -1;
  __syncthreads();

  // each CTA's head record, from the final segments and blocks
  for (int32_t c = tid; c < r.num_ctas; c += kReplanThreads)
    r.cta_heads[c] = cta_head(r.segs, r.blocks, r.cta_seg_begin[c], r.cta_seg_begin[c + 1]);
}

}  // namespace

cudaError_t launch_replan(const ReplanArgs &r, cudaStream_t stream) {
  if (r.nb == 0) return cudaSuccess;
  return launch_dependent(replan_kernel, dim3(1), dim3(kReplanThreads), 0, stream, r);
}

}  // namespace akp
