// Work-list arithmetic of replayable plans, shared by the device planner
// (replan.cu, run before every attention launch) and its host mirror
// (planner.cpp), so that both deal the same tiles to the same CTAs.
//
// A replayable plan fixes the query layout (qo_indptr) and therefore the row
// blocks; the request lengths are read on the device at every run, within the
// bounds the plan was built for.  For the lengths of one run:
//   - block bi's key range [klo, khi) follows from its rows as in the static
//     planner (bottom-right causal alignment, optional window);
//   - its tiles take the global positions [start[bi], start[bi+1]) of the
//     exclusive prefix sum `start` of the tile counts (T = start[nb] tiles);
//   - with C' = min(C, T) working CTAs, CTA c takes positions
//     [c*P/C', (c+1)*P/C') (equal shares, rounded down), so a block is cut
//     wherever a share ends and each piece is one segment.  On shares of 32
//     tiles or more every block is first given `charge` positions without a
//     tile (P = T + charge * nb): the CTA whose share reaches into a block
//     pays for its epilogue and Q staging with that much less work, as in the
//     static deal.
#pragma once
#include <cstdint>

#include "plan.hpp"

#ifdef __CUDACC__
#define AKP_HD __host__ __device__ __forceinline__
#else
#define AKP_HD inline
#endif

namespace akp {

// Key range of a block's rows for request length L.
AKP_HD void block_keys(const BlockDesc &bd, int32_t L, int32_t group, int32_t window,
                       int32_t *klo, int32_t *khi) {
  const int64_t i_first = (int64_t)L - bd.n + bd.row0 / group;
  const int64_t i_last = (int64_t)L - bd.n + (bd.row0 + bd.nrows - 1) / group;
  int64_t lo = 0;
  if (window > 0 && i_first - window + 1 > 0) lo = i_first - window + 1;
  *klo = (int32_t)lo;
  *khi = (int32_t)(i_last + 1);
}

// Key tiles of `tile` keys touched by keys [klo, khi) (klo < khi).
AKP_HD int32_t block_tile_count(int32_t klo, int32_t khi, int32_t tile) {
  return (khi - 1) / tile - klo / tile + 1;
}

// Positions a CTA pays for reaching into a block (its epilogue, the next Q),
// on shares of at least 8 such charges; 0 (plain tile shares) below.
constexpr int32_t kReplanSwitchTiles = 4;
AKP_HD int32_t switch_charge(int64_t T, int64_t ctas) {
  return T >= 8 * kReplanSwitchTiles * ctas ? kReplanSwitchTiles : 0;
}

// First global position of block bi: its tiles' prefix plus a charge per
// earlier block (the block's tiles start `charge` positions later).
AKP_HD int64_t block_pos(const int32_t *start, int32_t bi, int32_t charge) {
  return (int64_t)start[bi] + (int64_t)charge * bi;
}

// First global position of CTA c's share (c = ctas gives the total P).
AKP_HD int64_t share_begin(int64_t c, int64_t T, int64_t ctas) { return c * T / ctas; }

// CTA whose share holds global tile position x (0 <= x < T, ctas <= T): the
// largest c with floor(c*T/ctas) <= x.
AKP_HD int32_t share_owner(int64_t x, int64_t T, int64_t ctas) {
  return (int32_t)(((x + 1) * ctas - 1) / T);
}

// Block holding global position x: the largest i in [0, nb) with
// block_pos(i) <= x (positions strictly increasing, x < the total).
AKP_HD int32_t block_at(const int32_t *start, int32_t nb, int64_t x, int32_t charge) {
  int32_t lo = 0, hi = nb - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (block_pos(start, mid, charge) <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Segment of block bi inside CTA c's share [a, e), with the block at global
// positions [gs, ge), its tiles at [gs + charge, ge); tile_begin == tile_end
// when the share holds none of them (it ends in the block's charge).
AKP_HD SegDesc share_segment(int32_t bi, const BlockDesc &bd, int64_t gs, int64_t ge, int64_t a,
                             int64_t e, int32_t c, int64_t P, int64_t ctas, int32_t tile,
                             int32_t charge) {
  const int32_t tb = bd.klo / tile;
  const int64_t ts = gs + charge;
  const int64_t lo = a > ts ? a : ts;
  const int64_t hi = e < ge ? e : ge;
  SegDesc s;
  s.block = bi;
  s.tile_begin = tb + (int32_t)(lo - ts);
  s.tile_end = hi > lo ? tb + (int32_t)(hi - ts) : s.tile_begin;
  s.split = c - share_owner(ts, P, ctas);
  return s;
}

// Splits of block bi (global positions [gs, ge), tiles from gs + charge).
AKP_HD int32_t share_splits(int64_t gs, int64_t ge, int64_t P, int64_t ctas, int32_t charge) {
  return share_owner(ge - 1, P, ctas) - share_owner(gs + charge, P, ctas) + 1;
}

// The head record of a CTA whose segments are [s0, s1) (see CtaHead).
AKP_HD CtaHead cta_head(const SegDesc *segs, const BlockDesc *blocks, int32_t s0, int32_t s1) {
  CtaHead h{};
  h.seg_begin = s0;
  h.seg_end = s1;
  for (int32_t s = s0; s < s1; ++s) h.total += segs[s].tile_end - segs[s].tile_begin;
  if (s0 < s1) {
    h.seg = segs[s0];
    h.blk = blocks[h.seg.block];
  }
  return h;
}

// Arguments of the device planner (replan.cu).
struct ReplanArgs {
  BlockDesc *blocks;           // [nb]; b, g, row0, nrows, n, tok0 fixed
  SegDesc *segs;               // capacity nb + num_ctas
  int32_t *cta_seg_begin;      // [num_ctas + 1]
  CtaHead *cta_heads;          // [num_ctas]
  int32_t *tile_start;         // scratch [nb + 1]
  int32_t *part_start;         // scratch [nb + 1]
  const int32_t *seq_lens;     // [B] lengths of this run (caller's device array)
  const int32_t *seq_bounds;   // [B] upper bounds the plan was built for
  int32_t *err;                // device error word (bit 4: a length out of bounds)
  int32_t nb, num_ctas, group, window, key_tile;
};

}  // namespace akp
