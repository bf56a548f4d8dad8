// Internal plan layout shared by the host planner, the C ABI and the kernels.
// Not part of the public ABI (see include/attn_paged.h).
#pragma once
#include <cstddef>
#include <cstdint>
#include <vector>

#include "attn_paged.h"

namespace akp {

constexpr int kDqk = 192;       // query/key head dim
constexpr int kDqkSym = 128;    // query/key head dim of the symmetric pair 128/128
constexpr int kDv = 128;        // value head dim
constexpr int kKeyTile = 64;    // keys per pipeline tile (decode / verify kernel)
constexpr int kPrefillKeyTile = 128;   // keys per tile of the prefill kernel

// Query rows per row block.  A block packs up to block_rows query rows of one
// (request, KV head): row r <-> (token r / G, head g*G + r % G); decode blocks
// hold G rows, verify blocks n*G.  block_rows is 64 (M=64 MMAs) when no
// (request, KV head) has more than 64 query rows, 128 when none has more than
// 128, else 256: the prefill kernel's two 128-row Q tiles over 128-key tiles.

// One row block: rows [row0, row0 + nrows) of (b, g).  Keys [klo, khi) are
// the union of what its rows can see.  srow: with a staging scratch (prefill
// plans, see StageUnit), key j of (b, g) is scratch row srow + j; else 0.
struct BlockDesc {
  int32_t b, g, row0, nrows;
  int32_t L, n, tok0, klo;        // seq len, new tokens, first flat token, first key
  int32_t khi, num_splits, part_row_base, srow;
};
static_assert(sizeof(BlockDesc) == 48, "BlockDesc layout");

// One work segment: key tiles [tile_begin, tile_end) of one block.
// split = index of this segment among the block's segments.
struct SegDesc {
  int32_t block, tile_begin, tile_end, split;
};

// What a CTA reads first: its segment range, its key-tile count, and its
// first segment with that segment's block, in one 80-byte record, so that the
// kernel's start costs one memory round trip instead of three dependent ones.
struct CtaHead {
  int32_t seg_begin, seg_end, total, pad;
  SegDesc seg;
  BlockDesc blk;
};
static_assert(sizeof(CtaHead) == 80, "CtaHead layout");

// Prefill plans stage the keys their blocks read into a scratch of 16-bit
// rows (E4M3 widened to fp16, BF16 copied) once per call, which the prefill
// kernel then loads as whole tiles by TMA.  One unit per (request, KV head)
// with prefill blocks: keys [j0, j0 + 128 * tiles) go to scratch rows
// [row_base, ...); keys outside [klo, khi) (the union of the unit's blocks'
// ranges) are written as zeros.  tile_off: the unit's first tile among all
// units' tiles.
struct StageUnit {
  int32_t b, g, j0, klo, khi, tiles, row_base, tile_off;
};
static_assert(sizeof(StageUnit) == 32, "StageUnit layout");
constexpr int kStageTile = 128;      // keys per staged tile (the prefill key tile)

// One merge item: rows [row_begin, row_begin + 8) of a multi-split block.
struct MergeItem {
  int32_t block, row_begin;
};
constexpr int kMergeRowsPerCta = 8;

struct HostPlan {
  attn_problem_t prob{};
  std::vector<int32_t> qo_indptr, seq_lens;
  int32_t group = 1;             // G = Hq / Hkv
  int32_t block_rows = 128;      // 64 or 128 (the MMA M), or 256 (prefill kernel)
  int32_t key_tile = kKeyTile;   // keys per tile: 64, or 128 for the prefill kernel
  bool prefill = false;          // block_rows == 256: attn_prefill.cu runs the plan
  bool one_copy = false;         // every block has more than block_rows / 2 rows
  int32_t num_sms = 0, num_ctas = 0, threads = 0;
  std::vector<BlockDesc> blocks;
  std::vector<SegDesc> segs;
  std::vector<int32_t> seg_cta;        // CTA of each segment
  std::vector<int32_t> cta_seg_begin;  // [num_ctas + 1]
  std::vector<CtaHead> cta_heads;      // [num_ctas]
  std::vector<MergeItem> merge_items;
  int64_t part_rows = 0;
  // staging scratch (prefill plans that are not replayable; empty otherwise)
  std::vector<StageUnit> stage_units;
  int64_t stage_rows = 0, stage_tiles = 0;
  size_t partial_bytes = 0;      // split partials: part_o then part_lse
  size_t stage_bytes = 0;        // staged K rows then staged V rows, after the partials
  size_t workspace_bytes = 0;    // partial_bytes + stage_bytes
  int32_t multi_split_blocks = 0;
  bool use_tma = false;          // K/V tiles as TMA boxes (else gathered by threads)
  // Replayable plans: seq_lens holds the per-request upper bounds, the work
  // list is rebuilt from each run's lengths (replan.hpp); segs, part_rows and
  // merge_items are sized for any lengths within the bounds.
  bool replayable = false;
  int64_t seg_capacity = 0;
};

// Device-side copy of a plan (owned by attn_plan_s).
struct DevicePlan {
  BlockDesc *blocks = nullptr;
  SegDesc *segs = nullptr;
  int32_t *cta_seg_begin = nullptr;
  CtaHead *cta_heads = nullptr;
  MergeItem *merge_items = nullptr;
  StageUnit *stage_units = nullptr;
  int32_t *err = nullptr;  // device error word
  // replayable plans only
  int32_t *seq_bounds = nullptr;   // [B]
  int32_t *tile_start = nullptr;   // scratch [blocks + 1]
  int32_t *part_start = nullptr;   // scratch [blocks + 1]
};

// Validate `p` and build the schedule for a device with num_sms SMs.
attn_status_t build_host_plan(const attn_problem_t *p, int32_t num_sms, HostPlan *out);

// A replayable plan for the query layout of `p`, whose seq_lens are upper
// bounds: the blocks of build_host_plan, one CTA per SM (at most one per key
// tile), capacities for any lengths within the bounds, and the work list of
// the bounds themselves.
attn_status_t build_replayable_plan(const attn_problem_t *p, int32_t num_sms, HostPlan *out);

// Host mirror of the device planner: rebuild a replayable plan's work list for
// the lengths seq_lens[B], clamped into [n_b, bound_b] as on the device.
// Returns the error bits the device planner would set (4: a length clamped).
int32_t replan_host(HostPlan *hp, const int32_t *seq_lens);

// Workspace carve-up: partial outputs then partial lse, each 256-B aligned.
inline size_t part_o_bytes(int64_t part_rows) {
  return ((size_t)part_rows * kDv * sizeof(float) + 255) & ~(size_t)255;
}
inline size_t part_lse_bytes(int64_t part_rows) {
  return ((size_t)part_rows * sizeof(float) + 255) & ~(size_t)255;
}
// Staging scratch: K rows (dqk 16-bit values each), then V rows (kDv each).
inline size_t stage_k_bytes(int64_t rows, int dqk) {
  return ((size_t)rows * dqk * 2 + 255) & ~(size_t)255;
}
inline size_t stage_v_bytes(int64_t rows) {
  return ((size_t)rows * kDv * 2 + 255) & ~(size_t)255;
}

}  // namespace akp

struct attn_plan_s {
  akp::HostPlan host;
  akp::DevicePlan dev;
  int device = -1;     // -1: host-only plan (attn_plan_host)
};
