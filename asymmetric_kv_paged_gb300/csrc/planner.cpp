// Host planner: validates a problem and turns it into row blocks, key-tile
// segments per CTA, and a workspace layout.
//
// The split-KV schedule is the point of the pages' verify fix: the Triton
// kernel they describe dropped split-KV whenever a request carried several
// query tokens and left most SMs idle (MiMo-V2.6-Flash-RL model card, "What
// the kernels do").  Here every (request, KV head) key range is cut into
// tiles, and the tiles of all blocks are dealt to CTAs in order so that each
// CTA gets the same number of tiles, whatever the mode.  A block whose tiles
// land on several CTAs becomes a multi-split block whose partials are merged
// by log-sum-exp.  All query rows of a block (all draft tokens x all heads of
// the group) ride on one pass over the keys ("one program per whole verify").
#include <algorithm>
#include <cstring>

#include "plan.hpp"
#include "replan.hpp"

namespace akp {

namespace {
void fill_cta_heads(HostPlan *hp) {
  hp->cta_heads.resize(hp->num_ctas);
  for (int32_t c = 0; c < hp->num_ctas; ++c)
    hp->cta_heads[c] = cta_head(hp->segs.data(), hp->blocks.data(), hp->cta_seg_begin[c],
                                hp->cta_seg_begin[c + 1]);
}

// Staging units of a prefill plan: one per (request, KV head), over the
// 128-key tiles that hold the union of its blocks' key ranges (blocks come in
// (b, g, row0) order, so a unit's blocks are consecutive).  Each block learns
// where its keys sit in the scratch (srow).  Without a prefill plan, or if
// the scratch rows would overflow the int32 coordinates of a TMA copy, there
// is no scratch and the prefill kernel reads the cache itself.
void build_stage(HostPlan *hp) {
  hp->stage_units.clear();
  hp->stage_rows = hp->stage_tiles = 0;
  for (BlockDesc &bd : hp->blocks) bd.srow = 0;
  if (!hp->prefill || hp->replayable) return;
  const int64_t nb = (int64_t)hp->blocks.size();
  for (int64_t first = 0; first < nb;) {
    const BlockDesc &b0 = hp->blocks[first];
    int64_t end = first;
    int32_t klo = b0.klo, khi = b0.khi;
    while (end < nb && hp->blocks[end].b == b0.b && hp->blocks[end].g == b0.g) {
      klo = std::min(klo, hp->blocks[end].klo);
      khi = std::max(khi, hp->blocks[end].khi);
      ++end;
    }
    StageUnit u{};
    u.b = b0.b;
    u.g = b0.g;
    u.j0 = klo / kStageTile * kStageTile;
    u.klo = klo;
    u.khi = khi;
    u.tiles = (khi - 1) / kStageTile - klo / kStageTile + 1;
    if (hp->stage_rows + (int64_t)u.tiles * kStageTile > INT32_MAX - kStageTile) {
      hp->stage_units.clear();
      hp->stage_rows = hp->stage_tiles = 0;
      for (BlockDesc &bd : hp->blocks) bd.srow = 0;
      return;
    }
    u.row_base = (int32_t)hp->stage_rows;
    u.tile_off = (int32_t)hp->stage_tiles;
    for (int64_t bi = first; bi < end; ++bi) hp->blocks[bi].srow = u.row_base - u.j0;
    hp->stage_rows += (int64_t)u.tiles * kStageTile;
    hp->stage_tiles += u.tiles;
    hp->stage_units.push_back(u);
    first = end;
  }
}

// Workspace: split partials, then (prefill plans) the staging scratch.
void size_workspace(HostPlan *hp) {
  hp->partial_bytes =
      hp->part_rows ? part_o_bytes(hp->part_rows) + part_lse_bytes(hp->part_rows) : 0;
  hp->stage_bytes = hp->stage_rows ? stage_k_bytes(hp->stage_rows, hp->prob.head_dim_qk) +
                                         stage_v_bytes(hp->stage_rows)
                                   : 0;
  hp->workspace_bytes = hp->partial_bytes + hp->stage_bytes;
}
}  // namespace


attn_status_t build_host_plan(const attn_problem_t *p, int32_t num_sms, HostPlan *out) {
  if (!p || !out || num_sms <= 0) return ATTN_ERR_INVALID_ARG;
  if (p->batch < 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 || p->page_size <= 0 ||
      p->num_pages <= 0 || p->page_table_stride <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (p->batch > 0 && (!p->qo_indptr_host || !p->seq_lens_host)) return ATTN_ERR_INVALID_ARG;
  // Head-dim pairs: 192/128 (MiMo's layers), and 128/128 for layers whose
  // own pair is symmetric (sglang PR #32818, "Three changes", item 1: a model
  // is asymmetric when head_dim != v_head_dim or swa_head_dim !=
  // swa_v_head_dim, so its SWA layers may carry a pair of their own).
  if ((p->head_dim_qk != kDqk && p->head_dim_qk != kDqkSym) || p->head_dim_v != kDv)
    return ATTN_ERR_UNSUPPORTED;
  if (p->num_q_heads % p->num_kv_heads != 0) return ATTN_ERR_UNSUPPORTED;
  if (p->kv_dtype != ATTN_KV_BF16 && p->kv_dtype != ATTN_KV_FP8_E4M3) return ATTN_ERR_UNSUPPORTED;

  HostPlan hp;
  hp.prob = *p;
  hp.num_sms = num_sms;
  hp.group = p->num_q_heads / p->num_kv_heads;
  hp.qo_indptr.assign(p->qo_indptr_host ? p->qo_indptr_host : nullptr,
                      p->qo_indptr_host ? p->qo_indptr_host + p->batch + 1 : nullptr);
  if (p->batch == 0) hp.qo_indptr.assign(1, 0);
  hp.seq_lens.assign(p->seq_lens_host ? p->seq_lens_host : nullptr,
                     p->seq_lens_host ? p->seq_lens_host + p->batch : nullptr);
  hp.prob.qo_indptr_host = nullptr;
  hp.prob.seq_lens_host = nullptr;
  if (hp.qo_indptr[0] != 0) return ATTN_ERR_INVALID_ARG;
  for (int32_t b = 0; b < p->batch; ++b) {
    int64_t n = (int64_t)hp.qo_indptr[b + 1] - hp.qo_indptr[b];
    int64_t L = hp.seq_lens[b];
    if (n < 0 || L < n) return ATTN_ERR_INVALID_ARG;
    if ((L + p->page_size - 1) / p->page_size > p->page_table_stride) return ATTN_ERR_INVALID_ARG;
  }
  // Flat row and tile counts must stay inside int32 device arithmetic.
  if ((int64_t)hp.qo_indptr[p->batch] * p->num_q_heads > INT32_MAX / p->head_dim_qk)
    return ATTN_ERR_UNSUPPORTED;

  hp.threads = 352;
  int64_t max_rows = 0;
  for (int32_t b = 0; b < p->batch; ++b)
    max_rows = std::max<int64_t>(max_rows, (int64_t)(hp.qo_indptr[b + 1] - hp.qo_indptr[b]) * hp.group);
  // M = 64 halves the Q and P tiles, so one more K/V stage fits (and Q can be
  // double-buffered); for blocks of up to 64 rows that beats M = 128's second
  // row copy, measured on 8- and 64-row blocks.
  // (the prefill kernel is built for the 192/128 pair only)
  hp.block_rows = max_rows <= 64 ? 64 : max_rows <= 128 || p->head_dim_qk != kDqk ? 128 : 256;
  hp.prefill = hp.block_rows == 256;
  hp.key_tile = hp.prefill ? kPrefillKeyTile : kKeyTile;
  const int32_t rows_per_block = hp.block_rows;
  const int32_t tile = hp.key_tile;
  const int32_t G = hp.group;

  // Row blocks.
  int64_t total_tiles = 0;
  for (int32_t b = 0; b < p->batch; ++b) {
    const int32_t n = hp.qo_indptr[b + 1] - hp.qo_indptr[b];
    const int32_t L = hp.seq_lens[b];
    if (n == 0) continue;
    const int32_t R = n * G;
    for (int32_t g = 0; g < p->num_kv_heads; ++g) {
      for (int32_t row0 = 0; row0 < R; row0 += rows_per_block) {
        BlockDesc bd{};
        bd.b = b;
        bd.g = g;
        bd.row0 = row0;
        bd.nrows = std::min(rows_per_block, R - row0);
        bd.L = L;
        bd.n = n;
        bd.tok0 = hp.qo_indptr[b];
        const int32_t t_first = row0 / G;
        const int32_t t_last = (row0 + bd.nrows - 1) / G;
        const int64_t i_first = (int64_t)L - n + t_first;
        const int64_t i_last = (int64_t)L - n + t_last;
        int64_t lo = 0;
        if (p->window > 0) lo = std::max<int64_t>(0, i_first - p->window + 1);
        bd.klo = (int32_t)lo;
        bd.khi = (int32_t)(i_last + 1);
        total_tiles += (bd.khi - 1) / tile - bd.klo / tile + 1;
        hp.blocks.push_back(bd);
      }
    }
  }

  // Blocks of more than half the MMA rows hold one copy of each row; on M = 64
  // the split-KV kernel then runs two threads per row (verify blocks).
  hp.one_copy = !hp.blocks.empty();
  for (const BlockDesc &bd : hp.blocks) hp.one_copy = hp.one_copy && 2 * bd.nrows > rows_per_block;

  // Deal tiles to CTAs in block order, cutting a block where a CTA's share
  // ends.  Each new CTA's share is the remaining tiles over the remaining
  // CTAs, so rounding never piles up on the last one; a block remainder of at
  // most `slack` tiles (1/32 of a share; two for prefill plans) stays on the
  // current CTA rather than becoming a split of its own.
  const int64_t nb = (int64_t)hp.blocks.size();
  constexpr int64_t kWholeBlockTiles = 8;
  // A CTA that goes on to a further segment pays for the switch (the finished
  // segment's epilogue, the next block's Q) with this many tiles of its share:
  // measured, two-segment CTAs otherwise ended ~3-5 us after the others
  // (on the batched decode 4 tiles measured ~1.5% faster than 3, 5 and 6 no
  // better than 4).
  constexpr int64_t kSegSwitchTiles = 4;
  if (nb > 0) {
    const int64_t min_tiles = 2;
    int64_t remaining = total_tiles;
    int32_t cta = -1;
    int64_t room = 0, target = 0, slack = 0;
    bool charge = false;          // this CTA's share pays for its segment switches
    for (int64_t bi = 0; bi < nb; ++bi) {
      BlockDesc &bd = hp.blocks[bi];
      int32_t t0 = bd.klo / tile;
      const int32_t tend = (bd.khi - 1) / tile + 1;
      int32_t split = 0;
      while (t0 < tend) {
        if (room <= 0) {
          ++cta;
          const int64_t ctas_left = std::max<int64_t>(1, (int64_t)num_sms - cta);
          target = std::max<int64_t>(min_tiles, (remaining + ctas_left - 1) / ctas_left);
          // Large shares count the switches still ahead (about one per block
          // not yet begun) as work, so that the CTAs after a switch are not
          // left with the tiles the switching ones gave up; shares of a few
          // tiles, where most CTAs switch, stay even in tiles.
          charge = cta + 1 < num_sms && target >= 8 * kSegSwitchTiles;
          if (charge)
            target = (remaining + kSegSwitchTiles * (nb - bi - 1) + ctas_left - 1) / ctas_left;
          // A prefill tile (128 keys x 256 rows) costs far more than the
          // split it would save: there the slack is at most two tiles
          // (measured: 1/32 of a share left CTAs 2.5% apart in tiles and time).
          slack = hp.prefill ? std::min<int64_t>(2, target / 32) : target / 32;
          room = target;
        }
        const int64_t left = tend - t0;
        // A small block (at most kWholeBlockTiles, and at most two shares) is
        // not split while there are CTAs enough for every block still to
        // place: a fresh CTA takes it whole, a CTA it does not fit in leaves it
        // to the next one.  For such a block a split's extra segment and merge
        // cost more than the room left unused.
        const bool whole = t0 == bd.klo / tile && left <= kWholeBlockTiles &&
                           left <= 2 * target && nb - bi <= (int64_t)num_sms - cta - 1;
        if (whole && room < target && left > room + slack) {
          room = 0;
          continue;
        }
        const int64_t take = (whole || left <= room + slack) ? left : room;
        SegDesc s{(int32_t)bi, t0, (int32_t)(t0 + take), split++};
        hp.segs.push_back(s);
        hp.seg_cta.push_back(cta);
        room -= take;
        // the CTA's next tiles start a new segment (the last CTA takes all that is left)
        if (room > 0 && charge) room -= kSegSwitchTiles;
        remaining -= take;
        t0 += (int32_t)take;
      }
      bd.num_splits = split;
    }
    hp.num_ctas = cta + 1;
  }
  hp.cta_seg_begin.assign(hp.num_ctas + 1, 0);
  for (size_t s = 0; s < hp.segs.size(); ++s) hp.cta_seg_begin[hp.seg_cta[s] + 1]++;
  for (int32_t c = 0; c < hp.num_ctas; ++c) hp.cta_seg_begin[c + 1] += hp.cta_seg_begin[c];

  // Partials and merge items for multi-split blocks.
  for (int64_t bi = 0; bi < nb; ++bi) {
    BlockDesc &bd = hp.blocks[bi];
    bd.part_row_base = -1;
    if (bd.num_splits > 1) {
      bd.part_row_base = (int32_t)hp.part_rows;
      hp.part_rows += (int64_t)bd.num_splits * bd.nrows;
      hp.multi_split_blocks++;
      for (int32_t r = 0; r < bd.nrows; r += kMergeRowsPerCta)
        hp.merge_items.push_back(MergeItem{(int32_t)bi, r});
    }
  }
  if (hp.part_rows > INT32_MAX / kDv) return ATTN_ERR_UNSUPPORTED;
  build_stage(&hp);
  size_workspace(&hp);
  fill_cta_heads(&hp);
  *out = std::move(hp);
  return ATTN_OK;
}

// Replayable plans trade the static dealing above (whole small blocks, slack)
// for one a single CTA can redo on the device in microseconds: equal shares of
// the tiles in block order (replan.hpp).
attn_status_t build_replayable_plan(const attn_problem_t *p, int32_t num_sms, HostPlan *out) {
  HostPlan hp;
  attn_status_t st = build_host_plan(p, num_sms, &hp);
  if (st != ATTN_OK) return st;
  const int64_t nb = (int64_t)hp.blocks.size();
  // no run has more tiles than this: khi never exceeds its value at the bounds
  int64_t max_tiles = 0;
  int32_t max_rows = 0;
  for (const BlockDesc &bd : hp.blocks) {
    max_tiles += (bd.khi - 1) / hp.key_tile + 1;
    max_rows = std::max(max_rows, bd.nrows);
  }
  if (max_tiles >= INT32_MAX / 2) return ATTN_ERR_UNSUPPORTED;
  hp.replayable = true;
  hp.num_ctas = (int32_t)std::min<int64_t>(num_sms, max_tiles);
  hp.seg_capacity = nb + hp.num_ctas;
  // a multi-split block keeps nrows partial rows per split, and there are at
  // most nb + num_ctas - 1 segments in all
  hp.part_rows = (int64_t)max_rows * hp.seg_capacity;
  if (hp.part_rows > INT32_MAX / kDv) return ATTN_ERR_UNSUPPORTED;
  build_stage(&hp);     // no scratch: the work list changes from run to run
  size_workspace(&hp);
  // merge items for every block: the merge skips blocks a run leaves whole
  hp.merge_items.clear();
  for (int64_t bi = 0; bi < nb; ++bi)
    for (int32_t r = 0; r < hp.blocks[bi].nrows; r += kMergeRowsPerCta)
      hp.merge_items.push_back(MergeItem{(int32_t)bi, r});
  replan_host(&hp, hp.seq_lens.data());
  *out = std::move(hp);
  return ATTN_OK;
}

int32_t replan_host(HostPlan *hp, const int32_t *seq_lens) {
  int32_t err = 0;
  const int32_t nb = (int32_t)hp->blocks.size();
  std::vector<int32_t> start(nb + 1, 0);
  for (int32_t bi = 0; bi < nb; ++bi) {
    BlockDesc &bd = hp->blocks[bi];
    const int32_t bound = hp->seq_lens[bd.b];
    int32_t L = seq_lens[bd.b];
    if (L < bd.n || L > bound) {
      err |= 4;
      L = L < bd.n ? bd.n : bound;
    }
    int32_t klo, khi;
    block_keys(bd, L, hp->group, hp->prob.window, &klo, &khi);
    bd.L = L;
    bd.klo = klo;
    bd.khi = khi;
    start[bi + 1] = start[bi] + block_tile_count(klo, khi, hp->key_tile);
  }
  const int64_t T = start[nb];
  const int64_t ctas = std::min<int64_t>(T, hp->num_ctas);
  const int32_t charge = switch_charge(T, ctas);
  const int64_t P = T + (int64_t)charge * nb;
  const int32_t *st = start.data();
  hp->segs.clear();
  hp->seg_cta.clear();
  hp->cta_seg_begin.assign(hp->num_ctas + 1, 0);
  for (int32_t c = 0; c < hp->num_ctas; ++c) {
    if (c < ctas) {
      const int64_t a = share_begin(c, P, ctas), e = share_begin(c + 1, P, ctas);
      for (int32_t bi = block_at(st, nb, a, charge); bi < nb && block_pos(st, bi, charge) < e;
           ++bi) {
        const SegDesc sd = share_segment(bi, hp->blocks[bi], block_pos(st, bi, charge),
                                         block_pos(st, bi + 1, charge), a, e, c, P, ctas,
                                         hp->key_tile, charge);
        if (sd.tile_end == sd.tile_begin) continue;   // the share ends in the block's charge
        hp->segs.push_back(sd);
        hp->seg_cta.push_back(c);
      }
    }
    hp->cta_seg_begin[c + 1] = (int32_t)hp->segs.size();
  }
  int64_t part = 0;
  hp->multi_split_blocks = 0;
  for (int32_t bi = 0; bi < nb; ++bi) {
    BlockDesc &bd = hp->blocks[bi];
    bd.num_splits = share_splits(block_pos(st, bi, charge), block_pos(st, bi + 1, charge), P, ctas,
                                 charge);
    bd.part_row_base = -1;
    if (bd.num_splits > 1) {
      bd.part_row_base = (int32_t)part;
      part += (int64_t)bd.num_splits * bd.nrows;
      hp->multi_split_blocks++;
    }
  }
  fill_cta_heads(hp);
  return err;
}

}  // namespace akp
