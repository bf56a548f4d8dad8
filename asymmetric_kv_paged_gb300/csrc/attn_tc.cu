// Split-KV paged attention on the Blackwell tensor-core path (tcgen05 + TMEM)
// for row blocks of up to 128 query rows: decode, multi-token verify, and
// prefill chunks small enough (larger ones run attn_prefill.cu).
//
// A CTA walks the key tiles (64 keys) of its work segments.  Each segment
// belongs to one row block: up to 128 query rows of one (request, KV head),
// row r <-> (token r / G, head g*G + r % G), so every draft token and every
// head of the group shares one pass over the keys ("one program per whole
// verify", and the 8-token x 16-head packing of the prefill kernel on the
// MiMo-V2.6-Flash-RL model card, "What the kernels do").  When no block has
// more than 64 rows the kernel issues M=64 MMAs (smaller Q tile: a fourth K/V
// stage and a second Q buffer fit); blocks smaller than the MMA are copied
// across its rows, each copy taking a slice of every key tile.
//
// Warp roles (352 threads):
//   warps 0-3  softmax + epilogue: MMA row p lives in TMEM lane p (M=128) or
//              in lane 32*(p/16) + p%16 (M=64), and that lane's thread owns it
//              (HALF instantiations: lanes l and l+16 share row 16w + l%16,
//              32 key columns each);
//   warps 4-7  converters: stage Q per block; turn raw FP8 K/V tiles into
//              exact bf16 operand tiles; zero V rows of keys outside the
//              block's range on edge tiles (unused slots may hold NaN:
//              sammysun0711/sglang PR #35, FlyPA V-tail masking); or, for
//              page sizes TMA cannot tile, gather K/V rows themselves;
//   warp  8    TMEM allocation; issues the S = Q.K^T MMAs (one thread);
//   warp  9    TMA producer: page-table lookup, then 3D tensor-map loads of
//              the K/V boxes (BF16: straight into the 128-byte swizzled
//              operand layout; FP8: raw rows into a staging ring); for the
//              gather path, the page lookups into a ring of resolved slots;
//   warp 10    issues the O += P.V MMAs (one thread).
// A CTA starts from its head record (segment range, tile count, first segment
// and block) and is launched as a programmatic dependent (griddepcontrol).
// TMEM: S double buffer (2 x 64 columns), O (128 columns), P double buffer (2 x 32).
// Every wait is bounded in time; a broken invariant ends the kernel with bit 1
// of the plan's error word set instead of hanging the GPU.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "attn_paged_debug.h"
#include "e4m3.cuh"
#include "kernels.hpp"
#include "stamps.cuh"
#include "tc_common.cuh"

namespace akp {

#ifdef AKP_STAMPS
__device__ unsigned long long g_stamps[kStampCtas * kStampEvents];
#endif

namespace {

constexpr int kN = kKeyTile;                 // keys per tile (64)
constexpr int kThreads = 11 * 32;
constexpr int kBlk = kN * 128;               // one 64-column block of a 64-row tile: 8 KB
// Tile sizes for query/key head dim DQK (192, or 128 for layers with a
// symmetric head-dim pair; the value head dim is 128 either way).
template <int DQK>
struct Dims {
  static_assert(DQK % 64 == 0, "the K tile is made of 64-column blocks");
  static constexpr int kOpK = (DQK / 64) * kBlk;       // K operand tile: 24 KB at 192
  static constexpr int kOpBytes = kOpK + 2 * kBlk;      // + V operand tile: 40 KB at 192
  static constexpr int kRawK = kN * DQK;                // raw E4M3 K rows: 12 KB at 192
  static constexpr int kRawBytes = kRawK + kN * kDv;    // + raw V rows: 20 KB at 192
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 128;             // O: 128 fp32 columns
constexpr uint32_t kTmemP = 256;             // P double buffer: 2 x 32 columns (bf16 pairs)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;    // base-2 growth allowed before O is rescaled

// Gather mode only: the barriers of the slot ring, kept in dynamic shared
// memory behind the ring so the TMA kernels' static layout is unchanged.
struct SlotBars {
  uint64_t full[8], empty[8];
};

// Shared-memory layout for MR MMA rows (64 or 128): Q as three 64-column
// blocks of MR rows (two buffers where they fit), the K/V operand ring, the
// FP8 staging ring and the epilogue's copy-combine buffer.  P lives in TMEM.
template <bool FP8, int MR, bool TMA, int DQK>
struct Layout {
  static constexpr int kOpBytes = Dims<DQK>::kOpBytes;
  static constexpr int kRawBytes = Dims<DQK>::kRawBytes;
  static constexpr int kQBlock = MR * 128;    // one 64-column block of Q
  static constexpr int kQBytes = (DQK / 64) * kQBlock;
  // Q is double-buffered where it fits (BF16, M = 64): the next segment's
  // rows are staged while the current one runs.
  static constexpr int kQBufs = (!FP8 && MR == 64) ? 2 : 1;
  // copy-combine buffer of the epilogue: MR rows x 32 fp32 columns
  static constexpr int kCombBytes = MR * 32 * 4;
  static constexpr int kOpStages = FP8 ? (MR == 64 ? 3 : 2) : (TMA || MR == 64 ? 4 : 3);
  static constexpr int kRawStages = FP8 ? 3 : 0;
  static constexpr int kOffOp = kQBufs * kQBytes;
  static constexpr int kOffRaw = kOffOp + kOpStages * kOpBytes;
  static constexpr int kOffComb = kOffRaw + kRawStages * kRawBytes;
  // gather mode: a ring of kSlotRing tiles of resolved cache slots (one int64
  // per key, -1 for none), filled ahead by the producer warp
  static constexpr int kSlotRing = TMA ? 0 : 8;
  static constexpr int kOffSlots = kOffComb + kCombBytes;
  static constexpr int kOffSlotBars = kOffSlots + kSlotRing * kN * 8;
  static constexpr int kUsed = kOffSlotBars + (TMA ? 0 : (int)sizeof(SlotBars));
  static constexpr int kSmem = kUsed + 1024;  // room to align the base to 1024 B
  static constexpr int kTmaStages = FP8 ? kRawStages : kOpStages;
  // 227 KB per CTA, less the 2 KB of static shared memory.
  static_assert(kSmem + 2048 <= 227 * 1024, "shared memory layout too large");
};

struct Bars {
  uint64_t tma_full[4], tma_empty[4], edge_full[4];
  uint64_t op_full[4], op_empty[4];
  // FP8 + TMA only: V of a stage converted (v_full) and K of a stage read by
  // the Q.K^T MMAs (k_empty); op_full / op_empty then cover K / V alone
  uint64_t v_full[4], k_empty[4];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], pv_done[2];
  uint64_t o_free, final_done, sm_sync;
};


// Walks the CTA's tiles in order: segment, tile id, first/last flags.  The
// current segment and its block are cached in registers, so a tile step reads
// no memory unless it crosses into the next segment.
struct Cursor {
  const SegDesc *segs;
  const BlockDesc *blocks;
  int seg, seg_end, tile, si;
  SegDesc sd;
  BlockDesc bd;
  __device__ void init(const SegDesc *s, const BlockDesc *b, const CtaHead &h) {
    segs = s;
    blocks = b;
    seg = h.seg_begin;
    seg_end = h.seg_end;
    si = 0;
    sd = h.seg;       // the first segment and its block come with the head record
    bd = h.blk;
    pin_all();
  }
  __device__ void load() {
    sd = segs[seg];
    bd = blocks[sd.block];
    pin_all();
  }
  __device__ void pin_all() {
    // Pin every field in a register: without this the compiler may re-read a
    // field from global memory at each later use (it may assume the kernel's
    // float / bf16 stores cannot alias these ints), and under the K/V stream
    // such a re-read costs a DRAM round trip on every tile.
    pin(sd.block); pin(sd.tile_begin); pin(sd.tile_end); pin(sd.split);
    pin(bd.b); pin(bd.g); pin(bd.row0); pin(bd.nrows); pin(bd.L); pin(bd.n);
    pin(bd.tok0); pin(bd.klo); pin(bd.khi); pin(bd.num_splits); pin(bd.part_row_base);
    tile = sd.tile_begin;
  }
  static __device__ __forceinline__ void pin(int32_t &x) { asm volatile("" : "+r"(x)); }
  __device__ bool first() const { return tile == sd.tile_begin; }
  __device__ bool last() const { return tile + 1 == sd.tile_end; }
  __device__ void next() {
    if (++tile == sd.tile_end && seg + 1 < seg_end) {
      ++seg;
      ++si;
      load();
    }
  }
};

// Rows of a block are replicated across the 128 MMA rows when the block has
// at most 64 rows: row position p holds block row p % rows_pad, so each copy
// (p / rows_pad) of a row gets its own softmax thread, its own slice of every
// key tile and its own O accumulator; copies are combined once per segment.
__device__ __forceinline__ int rows_pad_of(int nrows) {
  return nrows <= 8 ? 8 : nrows <= 16 ? 16 : nrows <= 32 ? 32 : nrows <= 64 ? 64 : 128;
}

// Row positions of a segment.  Copies pay off over long segments (each
// tile's softmax is spread over more threads) but their combine makes the
// segment's epilogue ~4 us instead of ~1.5; a segment of at most 8 tiles
// keeps one copy of each row (the latency-bound small batches: tiny decode
// 23 -> 18 us, SWA with sinks 21.5 -> 16.8 us, the batched decode 1% faster).
template <int MR>
__device__ __forceinline__ int rows_pad_for(int nrows, int seg_tiles) {
  return seg_tiles <= 8 ? MR : rows_pad_of(nrows);
}


__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(tc::smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(tc::smem_u32(bar))
      : "memory");
}

// HALF (M = 64 only): every block of the plan has more than 32 rows, so each
// row has one copy, and lanes l and l + 16 of a softmax warp share row
// 16w + l % 16, each taking 32 of the tile's 64 key columns (the two-half
// 16-lane TMEM shapes): every lane works, on half the columns.
template <bool FP8, bool TMA, int MR, int DQK, bool HALF>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const RunArgs args, const __grid_constant__ TmaMaps maps) {
  static_assert(!HALF || MR == 64, "two threads per row only with the M = 64 layout");
  // A plain local copy of the arguments: the role lambdas capture by reference,
  // and a reference into kernel-parameter space would turn every field read
  // inside them into a memory load that the K/V stream keeps evicting.
  const RunArgs a = args;
  using Lay = Layout<FP8, MR, TMA, DQK>;
  // this instantiation's query/key head dim and tile sizes
  constexpr int kDqk = DQK;
  constexpr int kOpK = Dims<DQK>::kOpK;
  constexpr int kOpBytes = Dims<DQK>::kOpBytes;
  constexpr int kRawK = Dims<DQK>::kRawK;
  constexpr int kRawBytes = Dims<DQK>::kRawBytes;
  constexpr int kRows = MR;                 // MMA rows (M)
  constexpr int kQBlock = Lay::kQBlock;
  constexpr int NS = Lay::kOpStages;
  constexpr int NT = Lay::kTmaStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ Bars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float sm_m[128], sm_l[128];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  if (tid == 0) AKP_STAMP(kStampStart);
  // Launched as a programmatic dependent (of the device planner or the KV
  // append, when they precede it): nothing they write is read before this wait.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  // The split merge (a programmatic dependent of this kernel) may be scheduled
  // from here on: it reads the plan's blocks before its own wait, so only once
  // the planner that writes them has completed; it waits for this grid's
  // completion before it reads anything written here.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // the CTA's head record: segment range, tile count, first segment and block
  const CtaHead head = a.cta_heads[blockIdx.x];
  const int seg_begin = head.seg_begin;
  const int seg_end = head.seg_end;
  if (seg_begin >= seg_end) return;
  const int total = head.total;
  if (tid == 0) {
    AKP_STAMP(kStampHead);
    AKP_STAMP_VALUE(kStampSegs, seg_end - seg_begin);
    AKP_STAMP_VALUE(kStampTiles, total);
    AKP_STAMP_SMID(kStampSm);
  }
  if constexpr (HALF) {
    // Verify plans: while the barriers are set up, the producer warp warms
    // the page-table entries of the CTA's first four tiles and the converter
    // warps the first block's Q rows (L2 prefetches, within the block's own
    // entries and rows), so that neither the first TMA issue nor the first Q
    // staging waits on a DRAM round trip (c3a 59.8 -> 56.0 us with L2
    // flushed; the page-table prefetch in the decode instantiation measured
    // 1 us slower on the batched decode).
    if (warp == 9) {
      const BlockDesc &b0 = head.blk;
      const int lane = tid & 31;
      const int key0 = head.seg.tile_begin * kN;
      const int e0 = key0 / a.page_size;
      const int e1 = min(b0.khi - 1, key0 + 4 * kN - 1) / a.page_size;
      const int32_t *pt_row = a.page_table + (int64_t)b0.b * a.pt_stride;
      const int line0 = (int)(reinterpret_cast<uintptr_t>(pt_row + e0) >> 7);
      const int nline = (int)(reinterpret_cast<uintptr_t>(pt_row + e1) >> 7) - line0 + 1;
      if (lane < nline)
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(pt_row + min(e0 + lane * 32, e1)) : "memory");
    } else if (warp >= 4 && warp < 8) {
      const BlockDesc &b0 = head.blk;
      const int ct = tid - 128;
      for (int i = ct; i < b0.nrows * (kDqk / 64); i += 128) {
        const int r = i / (kDqk / 64), part = i % (kDqk / 64);
        const int flat = b0.row0 + r;
        const uint16_t *row = static_cast<const uint16_t *>(a.q) +
                              ((int64_t)(b0.tok0 + flat / a.group) * a.hq + b0.g * a.group + flat % a.group) * kDqk;
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(row + part * 64) : "memory");
      }
    }
  }

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < 4; ++s) {
      tc::mbar_init(&bars.tma_full[s], 1);
      tc::mbar_init(&bars.tma_empty[s], 128);
      tc::mbar_init(&bars.edge_full[s], 1);
      tc::mbar_init(&bars.op_full[s], 128);
      tc::mbar_init(&bars.op_empty[s], 1);
      tc::mbar_init(&bars.v_full[s], 128);
      tc::mbar_init(&bars.k_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bars.q_full[i], 128);
      tc::mbar_init(&bars.q_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars.s_full[b], 1);
      tc::mbar_init(&bars.s_empty[b], 128);
      tc::mbar_init(&bars.p_full[b], 128);
      tc::mbar_init(&bars.pv_done[b], 1);
    }
    tc::mbar_init(&bars.o_free, 128);
    tc::mbar_init(&bars.final_done, 2);
    tc::mbar_init(&bars.sm_sync, 128);
    if (!TMA) {
      SlotBars *sb = reinterpret_cast<SlotBars *>(smem + Lay::kOffSlotBars);
      for (int r = 0; r < 8; ++r) {
        tc::mbar_init(&sb->full[r], 32);
        tc::mbar_init(&sb->empty[r], 128);
      }
    }
    tc::fence_mbar_init();
  }
  if (warp == 8) tc::tmem_alloc(&tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t sbase = tc::smem_u32(smem);
  if (tid == 0) AKP_STAMP(kStampReady);
  SlotBars *slot_bars = reinterpret_cast<SlotBars *>(smem + Lay::kOffSlotBars);

  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    if (!TMA) {
      // Gather mode: the warp resolves every key's cache slot (page lookup)
      // and fills the slot ring up to kSlotRing tiles ahead of the converters,
      // four tiles per round trip to memory: each lane looks up two keys of
      // each of the four tiles before storing any of them.
      constexpr int R = Lay::kSlotRing > 0 ? Lay::kSlotRing : 1;   // 0 in TMA kernels (unused)
      constexpr int kBatchTiles = 4;
      const int ln = tid & 31;
      int64_t *ring = reinterpret_cast<int64_t *>(smem + Lay::kOffSlots);
      Cursor cur;
      cur.init(a.segs, a.blocks, head);
      bool ok = true;
      for (int k0 = 0; k0 < total && ok; k0 += kBatchTiles) {
        int64_t sl[kBatchTiles][2];
#pragma unroll
        for (int u = 0; u < kBatchTiles; ++u) {
          const BlockDesc &bd = cur.bd;
          const int32_t *pt_row = a.page_table + (int64_t)bd.b * a.pt_stride;
          const int key0 = cur.tile * kN;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int j = key0 + 2 * ln + q;
            sl[u][q] = -1;
            if (k0 + u < total && j >= bd.klo && j < bd.khi) {
              const int32_t page = __ldg(pt_row + j / a.page_size);
              if (page >= 0 && page < a.num_pages)
                sl[u][q] = (int64_t)page * a.page_size + j % a.page_size;
              else
                atomicOr(a.err, 1);
            }
          }
          if (k0 + u < total) cur.next();
        }
#pragma unroll
        for (int u = 0; u < kBatchTiles; ++u) {
          const int k = k0 + u;
          if (k >= total) break;
          const int r = k % R;
          if (k >= R && !tc::mbar_wait_warp(&slot_bars->empty[r], ((k / R) - 1) & 1, &abort_flag)) {
            ok = false;
            break;
          }
          ring[r * kN + 2 * ln] = sl[u][0];
          ring[r * kN + 2 * ln + 1] = sl[u][1];
          tc::mbar_arrive(&slot_bars->full[r]);
          if (k == 0 && ln == 0) AKP_STAMP(kStampFirstLoad);
        }
      }
    }
    if (TMA && (tid & 31) == 0) {
      const int box = a.page_size >= kN ? kN : a.page_size;   // key rows per box
      const int nbox = kN / box;
      const int oob = a.num_pages * a.page_size;              // first slot past the pool
      constexpr uint32_t kTileBytes = FP8 ? kRawBytes : kOpBytes;
      Cursor cur;
      cur.init(a.segs, a.blocks, head);
      for (int k = 0; k < total; ++k, cur.next()) {
        const int t = k % NT;
        const BlockDesc &bd = cur.bd;
        const int32_t *pt_row = a.page_table + (int64_t)bd.b * a.pt_stride;
        const int key0 = cur.tile * kN;
        // page-table lookups first: their latency overlaps the wait for a free stage
        int slot[kN / 8];
#pragma unroll
        for (int i = 0; i < kN / 8; ++i) {
          slot[i] = oob;  // boxes with no visible key read past the pool: zero fill
          const int j = key0 + i * box;
          if (i < nbox && j + box > bd.klo && j < bd.khi) {
            const int32_t page = __ldg(pt_row + j / a.page_size);
            if (page >= 0 && page < a.num_pages)
              slot[i] = page * a.page_size + j % a.page_size;
            else
              atomicOr(a.err, 1);
          }
        }
        if (k == 0) AKP_STAMP(kStampLookup);
        uint64_t *empty = FP8 ? &bars.tma_empty[t] : &bars.op_empty[t];
        if (k >= NT && !tc::mbar_wait(empty, ((k / NT) - 1) & 1, &abort_flag)) break;
        // BF16: a tile with keys outside the block's range lands on edge_full, which
        // only the converters wait on (they zero those V rows); every other tile
        // lands on tma_full, which only the Q.K^T issuer waits on.
        const bool edge = !FP8 && (key0 < bd.klo || key0 + kN > bd.khi);
        uint64_t *full = edge ? &bars.edge_full[t] : &bars.tma_full[t];
        mbar_expect_tx(full, kTileBytes);
        const uint32_t dst = sbase + (FP8 ? Lay::kOffRaw + t * kRawBytes : Lay::kOffOp + t * kOpBytes);
#pragma unroll
        for (int i = 0; i < kN / 8; ++i) {
          if (i >= nbox) break;
          if (FP8) {
            tma_load_3d(dst + i * box * kDqk, &maps.k, 0, bd.g, slot[i], full);
            tma_load_3d(dst + kRawK + i * box * kDv, &maps.v, 0, bd.g, slot[i], full);
          } else {
#pragma unroll
            for (int c = 0; c < kDqk / 64; ++c)
              tma_load_3d(dst + c * kBlk + i * box * 128, &maps.k, 64 * c, bd.g, slot[i],
                          full);
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_load_3d(dst + kOpK + c * kBlk + i * box * 128, &maps.v, 64 * c, bd.g, slot[i],
                          full);
          }
        }
        if (k == 0) AKP_STAMP(kStampFirstLoad);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ converters
    const int ct = tid - 128;
    const uint8_t *kc = static_cast<const uint8_t *>(a.k_cache);
    const uint8_t *vc = static_cast<const uint8_t *>(a.v_cache);
    Cursor cur;
    cur.init(a.segs, a.blocks, head);
    // Stage the Q rows of the cursor's segment (row position p holds block
    // row p % rows_pad).  The loads go out 8-12 at a time: under a saturated
    // K/V stream each round trip to memory takes microseconds.
    auto stage_q = [&](const Cursor &c) -> bool {
      constexpr int QB = Lay::kQBufs;
      const BlockDesc &bd = c.bd;
      const int qb = c.si % QB;
      if (c.si >= QB && !tc::mbar_wait_warp(&bars.q_empty[qb], ((c.si / QB) - 1) & 1, &abort_flag))
        return false;
      uint8_t *qs = smem + qb * Lay::kQBytes;
      const int rows_pad = rows_pad_for<kRows>(bd.nrows, c.sd.tile_end - c.sd.tile_begin);
      constexpr int kQch = kDqk / 8;       // 16-byte chunks per Q row
      constexpr int kIters = kRows * kQch / 128;
      constexpr int kBatch = kRows == 64 && kIters % 12 == 0 ? 12 : 8;
      static_assert(kIters % kBatch == 0, "Q staging batches");
#pragma unroll 1
      for (int i0 = 0; i0 < kIters; i0 += kBatch) {
        uint4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int idx = ct + (i0 + u) * 128;
          const int p = idx / kQch;        // MMA row position
          const int r = p % rows_pad;      // block row it holds
          const int ch = idx % kQch;
          v[u] = make_uint4(0u, 0u, 0u, 0u);
          if (r < bd.nrows) {
            const int flat = bd.row0 + r;
            const int tok = bd.tok0 + flat / a.group;
            const int h = bd.g * a.group + flat % a.group;
            v[u] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.q) +
                                                         ((int64_t)tok * a.hq + h) * kDqk) + ch);
          }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int idx = ct + (i0 + u) * 128;
          const int p = idx / kQch;
          const int ch = idx % kQch;
          *reinterpret_cast<uint4 *>(qs + (ch >> 3) * kQBlock + tc::sw128_offset(p, ch & 7)) = v[u];
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&bars.q_full[qb]);
      if (ct == 0 && c.si == 0) AKP_STAMP(kStampFirstQ);
      return true;
    };
    if constexpr (FP8 && TMA) {
      // FP8 rows staged by TMA: [64 keys x 192 B] K then [64 keys x 128 B] V.
      // Both halves are read into registers and the raw stage goes back to
      // the TMA producer at once (after a proxy fence: the refill must not
      // overtake these reads); then K and V are converted into the operand
      // stage, whose two halves are released separately: K once Q.K^T has
      // read it (k_empty), V once P.V has (op_empty).
      for (int k = 0; k < total; ++k, cur.next()) {
        const BlockDesc &bd = cur.bd;
        if (cur.first() && !stage_q(cur)) break;
        const int s = k % NS, t = k % NT;
        const int key0 = cur.tile * kN;
        constexpr int kKch = kDqk / 16;            // 16-byte source chunks per K row
        constexpr int kVch = kDv / 16;
        constexpr int kPerK = kN * kKch / 128;
        constexpr int kPerV = kN * kVch / 128;
        if (!tc::mbar_wait_warp(&bars.tma_full[t], (k / NT) & 1, &abort_flag)) break;
        const uint8_t *raw = smem + Lay::kOffRaw + t * kRawBytes;
        uint4 bk[kPerK], bv[kPerV];
#pragma unroll
        for (int u = 0; u < kPerK; ++u) {
          const int c = ct + u * 128;
          bk[u] = *reinterpret_cast<const uint4 *>(raw + (c / kKch) * kDqk + (c % kKch) * 16);
        }
#pragma unroll
        for (int u = 0; u < kPerV; ++u) {
          const int c = ct + u * 128;
          bv[u] = *reinterpret_cast<const uint4 *>(raw + kRawK + (c / kVch) * kDv + (c % kVch) * 16);
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&bars.tma_empty[t]);
        uint8_t *dst = smem + Lay::kOffOp + s * kOpBytes;
        if (k >= NS && !tc::mbar_wait_warp(&bars.k_empty[s], ((k / NS) - 1) & 1, &abort_flag))
          break;
#pragma unroll
        for (int u = 0; u < kPerK; ++u) {
          const int c = ct + u * 128;
          const int kk = c / kKch, c16 = 2 * (c % kKch);
          const int j = key0 + kk;
          uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
          if (j >= bd.klo && j < bd.khi) e4m3x16_to_bf16(bk[u], lo, hi);
          *reinterpret_cast<uint4 *>(dst + (c16 >> 3) * kBlk + tc::sw128_offset(kk, c16 & 7)) = lo;
          *reinterpret_cast<uint4 *>(dst + ((c16 + 1) >> 3) * kBlk +
                                     tc::sw128_offset(kk, (c16 + 1) & 7)) = hi;
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&bars.op_full[s]);
        if (k >= NS && !tc::mbar_wait_warp(&bars.op_empty[s], ((k / NS) - 1) & 1, &abort_flag))
          break;
        dst += kOpK;
#pragma unroll
        for (int u = 0; u < kPerV; ++u) {
          const int c = ct + u * 128;
          const int kk = c / kVch, c16 = 2 * (c % kVch);
          const int j = key0 + kk;
          uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
          if (j >= bd.klo && j < bd.khi) e4m3x16_to_bf16(bv[u], lo, hi);
          *reinterpret_cast<uint4 *>(dst + (c16 >> 3) * kBlk + tc::sw128_offset(kk, c16 & 7)) = lo;
          *reinterpret_cast<uint4 *>(dst + ((c16 + 1) >> 3) * kBlk +
                                     tc::sw128_offset(kk, (c16 + 1) & 7)) = hi;
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&bars.v_full[s]);
      }
    } else {
    uint32_t edge_parity = 0;   // BF16 + TMA: completed edge tiles per stage (one bit each)
    for (int k = 0; k < total; ++k, cur.next()) {
      const BlockDesc &bd = cur.bd;
      if (cur.first() && !stage_q(cur)) break;
      const int s = k % NS;
      const int key0 = cur.tile * kN;
      uint8_t *op = smem + Lay::kOffOp + s * kOpBytes;
      if (TMA && !FP8) {
        // BF16 tile landed by TMA in operand layout.  Interior tiles go straight
        // to the Q.K^T issuer; on edge tiles zero the V rows outside the range first.
        if (key0 >= bd.klo && key0 + kN <= bd.khi) continue;
        if (!tc::mbar_wait(&bars.edge_full[s], (edge_parity >> s) & 1, &abort_flag)) break;
        edge_parity ^= 1u << s;
        {
          for (int idx = ct; idx < kN * 16; idx += 128) {
            const int kk = idx >> 4;
            const int j = key0 + kk;
            if (j < bd.klo || j >= bd.khi) {
              const int c = (idx >> 3) & 1;
              *reinterpret_cast<uint4 *>(op + kOpK + c * kBlk + tc::sw128_offset(kk, idx & 7)) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&bars.op_full[s]);
        continue;
      }
      constexpr int kEs = FP8 ? 1 : 2;
      constexpr int kKch = kDqk * kEs / 16;  // source 16-byte chunks per K row
      constexpr int kVch = kDv * kEs / 16;
      constexpr int kPer = kN * (kKch + kVch) / 128;
      // Gather (page sizes TMA cannot tile): two threads per key.  The key's
      // cache slot comes from the ring the producer warp fills ahead; the row
      // loads go out before the wait for a free operand stage, so their
      // latency overlaps it.  Chunk u of this thread: (is K, key within the
      // tile, 16-byte chunk of the row).
      auto chunk_of = [&](int u, bool &is_k, int &kk, int &ch) {
        kk = ct >> 1;
        const int part = ct & 1;
        is_k = u < kKch / 2;
        ch = is_k ? part * (kKch / 2) + u : part * (kVch / 2) + (u - kKch / 2);
      };
      uint4 buf[kPer];
      {
        constexpr int R = Lay::kSlotRing > 0 ? Lay::kSlotRing : 1;   // 0 in TMA kernels (unused)
        const int r = k % R;
        if (!tc::mbar_wait_warp(&slot_bars->full[r], (k / R) & 1, &abort_flag)) break;
        const int64_t slot = reinterpret_cast<const int64_t *>(smem + Lay::kOffSlots)[r * kN + (ct >> 1)];
        tc::mbar_arrive(&slot_bars->empty[r]);
        const int64_t srow = (slot >= 0 ? slot : 0) * a.hkv + bd.g;
        const uint4 *krow = reinterpret_cast<const uint4 *>(kc + srow * (kDqk * kEs));
        const uint4 *vrow = reinterpret_cast<const uint4 *>(vc + srow * (kDv * kEs));
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          bool is_k;
          int kk, ch;
          chunk_of(u, is_k, kk, ch);
          buf[u] = slot >= 0 ? __ldg((is_k ? krow : vrow) + ch) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (k >= NS && !tc::mbar_wait(&bars.op_empty[s], ((k / NS) - 1) & 1, &abort_flag)) break;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        bool is_k;
        int kk, ch;
        chunk_of(u, is_k, kk, ch);
        const int j = key0 + kk;
        const bool keep = j >= bd.klo && j < bd.khi;
        uint8_t *dst = op + (is_k ? 0 : kOpK);
        if (FP8) {
          uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
          if (keep) e4m3x16_to_bf16(buf[u], lo, hi);
          const int c16 = 2 * ch;
          *reinterpret_cast<uint4 *>(dst + (c16 >> 3) * kBlk + tc::sw128_offset(kk, c16 & 7)) = lo;
          *reinterpret_cast<uint4 *>(dst + ((c16 + 1) >> 3) * kBlk +
                                     tc::sw128_offset(kk, (c16 + 1) & 7)) = hi;
        } else {
          *reinterpret_cast<uint4 *>(dst + (ch >> 3) * kBlk + tc::sw128_offset(kk, ch & 7)) =
              keep ? buf[u] : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&bars.op_full[s]);
    }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ S = Q.K^T issuer
    // One thread issues every Q.K^T MMA, in tile order.  P.V goes out from a
    // thread of its own (warp 10): an MMA issue blocks the issuing thread for
    // as long as the tensor pipe takes to accept it, so with one issuer P.V of
    // tile k would queue behind the whole Q.K^T of tile k+1.
    if ((tid & 31) == 0) {
      const uint32_t id_s = tc::idesc_f16(1, 0, 0, kRows, kN);
      Cursor cs;
      cs.init(a.segs, a.blocks, head);
      // BF16 + TMA: interior tiles are consumed straight off the TMA barrier;
      // edge tiles wait for the converters, whose barrier then completes only
      // on edge tiles (one parity bit per stage).
      uint32_t edge_parity = 0, inner_parity = 0;
      for (int ks = 0; ks < total; ++ks, cs.next()) {
        const int s = ks % NS;
        const int b = ks & 1;
        const int key0 = cs.tile * kN;
        constexpr int QB = Lay::kQBufs;
        const int qb = cs.si % QB;
        if (cs.first() && !tc::mbar_wait(&bars.q_full[qb], (cs.si / QB) & 1, &abort_flag)) break;
        bool ok;
        if (TMA && !FP8) {
          if (key0 < cs.bd.klo || key0 + kN > cs.bd.khi) {
            ok = tc::mbar_wait(&bars.op_full[s], (edge_parity >> s) & 1, &abort_flag);
            edge_parity ^= 1u << s;
          } else {
            ok = tc::mbar_wait(&bars.tma_full[s], (inner_parity >> s) & 1, &abort_flag);
            inner_parity ^= 1u << s;
          }
        } else {
          ok = tc::mbar_wait(&bars.op_full[s], (ks / NS) & 1, &abort_flag);
        }
        if (!ok) break;
        if (ks >= 2 && !tc::mbar_wait(&bars.s_empty[b], ((ks >> 1) - 1) & 1, &abort_flag)) break;
        tc::tc_fence_after();
        const uint32_t kb = sbase + Lay::kOffOp + s * kOpBytes;
#pragma unroll
        for (int kq = 0; kq < kDqk / 16; ++kq) {
          const uint32_t koff = (kq & 3) * 32;
          const uint64_t ad = tc::smem_desc_sw128(sbase + qb * Lay::kQBytes + (kq >> 2) * kQBlock + koff,
                                                  16, 1024);
          const uint64_t bdsc = tc::smem_desc_sw128(kb + (kq >> 2) * kBlk + koff, 16, 1024);
          tc::mma_f16_ss(tmem + b * kN, ad, bdsc, id_s, kq > 0 ? 1u : 0u);
        }
        tc::mma_commit(&bars.s_full[b]);
        if (ks == 0) AKP_STAMP(kStampFirstQK);
        if (FP8 && TMA) tc::mma_commit(&bars.k_empty[s]);
        if (cs.last()) tc::mma_commit(&bars.q_empty[qb]);
      }
      tc::mma_commit(&bars.final_done);
      tc::mbar_wait(&bars.final_done, 0, &abort_flag);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ O += P.V issuer
    if ((tid & 31) == 0) {
      const uint32_t id_pv = tc::idesc_f16(1, 0, 1, kRows, kDv);
      Cursor cp;
      cp.init(a.segs, a.blocks, head);
      for (int kp = 0; kp < total; ++kp, cp.next()) {
        const int b = kp & 1;
        const int s = kp % NS;
        const bool first = cp.first();
        if (!tc::mbar_wait(&bars.p_full[b], (kp >> 1) & 1, &abort_flag)) break;
        if (FP8 && TMA && !tc::mbar_wait(&bars.v_full[s], (kp / NS) & 1, &abort_flag)) break;
        // the first P.V of a segment overwrites O: the epilogue of the
        // previous segment must have read it
        if (first && cp.si > 0 && !tc::mbar_wait(&bars.o_free, (cp.si - 1) & 1, &abort_flag))
          break;
        tc::tc_fence_after();
        const uint32_t vb = sbase + Lay::kOffOp + s * kOpBytes + kOpK;
#pragma unroll
        for (int kk = 0; kk < kN / 16; ++kk) {
          const uint64_t bdsc = tc::smem_desc_sw128(vb + kk * 16 * 128, kBlk, 1024);
          tc::mma_f16_ts(tmem + kTmemO, tmem + kTmemP + b * 32 + kk * 8, bdsc, id_pv,
                         (!first || kk > 0) ? 1u : 0u);
        }
        // P.V of tile k completes after Q.K^T of tile k (P needed S): the
        // stage's V (and K, where K has no barrier of its own) may be
        // overwritten now
        tc::mma_commit(&bars.op_empty[s]);
        tc::mma_commit(&bars.pv_done[b]);
        if (kp == total - 1) AKP_STAMP(kStampLastPV);
      }
      tc::mma_commit(&bars.final_done);
      tc::mbar_wait(&bars.final_done, 0, &abort_flag);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = tid;
    const int lane = t & 31;
    // MMA row position held in this thread's TMEM lane: with M = 128 row p is
    // lane p; with M = 64 rows 16w..16w+15 sit in lanes 0-15 of warp w's
    // subpartition and lanes 16-31 hold no row (pos = -1).
    const int pos = kRows == 128 ? t : (HALF || lane < 16 ? warp * 16 + (lane & 15) : -1);
    const int half = HALF ? lane >> 4 : 0;   // which 32 of the row's 64 columns
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    Cursor cur;
    cur.init(a.segs, a.blocks, head);
    float m_run = -INFINITY, l_run = 0.f;
    int row_lo = 0, row_hi = 0, rr = 0, rows_pad = kRows, col0 = 0, off = 0, len = kN, nc = kN;
    int zero_pending = 0;
    int row_tok = 0, row_h = 0;
    float sink2 = -INFINITY;
    bool valid = false, warp_live = false;
    uint32_t sync_phase = 0;
    // Bounded wait with a warp-uniform outcome: the TMEM loads that follow are
    // warp-collective, so a warp must never split on a give-up.
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity, &abort_flag));
    };
    // bounded rendezvous of the 128 softmax threads; the four warps reach it
    // together, so it polls instead of sleeping (a suspended wait resumes
    // well after the phase completes)
    auto group_sync = [&]() -> bool {
      tc::mbar_arrive(&bars.sm_sync);
      const bool ok =
          __all_sync(0xffffffffu, tc::mbar_wait_spin(&bars.sm_sync, sync_phase, &abort_flag));
      sync_phase ^= 1;
      return ok;
    };
    // One key tile: S slice from TMEM -> mask -> P slice to TMEM.
    // A thread owns nc (16, 32 or 64) key columns of its row, read from TMEM in
    // 16-column chunks; the load of chunk c+1 is in flight while chunk c is
    // processed.  The loops are not unrolled beyond that pair, so this hot code
    // stays small: each SM sub-partition's instruction cache also holds the
    // converter and MMA loops, and a fully unrolled 64-column body thrashes it.
    //
    // P is computed against the running maximum m_run in a single pass over S,
    // tracking the tile maximum on the way.  Only when some value exceeds
    // m_run by more than the rescale threshold (rare once the maximum has
    // settled) is O rescaled and the pass repeated against the new maximum.
    // The first tile of a segment (m_run = -inf) takes a max pass first.
    // Columns outside the thread's visible range read as -inf.  The score
    // scale is positive (the entry points reject anything else), so maxima are
    // taken on the raw dot products and -inf stays -inf once scaled.
    auto mask16 = [&](uint32_t (&raw)[16], int c, int j_lo, int j_hi) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int jj = 16 * c + j;
        raw[j] = ((jj >= j_lo) & (jj < j_hi)) ? raw[j] : 0xFF800000u;
      }
    };
    auto tile_body = [&](int k) -> bool {
      const int b = k & 1;
      // visible columns of this thread in the warp's nc-column window: its own
      // slice [off, off + len) clipped to the row's keys [row_lo, row_hi)
      const int key0 = cur.tile * kN + col0;
      const int j_lo = max(off, row_lo - key0);
      const int j_hi = min(off + len, row_hi - key0);
      const uint32_t taddr = tmem + lane_base + b * kN + col0;
      const int nch = nc >> 4;
      const float sc = a.scale_log2;
      // P buffer b is free once P.V of tile k-2 is done
      if (k >= 2 && !wait(&bars.pv_done[b], ((k - 2) >> 1) & 1))
        return false;
      if (!warp_live) {
        tc::tc_fence_before();
        tc::mbar_arrive(&bars.s_empty[b]);
        return true;
      }
      // interior tiles (every column of every thread visible) skip the mask
      const bool full = __all_sync(0xffffffffu, j_lo <= 0 && j_hi >= nc);
      uint32_t ra[16], rb[16];
      // The TMEM loads are warp-collective: the whole warp takes the max pass
      // when any of its rows needs it, and only those rows adopt its result.
      const bool want_max = valid && (cur.first() || m_run == -INFINITY);
      if (HALF && __any_sync(0xffffffffu, want_max)) {
        uint32_t r[32];
        tc::tmem_ld_16x32bx2_x32<32>(taddr, r);
        tc::tmem_wait_ld_regs32(r);
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int jj = 32 * half + j;
          const float x0 = (jj >= j_lo) & (jj < j_hi) ? __uint_as_float(r[j]) : -INFINITY;
          const float x1 = (jj + 1 >= j_lo) & (jj + 1 < j_hi) ? __uint_as_float(r[j + 1]) : -INFINITY;
          mx[(j >> 1) & 1] = tc::max3(mx[(j >> 1) & 1], x0, x1);
        }
        float m = fmaxf(mx[0], mx[1]);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (want_max) m_run = m * sc;
      } else if (!HALF && __any_sync(0xffffffffu, want_max)) {
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          tc::tmem_ld16(taddr + 16 * c, ra);
          tc::tmem_wait_ld_regs(ra);
          mask16(ra, c, j_lo, j_hi);
#pragma unroll
          for (int j = 0; j < 16; j += 2)
            mx[(j >> 1) & 3] = tc::max3(mx[(j >> 1) & 3], __uint_as_float(ra[j]), __uint_as_float(ra[j + 1]));
        }
        if (want_max) m_run = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
      }
      // P of this thread's row: 16-bit pairs in TMEM columns kTmemP + 32b + key/2
      const uint32_t pcol = tmem + lane_base + kTmemP + b * 32;
      const int g0 = col0 >> 4;          // first 16-key group of the window
      if (zero_pending > 0) {
        // P columns outside the window stay zero for the whole segment: write
        // them once per buffer (the first two tiles), not on every tile
        --zero_pending;
        const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll 1
        for (int gi = 0; gi < kN / 16; ++gi)
          if (gi < g0 || gi >= g0 + nch) tc::tmem_st8(pcol + 8 * gi, z);
      }
      // exp pass over chunk c held in raw: P = 2^(s * sc - m) to smem, row sums
      // and the raw maximum
      float rs[4], mx[4];
      const auto exp16 = [&](uint32_t (&raw)[16], int c, float neg_m) {
        if (!full) mask16(raw, c, j_lo, j_hi);
        uint32_t pk[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float x0 = __uint_as_float(raw[j]), x1 = __uint_as_float(raw[j + 1]);
          mx[(j >> 1) & 3] = tc::max3(mx[(j >> 1) & 3], x0, x1);
          float y0, y1;
          tc::ffma2(y0, y1, x0, x1, sc, neg_m);
          const float p0 = ex2(y0), p1 = ex2(y1);
          if (j & 2)
            tc::fadd2(rs[2], rs[3], p0, p1);
          else
            tc::fadd2(rs[0], rs[1], p0, p1);
          pk[j / 2] = cvt_pair(p0, p1);
        }
        tc::tmem_st8(pcol + 8 * (g0 + c), pk);
      };
#pragma unroll 1
      for (int pass = 0;; ++pass) {
        const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          rs[i] = 0.f;
          mx[i] = -INFINITY;
        }
        if constexpr (HALF) {
          // this thread's 32 columns in one TMEM round trip; P goes back as 16
          // pairs, the halves 16 pair columns apart
          uint32_t r[32];
          tc::tmem_ld_16x32bx2_x32<32>(taddr, r);
          tc::tmem_wait_ld_regs32(r);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int jj = 32 * half + j;
            float x0 = __uint_as_float(r[j]), x1 = __uint_as_float(r[j + 1]);
            if (!full) {
              x0 = (jj >= j_lo) & (jj < j_hi) ? x0 : -INFINITY;
              x1 = (jj + 1 >= j_lo) & (jj + 1 < j_hi) ? x1 : -INFINITY;
            }
            mx[(j >> 1) & 3] = tc::max3(mx[(j >> 1) & 3], x0, x1);
            float y0, y1;
            tc::ffma2(y0, y1, x0, x1, sc, neg_m);
            const float p0 = ex2(y0), p1 = ex2(y1);
            if (j & 2)
              tc::fadd2(rs[2], rs[3], p0, p1);
            else
              tc::fadd2(rs[0], rs[1], p0, p1);
            pk[j / 2] = cvt_pair(p0, p1);
          }
          tc::tmem_st_16x32bx2_x16<16>(pcol, pk);
        } else {
          tc::tmem_ld16(taddr, ra);
          tc::tmem_wait_ld_regs(ra);
#pragma unroll 1
          for (int c = 0; c < nch; c += 2) {
            if (c + 1 < nch) tc::tmem_ld16(taddr + 16 * (c + 1), rb);
            exp16(ra, c, neg_m);
            if (c + 1 < nch) {
              tc::tmem_wait_ld_regs(rb);
              if (c + 2 < nch) tc::tmem_ld16(taddr + 16 * (c + 2), ra);
              exp16(rb, c + 1, neg_m);
              if (c + 2 < nch) tc::tmem_wait_ld_regs(ra);
            }
          }
        }
        float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
        // the two halves of a row agree on its tile maximum
        if (HALF) m_tile = fmaxf(m_tile, __shfl_xor_sync(0xffffffffu, m_tile, 16));
        const bool need = m_tile > m_run + kRescaleThreshold;
        if (pass > 0 || !__any_sync(0xffffffffu, need)) break;
        // rare: the maximum grew past the threshold; rescale O and redo
        if (!wait(&bars.pv_done[(k - 1) & 1], ((k - 1) >> 1) & 1))
          return false;
        tc::tc_fence_after();
        const float alpha = need ? ex2(m_run - m_tile) : 1.f;
#pragma unroll 1
        for (int c = 0; c < kDv / 32; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(tmem + lane_base + kTmemO + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tc::tmem_st32(tmem + lane_base + kTmemO + c * 32, o);
        }
        tc::tmem_wait_st();
        l_run *= alpha;
        if (need) m_run = m_tile;
      }
      tc::tmem_wait_st();                // P is in TMEM before p_full is signalled
      tc::tc_fence_before();
      tc::mbar_arrive(&bars.s_empty[b]);
      l_run += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      return true;
    };

    for (int k = 0; k < total; ++k, cur.next()) {
      const BlockDesc &bd = cur.bd;
      if (cur.first()) {
        // HALF plans: one copy per row
        rows_pad = HALF ? kRows : rows_pad_for<kRows>(bd.nrows, cur.sd.tile_end - cur.sd.tile_begin);
        rr = pos >= 0 ? pos % rows_pad : 0;
        valid = pos >= 0 && rr < bd.nrows;
        // copy c = pos / rows_pad of a row owns key columns [c*len, (c+1)*len) of
        // every tile; a warp reads the columns of the copies it holds
        constexpr int ppw = kRows / 4;           // row positions per warp
        len = kN * rows_pad / kRows;
        if (rows_pad <= ppw) {                   // several copies per warp: 16 columns
          nc = 16;
          col0 = 16 * warp;
          off = (pos >= 0 ? pos / rows_pad : 0) * len - col0;
        } else {                                 // part of one copy per warp
          nc = len;
          col0 = ((warp * ppw) / rows_pad) * len;
          off = 0;
        }
        warp_live = __any_sync(0xffffffffu, valid);
        row_lo = row_hi = 0;
        sink2 = -INFINITY;
        if (valid) {
          // the row's query token and head, and its sink logit in base 2: read
          // now, their latency hidden behind the segment's tiles
          const int flat = bd.row0 + rr;
          row_tok = bd.tok0 + flat / a.group;
          row_h = bd.g * a.group + flat % a.group;
          if (a.sinks) sink2 = a.sinks[row_h] * kLog2e;
          const int i = bd.L - bd.n + (bd.row0 + rr) / a.group;
          row_hi = i + 1;
          row_lo = a.window > 0 ? max(0, i - a.window + 1) : 0;
        }
        m_run = -INFINITY;
        l_run = 0.f;
        zero_pending = nc < kN ? 2 : 0;
      }
      const int b = k & 1;
      if (!wait(&bars.s_full[b], (k >> 1) & 1)) break;
      if (t == 0 && k == 0) AKP_STAMP(kStampFirstS);
      tc::tc_fence_after();
      if (!tile_body(k)) break;
      tc::tc_fence_before();
      tc::mbar_arrive(&bars.p_full[b]);
      if (!cur.last()) continue;

      // ---------------- end of segment: normalise and write the block's rows
      if (!wait(&bars.pv_done[b], (k >> 1) & 1)) break;
      if (t == 0) AKP_STAMP(kStampEpiBegin);
      if constexpr (HALF) {
        // the row's two halves: one denominator; the lower half writes the row
        // (its lane holds the row's O)
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
        valid = valid && half == 0;
      }
      tc::tc_fence_after();
      const SegDesc &sd = cur.sd;
      const bool single = bd.num_splits == 1;
      if (rows_pad == kRows) {
        // one copy per row: the thread owns its row position outright
        if (warp_live) {
          int tok = 0, h = 0;
          if (valid) {
            const int flat = bd.row0 + pos;
            tok = bd.tok0 + flat / a.group;
            h = bd.g * a.group + flat % a.group;
          }
          float scale_o = 0.f, lse = -INFINITY;
          if (single) {
            const float sig = valid ? sink2 : -INFINITY;
            const float MM = fmaxf(m_run, sig);
            if (MM != -INFINITY) {
              const float Z = l_run * exp2f(m_run - MM) + exp2f(sig - MM);
              scale_o = exp2f(m_run - MM) * a.v_scale / Z;
              lse = (MM + log2f(Z)) * kLn2;
            }
          } else {
            scale_o = l_run > 0.f ? a.v_scale / l_run : 0.f;
            lse = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
          }
          const int prow = bd.part_row_base + sd.split * bd.nrows + pos;
#pragma unroll
          for (int c = 0; c < kDv / 32; ++c) {
            uint32_t o[32];
            tc::tmem_ld32(tmem + lane_base + kTmemO + c * 32, o);
            tc::tmem_wait_ld();
            if (!valid) continue;
            if (single) {
              uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) +
                                                     ((int64_t)tok * a.hq + h) * kDv + c * 32);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  w[e] = cvt_pair(__uint_as_float(o[8 * q + 2 * e]) * scale_o,
                                  __uint_as_float(o[8 * q + 2 * e + 1]) * scale_o);
                dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
              float4 *dst = reinterpret_cast<float4 *>(a.part_o + (int64_t)prow * kDv + c * 32);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(__uint_as_float(o[4 * q]) * scale_o,
                                     __uint_as_float(o[4 * q + 1]) * scale_o,
                                     __uint_as_float(o[4 * q + 2]) * scale_o,
                                     __uint_as_float(o[4 * q + 3]) * scale_o);
            }
          }
          if (valid) {
            if (single) {
              if (a.lse_out) a.lse_out[(int64_t)tok * a.hq + h] = lse;
            } else {
              a.part_lse[prow] = lse;
            }
          }
        }
      } else {
        // Several copies per row (copy c of block row r sits at position
        // c * rows_pad + r).  Each copy works out the row's common maximum and
        // normaliser from the copies' statistics, scales its own O row by its
        // share, and the copies are then summed through shared memory 32
        // columns at a time (rows of 32 floats, XOR-swizzled by row: no bank
        // conflicts).
        const int copies = kRows / rows_pad;
        if (pos >= 0) {
          sm_m[pos] = valid ? m_run : -INFINITY;
          sm_l[pos] = valid ? l_run : 0.f;
        }
        if (!group_sync()) break;
        float f = 0.f, lse = -INFINITY;
        if (valid) {
          float M = -INFINITY;
          for (int c = 0; c < copies; ++c) M = fmaxf(M, sm_m[c * rows_pad + rr]);
          float L = 0.f;
          if (M != -INFINITY)
            for (int c = 0; c < copies; ++c) {
              const float mc = sm_m[c * rows_pad + rr];
              if (mc != -INFINITY) L += sm_l[c * rows_pad + rr] * exp2f(mc - M);
            }
          const float mine = m_run == -INFINITY ? 0.f : 1.f;
          if (single) {
            const float MM = fmaxf(M, sink2);
            if (MM != -INFINITY) {
              const float Z = L * exp2f(M - MM) + exp2f(sink2 - MM);
              f = mine * exp2f(m_run - MM) * a.v_scale / Z;
              lse = (MM + log2f(Z)) * kLn2;
            }
          } else if (L > 0.f) {
            f = mine * exp2f(m_run - M) * a.v_scale / L;
            lse = M + log2f(L);
          }
          if (pos < rows_pad) {          // copy 0 writes the row's log-sum-exp
            if (single) {
              if (a.lse_out) a.lse_out[(int64_t)row_tok * a.hq + row_h] = lse;
            } else {
              a.part_lse[bd.part_row_base + sd.split * bd.nrows + rr] = lse;
            }
          }
        }
        float *buf = reinterpret_cast<float *>(smem + Lay::kOffComb);
        const int nout = rows_pad / 4;   // (row, column) outputs per thread per chunk
        bool sync_ok = true;
#pragma unroll 1
        for (int c = 0; c < kDv / 32; ++c) {
          if (warp_live) {
            uint32_t o[32];
            tc::tmem_ld32(tmem + lane_base + kTmemO + c * 32, o);
            tc::tmem_wait_ld();
            if (pos >= 0)
#pragma unroll
              for (int j = 0; j < 32; ++j) buf[pos * 32 + (j ^ (pos & 31))] = f * __uint_as_float(o[j]);
          }
          sync_ok = group_sync() && sync_ok;
#pragma unroll 1
          for (int i = 0; i < nout; ++i) {
            const int row = (t >> 5) + 4 * i;
            if (!sync_ok || row >= bd.nrows) continue;
            float v = 0.f;
#pragma unroll 4
            for (int cp2 = 0; cp2 < copies; ++cp2) {
              const int p2 = cp2 * rows_pad + row;
              v += buf[p2 * 32 + (lane ^ (p2 & 31))];
            }
            if (single) {
              const int flat = bd.row0 + row;
              const int tok = bd.tok0 + flat / a.group;
              const int h = bd.g * a.group + flat % a.group;
              static_cast<__nv_bfloat16 *>(a.out)[((int64_t)tok * a.hq + h) * kDv + 32 * c + lane] =
                  __float2bfloat16_rn(v);
            } else {
              const int prow = bd.part_row_base + sd.split * bd.nrows + row;
              a.part_o[(int64_t)prow * kDv + 32 * c + lane] = v;
            }
          }
          sync_ok = group_sync() && sync_ok;
        }
        if (!sync_ok) break;
      }
      if (t == 0) AKP_STAMP(kStampEpiEnd);
      tc::tc_fence_before();
      tc::mbar_arrive(&bars.o_free);
    }
  }

  __syncthreads();
  if (tid == 0) AKP_STAMP(kStampEnd);
  if (tid == 0 && abort_flag) atomicOr(a.err, 2);
  if (warp == 8) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool FP8, bool TMA, int MR, int DQK, bool HALF>
cudaError_t launch_one(const HostPlan &hp, const RunArgs &a, const TmaMaps &m, cudaStream_t st) {
  return launch_dependent(attn_tc_kernel<FP8, TMA, MR, DQK, HALF>, dim3(hp.num_ctas),
                          dim3(kThreads), Layout<FP8, MR, TMA, DQK>::kSmem, st, a, m);
}

template <bool FP8, bool TMA, int MR, int DQK, bool HALF>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(attn_tc_kernel<FP8, TMA, MR, DQK, HALF>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Layout<FP8, MR, TMA, DQK>::kSmem);
}

template <int MR, int DQK, bool HALF>
cudaError_t launch_rows(const HostPlan &hp, const RunArgs &a, const TmaMaps &m, cudaStream_t st) {
  const bool fp8 = hp.prob.kv_dtype == ATTN_KV_FP8_E4M3;
  if (hp.use_tma)
    return fp8 ? launch_one<true, true, MR, DQK, HALF>(hp, a, m, st)
               : launch_one<false, true, MR, DQK, HALF>(hp, a, m, st);
  return fp8 ? launch_one<true, false, MR, DQK, HALF>(hp, a, m, st)
             : launch_one<false, false, MR, DQK, HALF>(hp, a, m, st);
}

template <int MR, int DQK, bool HALF>
cudaError_t prepare_rows(const HostPlan &hp) {
  const bool fp8 = hp.prob.kv_dtype == ATTN_KV_FP8_E4M3;
  if (hp.use_tma)
    return fp8 ? prepare_one<true, true, MR, DQK, HALF>() : prepare_one<false, true, MR, DQK, HALF>();
  return fp8 ? prepare_one<true, false, MR, DQK, HALF>() : prepare_one<false, false, MR, DQK, HALF>();
}

// M = 64 plans whose blocks all have more than 32 rows run the two-threads-
// per-row instantiation.
template <int DQK>
cudaError_t launch_dqk(const HostPlan &hp, const RunArgs &a, const TmaMaps &m, cudaStream_t st) {
  if (hp.block_rows != 64) return launch_rows<128, DQK, false>(hp, a, m, st);
  return hp.one_copy ? launch_rows<64, DQK, true>(hp, a, m, st)
                     : launch_rows<64, DQK, false>(hp, a, m, st);
}

template <int DQK>
cudaError_t prepare_dqk(const HostPlan &hp) {
  if (hp.block_rows != 64) return prepare_rows<128, DQK, false>(hp);
  return hp.one_copy ? prepare_rows<64, DQK, true>(hp) : prepare_rows<64, DQK, false>(hp);
}

}  // namespace

bool tc_tma_page_size(int32_t page_size, int32_t num_pages) {
  if ((int64_t)num_pages * page_size >= INT32_MAX) return false;
  return page_size % kN == 0 || (kN % page_size == 0 && page_size >= 8);
}

cudaError_t launch_attn_tc(const HostPlan &hp, const RunArgs &a, const TmaMaps &m,
                           cudaStream_t stream) {
  if (hp.num_ctas == 0) return cudaSuccess;
  return hp.prob.head_dim_qk == kDqkSym ? launch_dqk<kDqkSym>(hp, a, m, stream)
                                        : launch_dqk<kDqk>(hp, a, m, stream);
}

cudaError_t prepare_attn_tc(const HostPlan &hp) {
  return hp.prob.head_dim_qk == kDqkSym ? prepare_dqk<kDqkSym>(hp) : prepare_dqk<kDqk>(hp);
}

}  // namespace akp

extern "C" attn_status_t attn_debug_stamps(uint64_t *host, int32_t clear) {
#ifdef AKP_STAMPS
  static_assert(akp::kStampCtas == ATTN_DEBUG_STAMP_CTAS &&
                    akp::kStampEvents == ATTN_DEBUG_STAMP_EVENTS,
                "stamp array shape");
  if (!host) return ATTN_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaMemcpyFromSymbol(host, akp::g_stamps, sizeof(akp::g_stamps)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (clear) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, akp::g_stamps) != cudaSuccess ||
        cudaMemset(p, 0, sizeof(akp::g_stamps)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
#else
  (void)host;
  (void)clear;
  return ATTN_ERR_UNSUPPORTED;
#endif
}
