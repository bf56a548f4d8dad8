// Prefill attention on the Blackwell tensor-core path (tcgen05 + TMEM) for row
// blocks of more than 128 query rows: the chunked-prefill shape of the
// MiMo-V2.6-Flash-RL model card ("What the kernels do": a 4096-token chunk
// after 26K cached tokens, many tokens x all GQA heads of a KV head per CTA).
//
// A row block holds up to 256 query rows of one (request, KV head), as two
// 128-row Q tiles that share every 128-key K/V tile: each key tile is fetched
// and (for FP8 caches) widened once per 256 rows, and each tcgen05.mma runs at
// N = 128, the shape that keeps the tensor pipe at its full rate.
//
// Warp roles (512 threads, four warpgroups; registers are moved from the load
// and MMA warpgroups to the softmax ones after the start):
//   warps 0-3   softmax + epilogue of Q tile 0 (row p in TMEM lane p);
//   warps 4-7   the same for Q tile 1;
//   warps 8-11  load warps: the Q rows of each new block (for FP8 caches
//               scaled per row by a power of two, see q_row_shift), and the
//               K/V tiles.  With a staging scratch (kv_stage.cu: every key of
//               the block's (request, KV head) already a 16-bit row, E4M3
//               widened exactly to fp16) one thread issues each tile as TMA
//               boxes in the operand layout.  Without one, per key tile: the
//               page lookup of each key, K and V rows read from the cache with
//               16-byte loads (one thread per key), widened in registers, and
//               stored into the 128-byte-swizzled operand tiles.  (The MMAs of
//               an FP8 cache run in fp16.)
//   warp  12    TMEM allocation; one thread issues the MMAs of Q tile 0;
//   warp  13    one thread issues the MMAs of Q tile 1;
//   warps 14-15 idle (they complete the fourth warpgroup).
// Shared memory: Q 2 x 48 KB, K 2 x 48 KB (double-buffered), V 32 KB.
// TMEM (512 columns): S of Q tile t at columns [128t, 128t + 128), O of Q
// tile t at [256 + 128t, 384 + 128t); P (16-bit pairs) overwrites the last 64
// columns of its S once the softmax has read them.
// Per Q tile t and key tile k: S_t = Q_t.K^T, softmax, O_t += P_t.V.  S_t of
// tile k+1 is issued right behind P_t.V of tile k (P_t lives in S_t's
// columns; one thread's MMAs run in issue order); the two Q tiles' chains run
// from separate issuing threads, so one tile's MMAs fill the tensor pipe while
// the other waits for its softmax.  Every wait is
// bounded in time; a broken invariant ends the kernel with bit 1 of the plan's
// error word set instead of hanging the GPU.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>

#include "e4m3.cuh"
#include "kernels.hpp"
#include "tc_common.cuh"

namespace akp {
namespace {

constexpr int kPN = kPrefillKeyTile;          // keys per tile (128)
constexpr int kPM = 128;                      // rows per Q tile (MMA M)
constexpr int kMmaWarp = 12;                  // warps 12 and 13 issue the MMAs
constexpr int kPThreads = 16 * 32;            // four full warpgroups (register split)
constexpr int kLoadThreads = 128;
constexpr int kLoadWarps = kLoadThreads / 32;
constexpr int kTileBlk = 128 * 128;           // one 64-column block of a 128-row tile: 16 KB
constexpr int kQTile = 3 * kTileBlk;          // 48 KB
constexpr int kKStage = 3 * kTileBlk;         // 48 KB
constexpr int kVStage = 2 * kTileBlk;         // 32 KB
constexpr int kOffK = 2 * kQTile;
constexpr int kOffV = kOffK + 2 * kKStage;
constexpr int kSmem = kOffV + kVStage + 1024;  // + room to align the base to 1024 B
// with the static shared memory (barriers: < 1 KB)
static_assert(kSmem + 1024 <= 227 * 1024, "shared memory layout too large");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;     // base-2 growth allowed before O is rescaled

struct PBars {
  uint64_t k_full[2], k_empty[2], v_full, v_empty, q_full, q_empty;
  // P of keys 64-127 (p_hi) is published before P of keys 0-63 (p_full), so
  // that half of P.V overlaps the rest of the softmax
  uint64_t s_full[2], p_hi[2], p_full[2], pv_done[2], o_free[2];
  uint64_t done[2];
};

// Walks the CTA's key tiles in order (segment, absolute tile id); the current
// segment and its block sit in registers.
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
    // keep every field in a register (see attn_tc.cu: re-reads from global
    // memory would sit behind the K/V traffic)
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

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t f16_pair(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}


// FP8 caches: Q rows go to fp16 scaled by 2^sh, the power of two that puts
// the row's largest |q| in [2^14, 2^15) (bf16 exponent field e of that
// maximum: sh = 141 - e, at most 126 for zero or subnormal rows).  Every bf16
// element down to 2^-31 of the maximum is then exact in fp16.  The load warps
// (which scale the row) and the row's softmax thread (which divides the scores
// by 2^sh) both derive sh from the row itself with this function.
__device__ __forceinline__ int q_row_shift(const uint4 *row) {
  uint32_t e = 0;
#pragma unroll 1
  for (int c0 = 0; c0 < kDqk / 8; c0 += 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldg(row + c0 + u);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) e = max(e, max((w[q] >> 7) & 0xFFu, (w[q] >> 23) & 0xFFu));
    }
  }
  return min(141 - (int)e, 126);
}

// STAGED: the K/V tiles are TMA boxes of the staging scratch (kv_stage.cu),
// issued by one thread of the load warps; else the load warps read the paged
// caches themselves (plans without a scratch: replayable plans, runs without
// a workspace).
template <bool FP8, bool STAGED>
__global__ void __launch_bounds__(kPThreads, 1)
    attn_prefill_kernel(const RunArgs args, const __grid_constant__ TmaMaps stage) {
  const RunArgs a = args;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ PBars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
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
    abort_flag = 0;
    // a K or V stage is filled by the four load warps, or by one TMA issue
    constexpr uint32_t kFill = STAGED ? 1 : kLoadWarps;
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bars.k_full[i], kFill);
      tc::mbar_init(&bars.k_empty[i], 2);
      tc::mbar_init(&bars.done[i], 1);
      tc::mbar_init(&bars.s_full[i], 1);
      tc::mbar_init(&bars.p_full[i], 4);       // the Q tile's four softmax warps
      tc::mbar_init(&bars.p_hi[i], 4);
      tc::mbar_init(&bars.pv_done[i], 1);
      tc::mbar_init(&bars.o_free[i], 4);
    }
    tc::mbar_init(&bars.v_full, kFill);
    tc::mbar_init(&bars.v_empty, 2);
    tc::mbar_init(&bars.q_full, kLoadWarps);
    tc::mbar_init(&bars.q_empty, 2);
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) tc::tmem_alloc(&tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t sbase = tc::smem_u32(smem);
  // Register split per warpgroup, set first thing in each role (per SM
  // sub-partition one warp of each: 168 + 168 + 120 + 56 = 512 registers a
  // lane, the 128 x 4 of the launch): the softmax warps hold a whole
  // 128-column S row in registers.

  if (warp >= 8 && warp < kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 120;\n" ::: "memory");
    // ------------------------------------------------------------ load warps
    // Thread `key` owns that key of every tile: its page lookup, its K and V
    // rows (16-byte loads), the E4M3 -> bf16 widening and the stores into the
    // swizzled operand tiles (8 consecutive keys per 8-lane phase of a 16-byte
    // shared store: 8 distinct bank groups).
    const int lt = tid - 256;
    const int key = lt;
    constexpr int kEs = FP8 ? 1 : 2;
    const uint8_t *kc = static_cast<const uint8_t *>(a.k_cache);
    const uint8_t *vc = static_cast<const uint8_t *>(a.v_cache);
    // K-stream position: segment, tile, and the block fields a page lookup
    // needs (loaded from the plan when the stream enters a segment).
    struct KPos {
      int seg, tile, tile_end, b, g, klo, khi;
    };
    auto kpos_load = [&](KPos &p, int seg) {
      const SegDesc sd = a.segs[seg];
      const BlockDesc bd = a.blocks[sd.block];
      p.seg = seg;
      p.tile = sd.tile_begin;
      p.tile_end = sd.tile_end;
      p.b = bd.b;
      p.g = bd.g;
      p.klo = bd.klo;
      p.khi = bd.khi;
    };
    auto kpos_next = [&](KPos &p) {
      if (++p.tile == p.tile_end && p.seg + 1 < seg_end) kpos_load(p, p.seg + 1);
    };
    // Cache slot of this thread's key in the position's tile, -1 outside the
    // block's key range.  Branch-free on the page id, so the warp does not stop
    // for the page-table load until the slot is used; a page id outside the
    // pool reads as zeros and is reported once at the end.
    int bad_page = 0;
    auto lookup = [&](const KPos &p) -> int64_t {
      const int j = p.tile * kPN + key;
      const bool in = j >= p.klo && j < p.khi;
      int32_t page = 0;
      if (in) page = __ldg(a.page_table + (int64_t)p.b * a.pt_stride + j / a.page_size);
      const bool ok = in && page >= 0 && page < a.num_pages;
      bad_page |= (int)(in && !ok);
      return ok ? (int64_t)page * a.page_size + j % a.page_size : -1;
    };
    auto row_ptr = [&](const uint8_t *cache, int64_t slot, int g, int d) {
      return reinterpret_cast<const uint4 *>(cache + ((slot >= 0 ? slot : 0) * a.hkv + g) * (d * kEs));
    };
    // N 16-byte chunks of a row, from chunk c0; zeros for slot -1
    auto load = [&](uint4 *dst, int n, const uint4 *row, int64_t slot) {
#pragma unroll
      for (int i = 0; i < n; ++i) dst[i] = slot >= 0 ? __ldg(row + i) : make_uint4(0u, 0u, 0u, 0u);
    };
    // one 16-byte bf16 chunk `ch` (0..23 for K, 0..15 for V) of this key's row
    auto put = [&](uint32_t base, int ch, uint4 v) {
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(
                       base + (ch >> 3) * kTileBlk + tc::sw128_offset(key, ch & 7)),
                   "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    };
    // E4M3 chunks (16 codes each) -> two fp16 chunks each (exact; one
    // conversion instruction per pair of codes): Q.K^T and P.V run in fp16
    // for FP8 caches (Q scaled per row, see stage_q; P keeps 11 mantissa bits)
    auto put_fp8 = [&](uint32_t base, const uint4 *src, int n, bool to_bf16) {
#pragma unroll
      for (int i = 0; i < n; ++i) {
        uint4 lo, hi;
        if (to_bf16)
          e4m3x16_to_bf16(src[i], lo, hi);
        else
          e4m3x16_to_f16(src[i], lo, hi);
        put(base, 2 * i, lo);
        put(base, 2 * i + 1, hi);
      }
    };
    // Q rows of the cursor's block: row r of the block is Q tile r / 128, MMA
    // row r % 128; rows past the block are zero.  Loads go out 4 at a time.
    auto stage_q = [&](int seg) -> bool {
      const BlockDesc bd = a.blocks[a.segs[seg].block];
      const int si = seg - seg_begin;
      if (si > 0 && !tc::mbar_wait_warp(&bars.q_empty, (si - 1) & 1, &abort_flag)) return false;
      if constexpr (FP8) {
        // Q.K^T runs in fp16 against K widened exactly from E4M3, each Q row
        // scaled by 2^sh (q_row_shift).  One thread per row (rows lt and
        // lt + 128): a pass for the shift, then one that scales, converts and
        // stores.
#pragma unroll 1
        for (int rr = 0; rr < 2; ++rr) {
          const int r = lt + rr * kLoadThreads;
          const bool live = r < bd.nrows;
          const int flat = bd.row0 + (live ? r : 0);
          const uint4 *src = reinterpret_cast<const uint4 *>(
              static_cast<const uint16_t *>(a.q) +
              ((int64_t)(bd.tok0 + flat / a.group) * a.hq + bd.g * a.group + flat % a.group) * kDqk);
          const int sh = live ? q_row_shift(src) : 0;
          const float f = __int_as_float((sh + 127) << 23);
#pragma unroll 1
          for (int c0 = 0; c0 < 24; c0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = live ? __ldg(src + c0 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
              uint32_t h[4];
#pragma unroll
              for (int q = 0; q < 4; ++q)
                h[q] = f16_pair(__uint_as_float(w[q] << 16) * f, __uint_as_float(w[q] & 0xFFFF0000u) * f);
              const int ch = c0 + u;
              const uint32_t dst = sbase + (r >> 7) * kQTile + (ch >> 3) * kTileBlk +
                                   tc::sw128_offset(r & 127, ch & 7);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(h[0]),
                           "r"(h[1]), "r"(h[2]), "r"(h[3])
                           : "memory");
            }
          }
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive_warp(&bars.q_full);
        return true;
      }
      constexpr int kIters = 2 * kPM * 24 / kLoadThreads;   // 48
      constexpr int kBatch = 4;      // the next tile's K/V rows are held in registers meanwhile
#pragma unroll 1
      for (int i0 = 0; i0 < kIters; i0 += kBatch) {
        uint4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int idx = lt + (i0 + u) * kLoadThreads;
          const int r = idx / 24, ch = idx % 24;
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
          const int idx = lt + (i0 + u) * kLoadThreads;
          const int r = idx / 24, ch = idx % 24;
          const uint32_t dst = sbase + (r >> 7) * kQTile + (ch >> 3) * kTileBlk +
                               tc::sw128_offset(r & 127, ch & 7);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(v[u].x),
                       "r"(v[u].y), "r"(v[u].z), "r"(v[u].w)
                       : "memory");
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive_warp(&bars.q_full);
      return true;
    };

    if constexpr (STAGED) {
      // K(k) and V(k-1) per iteration, as in the paths below, but as TMA
      // boxes of the staging scratch (64 columns x 128 keys, 128-byte
      // swizzle: the operand layout) issued by lane 0 of the first load warp;
      // all four load warps stage the Q rows when a segment starts.  Key j of
      // the block's (b, g) is scratch row srow + j.
      const bool issuer = lt == 0;
      int sg = seg_begin;
      SegDesc ssd = head.seg;
      int s_row = head.blk.srow;
      int s_tile = ssd.tile_begin;
      bool s_first = true;
      int v_row = 0;
      if (issuer) {
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&stage.k)) : "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&stage.v)) : "memory");
      }
      for (int k = 0; k <= total; ++k) {
        bool ok = true;
        if (k < total) {
          if (s_first && !stage_q(sg)) break;
          if (issuer) {
            const int s = k & 1;
            ok = k < 2 || tc::mbar_wait(&bars.k_empty[s], ((k >> 1) - 1) & 1, &abort_flag);
            if (ok) {
              tc::mbar_arrive_expect_tx(&bars.k_full[s], kKStage);
              const int y = s_row + s_tile * kPN;
#pragma unroll
              for (int c = 0; c < 3; ++c)
                tc::tma_load_2d(sbase + kOffK + s * kKStage + c * kTileBlk, &stage.k, c * 64, y,
                                &bars.k_full[s]);
            }
          }
        }
        if (k >= 1 && issuer && ok) {
          ok = k < 2 || tc::mbar_wait(&bars.v_empty, (k - 2) & 1, &abort_flag);
          if (ok) {
            tc::mbar_arrive_expect_tx(&bars.v_full, kVStage);
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tc::tma_load_2d(sbase + kOffV + c * kTileBlk, &stage.v, c * 64, v_row, &bars.v_full);
          }
        }
        if (__any_sync(0xffffffffu, !ok)) break;
        if (k < total) {
          v_row = s_row + s_tile * kPN;
          s_first = false;
          if (++s_tile == ssd.tile_end && sg + 1 < seg_end) {
            ++sg;
            ssd = a.segs[sg];
            s_row = a.blocks[ssd.block].srow;
            s_tile = ssd.tile_begin;
            s_first = true;
          }
        }
      }
    } else {
      // The K stream runs one tile ahead of the V stream: iteration k stores
      // K(k) (once Q.K^T of tile k-2 has freed its stage) and then V(k-1) (once
      // P.V of tile k-2 is done), so a tile's K never waits behind the previous
      // tile's P.V.  Page lookups run two tiles ahead of the K stream.
      // Per tile in flight ([0]: tile k, [1]: k+1, [2]: k+2): its cache slot,
      // and its KV head, segment and whether it starts the segment packed as
      // segment << 17 | first << 16 | head.
      KPos kp;
      kpos_load(kp, seg_begin);
      int64_t slot[3];
      int info[3];
      auto pack = [](int seg, bool first, int g) { return (seg << 17) | ((int)first << 16) | g; };
      slot[0] = lookup(kp);
      info[0] = pack(kp.seg, true, kp.g);
      for (int i = 1; i < 3; ++i) {
        slot[i] = -1;
        info[i] = 0;
        if (i < total) {
          const int prev_seg = kp.seg;
          kpos_next(kp);
          slot[i] = lookup(kp);
          info[i] = pack(kp.seg, kp.seg != prev_seg, kp.g);
        }
      }
      auto shift = [&](int k) {    // tile k+1 becomes [0]; look up tile k+3 into [2]
        slot[0] = slot[1];
        info[0] = info[1];
        slot[1] = slot[2];
        info[1] = info[2];
        slot[2] = -1;
        if (k + 3 < total) {
          const int prev_seg = kp.seg;
          kpos_next(kp);
          slot[2] = lookup(kp);
          info[2] = pack(kp.seg, kp.seg != prev_seg, kp.g);
        }
      };
      auto head_of = [](int in) { return in & 0xFFFF; };
      auto starts = [](int in) { return ((in >> 16) & 1) != 0; };
      auto seg_of = [](int in) { return in >> 17; };
      if constexpr (FP8) {
        // raw E4M3 rows in registers: K of tile k, V of tile k-1 (20 x 16 bytes)
        constexpr int KCH = kDqk / 16, VCH = kDv / 16;
        uint4 kr[KCH], vr[VCH];
        int64_t v_slot = -1;
        int v_g = 0;
        load(kr, KCH, row_ptr(kc, slot[0], head_of(info[0]), kDqk), slot[0]);
        for (int k = 0; k <= total; ++k) {
          if (k < total) {
            if (starts(info[0]) && !stage_q(seg_of(info[0]))) break;
            const int s = k & 1;
            if (k >= 2 && !tc::mbar_wait_warp(&bars.k_empty[s], ((k >> 1) - 1) & 1, &abort_flag)) break;
            put_fp8(sbase + kOffK + s * kKStage, kr, KCH, false);
            tc::fence_proxy_async_smem();
            tc::mbar_arrive_warp(&bars.k_full[s]);
            if (k + 1 < total) load(kr, KCH, row_ptr(kc, slot[1], head_of(info[1]), kDqk), slot[1]);
          }
          if (k >= 1) {
            if (k >= 2 && !tc::mbar_wait_warp(&bars.v_empty, (k - 2) & 1, &abort_flag)) break;
            put_fp8(sbase + kOffV, vr, VCH, false);
            tc::fence_proxy_async_smem();
            tc::mbar_arrive_warp(&bars.v_full);
          }
          if (k < total) {
            v_slot = slot[0];
            v_g = head_of(info[0]);
            load(vr, VCH, row_ptr(vc, v_slot, v_g, kDv), v_slot);
            shift(k);
          }
        }
      } else {
        // BF16 rows are twice as wide: each goes through registers in pieces of
        // 12 and 8 chunks, loaded just before they are stored.
        uint4 buf[12];
        int64_t v_slot = -1;
        int v_g = 0;
        for (int k = 0; k <= total; ++k) {
          if (k < total) {
            if (starts(info[0]) && !stage_q(seg_of(info[0]))) break;
            const uint4 *krow = row_ptr(kc, slot[0], head_of(info[0]), kDqk);
            const int s = k & 1;
            load(buf, 12, krow, slot[0]);
            if (k >= 2 && !tc::mbar_wait_warp(&bars.k_empty[s], ((k >> 1) - 1) & 1, &abort_flag)) break;
            const uint32_t kb = sbase + kOffK + s * kKStage;
  #pragma unroll
            for (int i = 0; i < 12; ++i) put(kb, i, buf[i]);
            load(buf, 12, krow + 12, slot[0]);
  #pragma unroll
            for (int i = 0; i < 12; ++i) put(kb, 12 + i, buf[i]);
            tc::fence_proxy_async_smem();
            tc::mbar_arrive_warp(&bars.k_full[s]);
          }
          if (k >= 1) {
            const uint4 *vrow = row_ptr(vc, v_slot, v_g, kDv);
            load(buf, 8, vrow, v_slot);
            if (k >= 2 && !tc::mbar_wait_warp(&bars.v_empty, (k - 2) & 1, &abort_flag)) break;
  #pragma unroll
            for (int i = 0; i < 8; ++i) put(sbase + kOffV, i, buf[i]);
            load(buf, 8, vrow + 8, v_slot);
  #pragma unroll
            for (int i = 0; i < 8; ++i) put(sbase + kOffV, 8 + i, buf[i]);
            tc::fence_proxy_async_smem();
            tc::mbar_arrive_warp(&bars.v_full);
          }
          if (k < total) {
            v_slot = slot[0];
            v_g = head_of(info[0]);
            shift(k);
          }
        }
      }
      if (bad_page) atomicOr(a.err, 1);
    }
  } else if (warp >= kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;\n" ::: "memory");
    if (warp > kMmaWarp + 1) goto done;   // warps 14-15: idle
    // ------------------------------------------------------------ MMA issuers
    // One thread per Q tile (warp 12: Q tile 0, warp 13: Q tile 1), so that the
    // two tiles' chains S_t -> softmax_t -> P_t.V -> next S_t never wait on
    // each other: while one thread waits for its softmax or for its P.V to
    // finish, the other keeps the tensor pipe fed.  The K, V and Q stages go
    // back to the load warps once both threads have committed (count 2); the
    // thread of Q tile 1 commits on tiles without Q tile 1 rows too.  The
    // threads sleep on their barriers (mbarrier try_wait) rather than poll
    // them: a polling thread takes issue slots from the softmax warps of its
    // SM sub-partition, whose P it is waiting for (polling measured 2.5%
    // slower on the chunked prefill).
    if ((tid & 31) == 0) {
      const int t = warp - kMmaWarp;
      const uint32_t id_s = tc::idesc_f16(FP8 ? 0 : 1, 0, 0, kPM, kPN);     // fp16 for FP8 caches
      const uint32_t id_pv = tc::idesc_f16(FP8 ? 0 : 1, 0, 1, kPM, kDv);   // P.V in fp16 for FP8 caches
      const uint32_t q_smem = sbase + t * kQTile;
      const uint32_t s_tmem = tmem + kPN * t;
      const uint32_t o_tmem = tmem + kTmemO + kDv * t;
      Cursor cm;
      cm.init(a.segs, a.blocks, head);
      int ct = 0;      // key tiles with rows in this Q tile
      int segs_t = 0;  // finished segments with rows in this Q tile
      for (int k = 0; k < total; ++k, cm.next()) {
        const bool has1 = cm.bd.nrows > kPM;
        const bool mine = t == 0 || has1;
        const bool first = cm.first();
        const int s = k & 1;
        if (first && !tc::mbar_wait(&bars.q_full, cm.si & 1, &abort_flag)) break;
        if (!tc::mbar_wait(&bars.k_full[s], (k >> 1) & 1, &abort_flag)) break;
        if (mine) {
          // S_t of this tile overwrites P_t of the previous one, which P_t.V
          // reads: that MMA was issued before these by this same thread, and
          // the tensor pipe runs one thread's MMAs in issue order, so there
          // is nothing to wait for.  The two Q tiles' chains are not paced
          // against each other: each thread issues as soon as its own inputs
          // are ready (making S1 of a tile wait for S0 of it, and S0 for S1 of
          // the previous tile, measured 4% slower once K/V came by TMA).
          tc::tc_fence_after();
#pragma unroll
          for (int kq = 0; kq < kDqk / 16; ++kq) {
            const uint32_t koff = (kq & 3) * 32 + (kq >> 2) * kTileBlk;
            const uint64_t ad = tc::smem_desc_sw128(q_smem + koff, 16, 1024);
            const uint64_t bd = tc::smem_desc_sw128(sbase + kOffK + s * kKStage + koff, 16, 1024);
            tc::mma_f16_ss(s_tmem, ad, bd, id_s, kq > 0 ? 1u : 0u);
          }
          tc::mma_commit(&bars.s_full[t]);
        }
        tc::mma_commit(&bars.k_empty[s]);
        if (cm.last()) tc::mma_commit(&bars.q_empty);
        if (!tc::mbar_wait(&bars.v_full, k & 1, &abort_flag)) break;
        if (mine) {
          if (!tc::mbar_wait(&bars.p_hi[t], ct & 1, &abort_flag)) break;
          // the first P.V of a segment overwrites O: the previous epilogue must have read it
          if (first && segs_t > 0 && !tc::mbar_wait(&bars.o_free[t], (segs_t - 1) & 1, &abort_flag))
            break;
          // keys 64-127 first (their P is ready first), then keys 0-63
          auto pv = [&](int kk, bool acc) {
            const uint64_t bd = tc::smem_desc_sw128(sbase + kOffV + kk * 16 * 128, kTileBlk, 1024);
            tc::mma_f16_ts(o_tmem, s_tmem + kPN / 2 + kk * 8, bd, id_pv, acc ? 1u : 0u);
          };
          tc::tc_fence_after();
#pragma unroll
          for (int kk = kPN / 32; kk < kPN / 16; ++kk) pv(kk, !first || kk > kPN / 32);
          if (!tc::mbar_wait(&bars.p_full[t], ct & 1, &abort_flag)) break;
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kPN / 32; ++kk) pv(kk, true);
          tc::mma_commit(&bars.pv_done[t]);
          ++ct;
          if (cm.last()) ++segs_t;
        }
        tc::mma_commit(&bars.v_empty);
      }
      // every MMA issued must be complete before TMEM is released, also
      // after a give-up (a wait of its own, bounded, that ignores the abort)
      tc::mma_commit(&bars.done[t]);
      int no_abort = 0;
      tc::mbar_wait(&bars.done[t], 0, &no_abort, 100000000ull);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 168;\n" ::: "memory");
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;               // Q tile
    const int wq = warp & 3;               // TMEM lane quadrant
    const int lane = tid & 31;
    const int p = wq * 32 + lane;          // MMA row (TMEM lane)
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + kPN * t;
    const uint32_t o_addr = tmem + lane_base + kTmemO + kDv * t;
    float sc = a.scale_log2;               // base-2 score scale of this thread's row
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity, &abort_flag));
    };
    // The softmax keeps only what it needs of the current segment in
    // registers (its S row lives in them too): the tile range, and per block
    // the row's parameters, taken when the segment starts.
    int seg = seg_begin;
    SegDesc sd = a.segs[seg];
    int tile = sd.tile_begin;
    auto advance = [&]() {
      if (++tile == sd.tile_end && seg + 1 < seg_end) {
        ++seg;
        sd = a.segs[seg];
        tile = sd.tile_begin;
      }
    };
    int nrows = 0, prow = 0;
    bool single = true, valid = false;
    float m_run = -INFINITY, l_run = 0.f, sink2 = -INFINITY;
    int row_lo = 0, row_hi = 0, row_tok = 0, row_h = 0;
    int c = 0;                             // key tiles of this Q tile so far
    for (int k = 0; k < total; ++k, advance()) {
      const bool last = tile + 1 == sd.tile_end;
      if (tile == sd.tile_begin) {
        const BlockDesc bd = a.blocks[sd.block];
        const int r = kPM * t + p;
        nrows = bd.nrows;
        single = bd.num_splits == 1;
        prow = bd.part_row_base + sd.split * bd.nrows + r;
        valid = r < bd.nrows;
        row_lo = row_hi = 0;
        sink2 = -INFINITY;
        if (valid) {
          const int flat = bd.row0 + r;
          row_tok = bd.tok0 + flat / a.group;
          row_h = bd.g * a.group + flat % a.group;
          if (a.sinks) sink2 = a.sinks[row_h] * kLog2e;
          if (FP8) {
            // the scores of this row come from Q scaled by 2^sh (see q_row_shift)
            const int sh = q_row_shift(reinterpret_cast<const uint4 *>(
                static_cast<const uint16_t *>(a.q) + ((int64_t)row_tok * a.hq + row_h) * kDqk));
            sc = a.scale_log2 * __int_as_float((127 - sh) << 23);
          }
          const int i = bd.L - bd.n + flat / a.group;
          row_hi = i + 1;
          row_lo = a.window > 0 ? max(0, i - a.window + 1) : 0;
        }
        m_run = -INFINITY;
        l_run = 0.f;
      }
      if (t == 1 && nrows <= kPM) continue;

      if (!wait(&bars.s_full[t], c & 1)) break;
      tc::tc_fence_after();
      const int key0 = tile * kPN;
      const int j_lo = max(0, row_lo - key0);
      const int j_hi = min(kPN, row_hi - key0);
      const bool full = __all_sync(0xffffffffu, j_lo <= 0 && j_hi >= kPN);
      // The whole 128-column S row comes into registers with one TMEM round
      // trip (four loads in flight).  P_t (key j's bf16/fp16 value in the low
      // or high half of column 64 + j/2) then overwrites S columns 64-127.
      uint32_t s0[32], s1[32], s2[32], s3[32];
      tc::tmem_ld32(s_addr, s0);
      tc::tmem_ld32(s_addr + 32, s1);
      tc::tmem_ld32(s_addr + 64, s2);
      tc::tmem_ld32(s_addr + 96, s3);
      tc::tmem_wait_ld_regs64(s0, s1);
      tc::tmem_wait_ld_regs64(s2, s3);
      auto mask32 = [&](uint32_t (&raw)[32], int c0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int jj = c0 + j;
          raw[j] = ((jj >= j_lo) & (jj < j_hi)) ? raw[j] : 0xFF800000u;
        }
      };
      if (!full) {
        mask32(s0, 0);
        mask32(s1, 32);
        mask32(s2, 64);
        mask32(s3, 96);
      }
      float mx[2] = {-INFINITY, -INFINITY};
      auto max32 = [&](const uint32_t (&raw)[32]) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          mx[0] = tc::max3(mx[0], __uint_as_float(raw[j]), __uint_as_float(raw[j + 1]));
          mx[1] = tc::max3(mx[1], __uint_as_float(raw[j + 2]), __uint_as_float(raw[j + 3]));
        }
      };
      max32(s0);
      max32(s1);
      const float m_lo = fmaxf(mx[0], mx[1]) * sc;
      // Keys 64-127 are exponentiated against m_base, the running maximum (on
      // a row's first tile the maximum of keys 0-63), while their own maximum
      // is taken, so their exponents need not wait for a maximum pass.  Only
      // when the tile's maximum exceeds m_base by more than the threshold
      // (rare once the maximum has settled) is O rescaled and the pass redone
      // from S, which is still in TMEM.  Until then P may exceed 1 (up to 2^8).
      float m_base = m_run != -INFINITY ? m_run : m_lo;
      float rs[2] = {0.f, 0.f};
      float mh[2] = {-INFINITY, -INFINITY};
      uint32_t pk2[16], pk3[16];
      auto exp_pack = [&](const uint32_t (&raw)[32], uint32_t (&pk)[16], float nm, bool track) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float x0 = __uint_as_float(raw[j]), x1 = __uint_as_float(raw[j + 1]);
          if (track) mh[(j >> 1) & 1] = tc::max3(mh[(j >> 1) & 1], x0, x1);
          float y0, y1;
          tc::ffma2(y0, y1, x0, x1, sc, nm);
          const float p0 = ex2(y0), p1 = ex2(y1);
          tc::fadd2(rs[0], rs[1], p0, p1);
          pk[j >> 1] = FP8 ? f16_pair(p0, p1) : bf16_pair(p0, p1);
        }
      };
      exp_pack(s2, pk2, m_base == -INFINITY ? 0.f : -m_base, true);
      exp_pack(s3, pk3, m_base == -INFINITY ? 0.f : -m_base, true);
      const float m_tile = fmaxf(m_lo, fmaxf(mh[0], mh[1]) * sc);
      const bool need = m_tile > m_base + kRescaleThreshold;   // never for m_tile = -inf
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? m_tile : m_base;
        // O holds earlier tiles' sums only where the running maximum is finite
        const bool rescale = need && m_run != -INFINITY;
        if (__any_sync(0xffffffffu, rescale)) {
          if (!wait(&bars.pv_done[t], (c - 1) & 1)) break;
          tc::tc_fence_after();
          const float alpha = rescale ? ex2(m_run - m_new) : 1.f;
#pragma unroll 1
          for (int q = 0; q < kDv / 16; ++q) {
            uint32_t o[16];
            tc::tmem_ld16(o_addr + q * 16, o);
            tc::tmem_wait_ld_regs(o);
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tc::tmem_st16(o_addr + q * 16, o);
          }
          tc::tmem_wait_st();
          l_run *= alpha;
        }
        m_base = m_new;
        tc::tmem_ld32(s_addr + 64, s2);
        tc::tmem_ld32(s_addr + 96, s3);
        tc::tmem_wait_ld_regs64(s2, s3);
        if (!full) {
          mask32(s2, 64);
          mask32(s3, 96);
        }
        rs[0] = rs[1] = 0.f;
        exp_pack(s2, pk2, m_base == -INFINITY ? 0.f : -m_base, false);
        exp_pack(s3, pk3, m_base == -INFINITY ? 0.f : -m_base, false);
      }
      m_run = m_base;
      // P_t: key j's 16-bit value in the low (even j) or high half of TMEM
      // column 64 + j/2 of S_t; keys 64-127 first, so that half of P.V starts
      // while keys 0-63 are exponentiated
      tc::tmem_st16(s_addr + kPN / 2 + 32, pk2);
      tc::tmem_st16(s_addr + kPN / 2 + 48, pk3);
      tc::tmem_wait_st();
      tc::tc_fence_before();
      tc::mbar_arrive_warp(&bars.p_hi[t]);
      const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
      auto exp32 = [&](const uint32_t (&raw)[32], int c0) {
#pragma unroll
        for (int h = 0; h < 32; h += 16) {
          uint32_t pk[8];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            float y0, y1;
            tc::ffma2(y0, y1, __uint_as_float(raw[h + j]), __uint_as_float(raw[h + j + 1]), sc, neg_m);
            const float p0 = ex2(y0), p1 = ex2(y1);
            tc::fadd2(rs[0], rs[1], p0, p1);
            pk[j >> 1] = FP8 ? f16_pair(p0, p1) : bf16_pair(p0, p1);
          }
          tc::tmem_st8(s_addr + kPN / 2 + (c0 + h) / 2, pk);
        }
      };
      exp32(s0, 0);
      exp32(s1, 32);
      tc::tmem_wait_st();                  // P is in TMEM before p_full is signalled
      tc::tc_fence_before();
      tc::mbar_arrive_warp(&bars.p_full[t]);
      l_run += rs[0] + rs[1];
      const int cdone = c++;
      if (!last) continue;

      // ---------------- end of segment: normalise and write the rows
      if (!wait(&bars.pv_done[t], cdone & 1)) break;
      tc::tc_fence_after();
      float scale_o = 0.f, lse = -INFINITY;
      if (single) {
        const float MM = fmaxf(m_run, sink2);
        if (MM != -INFINITY) {
          const float Z = l_run * exp2f(m_run - MM) + exp2f(sink2 - MM);
          scale_o = exp2f(m_run - MM) * a.v_scale / Z;
          lse = (MM + log2f(Z)) * kLn2;
        }
      } else if (l_run > 0.f) {
        scale_o = a.v_scale / l_run;
        lse = m_run + log2f(l_run);
      }
#pragma unroll 1
      for (int q = 0; q < kDv / 32; ++q) {
        uint32_t o[32];
        tc::tmem_ld32(o_addr + q * 32, o);
        tc::tmem_wait_ld();
        if (!valid) continue;
        if (single) {
          uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) +
                                                 ((int64_t)row_tok * a.hq + row_h) * kDv + q * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(
                bf16_pair(__uint_as_float(o[8 * e + 0]) * scale_o, __uint_as_float(o[8 * e + 1]) * scale_o),
                bf16_pair(__uint_as_float(o[8 * e + 2]) * scale_o, __uint_as_float(o[8 * e + 3]) * scale_o),
                bf16_pair(__uint_as_float(o[8 * e + 4]) * scale_o, __uint_as_float(o[8 * e + 5]) * scale_o),
                bf16_pair(__uint_as_float(o[8 * e + 6]) * scale_o, __uint_as_float(o[8 * e + 7]) * scale_o));
        } else {
          float4 *dst = reinterpret_cast<float4 *>(a.part_o + (int64_t)prow * kDv + q * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(o[4 * e]) * scale_o, __uint_as_float(o[4 * e + 1]) * scale_o,
                                 __uint_as_float(o[4 * e + 2]) * scale_o, __uint_as_float(o[4 * e + 3]) * scale_o);
        }
      }
      if (valid) {
        if (single) {
          if (a.lse_out) a.lse_out[(int64_t)row_tok * a.hq + row_h] = lse;
        } else {
          a.part_lse[prow] = lse;
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive_warp(&bars.o_free[t]);
    }
  }

done:
  __syncthreads();
  if (tid == 0 && abort_flag) atomicOr(a.err, 2);
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attn_prefill(const HostPlan &hp, const RunArgs &a, const TmaMaps *stage,
                                cudaStream_t stream) {
  if (hp.num_ctas == 0) return cudaSuccess;
  const dim3 grid(hp.num_ctas), block(kPThreads);
  const TmaMaps none{};
  const bool fp8 = hp.prob.kv_dtype == ATTN_KV_FP8_E4M3;
  if (stage)
    return fp8 ? launch_dependent(attn_prefill_kernel<true, true>, grid, block, kSmem, stream, a, *stage)
               : launch_dependent(attn_prefill_kernel<false, true>, grid, block, kSmem, stream, a,
                                  *stage);
  return fp8 ? launch_dependent(attn_prefill_kernel<true, false>, grid, block, kSmem, stream, a, none)
             : launch_dependent(attn_prefill_kernel<false, false>, grid, block, kSmem, stream, a,
                                none);
}

cudaError_t prepare_attn_prefill(const HostPlan &hp) {
  const bool fp8 = hp.prob.kv_dtype == ATTN_KV_FP8_E4M3;
  cudaError_t e = cudaFuncSetAttribute(fp8 ? attn_prefill_kernel<true, true> : attn_prefill_kernel<false, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fp8 ? attn_prefill_kernel<true, false> : attn_prefill_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  return e;
}

}  // namespace akp
