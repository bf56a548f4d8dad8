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
// Warp roles (416 threads; at most four warps per SM sub-partition, so each
// thread may hold 128 registers):
//   warps 0-3   softmax + epilogue of Q tile 0 (row p in TMEM lane p);
//   warps 4-7   the same for Q tile 1;
//   warps 8-11  load warps: per key tile, the page lookup of each key, K and V
//               rows read from the cache with 16-byte loads (one thread per
//               key), E4M3 widened exactly to bf16 in registers, and the rows
//               stored into the 128-byte-swizzled operand tiles; the Q rows of
//               each new block;
//   warp  12    TMEM allocation; one thread issues every MMA.
// Shared memory: Q 2 x 48 KB, K 2 x 48 KB (double-buffered), V 32 KB.
// TMEM (512 columns): S of Q tile t at columns [128t, 128t + 128), O of Q
// tile t at [256 + 128t, 384 + 128t); P (bf16 pairs) overwrites the first 64
// columns of its S once the softmax has read them.
// Tensor-pipe order per key tile k: S0 = Q0.K^T, S1 = Q1.K^T, O0 += P0.V,
// O1 += P1.V.  S_t of tile k+1 is issued only once P_t.V of tile k is done
// (P_t lives in S_t's columns); the other Q tile's MMA queued in between hides
// that wait.  Every wait is bounded in time; a broken invariant ends the
// kernel with bit 1 of the plan's error word set instead of hanging the GPU.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "e4m3.cuh"
#include "kernels.hpp"
#include "tc_common.cuh"

namespace akp {
namespace {

constexpr int kPN = kPrefillKeyTile;          // keys per tile (128)
constexpr int kPM = 128;                      // rows per Q tile (MMA M)
constexpr int kMmaWarp = 12;
constexpr int kPThreads = 13 * 32;
constexpr int kLoadThreads = 128;
constexpr int kTileBlk = 128 * 128;           // one 64-column block of a 128-row tile: 16 KB
constexpr int kQTile = 3 * kTileBlk;          // 48 KB
constexpr int kKStage = 3 * kTileBlk;         // 48 KB
constexpr int kVStage = 2 * kTileBlk;         // 32 KB
constexpr int kOffK = 2 * kQTile;
constexpr int kOffV = kOffK + 2 * kKStage;
constexpr int kSmem = kOffV + kVStage + 1024;  // + room to align the base to 1024 B
static_assert(kSmem + 1024 <= 227 * 1024, "shared memory layout too large");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;     // base-2 growth allowed before O is rescaled

struct PBars {
  uint64_t k_full[2], k_empty[2], v_full, v_empty, q_full, q_empty;
  uint64_t s_full[2], p_full[2], pv_done[2], o_free[2];
  uint64_t done;
};

// Walks the CTA's key tiles in order (segment, absolute tile id); the current
// segment and its block sit in registers.
struct Cursor {
  const SegDesc *segs;
  const BlockDesc *blocks;
  int seg, seg_end, tile, si;
  SegDesc sd;
  BlockDesc bd;
  __device__ void init(const SegDesc *s, const BlockDesc *b, int first, int end) {
    segs = s;
    blocks = b;
    seg = first;
    seg_end = end;
    si = 0;
    load();
  }
  __device__ void load() {
    sd = segs[seg];
    bd = blocks[sd.block];
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

// Columns outside [j_lo, j_hi) of a 16-column chunk c become -inf.
__device__ __forceinline__ void mask16(uint32_t (&raw)[16], int c, int j_lo, int j_hi) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int jj = 16 * c + j;
    raw[j] = ((jj >= j_lo) & (jj < j_hi)) ? raw[j] : 0xFF800000u;
  }
}

template <bool FP8>
__global__ void __launch_bounds__(kPThreads, 1) attn_prefill_kernel(const RunArgs args) {
  const RunArgs a = args;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ PBars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  // the split merge (a programmatic dependent) may be scheduled now; it waits
  // for this grid's completion before it reads anything written here
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int seg_begin = a.cta_seg_begin[blockIdx.x];
  const int seg_end = a.cta_seg_begin[blockIdx.x + 1];
  if (seg_begin >= seg_end) return;
  int total = 0;
  for (int s = seg_begin; s < seg_end; ++s) total += a.segs[s].tile_end - a.segs[s].tile_begin;

  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bars.k_full[i], kLoadThreads);
      tc::mbar_init(&bars.k_empty[i], 1);
      tc::mbar_init(&bars.s_full[i], 1);
      tc::mbar_init(&bars.p_full[i], kPM);
      tc::mbar_init(&bars.pv_done[i], 1);
      tc::mbar_init(&bars.o_free[i], kPM);
    }
    tc::mbar_init(&bars.v_full, kLoadThreads);
    tc::mbar_init(&bars.v_empty, 1);
    tc::mbar_init(&bars.q_full, kLoadThreads);
    tc::mbar_init(&bars.q_empty, 1);
    tc::mbar_init(&bars.done, 1);
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) tc::tmem_alloc(&tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t sbase = tc::smem_u32(smem);

  if (warp >= 8 && warp < kMmaWarp) {
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
    // cache slot of this thread's key in the cursor's tile, -1 outside the
    // block's key range (or for a page id outside the pool: flagged, read as 0)
    auto lookup = [&](const Cursor &c) -> int64_t {
      const int j = c.tile * kPN + key;
      if (j < c.bd.klo || j >= c.bd.khi) return -1;
      const int32_t page = __ldg(a.page_table + (int64_t)c.bd.b * a.pt_stride + j / a.page_size);
      if (page < 0 || page >= a.num_pages) {
        atomicOr(a.err, 1);
        return -1;
      }
      return (int64_t)page * a.page_size + j % a.page_size;
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
    // E4M3 chunks (16 codes each) -> two bf16 chunks each
    auto put_fp8 = [&](uint32_t base, int c0, const uint4 *src, int n) {
#pragma unroll
      for (int i = 0; i < n; ++i) {
        uint4 lo, hi;
        e4m3x16_to_bf16(src[i], lo, hi);
        put(base, 2 * (c0 + i), lo);
        put(base, 2 * (c0 + i) + 1, hi);
      }
    };
    // Q rows of the cursor's block: row r of the block is Q tile r / 128, MMA
    // row r % 128; rows past the block are zero.  Loads go out 4 at a time.
    auto stage_q = [&](const Cursor &c) -> bool {
      const BlockDesc &bd = c.bd;
      if (c.si > 0 && !tc::mbar_wait_warp(&bars.q_empty, (c.si - 1) & 1, &abort_flag)) return false;
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
      tc::mbar_arrive(&bars.q_full);
      return true;
    };

    Cursor cur;
    cur.init(a.segs, a.blocks, seg_begin, seg_end);
    if constexpr (FP8) {
      // One cursor, moved to tile k+1 as soon as tile k's Q rows are staged:
      // the next tile's page lookup and row loads go out while this tile's K
      // and V are stored (a whole E4M3 row pair is 20 registers of 16 bytes).
      constexpr int KCH = kDqk / 16, VCH = kDv / 16;
      uint4 kr[KCH], vr[VCH];
      {
        const int64_t slot = lookup(cur);
        load(kr, KCH, row_ptr(kc, slot, cur.bd.g, kDqk), slot);
        load(vr, VCH, row_ptr(vc, slot, cur.bd.g, kDv), slot);
      }
      for (int k = 0; k < total; ++k) {
        if (cur.first() && !stage_q(cur)) break;
        const bool has_next = k + 1 < total;
        if (has_next) cur.next();
        const int64_t slot_next = has_next ? lookup(cur) : -1;
        const int s = k & 1;
        if (k >= 2 && !tc::mbar_wait_warp(&bars.k_empty[s], ((k >> 1) - 1) & 1, &abort_flag)) break;
        put_fp8(sbase + kOffK + s * kKStage, 0, kr, KCH);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&bars.k_full[s]);
        if (has_next) load(kr, KCH, row_ptr(kc, slot_next, cur.bd.g, kDqk), slot_next);
        if (k >= 1 && !tc::mbar_wait_warp(&bars.v_empty, (k - 1) & 1, &abort_flag)) break;
        put_fp8(sbase + kOffV, 0, vr, VCH);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&bars.v_full);
        if (has_next) load(vr, VCH, row_ptr(vc, slot_next, cur.bd.g, kDv), slot_next);
      }
    } else {
      // BF16 rows are twice as wide: each row goes through registers in
      // 12- and 8-chunk pieces, the first piece loaded before the stage wait.
      uint4 buf[12];
      for (int k = 0; k < total; ++k, cur.next()) {
        if (cur.first() && !stage_q(cur)) break;
        const int64_t slot = lookup(cur);
        const uint4 *krow = row_ptr(kc, slot, cur.bd.g, kDqk);
        const uint4 *vrow = row_ptr(vc, slot, cur.bd.g, kDv);
        const int s = k & 1;
        load(buf, 12, krow, slot);
        if (k >= 2 && !tc::mbar_wait_warp(&bars.k_empty[s], ((k >> 1) - 1) & 1, &abort_flag)) break;
        const uint32_t kb = sbase + kOffK + s * kKStage;
#pragma unroll
        for (int i = 0; i < 12; ++i) put(kb, i, buf[i]);
        load(buf, 12, krow + 12, slot);
#pragma unroll
        for (int i = 0; i < 12; ++i) put(kb, 12 + i, buf[i]);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&bars.k_full[s]);
        load(buf, 8, vrow, slot);
        if (k >= 1 && !tc::mbar_wait_warp(&bars.v_empty, (k - 1) & 1, &abort_flag)) break;
#pragma unroll
        for (int i = 0; i < 8; ++i) put(sbase + kOffV, i, buf[i]);
        load(buf, 8, vrow + 8, slot);
#pragma unroll
        for (int i = 0; i < 8; ++i) put(sbase + kOffV, 8 + i, buf[i]);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&bars.v_full);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if ((tid & 31) == 0) {
      const uint32_t id_s = tc::idesc_f16(1, 0, 0, kPM, kPN);
      const uint32_t id_pv = tc::idesc_f16(1, 0, 1, kPM, kDv);
      auto qk = [&](int t, int s) {
#pragma unroll
        for (int kq = 0; kq < kDqk / 16; ++kq) {
          const uint32_t koff = (kq & 3) * 32 + (kq >> 2) * kTileBlk;
          const uint64_t ad = tc::smem_desc_sw128(sbase + t * kQTile + koff, 16, 1024);
          const uint64_t bd = tc::smem_desc_sw128(sbase + kOffK + s * kKStage + koff, 16, 1024);
          tc::mma_f16_ss(tmem + kPN * t, ad, bd, id_s, kq > 0 ? 1u : 0u);
        }
      };
      auto pv = [&](int t, bool first) {
#pragma unroll
        for (int kk = 0; kk < kPN / 16; ++kk) {
          const uint64_t bd = tc::smem_desc_sw128(sbase + kOffV + kk * 16 * 128, kTileBlk, 1024);
          tc::mma_f16_ts(tmem + kTmemO + kDv * t, tmem + kPN * t + kk * 8, bd, id_pv,
                         (!first || kk > 0) ? 1u : 0u);
        }
      };
      Cursor cm;
      cm.init(a.segs, a.blocks, seg_begin, seg_end);
      int c1 = 0;      // key tiles that had a Q tile 1
      int segs1 = 0;   // finished segments that had a Q tile 1
      for (int k = 0; k < total; ++k, cm.next()) {
        const bool q1 = cm.bd.nrows > kPM;
        const bool first = cm.first();
        const int s = k & 1;
        if (first && !tc::mbar_wait(&bars.q_full, cm.si & 1, &abort_flag)) break;
        if (!tc::mbar_wait(&bars.k_full[s], (k >> 1) & 1, &abort_flag)) break;
        // S0 of this tile overwrites P0 of the previous one
        if (k > 0 && !tc::mbar_wait(&bars.pv_done[0], (k - 1) & 1, &abort_flag)) break;
        tc::tc_fence_after();
        qk(0, s);
        tc::mma_commit(&bars.s_full[0]);
        if (q1) {
          if (c1 > 0 && !tc::mbar_wait(&bars.pv_done[1], (c1 - 1) & 1, &abort_flag)) break;
          tc::tc_fence_after();
          qk(1, s);
          tc::mma_commit(&bars.s_full[1]);
        }
        tc::mma_commit(&bars.k_empty[s]);
        if (cm.last()) tc::mma_commit(&bars.q_empty);
        if (!tc::mbar_wait(&bars.p_full[0], k & 1, &abort_flag)) break;
        if (!tc::mbar_wait(&bars.v_full, k & 1, &abort_flag)) break;
        // the first P.V of a segment overwrites O: the previous epilogue must have read it
        if (first && cm.si > 0 && !tc::mbar_wait(&bars.o_free[0], (cm.si - 1) & 1, &abort_flag))
          break;
        tc::tc_fence_after();
        pv(0, first);
        tc::mma_commit(&bars.pv_done[0]);
        if (q1) {
          if (!tc::mbar_wait(&bars.p_full[1], c1 & 1, &abort_flag)) break;
          if (first && segs1 > 0 && !tc::mbar_wait(&bars.o_free[1], (segs1 - 1) & 1, &abort_flag))
            break;
          tc::tc_fence_after();
          pv(1, first);
          tc::mma_commit(&bars.pv_done[1]);
          ++c1;
          if (cm.last()) ++segs1;
        }
        tc::mma_commit(&bars.v_empty);
      }
      // every MMA issued must be complete before TMEM is released, also
      // after a give-up (a wait of its own, bounded, that ignores the abort)
      tc::mma_commit(&bars.done);
      int no_abort = 0;
      tc::mbar_wait(&bars.done, 0, &no_abort, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;               // Q tile
    const int wq = warp & 3;               // TMEM lane quadrant
    const int lane = tid & 31;
    const int p = wq * 32 + lane;          // MMA row (TMEM lane)
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + kPN * t;
    const uint32_t o_addr = tmem + lane_base + kTmemO + kDv * t;
    const float sc = a.scale_log2;
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity, &abort_flag));
    };
    Cursor cur;
    cur.init(a.segs, a.blocks, seg_begin, seg_end);
    float m_run = -INFINITY, l_run = 0.f, sink2 = -INFINITY;
    int row_lo = 0, row_hi = 0, row_tok = 0, row_h = 0, r = 0;
    bool valid = false;
    int c = 0;                             // key tiles of this Q tile so far
    for (int k = 0; k < total; ++k, cur.next()) {
      const BlockDesc &bd = cur.bd;
      if (t == 1 && bd.nrows <= kPM) continue;
      if (cur.first()) {
        r = kPM * t + p;
        valid = r < bd.nrows;
        row_lo = row_hi = 0;
        sink2 = -INFINITY;
        if (valid) {
          const int flat = bd.row0 + r;
          row_tok = bd.tok0 + flat / a.group;
          row_h = bd.g * a.group + flat % a.group;
          if (a.sinks) sink2 = a.sinks[row_h] * kLog2e;
          const int i = bd.L - bd.n + flat / a.group;
          row_hi = i + 1;
          row_lo = a.window > 0 ? max(0, i - a.window + 1) : 0;
        }
        m_run = -INFINITY;
        l_run = 0.f;
      }
      if (!wait(&bars.s_full[t], c & 1)) break;
      tc::tc_fence_after();
      const int key0 = cur.tile * kPN;
      const int j_lo = max(0, row_lo - key0);
      const int j_hi = min(kPN, row_hi - key0);
      const bool full = __all_sync(0xffffffffu, j_lo <= 0 && j_hi >= kPN);
      uint32_t ra[16], rb[16];
      // pass 1: the tile maximum of the row's visible columns
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      tc::tmem_ld16(s_addr, ra);
#pragma unroll 1
      for (int ch = 0; ch < kPN / 16; ch += 2) {
        tc::tmem_wait_ld_regs(ra);
        tc::tmem_ld16(s_addr + 16 * (ch + 1), rb);
        if (!full) mask16(ra, ch, j_lo, j_hi);
#pragma unroll
        for (int j = 0; j < 16; ++j) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(ra[j]));
        tc::tmem_wait_ld_regs(rb);
        if (ch + 2 < kPN / 16) tc::tmem_ld16(s_addr + 16 * (ch + 2), ra);
        if (!full) mask16(rb, ch + 1, j_lo, j_hi);
#pragma unroll
        for (int j = 0; j < 16; ++j) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(rb[j]));
      }
      const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
      // O is rescaled only when the maximum grows by more than the threshold;
      // until then P may exceed 1 (up to 2^8)
      const bool need = m_run != -INFINITY && m_tile > m_run + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        if (!wait(&bars.pv_done[t], (c - 1) & 1)) break;
        tc::tc_fence_after();
        const float alpha = need ? ex2(m_run - m_tile) : 1.f;
#pragma unroll 1
        for (int q = 0; q < kDv / 32; ++q) {
          uint32_t o[32];
          tc::tmem_ld32(o_addr + q * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tc::tmem_st32(o_addr + q * 32, o);
        }
        tc::tmem_wait_st();
        l_run *= alpha;
      }
      if (need || m_run == -INFINITY) m_run = m_tile;
      // pass 2: P = 2^(s * sc - m_run) as bf16 pairs into the S columns already read
      const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
      auto exp16 = [&](uint32_t (&raw)[16], int ch) {
        if (!full) mask16(raw, ch, j_lo, j_hi);
        uint32_t pk[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(raw[j]), sc, neg_m));
          const float p1 = ex2(fmaf(__uint_as_float(raw[j + 1]), sc, neg_m));
          rs[(j >> 1) & 3] += p0 + p1;
          pk[j >> 1] = bf16_pair(p0, p1);
        }
        tc::tmem_st8(s_addr + 8 * ch, pk);
      };
      tc::tmem_ld16(s_addr, ra);
#pragma unroll 1
      for (int ch = 0; ch < kPN / 16; ch += 2) {
        tc::tmem_wait_ld_regs(ra);
        tc::tmem_ld16(s_addr + 16 * (ch + 1), rb);
        exp16(ra, ch);
        tc::tmem_wait_ld_regs(rb);
        if (ch + 2 < kPN / 16) tc::tmem_ld16(s_addr + 16 * (ch + 2), ra);
        exp16(rb, ch + 1);
      }
      tc::tmem_wait_st();                  // P is in TMEM before p_full is signalled
      tc::tc_fence_before();
      tc::mbar_arrive(&bars.p_full[t]);
      l_run += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      const int cdone = c++;
      if (!cur.last()) continue;

      // ---------------- end of segment: normalise and write the rows
      if (!wait(&bars.pv_done[t], cdone & 1)) break;
      tc::tc_fence_after();
      const bool single = bd.num_splits == 1;
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
      const int prow = bd.part_row_base + cur.sd.split * bd.nrows + r;
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
      tc::mbar_arrive(&bars.o_free[t]);
    }
  }

  __syncthreads();
  if (tid == 0 && abort_flag) atomicOr(a.err, 2);
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attn_prefill(const HostPlan &hp, const RunArgs &a, cudaStream_t stream) {
  if (hp.num_ctas == 0) return cudaSuccess;
  if (hp.prob.kv_dtype == ATTN_KV_FP8_E4M3)
    attn_prefill_kernel<true><<<hp.num_ctas, kPThreads, kSmem, stream>>>(a);
  else
    attn_prefill_kernel<false><<<hp.num_ctas, kPThreads, kSmem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t prepare_attn_prefill(const HostPlan &hp) {
  return hp.prob.kv_dtype == ATTN_KV_FP8_E4M3
             ? cudaFuncSetAttribute(attn_prefill_kernel<true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)
             : cudaFuncSetAttribute(attn_prefill_kernel<false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

}  // namespace akp
