// Tensor-core split-KV attention for 128-row blocks (chunked prefill), on the
// Blackwell tcgen05 path: Q.K^T and P.V run on tcgen05.mma with operands in
// 128-byte swizzled shared memory and accumulators in tensor memory (TMEM).
//
// The pages' own prefill kernel (MiMo-V2.6-Flash-RL model card, "What the
// kernels do") is an sm_120 mma.sync design with one CTA per 8 tokens x 16 GQA
// heads and FP8 K/V converted in the load path; the row packing and the
// conversion point are kept, the rest is redesigned for sm_103a:
//   warps 0-3  softmax: thread r owns query row r = TMEM lane r; reads S from
//              TMEM, masks, keeps a lazily rescaled running max (O in TMEM is
//              only rescaled when the max grows by more than 2^8), writes P
//              (fp16/bf16) to shared memory, and runs the epilogue;
//   warps 4-7  loaders: gather K/V rows through the page table (16-byte
//              loads), convert E4M3 to fp16 exactly, and store them in the
//              swizzled operand layouts; also stage Q per block;
//   warp  8    allocates TMEM and issues every tcgen05.mma from one thread:
//              S(i+1) = Q.K(i+1)^T is issued before O += P(i).V(i) so the
//              softmax of tile i overlaps the next Q.K^T.
// TMEM: S double buffer (2 x 64 columns) + O (128 columns) = 256 columns.
// All waits are bounded in time: a broken invariant ends the kernel and sets
// bit 1 of the plan's error word instead of hanging the GPU.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <cstdint>

#include "kernels.hpp"
#include "tc_common.cuh"

namespace akp {
namespace {

constexpr int kRows = 128;
constexpr int kN = kKeyTile;                 // keys per tile
constexpr int kStages = 3;                   // K/V ring depth
constexpr int kThreads = 9 * 32;
constexpr int kQBlock = kRows * 128;         // one 64-column block of Q: 16 KB
constexpr int kQBytes = 3 * kQBlock;         // 48 KB
constexpr int kKBlock = kN * 128;            // one 64-column block of a K tile: 8 KB
constexpr int kKBytes = 3 * kKBlock;         // 24 KB
constexpr int kVBlock = kN * 128;            // one 64-wide dv block of a V tile: 8 KB
constexpr int kVBytes = 2 * kVBlock;         // 16 KB
constexpr int kPBytes = kRows * 128;         // P tile [128 rows x 64 keys]: 16 KB
constexpr int kOffK = kQBytes;
constexpr int kOffV = kOffK + kStages * kKBytes;
constexpr int kOffP = kOffV + kStages * kVBytes;
constexpr int kSmemUsed = kOffP + 2 * kPBytes;
constexpr int kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024 B
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemO = 128;             // O accumulator columns [128, 256)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;    // base-2 growth allowed before O is rescaled

struct Bars {
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], pv_done[2];
  uint64_t o_free, final_done;
};

// Walks the CTA's tiles in order: segment index, tile id, first/last flags.
struct Cursor {
  const SegDesc *segs;
  int seg, seg_end, tile, si;
  __device__ void init(const SegDesc *s, int b, int e) {
    segs = s;
    seg = b;
    seg_end = e;
    tile = s[b].tile_begin;
    si = 0;
  }
  __device__ bool first() const { return tile == segs[seg].tile_begin; }
  __device__ bool last() const { return tile + 1 == segs[seg].tile_end; }
  __device__ void next() {
    if (++tile == segs[seg].tile_end && seg + 1 < seg_end) {
      ++seg;
      ++si;
      tile = segs[seg].tile_begin;
    }
  }
};

__device__ __forceinline__ uint32_t cvt_pair(float lo, float hi, bool half) {
  if (half) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// 16 E4M3 codes -> 16 fp16 values (exact), as two 16-byte chunks.
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 raw, uint4 &lo, uint4 &hi) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t h[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __half2_raw a = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[q] & 0xFFFFu),
                                               __NV_E4M3);
    __half2_raw b = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[q] >> 16),
                                               __NV_E4M3);
    h[2 * q] = static_cast<uint32_t>(a.x) | (static_cast<uint32_t>(a.y) << 16);
    h[2 * q + 1] = static_cast<uint32_t>(b.x) | (static_cast<uint32_t>(b.y) << 16);
  }
  lo = make_uint4(h[0], h[1], h[2], h[3]);
  hi = make_uint4(h[4], h[5], h[6], h[7]);
}

__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&w[q]);
    __half2 h = __float22half2_rn(__bfloat1622float2(b));
    w[q] = *reinterpret_cast<uint32_t *>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const RunArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ Bars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int seg_begin = a.cta_seg_begin[blockIdx.x];
  const int seg_end = a.cta_seg_begin[blockIdx.x + 1];
  if (seg_begin >= seg_end) return;
  int total = 0;
  for (int s = seg_begin; s < seg_end; ++s) total += a.segs[s].tile_end - a.segs[s].tile_begin;

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&bars.kv_full[s], 128);
      tc::mbar_init(&bars.kv_empty[s], 1);
    }
    tc::mbar_init(&bars.q_full, 128);
    tc::mbar_init(&bars.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars.s_full[b], 1);
      tc::mbar_init(&bars.s_empty[b], 128);
      tc::mbar_init(&bars.p_full[b], 128);
      tc::mbar_init(&bars.pv_done[b], 1);
    }
    tc::mbar_init(&bars.o_free, 128);
    tc::mbar_init(&bars.final_done, 1);
    tc::fence_mbar_init();
  }
  if (warp == 8) tc::tmem_alloc(&tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t sbase = tc::smem_u32(smem);
  constexpr bool kHalf = FP8;  // operand type: fp16 for FP8 caches, bf16 otherwise

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ loaders
    const int lt = tid - 128;
    const uint8_t *kc = static_cast<const uint8_t *>(a.k_cache);
    const uint8_t *vc = static_cast<const uint8_t *>(a.v_cache);
    Cursor cur;
    cur.init(a.segs, seg_begin, seg_end);
    for (int k = 0; k < total; ++k, cur.next()) {
      const SegDesc sd = a.segs[cur.seg];
      const BlockDesc bd = a.blocks[sd.block];
      if (cur.first()) {
        if (cur.si > 0 && !tc::mbar_wait(&bars.q_empty, (cur.si - 1) & 1, &abort_flag)) break;
        // Q rows of the block -> 3 swizzled 64-column blocks
        for (int idx = lt; idx < kRows * 24; idx += 128) {
          const int r = idx / 24;
          const int ch = idx % 24;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (r < bd.nrows) {
            const int flat = bd.row0 + r;
            const int tok = bd.tok0 + flat / a.group;
            const int h = bd.g * a.group + flat % a.group;
            v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.q) +
                                                      ((int64_t)tok * a.hq + h) * kDqk) + ch);
            if (kHalf) v = bf16x8_to_f16x8(v);
          }
          *reinterpret_cast<uint4 *>(smem + (ch >> 3) * kQBlock + tc::sw128_offset(r, ch & 7)) = v;
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&bars.q_full);
      }
      const int s = k % kStages;
      if (k >= kStages && !tc::mbar_wait(&bars.kv_empty[s], ((k / kStages) - 1) & 1, &abort_flag))
        break;
      uint8_t *sk = smem + kOffK + s * kKBytes;
      uint8_t *sv = smem + kOffV + s * kVBytes;
      const int key0 = cur.tile * kN;
      const int32_t *pt_row = a.page_table + (int64_t)bd.b * a.pt_stride;
      constexpr int kEs = FP8 ? 1 : 2;
      constexpr int kKch = kDqk * kEs / 16;  // source 16-byte chunks per K row
      constexpr int kVch = kDv * kEs / 16;
      constexpr int kPer = kN * (kKch + kVch) / 128;
      uint4 buf[kPer];
      // issue every load of the tile first, then convert and store
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int c = lt + u * 128;
        const bool is_k = c < kN * kKch;
        const int cc = is_k ? c : c - kN * kKch;
        const int nch = is_k ? kKch : kVch;
        const int kk = cc / nch;
        const int ch = cc % nch;
        const int j = key0 + kk;
        buf[u] = make_uint4(0u, 0u, 0u, 0u);
        if (j >= bd.klo && j < bd.khi) {
          const int32_t page = __ldg(pt_row + j / a.page_size);
          if (page >= 0 && page < a.num_pages) {
            const int64_t slot = (int64_t)page * a.page_size + j % a.page_size;
            const uint8_t *src = is_k ? kc + (slot * a.hkv + bd.g) * (kDqk * kEs) + ch * 16
                                      : vc + (slot * a.hkv + bd.g) * (kDv * kEs) + ch * 16;
            buf[u] = __ldg(reinterpret_cast<const uint4 *>(src));
          } else {
            atomicOr(a.err, 1);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int c = lt + u * 128;
        const bool is_k = c < kN * kKch;
        const int cc = is_k ? c : c - kN * kKch;
        const int nch = is_k ? kKch : kVch;
        const int kk = cc / nch;
        const int ch = cc % nch;
        uint8_t *dst = is_k ? sk : sv;   // both: 64-column blocks of [64 rows x 128 B]
        if (FP8) {
          uint4 lo, hi;
          e4m3x16_to_f16(buf[u], lo, hi);
          const int c16 = 2 * ch;        // fp16 chunk index within the row
          *reinterpret_cast<uint4 *>(dst + (c16 >> 3) * kKBlock + tc::sw128_offset(kk, c16 & 7)) = lo;
          *reinterpret_cast<uint4 *>(dst + ((c16 + 1) >> 3) * kKBlock +
                                     tc::sw128_offset(kk, (c16 + 1) & 7)) = hi;
        } else {
          *reinterpret_cast<uint4 *>(dst + (ch >> 3) * kKBlock + tc::sw128_offset(kk, ch & 7)) =
              buf[u];
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&bars.kv_full[s]);
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if ((tid & 31) == 0) {
      const uint32_t id_s = tc::idesc_f16(kHalf ? 0 : 1, 0, 0, kRows, kN);
      const uint32_t id_pv = tc::idesc_f16(kHalf ? 0 : 1, 0, 1, kRows, kDv);
      Cursor cs, cp;
      cs.init(a.segs, seg_begin, seg_end);
      cp.init(a.segs, seg_begin, seg_end);
      bool ok = true;
      auto issue_pv = [&](int k) -> bool {
        const int b = k & 1;
        const int s = k % kStages;
        if (!tc::mbar_wait(&bars.p_full[b], (k >> 1) & 1, &abort_flag)) return false;
        const bool first = cp.first();
        if (first && cp.si > 0 && !tc::mbar_wait(&bars.o_free, (cp.si - 1) & 1, &abort_flag))
          return false;
        tc::tc_fence_after();
        const uint32_t pb = sbase + kOffP + b * kPBytes;
        const uint32_t vb = sbase + kOffV + s * kVBytes;
#pragma unroll
        for (int kk = 0; kk < kN / 16; ++kk) {
          const uint64_t ad = tc::smem_desc_sw128(pb + kk * 32, 16, 1024);
          const uint64_t bdsc = tc::smem_desc_sw128(vb + kk * 16 * 128, kVBlock, 1024);
          tc::mma_f16_ss(tmem + kTmemO, ad, bdsc, id_pv, (!first || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(&bars.kv_empty[s]);
        tc::mma_commit(&bars.pv_done[b]);
        cp.next();
        return true;
      };
      for (int k = 0; k < total && ok; ++k, cs.next()) {
        const int s = k % kStages;
        const int b = k & 1;
        if (cs.first() && !tc::mbar_wait(&bars.q_full, cs.si & 1, &abort_flag)) break;
        if (!tc::mbar_wait(&bars.kv_full[s], (k / kStages) & 1, &abort_flag)) break;
        if (k >= 2 && !tc::mbar_wait(&bars.s_empty[b], ((k >> 1) - 1) & 1, &abort_flag)) break;
        tc::tc_fence_after();
        const uint32_t kb = sbase + kOffK + s * kKBytes;
#pragma unroll
        for (int ks = 0; ks < kDqk / 16; ++ks) {
          const uint32_t koff = (ks & 3) * 32;
          const uint64_t ad = tc::smem_desc_sw128(sbase + (ks >> 2) * kQBlock + koff, 16, 1024);
          const uint64_t bdsc = tc::smem_desc_sw128(kb + (ks >> 2) * kKBlock + koff, 16, 1024);
          tc::mma_f16_ss(tmem + b * kN, ad, bdsc, id_s, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(&bars.s_full[b]);
        if (cs.last()) tc::mma_commit(&bars.q_empty);
        if (k >= 1) ok = issue_pv(k - 1);
      }
      if (ok && !abort_flag) issue_pv(total - 1);
      tc::mma_commit(&bars.final_done);
      tc::mbar_wait(&bars.final_done, 0, &abort_flag);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = tid;  // query row of the block == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    Cursor cur;
    cur.init(a.segs, seg_begin, seg_end);
    float m_run = -INFINITY, l_run = 0.f;
    int row_lo = 0, row_hi = 0, tok = 0, h = 0;
    bool valid = false;
    BlockDesc bd{};
    for (int k = 0; k < total; ++k, cur.next()) {
      const SegDesc sd = a.segs[cur.seg];
      const bool first = cur.first();
      if (first) {
        bd = a.blocks[sd.block];
        valid = r < bd.nrows;
        row_lo = row_hi = 0;
        if (valid) {
          const int flat = bd.row0 + r;
          const int t = flat / a.group;
          tok = bd.tok0 + t;
          h = bd.g * a.group + flat % a.group;
          const int i = bd.L - bd.n + t;
          row_hi = i + 1;
          row_lo = a.window > 0 ? max(0, i - a.window + 1) : 0;
        }
      }
      const int b = k & 1;
      if (!tc::mbar_wait(&bars.s_full[b], (k >> 1) & 1, &abort_flag)) break;
      tc::tc_fence_after();
      float sv[kN];
      {
        uint32_t raw[32];
        tc::tmem_ld32(tmem + lane_base + b * kN, raw);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(raw[j]);
        tc::tmem_ld32(tmem + lane_base + b * kN + 32, raw);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[32 + j] = __uint_as_float(raw[j]);
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&bars.s_empty[b]);

      const int key0 = cur.tile * kN;
      float m_tile = -INFINITY;
#pragma unroll
      for (int j = 0; j < kN; ++j) {
        const int key = key0 + j;
        const bool vis = key >= row_lo && key < row_hi;
        sv[j] = vis ? sv[j] * a.scale_log2 : -INFINITY;
        m_tile = fmaxf(m_tile, sv[j]);
      }
      if (first) {
        m_run = m_tile;
        l_run = 0.f;
      } else {
        const bool need = m_tile > m_run + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          if (!tc::mbar_wait(&bars.pv_done[(k - 1) & 1], ((k - 1) >> 1) & 1, &abort_flag)) break;
          tc::tc_fence_after();
          const float m_new = need ? m_tile : m_run;
          const float alpha = need ? exp2f(m_run - m_new) : 1.f;
#pragma unroll
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
          m_run = m_new;
        }
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      uint32_t pk[kN / 2];
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < kN; j += 2) {
        const float p0 = exp2f(sv[j] - m_use);
        const float p1 = exp2f(sv[j + 1] - m_use);
        rs += p0 + p1;
        pk[j / 2] = cvt_pair(p0, p1, kHalf);
      }
      l_run += rs;
      if (k >= 2 && !tc::mbar_wait(&bars.pv_done[b], ((k - 2) >> 1) & 1, &abort_flag)) break;
      uint8_t *pb = smem + kOffP + b * kPBytes;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(pb + tc::sw128_offset(r, c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(&bars.p_full[b]);

      if (cur.last()) {
        if (!tc::mbar_wait(&bars.pv_done[b], (k >> 1) & 1, &abort_flag)) break;
        tc::tc_fence_after();
        const bool single = bd.num_splits == 1;
        float scale_o = 0.f, lse = -INFINITY;
        if (single) {
          const float sig = (a.sinks && valid) ? a.sinks[h] * kLog2e : -INFINITY;
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
        const int prow = bd.part_row_base + sd.split * bd.nrows + r;
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
                                __uint_as_float(o[8 * q + 2 * e + 1]) * scale_o, false);
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
        tc::tc_fence_before();
        tc::mbar_arrive(&bars.o_free);
      }
    }
  }

  __syncthreads();
  if (tid == 0 && abort_flag) atomicOr(a.err, 2);
  if (warp == 8) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill_tc(const HostPlan &hp, const RunArgs &a, cudaStream_t stream) {
  if (hp.num_ctas == 0) return cudaSuccess;
  if (hp.prob.kv_dtype == ATTN_KV_FP8_E4M3)
    prefill_tc_kernel<true><<<hp.num_ctas, kThreads, kSmemBytes, stream>>>(a);
  else
    prefill_tc_kernel<false><<<hp.num_ctas, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t prepare_prefill_tc(const HostPlan &hp) {
  if (hp.prob.kv_dtype == ATTN_KV_FP8_E4M3)
    return cudaFuncSetAttribute(prefill_tc_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  return cudaFuncSetAttribute(prefill_tc_kernel<false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

}  // namespace akp
