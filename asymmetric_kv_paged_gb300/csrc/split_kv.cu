// Split-KV paged attention for QK head dim 192 / V head dim 128.
//
// One CTA walks the key tiles of its segments (see planner.cpp) through a
// multi-stage cp.async pipeline: page-table lookup -> 16-byte async copies of
// the 384-byte K rows and 256-byte V rows into XOR-swizzled shared memory ->
// (FP8 caches: exact E4M3 -> fp16 conversion in shared memory) -> Q.K^T on
// tensor cores -> mask -> online softmax (base 2) -> P.V on tensor cores.
// A segment that covers its whole block writes the final bf16 row (sink
// folded into the denominator); otherwise it writes a normalised fp32 partial
// and its base-2 log-sum-exp for the merge kernel.
//
// Page-table gather, FP8 conversion in the load path, split-KV that stays on
// for multi-token verify, and one pass over the keys for all draft tokens of a
// request follow the MiMo-V2.6-Flash-RL model card ("What the kernels do").
// Keys outside a block's visible range are never fetched (their shared-memory
// rows are zero-filled) and masked scores are replaced, not multiplied, so NaN
// in unused slots cannot leak (sammysun0711/sglang PR #35, FlyPA V-tail fix).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <cstdint>

#include "kernels.hpp"

namespace akp {

namespace {

constexpr int kStages = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16) * B(16x8), fp32 accumulate; element type bf16 or fp16.
template <bool kHalf>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (kHalf) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <bool kHalf>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kHalf) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}

// Byte offset of 16-byte chunk `ch` of row `row` in a swizzled tile whose rows
// are `row_bytes` long: the low three chunk bits are XORed with the row, so an
// 8x16-byte ldmatrix read touches 8 distinct bank groups.
__device__ __forceinline__ uint32_t swz(int row, int ch, int row_bytes) {
  return static_cast<uint32_t>(row * row_bytes + ((ch ^ (row & 7)) << 4));
}

// Static shape of one kernel instance.
template <int WM, int WN, bool FP8>
struct Cfg {
  static constexpr int kWarps = WM * WN;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kKw = kKeyTile / WN;   // keys per warp per tile
  static constexpr int kNt = kKw / 8;         // n8 score tiles per warp
  static constexpr int kElem = FP8 ? 1 : 2;   // cache element bytes
  static constexpr int kKRow = kDqk * kElem;  // bytes of one cached K row
  static constexpr int kVRow = kDv * kElem;
  // shared memory
  static constexpr int kStageK = kKeyTile * kKRow;
  static constexpr int kStageV = kKeyTile * kVRow;
  static constexpr int kStageBytes = kStageK + kStageV;
  static constexpr int kConvK = FP8 ? kKeyTile * kDqk * 2 : 0;  // fp16 compute tile
  static constexpr int kConvV = FP8 ? kKeyTile * kDv * 2 : 0;
  static constexpr int kComb = WN > 1 ? WN * 16 * (kDv + 2) * 4 : 0;
  static constexpr int kSmem = kStages * kStageBytes + kConvK + kConvV + kComb;
};

template <int WM, int WN, bool FP8>
__global__ void __launch_bounds__(Cfg<WM, WN, FP8>::kThreads, 1)
    split_kv_kernel(const RunArgs a) {
  using C = Cfg<WM, WN, FP8>;
  constexpr bool kHalf = FP8;  // FP8 caches compute in fp16 (exact E4M3 -> fp16)
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *const s_stage = smem;
  uint8_t *const s_convk = smem + kStages * C::kStageBytes;
  uint8_t *const s_convv = s_convk + C::kConvK;
  float *const s_comb = reinterpret_cast<float *>(s_convv + C::kConvV);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int wm = warp / WN;
  const int wn = warp % WN;
  const int qr = lane >> 2;  // fragment row within 8
  const int qc = lane & 3;   // fragment column pair

  const int seg_begin = a.cta_seg_begin[blockIdx.x];
  const int seg_end = a.cta_seg_begin[blockIdx.x + 1];
  if (seg_begin >= seg_end) return;
  int total = 0;
  for (int s = seg_begin; s < seg_end; ++s) total += a.segs[s].tile_end - a.segs[s].tile_begin;

  const uint8_t *kc = static_cast<const uint8_t *>(a.k_cache);
  const uint8_t *vc = static_cast<const uint8_t *>(a.v_cache);

  // ---------------- loader: one tile into one stage ----------------
  int ld_seg = seg_begin;
  int ld_tile = a.segs[seg_begin].tile_begin;
  int issued = 0;
  auto issue = [&]() {
    if (issued < total) {
      const SegDesc sd = a.segs[ld_seg];
      const BlockDesc bd = a.blocks[sd.block];
      uint8_t *stg = s_stage + (issued % kStages) * C::kStageBytes;
      const uint32_t sk = smem_u32(stg);
      const uint32_t sv = sk + C::kStageK;
      const int key0 = ld_tile * kKeyTile;
      const int32_t *pt_row = a.page_table + (int64_t)bd.b * a.pt_stride;
      constexpr int kKch = C::kKRow / 16;  // 16-B chunks per K row
      constexpr int kVch = C::kVRow / 16;
      constexpr int kChunks = kKeyTile * (kKch + kVch);
      static_assert(kChunks % C::kThreads == 0, "chunk split");
      int cached_key = -1;
      int64_t slot = 0;
      bool valid = false;
#pragma unroll 4
      for (int u = 0; u < kChunks / C::kThreads; ++u) {
        const int c = tid + u * C::kThreads;
        const bool is_k = c < kKeyTile * kKch;
        const int cc = is_k ? c : c - kKeyTile * kKch;
        const int nch = is_k ? kKch : kVch;
        const int kk = cc / nch;
        const int ch = cc % nch;
        const int j = key0 + kk;
        if (kk != cached_key) {
          cached_key = kk;
          valid = j >= bd.klo && j < bd.khi;
          if (valid) {
            const int32_t page = __ldg(pt_row + j / a.page_size);
            if (page < 0 || page >= a.num_pages) {
              atomicOr(a.err, 1);
              valid = false;
            } else {
              slot = (int64_t)page * a.page_size + (j % a.page_size);
            }
          }
        }
        const uint8_t *src;
        uint32_t dst;
        if (is_k) {
          src = kc + ((slot * a.hkv + bd.g) * C::kKRow + ch * 16);
          dst = FP8 ? sk + kk * C::kKRow + ch * 16 : sk + swz(kk, ch, C::kKRow);
        } else {
          src = vc + ((slot * a.hkv + bd.g) * C::kVRow + ch * 16);
          dst = FP8 ? sv + kk * C::kVRow + ch * 16 : sv + swz(kk, ch, C::kVRow);
        }
        cp_async16(dst, valid ? src : kc, valid ? 16 : 0);
      }
      // advance the loader cursor
      if (++ld_tile == sd.tile_end && ld_seg + 1 < seg_end) {
        ++ld_seg;
        ld_tile = a.segs[ld_seg].tile_begin;
      }
    }
    cp_async_commit();
    ++issued;
  };

  for (int s = 0; s < kStages - 1; ++s) issue();

  // ---------------- per-segment compute state ----------------
  uint32_t qf[kDqk / 16][4];
  float o[kDv / 8][4];
  float m_run[2], l_run[2];
  int row_lo[2], row_hi[2];
  int c_seg = seg_begin;
  int c_tile = a.segs[seg_begin].tile_begin;
  BlockDesc bd = a.blocks[a.segs[seg_begin].block];

  for (int k = 0; k < total; ++k) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    issue();

    const SegDesc sd = a.segs[c_seg];
    if (c_tile == sd.tile_begin) {
      // ---- begin a segment: rows, Q fragments, running state ----
      bd = a.blocks[sd.block];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = wm * 16 + qr + hr * 8;
        row_lo[hr] = 0;
        row_hi[hr] = 0;
        if (r < bd.nrows) {
          const int flat = bd.row0 + r;
          const int t = flat / a.group;
          const int i = bd.L - bd.n + t;
          row_hi[hr] = i + 1;
          row_lo[hr] = a.window > 0 ? max(0, i - a.window + 1) : 0;
        }
        m_run[hr] = -INFINITY;
        l_run[hr] = 0.f;
      }
#pragma unroll
      for (int nt = 0; nt < kDv / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
      const uint32_t *qrow[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = wm * 16 + qr + hr * 8;
        qrow[hr] = nullptr;
        if (r < bd.nrows) {
          const int flat = bd.row0 + r;
          const int tok = bd.tok0 + flat / a.group;
          const int h = bd.g * a.group + flat % a.group;
          qrow[hr] = reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(a.q) +
                                                        ((int64_t)tok * a.hq + h) * kDqk);
        }
      }
#pragma unroll
      for (int ks = 0; ks < kDqk / 16; ++ks) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int hr = e & 1;
          const int col = ks * 8 + qc + (e >> 1) * 4;  // in 32-bit words
          uint32_t v = qrow[hr] ? __ldg(qrow[hr] + col) : 0u;
          if constexpr (kHalf) {
            __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&v);
            __half2 h2 = __float22half2_rn(__bfloat1622float2(b));
            v = *reinterpret_cast<uint32_t *>(&h2);
          }
          qf[ks][e] = v;
        }
      }
    }

    // ---- FP8: convert the landed stage into the fp16 compute tile ----
    const uint8_t *stg = s_stage + (k % kStages) * C::kStageBytes;
    uint32_t tk, tv;
    if constexpr (FP8) {
      constexpr int kKch8 = kDqk / 16;  // 12 raw 16-B chunks per K row
      constexpr int kVch8 = kDv / 16;   // 8 per V row
      constexpr int kRaw = kKeyTile * (kKch8 + kVch8);
      for (int c = tid; c < kRaw; c += C::kThreads) {
        const bool is_k = c < kKeyTile * kKch8;
        const int cc = is_k ? c : c - kKeyTile * kKch8;
        const int nch = is_k ? kKch8 : kVch8;
        const int kk = cc / nch;
        const int ch = cc % nch;
        const uint4 raw = *reinterpret_cast<const uint4 *>(
            stg + (is_k ? kk * kDqk + ch * 16 : C::kStageK + kk * kDv + ch * 16));
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t hv[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
              static_cast<__nv_fp8x2_storage_t>(w[q] & 0xFFFFu), __NV_E4M3);
          __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
              static_cast<__nv_fp8x2_storage_t>(w[q] >> 16), __NV_E4M3);
          hv[2 * q] = static_cast<uint32_t>(lo.x) | (static_cast<uint32_t>(lo.y) << 16);
          hv[2 * q + 1] = static_cast<uint32_t>(hi.x) | (static_cast<uint32_t>(hi.y) << 16);
        }
        uint8_t *dstb = is_k ? s_convk : s_convv;
        const int rb = is_k ? kDqk * 2 : kDv * 2;
        *reinterpret_cast<uint4 *>(dstb + swz(kk, 2 * ch, rb)) =
            make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4 *>(dstb + swz(kk, 2 * ch + 1, rb)) =
            make_uint4(hv[4], hv[5], hv[6], hv[7]);
      }
      __syncthreads();
      tk = smem_u32(s_convk);
      tv = smem_u32(s_convv);
    } else {
      tk = smem_u32(stg);
      tv = tk + C::kStageK;
    }

    // ---- S = Q K^T for this warp's keys ----
    float acc[C::kNt][4];
#pragma unroll
    for (int nt = 0; nt < C::kNt; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
    const int kw0 = wn * C::kKw;  // warp's first key within the tile
#pragma unroll
    for (int ks = 0; ks < kDqk / 16; ++ks) {
#pragma unroll
      for (int np = 0; np < C::kNt / 2; ++np) {
        const int key = kw0 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int ch = 2 * ks + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tk + swz(key, ch, kDqk * 2), b0, b1, b2, b3);
        mma16816<kHalf>(acc[2 * np], qf[ks], b0, b1);
        mma16816<kHalf>(acc[2 * np + 1], qf[ks], b2, b3);
      }
    }

    // ---- mask + online softmax (base 2) ----
    const int key_base = c_tile * kKeyTile + kw0;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < C::kNt; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        const int j = key_base + nt * 8 + 2 * qc + (e & 1);
        const bool vis = j >= row_lo[hr] && j < row_hi[hr];
        const float s = vis ? acc[nt][e] * a.scale_log2 : -INFINITY;
        acc[nt][e] = s;
        mx[hr] = fmaxf(mx[hr], s);
      }
    float alpha[2], m_use[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
      const float m_new = fmaxf(m_run[hr], mx[hr]);
      m_use[hr] = m_new == -INFINITY ? 0.f : m_new;
      alpha[hr] = exp2f(m_run[hr] - m_use[hr]);
      m_run[hr] = m_new;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < C::kNt; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        const float p = exp2f(acc[nt][e] - m_use[hr]);
        acc[nt][e] = p;
        rs[hr] += p;
      }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) l_run[hr] = l_run[hr] * alpha[hr] + rs[hr];
#pragma unroll
    for (int nt = 0; nt < kDv / 8; ++nt) {
      o[nt][0] *= alpha[0];
      o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1];
      o[nt][3] *= alpha[1];
    }

    // ---- O += P V ----
#pragma unroll
    for (int kk = 0; kk < C::kKw / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = pack2<kHalf>(acc[2 * kk][0], acc[2 * kk][1]);
      pa[1] = pack2<kHalf>(acc[2 * kk][2], acc[2 * kk][3]);
      pa[2] = pack2<kHalf>(acc[2 * kk + 1][0], acc[2 * kk + 1][1]);
      pa[3] = pack2<kHalf>(acc[2 * kk + 1][2], acc[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < kDv / 16; ++dp) {
        const int key = kw0 + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int ch = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tv + swz(key, ch, kDv * 2), b0, b1, b2, b3);
        mma16816<kHalf>(o[2 * dp], pa, b0, b1);
        mma16816<kHalf>(o[2 * dp + 1], pa, b2, b3);
      }
    }

    // ---- end of segment: write the row results ----
    if (c_tile + 1 == sd.tile_end) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
        l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
      }
      if constexpr (WN > 1) {
        // combine the WN key-slices of the same 16 rows through shared memory
        float *cw = s_comb + wn * 16 * (kDv + 2);
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int r = qr + hr * 8;
#pragma unroll
          for (int nt = 0; nt < kDv / 8; ++nt) {
            cw[r * (kDv + 2) + nt * 8 + 2 * qc] = o[nt][2 * hr];
            cw[r * (kDv + 2) + nt * 8 + 2 * qc + 1] = o[nt][2 * hr + 1];
          }
          if (qc == 0) {
            cw[r * (kDv + 2) + kDv] = m_run[hr];
            cw[r * (kDv + 2) + kDv + 1] = l_run[hr];
          }
        }
        __syncthreads();
        // each thread finalises (row, 4 columns) pairs
        for (int idx = tid; idx < 16 * (kDv / 4); idx += C::kThreads) {
          const int r = idx / (kDv / 4);
          const int c4 = (idx % (kDv / 4)) * 4;
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < WN; ++w) M = fmaxf(M, s_comb[(w * 16 + r) * (kDv + 2) + kDv]);
          const float Mu = M == -INFINITY ? 0.f : M;
          float L = 0.f, v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int w = 0; w < WN; ++w) {
            const float *row = s_comb + (w * 16 + r) * (kDv + 2);
            const float f = exp2f(row[kDv] - Mu);
            L += row[kDv + 1] * f;
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] += row[c4 + e] * f;
          }
          if (r < bd.nrows) {
            const int flat = bd.row0 + r;
            const int tok = bd.tok0 + flat / a.group;
            const int h = bd.g * a.group + flat % a.group;
            if (bd.num_splits == 1) {
              const float sig = a.sinks ? a.sinks[h] * kLog2e : -INFINITY;
              const float MM = fmaxf(M, sig);
              float scale_o = 0.f, lse = -INFINITY;
              if (MM != -INFINITY) {
                const float Z = L * exp2f(M - MM) + exp2f(sig - MM);
                scale_o = exp2f(M - MM) * a.v_scale / Z;
                lse = (MM + log2f(Z)) * kLn2;
              }
              __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(
                  static_cast<uint16_t *>(a.out) + ((int64_t)tok * a.hq + h) * kDv + c4);
              dst[0] = __floats2bfloat162_rn(v[0] * scale_o, v[1] * scale_o);
              dst[1] = __floats2bfloat162_rn(v[2] * scale_o, v[3] * scale_o);
              if (a.lse_out && c4 == 0) a.lse_out[(int64_t)tok * a.hq + h] = lse;
            } else {
              const int prow = bd.part_row_base + sd.split * bd.nrows + r;
              const float inv = L > 0.f ? a.v_scale / L : 0.f;
              *reinterpret_cast<float4 *>(a.part_o + (int64_t)prow * kDv + c4) =
                  make_float4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
              if (c4 == 0) a.part_lse[prow] = L > 0.f ? M + log2f(L) : -INFINITY;
            }
          }
        }
        __syncthreads();
      } else {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int r = wm * 16 + qr + hr * 8;
          if (r >= bd.nrows) continue;
          const int flat = bd.row0 + r;
          const int tok = bd.tok0 + flat / a.group;
          const int h = bd.g * a.group + flat % a.group;
          const float M = m_run[hr];
          const float L = l_run[hr];
          if (bd.num_splits == 1) {
            const float sig = a.sinks ? a.sinks[h] * kLog2e : -INFINITY;
            const float MM = fmaxf(M, sig);
            float scale_o = 0.f, lse = -INFINITY;
            if (MM != -INFINITY) {
              const float Z = L * exp2f(M - MM) + exp2f(sig - MM);
              scale_o = exp2f(M - MM) * a.v_scale / Z;
              lse = (MM + log2f(Z)) * kLn2;
            }
            uint16_t *orow = static_cast<uint16_t *>(a.out) + ((int64_t)tok * a.hq + h) * kDv;
#pragma unroll
            for (int nt = 0; nt < kDv / 8; ++nt)
              *reinterpret_cast<__nv_bfloat162 *>(orow + nt * 8 + 2 * qc) = __floats2bfloat162_rn(
                  o[nt][2 * hr] * scale_o, o[nt][2 * hr + 1] * scale_o);
            if (a.lse_out && qc == 0) a.lse_out[(int64_t)tok * a.hq + h] = lse;
          } else {
            const int prow = bd.part_row_base + sd.split * bd.nrows + r;
            const float inv = L > 0.f ? a.v_scale / L : 0.f;
            float *prow_o = a.part_o + (int64_t)prow * kDv;
#pragma unroll
            for (int nt = 0; nt < kDv / 8; ++nt)
              *reinterpret_cast<float2 *>(prow_o + nt * 8 + 2 * qc) =
                  make_float2(o[nt][2 * hr] * inv, o[nt][2 * hr + 1] * inv);
            if (qc == 0) a.part_lse[prow] = L > 0.f ? M + log2f(L) : -INFINITY;
          }
        }
      }
    }

    // advance the compute cursor
    if (++c_tile == sd.tile_end && c_seg + 1 < seg_end) {
      ++c_seg;
      c_tile = a.segs[c_seg].tile_begin;
    }
  }
  cp_async_wait<0>();
}

template <int WM, int WN, bool FP8>
cudaError_t launch_one(const HostPlan &hp, const RunArgs &a, cudaStream_t stream) {
  using C = Cfg<WM, WN, FP8>;
  split_kv_kernel<WM, WN, FP8><<<hp.num_ctas, C::kThreads, C::kSmem, stream>>>(a);
  return cudaGetLastError();
}

template <int WM, int WN, bool FP8>
cudaError_t prepare_one() {
  using C = Cfg<WM, WN, FP8>;
  return cudaFuncSetAttribute(split_kv_kernel<WM, WN, FP8>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
}

}  // namespace

cudaError_t launch_split_kv(const HostPlan &hp, const RunArgs &a, cudaStream_t stream) {
  if (hp.num_ctas == 0) return cudaSuccess;
  const bool fp8 = hp.prob.kv_dtype == ATTN_KV_FP8_E4M3;
  switch (hp.shape) {
    case Shape::kRows16:
      return fp8 ? launch_one<1, 4, true>(hp, a, stream) : launch_one<1, 4, false>(hp, a, stream);
    case Shape::kRows64:
      return fp8 ? launch_one<4, 1, true>(hp, a, stream) : launch_one<4, 1, false>(hp, a, stream);
    case Shape::kRows128:
      if (hp.use_tc) return launch_prefill_tc(hp, a, stream);
      return fp8 ? launch_one<8, 1, true>(hp, a, stream) : launch_one<8, 1, false>(hp, a, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prepare_kernels(const HostPlan &hp) {
  const bool fp8 = hp.prob.kv_dtype == ATTN_KV_FP8_E4M3;
  switch (hp.shape) {
    case Shape::kRows16:
      return fp8 ? prepare_one<1, 4, true>() : prepare_one<1, 4, false>();
    case Shape::kRows64:
      return fp8 ? prepare_one<4, 1, true>() : prepare_one<4, 1, false>();
    case Shape::kRows128:
      if (hp.use_tc) return prepare_prefill_tc(hp);
      return fp8 ? prepare_one<8, 1, true>() : prepare_one<8, 1, false>();
  }
  return cudaErrorInvalidValue;
}

}  // namespace akp
