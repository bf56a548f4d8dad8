// Self-test of the tcgen05 building blocks used by the tensor-core attention
// kernel: 128-byte swizzled K-major and MN-major shared-memory operands,
// instruction descriptors, TMEM allocation, commit-to-mbarrier and tcgen05.ld.
// One CTA of 128 threads computes one small product and writes it in fp32.
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_paged_debug.h"
#include "tc_common.cuh"

namespace akp {
namespace {

constexpr int kThreads = 128;
constexpr int kSmemBytes = 161 * 1024;   // 160 KB used, +1 KB for 1024-byte alignment

// Copy a row-major 16-bit matrix [rows x cols] (cols a multiple of 64) into
// 128-byte swizzled column blocks of 64 elements: block c holds columns
// [64c, 64c+64) of every row, rows 128 bytes apart.
__device__ void stage_sw128(uint8_t *dst, const uint16_t *src, int rows, int cols) {
  const int chunks_per_row = cols / 8;
  for (int idx = threadIdx.x; idx < rows * chunks_per_row; idx += kThreads) {
    const int r = idx / chunks_per_row;
    const int ch = idx % chunks_per_row;
    const uint4 v = *reinterpret_cast<const uint4 *>(src + (size_t)r * cols + ch * 8);
    uint8_t *blk = dst + (ch / 8) * rows * 128;
    *reinterpret_cast<uint4 *>(blk + tc::sw128_offset(r, ch % 8)) = v;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(int mode, int variant, int ab_type, int n, const uint16_t *a,
                   const uint16_t *b, float *d, int32_t *status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte swizzle atoms must start on 1024-byte boundaries
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  uint8_t *sa = smem;               // A operand blocks
  uint8_t *sb = smem + 64 * 1024;   // B operand blocks
  const int warp = threadIdx.x / 32;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 512);

  if (mode == 0) {
    stage_sw128(sa, a, 128, 192);   // [128 x 192] K-major
    stage_sw128(sb, b, n, 192);     // [n x 192] K-major
  } else if (mode == 2 || mode == 5 || mode == 6) {
    stage_sw128(sa, a, 64, 192);    // [64 x 192] K-major
    stage_sw128(sb, b, 64, 192);    // [64 x 192] K-major
  } else if (mode == 1) {
    stage_sw128(sa, a, 128, 64);    // [128 x 64] K-major
    stage_sw128(sb, b, 64, 128);    // [64 keys x 128] stored key-major: MN-major B
  } else {
    stage_sw128(sb, b, 64, 128);    // modes 3/4: only V in shared memory
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int M = (mode == 2 || mode == 4 || mode == 5 || mode == 6) ? 64 : 128;
  if (mode == 3 || mode == 4) {
    // A = P [M x 64] into TMEM columns 256..287, each thread its own row's
    // lane (M = 64: rows 16w..16w+15 in lanes 0-15 of warp w's quadrant)
    const int lane = threadIdx.x & 31;
    const int row = M == 128 ? (int)threadIdx.x : (lane < 16 ? warp * 16 + lane : -1);
    uint32_t r[32];
    for (int j = 0; j < 32; ++j)
      r[j] = row >= 0 ? *reinterpret_cast<const uint32_t *>(a + (size_t)row * 64 + 2 * j) : 0u;
    tc::tmem_st32(tmem + ((uint32_t)(warp * 32) << 16) + 256, r);
    tc::tmem_wait_st();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
  }

  if (threadIdx.x == 0) {
    const uint32_t a0 = tc::smem_u32(sa);
    const uint32_t b0 = tc::smem_u32(sb);
    if (mode == 0) {
      const uint32_t idesc = tc::idesc_f16(ab_type, 0, 0, 128, n);
      for (int ks = 0; ks < 12; ++ks) {
        const uint32_t koff = (ks / 4) * 0u + (ks % 4) * 32u;
        const uint64_t ad = tc::smem_desc_sw128(a0 + (ks / 4) * 128 * 128 + koff, 16, 1024);
        const uint64_t bd = tc::smem_desc_sw128(b0 + (ks / 4) * n * 128 + koff, 16, 1024);
        tc::mma_f16_ss(tmem, ad, bd, idesc, ks > 0);
      }
    } else if (mode == 2 || mode == 5 || mode == 6) {
      const uint32_t idesc = tc::idesc_f16(ab_type, 0, 0, 64, 64);
      for (int ks = 0; ks < 12; ++ks) {
        const uint32_t koff = (ks % 4) * 32u;
        const uint64_t ad = tc::smem_desc_sw128(a0 + (ks / 4) * 64 * 128 + koff, 16, 1024);
        const uint64_t bd = tc::smem_desc_sw128(b0 + (ks / 4) * 64 * 128 + koff, 16, 1024);
        tc::mma_f16_ss(tmem, ad, bd, idesc, ks > 0);
      }
    } else if (mode >= 3) {
      const uint32_t idesc = tc::idesc_f16(ab_type, 0, 1, M, 128);
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bd = tc::smem_desc_sw128(b0 + kk * 16 * 128, 64 * 128, 1024);
        tc::mma_f16_ts(tmem, tmem + 256 + kk * 8, bd, idesc, kk > 0);
      }
    } else {
      const uint32_t idesc = tc::idesc_f16(ab_type, 0, 1, 128, 128);
      const uint32_t lbo = variant == 0 ? 64 * 128 : 1024;   // between 64-wide N blocks
      const uint32_t sbo = variant == 0 ? 1024 : 64 * 128;   // between 8-key groups
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = tc::smem_desc_sw128(a0 + kk * 32, 16, 1024);
        const uint64_t bd = tc::smem_desc_sw128(b0 + kk * 16 * 128, lbo, sbo);
        tc::mma_f16_ss(tmem, ad, bd, idesc, kk > 0);
      }
    }
    tc::mma_commit(&bar);
  }
  const bool ok = tc::mbar_wait(&bar, 0, &abort_flag);
  tc::tc_fence_after();
  const int ncols = mode == 0 ? n : (mode == 2 ? 64 : 128);
  (void)M;
  if (ok && mode == 6) {
    // the two-half 16-lane shapes: a 16x32bx2.x32 load with the halves 32
    // columns apart, dumped as d[warp][thread][register]; then a 16x32bx2.x16
    // store at column 64 with the halves 16 columns apart, and a 32x32b load
    // of columns 64-95 into d[4*32*32 + (warp*32 + lane)*32 + column]
    const int t = threadIdx.x & 31;
    uint32_t r[32];
    tc::tmem_ld_16x32bx2_x32<32>(tmem + ((uint32_t)(warp * 32) << 16), r);
    tc::tmem_wait_ld();
    for (int j = 0; j < 32; ++j) d[(warp * 32 + t) * 32 + j] = __uint_as_float(r[j]);
    uint32_t w16[16];
    for (int j = 0; j < 16; ++j) w16[j] = (uint32_t)(warp * 100000 + t * 100 + j);
    tc::tmem_st_16x32bx2_x16<16>(tmem + ((uint32_t)(warp * 32) << 16) + 64, w16);
    tc::tmem_wait_st();
    uint32_t q[32];
    tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 64, q);
    tc::tmem_wait_ld();
    for (int j = 0; j < 32; ++j) d[4 * 32 * 32 + (warp * 32 + t) * 32 + j] = (float)q[j];
  } else if (ok && mode == 5) {
    // the 16-lane shapes: every thread's 32 registers of a 16x256b.x8 load of
    // its warp's lanes 0-15, dumped as d[warp][thread][register]; then the
    // 16x128b.x8 store writes register pairs back (column 64 + ...) and a
    // 32x32b load of those columns lands in d[4*32*32 + lane*16 + column]
    const int t = threadIdx.x & 31;
    uint32_t r[32];
    tc::tmem_ld_16x256b_x8(tmem + ((uint32_t)(warp * 32) << 16), r);
    tc::tmem_wait_ld();
    for (int j = 0; j < 32; ++j) d[(warp * 32 + t) * 32 + j] = __uint_as_float(r[j]);
    uint32_t w16[16];
    for (int j = 0; j < 16; ++j) w16[j] = (uint32_t)(warp * 100000 + t * 100 + j);
    tc::tmem_st_16x128b_x8(tmem + ((uint32_t)(warp * 32) << 16) + 64, w16);
    tc::tmem_wait_st();
    uint32_t q[16];
    tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 64, q);
    tc::tmem_wait_ld();
    for (int j = 0; j < 16; ++j) d[4 * 32 * 32 + (warp * 32 + t) * 16 + j] = (float)q[j];
  } else if (ok) {
    const int row = threadIdx.x;   // TMEM lane = row; warp w owns lanes 32w..32w+31
    for (int c0 = 0; c0 < ncols; c0 += 32) {
      uint32_t r[32];
      tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, r);
      tc::tmem_wait_ld();
      for (int j = 0; j < 32; ++j) d[row * ncols + c0 + j] = __uint_as_float(r[j]);
    }
  } else if (threadIdx.x == 0) {
    *status = 1;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

}  // namespace
}  // namespace akp

extern "C" attn_status_t attn_debug_tc_gemm(int32_t mode, int32_t variant, int32_t ab_type,
                                            int32_t n, const void *a, const void *b, float *d,
                                            int32_t *status, void *stream) {
  if (mode < 0 || mode > 6) return ATTN_ERR_INVALID_ARG;
  if (mode == 0 && n != 64 && n != 128) return ATTN_ERR_INVALID_ARG;
  if (variant != 0 && variant != 1) return ATTN_ERR_INVALID_ARG;
  if (ab_type != 0 && ab_type != 1) return ATTN_ERR_INVALID_ARG;
  if (!a || !b || !d || !status) return ATTN_ERR_INVALID_ARG;
  if (cudaFuncSetAttribute(akp::tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           akp::kSmemBytes) != cudaSuccess)
    return ATTN_ERR_CUDA;
  akp::tc_gemm_kernel<<<1, akp::kThreads, akp::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(
      mode, variant, ab_type, n, static_cast<const uint16_t *>(a),
      static_cast<const uint16_t *>(b), d, status);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
