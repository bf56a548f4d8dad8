/*
 * attn_paged_debug.h - test entry points of libattn_paged.so.
 *
 * Not needed to run attention; they expose building blocks of the kernels so
 * that tests can check them in isolation.  Same status codes as attn_paged.h.
 */
#ifndef ATTN_PAGED_DEBUG_H
#define ATTN_PAGED_DEBUG_H

#include "attn_paged.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One tensor-core product on one CTA with the shared-memory layouts of the
 * tensor-core attention kernel (128-byte swizzled operands, accumulator in
 * tensor memory, fp32 result):
 *   mode 0: d[128 x n] = a[128 x 192] * b[n x 192]^T, n in {64, 128}
 *           (both operands K-major, as Q and K in Q.K^T);
 *   mode 1: d[128 x 128] = a[128 x 64] * b[64 x 128]
 *           (b stored row-major, i.e. MN-major, as V in P.V); variant 0/1
 *           picks which descriptor offset spans the two 64-wide column blocks
 *           of b (0: leading offset, 1: stride offset);
 *   mode 2: the M=64 form: a[64 x 192] * b[64 x 192]^T; d receives all 128
 *           TMEM lanes x 64 columns as d[128 x 64], so the test can check
 *           which lanes hold the 64 rows (unused lanes hold whatever TMEM had);
 *   mode 3: d[128 x 128] = a[128 x 64] * b[64 x 128] with a read from tensor
 *           memory (row r written by thread r into its lane, two elements per
 *           32-bit column, element 2j in the low half), b MN-major as in
 *           mode 1 variant 0 (the P.V form with P kept in TMEM);
 *   mode 4: mode 3 with M = 64: a[64 x 64], row r written into lane
 *           32*(r/16) + r%16; d receives all 128 lanes x 128 columns;
 *   mode 5: the product of mode 2, then read back with the 16-lane shapes:
 *           d[0 : 4096] = each thread's 32 registers of a 16x256b.x8 load
 *           (index (warp*32 + thread)*32 + register); then every thread
 *           stores the values warp*100000 + thread*100 + j (j < 16) with a
 *           16x128b.x8 store at column 64, and d[4096 : 6144] receives a
 *           32x32b load of those 16 columns (index (warp*32 + lane)*16 + col)
 *           as floats.  d must hold 6144 floats;
 *   mode 6: the product of mode 2, then read back with the two-half shapes:
 *           d[0 : 4096] = each thread's 32 registers of a 16x32bx2.x32 load
 *           with the halves 32 columns apart; then every thread stores
 *           warp*100000 + thread*100 + j (j < 16) with a 16x32bx2.x16 store at
 *           column 64, halves 16 apart, and d[4096 : 8192] receives a 32x32b
 *           load of columns 64-95 (index (warp*32 + lane)*32 + col) as
 *           floats.  d must hold 8192 floats.
 * a, b: device 16-bit matrices, row-major (ab_type 0 = fp16, 1 = bf16);
 * d: device fp32, row-major; status: device int32, set to 1 if the
 * completion wait timed out (left untouched otherwise).  Asynchronous on
 * `stream`.  Errors: INVALID_ARG, CUDA.
 */
attn_status_t attn_debug_tc_gemm(int32_t mode, int32_t variant, int32_t ab_type, int32_t n,
                                 const void *a, const void *b, float *d, int32_t *status,
                                 void *stream);

/*
 * Start-up and epilogue timestamps of the split-KV attention kernel, recorded
 * only by a profiling build of the library (compiled with AKP_STAMPS; the
 * default build returns ATTN_ERR_UNSUPPORTED and records nothing).  Each CTA
 * with index below ATTN_DEBUG_STAMP_CTAS writes, on every launch, the GPU's
 * global timer (ns) at fixed points of its run into row `cta` of a
 * [ATTN_DEBUG_STAMP_CTAS][ATTN_DEBUG_STAMP_EVENTS] array of uint64:
 *   0 first instruction, 1 head record read, 2 barriers and TMEM ready,
 *   3 first tile's K/V requested, 4 first Q block staged, 5 first Q.K^T
 *   issued, 6 first S tile ready, 7 last P.V issued, 8 / 9 begin / end of the
 *   last segment's epilogue, 10 all roles done;
 *   11 and 12 are counts, not times: the CTA's segments and key tiles;
 *   13 first tile's page-table entries read (page sizes TMA can tile);
 *   14 a value: the index of the SM the CTA ran on.
 * Entries a launch does not reach keep their previous value (0 after a clear).
 * attn_debug_stamps synchronises the current device, copies the array into
 * `host` (ATTN_DEBUG_STAMP_CTAS * ATTN_DEBUG_STAMP_EVENTS values, caller-owned)
 * and, if `clear` is nonzero, zeroes it on the device.
 * Errors: UNSUPPORTED (default build), INVALID_ARG (host NULL), CUDA.
 */
#define ATTN_DEBUG_STAMP_CTAS 160
#define ATTN_DEBUG_STAMP_EVENTS 16
attn_status_t attn_debug_stamps(uint64_t *host, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_PAGED_DEBUG_H */
