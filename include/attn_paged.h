/*
 * attn_paged.h - C ABI of the GB300 (sm_103a) paged-attention library for
 * models whose query/key head dim (192) differs from the value head dim (128).
 *
 * The operation (no page states a formula; this is the plainest reading of
 * what the pages name, and the design notes list every reading):
 *   For request b with n_b new tokens (qo_indptr[b+1] - qo_indptr[b]) and
 *   L_b = seq_lens[b] keys in the cache (the n_b new tokens included, as the
 *   last n_b keys), query token t in [0, n_b) and query head h:
 *     g  = h / (Hq / Hkv)          (GQA: consecutive q heads share KV head g)
 *     i  = L_b - n_b + t           (causal position of the token)
 *     visible keys j: 0 <= j <= i and, when window > 0, j > i - window
 *     k_j = K[page_table[b][j / P], j % P, g, :] * k_scale
 *     v_j = V[page_table[b][j / P], j % P, g, :] * v_scale
 *     s_j = softmax_scale * <q, k_j>
 *     out = sum_j e^{s_j - m} v_j / (sum_j e^{s_j - m} + e^{sinks[h] - m}),
 *     m = max(max_j s_j, sinks[h]); without sinks the sink term is absent.
 *     lse = m + ln(denominator)  (natural log)
 *
 * Where the operation comes from:
 *   - separate K and V caches of different row widths (192 vs 128): sglang
 *     PR #32818, "Route asymmetric-KV models to fa4 on SM100" (the
 *     trtllm_mha key_cache/value_cache size check, and has_asymmetric_kv);
 *   - paged KV with page size 1 or 128, CUDA-graph replay: sglang PR #41886,
 *     "Speed Tests and Profiling" and "Accuracy Tests";
 *   - decode, 8-token verify, full vs sliding window with sinks, ragged page
 *     boundaries: sglang PR #41886, "Accuracy Tests";
 *   - split-KV kept on for multi-token verify, one program per whole verify,
 *     FP8 E4M3 K/V converted in the load path, Q.K kept in 16-bit: the
 *     MiMo-V2.6-Flash-RL 2x RTX PRO 6000 model card, "What the kernels do"
 *     and "Things that were measured and did not help";
 *   - unused KV tails may hold NaN and must be masked, not multiplied:
 *     sammysun0711/sglang PR #35, "Modifications" (FlyPA V-tail masking).
 *
 * Conventions shared by every call:
 *   - All pointers named *_host are host memory; all others are device memory
 *     of the plan's device.  The caller owns every buffer it passes.
 *   - Functions return a status and never abort the process.
 *   - attn_run_paged never allocates, never synchronises and issues work only
 *     on the given stream, so it can be captured in a CUDA graph.
 */
#ifndef ATTN_PAGED_H
#define ATTN_PAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = -1,  /* a NULL pointer, inconsistent sizes, or a run
                                   argument that does not match the plan */
    ATTN_ERR_UNSUPPORTED = -2,  /* head dims other than 192/128 or 128/128, Hq % Hkv != 0 */
    ATTN_ERR_WORKSPACE = -3,    /* workspace smaller than attn_plan reported */
    ATTN_ERR_CUDA = -4          /* a CUDA runtime error (allocation in attn_plan,
                                   or a launch error in attn_run_paged) */
} attn_status_t;

typedef enum {
    ATTN_KV_BF16 = 0,      /* K/V elements are bfloat16 */
    ATTN_KV_FP8_E4M3 = 1   /* K/V elements are OCP FP8 E4M3 codes; value =
                              decoded code * k_scale (resp. v_scale) */
} attn_kv_dtype_t;

typedef struct attn_plan_s *attn_plan_t;

/*
 * Problem description, copied by attn_plan (the caller may free the host
 * arrays afterwards).
 *   batch               B >= 0 requests.
 *   num_q_heads         Hq; num_kv_heads Hkv; Hq % Hkv == 0.
 *   head_dim_qk         192 (the asymmetric pair 192/128), or 128 for a layer
 *                       whose own pair is symmetric (128/128): a model is
 *                       asymmetric when head_dim != v_head_dim or
 *                       swa_head_dim != swa_v_head_dim (sglang PR #32818,
 *                       "Three changes", item 1), so its sliding-window layers
 *                       may carry a pair of their own.  head_dim_v must be 128.
 *                       128/128 plans never use the 256-row prefill kernel.
 *   page_size           P >= 1 tokens per page.
 *   num_pages           pages in each of the K and V pools.
 *   page_table_stride   int32 entries per request row of the page table; must
 *                       be >= ceil(seq_lens[b] / P) for every b.
 *   kv_dtype            element type of both caches.
 *   window              <= 0: full causal attention; > 0: the query at
 *                       position i sees keys j with i - window < j <= i
 *                       (window keys, itself included).
 *   has_sinks           nonzero: attn_run_paged takes a per-head sink logit.
 *   qo_indptr_host      [B+1] int32, qo_indptr[0] = 0, non-decreasing.
 *   seq_lens_host       [B] int32, seq_lens[b] >= qo_indptr[b+1]-qo_indptr[b].
 */
typedef struct {
    int32_t batch, num_q_heads, num_kv_heads;
    int32_t head_dim_qk, head_dim_v;
    int32_t page_size, num_pages, page_table_stride;
    attn_kv_dtype_t kv_dtype;
    int32_t window;
    int32_t has_sinks;
    const int32_t *qo_indptr_host;
    const int32_t *seq_lens_host;
} attn_problem_t;

/*
 * Build a plan for one batch shape on CUDA device `device`.
 * Splits every (request, KV head) key range into work segments sized for the
 * device's SM count, uploads the work list to device memory owned by the plan,
 * and reports the workspace size attn_run_paged needs (may be 0).
 * Synchronous; allocates device memory.  Errors: INVALID_ARG (NULL pointers,
 * inconsistent lengths), UNSUPPORTED (head dims), CUDA (device errors).
 * On error *plan is set to NULL.
 */
attn_status_t attn_plan(const attn_problem_t *problem, int device, attn_plan_t *plan,
                        size_t *workspace_bytes);

/*
 * Build a replayable plan: one whose request lengths are read on the device
 * at every run, so that a CUDA graph captured once keeps serving a batch while
 * its requests grow (the decode and verify paths run under CUDA graph replay
 * in sglang PR #41886, "Accuracy Tests").
 *   bounds->qo_indptr_host   the batch's query layout, fixed for the plan's
 *                            lifetime (the device qo_indptr must equal it).
 *   bounds->seq_lens_host    per-request upper bounds of the lengths;
 *                            page_table_stride must cover them.
 * Other fields as for attn_plan.  Each run first launches a one-CTA planner
 * kernel that reads the caller's device seq_lens and rewrites the plan's work
 * list in device memory (key ranges, equal shares of the key tiles for one CTA
 * per SM, each block also counting 4 tiles on shares of 32 tiles or more,
 * splits, partial offsets); the attention kernel and the merge follow
 * on the same stream.  The workspace reported covers every length vector
 * within the bounds.  Results equal those of a plan built for the run's
 * lengths, up to the floating-point order of the split merge.
 * Synchronous; allocates device memory.  Errors as for attn_plan.
 */
attn_status_t attn_plan_replayable(const attn_problem_t *bounds, int device, attn_plan_t *plan,
                                   size_t *workspace_bytes);

/*
 * Run the planned attention on `stream`.
 *   q            bf16 [total_q, Hq, Dqk], row-major, contiguous (Dqk = the
 *                plan's head_dim_qk: 192 or 128).
 *   k_cache      [num_pages, P, Hkv, Dqk] of bf16 or E4M3 bytes.
 *   v_cache      [num_pages, P, Hkv, 128] of the same type.
 *   page_table   int32 [B, page_table_stride]; entries at or beyond
 *                ceil(seq_lens[b] / P) are never read, and with a window
 *                neither are the entries below floor(lo_b / P), where
 *                lo_b = max(0, seq_lens[b] - n_b - window + 1) is the first key
 *                request b's first query sees: a cache that evicts pages
 *                behind the window may leave anything there (-1 included).
 *                Page ids outside [0, num_pages) that are read are not
 *                dereferenced: the rows they would supply are read as zero
 *                and the plan's device error word records the fault
 *                (attn_get_device_error).
 *   seq_lens     int32 [B] device copy; qo_indptr int32 [B+1] device copy.
 *                Both must equal the host arrays the plan was built from: the
 *                kernels take lengths from the plan's own device copy.  For a
 *                replayable plan seq_lens is read at every run instead, and
 *                may hold any n_b <= seq_lens[b] <= bound_b; a length outside
 *                that range is clamped into it and sets bit 2 of the device
 *                error word.
 *   sinks        fp32 [Hq] sink logits in the units of the scaled scores, or
 *                NULL; must be non-NULL exactly when the plan has_sinks.
 *   window       must equal the plan's window.
 *   softmax_scale, k_scale, v_scale  as in the operation above (the kv scales
 *                are ignored for bf16 caches and should be 1).  All finite;
 *                softmax_scale > 0, and k_scale > 0 for an FP8 cache.
 *   out          bf16 [total_q, Hq, 128].
 *   lse_out      fp32 [total_q, Hq] natural-log denominators, or NULL.
 *   workspace    device scratch of at least workspace_bytes (may be NULL when
 *                the plan reported 0).  Its contents need no initialisation.
 * Slots of the caches that no query can see are never read, so they may hold
 * anything (NaN included).  Queries keep their full bf16 range for either
 * cache type.  Plans whose row blocks hold at most 128 rows (decode, verify)
 * widen E4M3 elements exactly to bf16 and form every product as bf16 x bf16
 * with fp32 accumulation.  Plans with larger blocks (chunked prefill) run
 * Q.K^T on an FP8 cache in fp16: each query row is multiplied by the power of
 * two that puts its largest |q| in [2^14, 2^15) (exact; every element down to
 * 2^-31 of that maximum stays exact in fp16), E4M3 is widened exactly to
 * fp16, and the scores are divided by the same power of two in fp32; P.V
 * is fp16 x fp16 with fp32 accumulation.  The E4M3 NaN codes (0x7F, 0xFF) in
 * a visible slot read as +-480 on the decode/verify plans and stay NaN on the
 * prefill plans.
 * Prefill plans that are not replayable first gather the keys their blocks
 * read into a staging scratch in the workspace (16-bit rows: E4M3 widened
 * exactly to fp16, BF16 copied; (Dqk + 128) * 2 bytes per key of each KV
 * head, over whole 128-key tiles), which the prefill kernel loads as TMA
 * tiles; attn_plan's workspace size includes it.
 * Runs of one plan must be ordered on one stream (they share the plan's
 * device error word); different plans are independent.
 * Errors: INVALID_ARG, WORKSPACE, CUDA (launch errors; nothing is waited for).
 */
attn_status_t attn_run_paged(attn_plan_t plan, const void *q, const void *k_cache,
                             const void *v_cache, const int32_t *page_table,
                             const int32_t *seq_lens, const int32_t *qo_indptr,
                             const float *sinks, int32_t window, float softmax_scale,
                             float k_scale, float v_scale, void *out, float *lse_out,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * The two launches attn_run_paged makes, one at a time, for callers that time
 * or interleave them: phase 0 is the split-KV attention kernel, phase 1 the
 * log-sum-exp merge of split partials (nothing is launched when the plan has
 * no block split over several CTAs).  Arguments, validation and errors are
 * those of attn_run_paged; phase 0 then phase 1 on one stream is exactly
 * attn_run_paged.  Other phase values: INVALID_ARG.
 */
attn_status_t attn_run_phase(attn_plan_t plan, int32_t phase, const void *q,
                             const void *k_cache, const void *v_cache,
                             const int32_t *page_table, const int32_t *seq_lens,
                             const int32_t *qo_indptr, const float *sinks, int32_t window,
                             float softmax_scale, float k_scale, float v_scale, void *out,
                             float *lse_out, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * Write the new tokens' K and V rows into the paged caches — the step that
 * precedes attention on every mode.  For request b and its new token t
 * (qo_indptr[b] <= tok = qo_indptr[b] + t < qo_indptr[b+1]) the position is
 * i = seq_lens[b] - n_b + t (the new tokens are the last n_b keys, as for
 * attn_run_paged), stored at page page_table[b][i / P], offset i % P, for
 * every KV head g:
 *   BF16 caches: k_cache[page][i % P][g][:] = k_new[tok][g][:] bit for bit;
 *   FP8 caches:  k_cache[...] = E4M3(k_new[tok][g][:] / k_scale), the
 *                division in fp32 (IEEE, round to nearest even) and the E4M3
 *                rounding to nearest even with saturation to +-448, which is
 *                how an FP8 E4M3 KV cache with a per-tensor scale stores its
 *                entries (model card MiMo-V2.6-Flash-RL-FP8KV-W4A8-2x-RTX-PRO-
 *                6000, "What the kernels do"); V likewise with v_scale.
 *   k_new, v_new bf16 [total_q][Hkv][Dqk] and [total_q][Hkv][128], contiguous.
 *   k_cache, v_cache, page_table, seq_lens, qo_indptr: as for attn_run_paged
 *                (device copies equal to the plan's host arrays).
 *   k_scale, v_scale  finite and > 0 for FP8 caches; ignored for BF16.
 * Only the written slots change.  A page id outside [0, num_pages) is not
 * dereferenced: that token's rows are skipped and the plan's device error
 * word records it (bit 0).  With a replayable plan seq_lens may change between
 * runs; a position outside the request's page-table row is skipped and sets
 * bit 2.  Runs on `stream`; no allocation, no synchronisation.
 * Errors: INVALID_ARG, CUDA.
 */
attn_status_t attn_append_kv(attn_plan_t plan, const void *k_new, const void *v_new,
                             void *k_cache, void *v_cache, const int32_t *page_table,
                             const int32_t *seq_lens, const int32_t *qo_indptr, float k_scale,
                             float v_scale, void *stream);

/*
 * Size of the library-owned scratch used by attn_run_paged_no_workspace.
 */
#define ATTN_NO_WORKSPACE_MAX_BYTES (16u * 1024u * 1024u)

/*
 * attn_run_paged for callers that cannot allocate device memory.
 *
 * The paper has no counterpart: this entry point exists for integration.
 * Some callers have no way to obtain the workspace attn_run_paged asks for:
 * plugins that a host framework hands tensor pointers but no allocator (the
 * framework owns every device byte through its own memory pool), and serving
 * loops that forbid cudaMalloc on the hot path, where it can synchronise the
 * device and take unbounded time.  This call takes the same arguments as
 * attn_run_paged minus the workspace and uses instead one scratch array of
 * ATTN_NO_WORKSPACE_MAX_BYTES bytes in device global memory that the library
 * owns: every GPU that loads the library holds that array until the process
 * exits.  Nothing is allocated, here or later.
 *   - The first call on a device looks up the array's device address on that
 *     device (a host-side query, no allocation); make that first call before
 *     any stream capture.  The address is kept for the life of the process
 *     and is stale after cudaDeviceReset (as are plans made before it).
 *   - Plans whose split partials exceed ATTN_NO_WORKSPACE_MAX_BYTES are
 *     rejected with ATTN_ERR_WORKSPACE before anything is launched.  A
 *     prefill plan's K/V staging scratch is not used: its prefill kernel
 *     reads the paged caches itself (same results).
 *   - All calls share the one array, and it keeps whatever the last call left
 *     in it; nothing in it needs to start at zero, because each call writes
 *     every partial it later reads.  Calls whose kernels overlap on the GPU
 *     (different streams, or different threads without ordering) race on the
 *     array and give wrong results: order them on one stream.
 * Other arguments, validation and errors are those of attn_run_paged.
 */
attn_status_t attn_run_paged_no_workspace(attn_plan_t plan, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *page_table,
                                          const int32_t *seq_lens, const int32_t *qo_indptr,
                                          const float *sinks, int32_t window,
                                          float softmax_scale, float k_scale, float v_scale,
                                          void *out, float *lse_out, void *stream);

/* Free a plan and its device memory (synchronises the plan's device).
 * NULL is accepted. */
attn_status_t attn_plan_destroy(attn_plan_t plan);

/*
 * Read and clear the plan's device error word (synchronous).  Bit 0: a page
 * id outside [0, num_pages) was met.  Bit 1: a pipeline wait of the attention
 * kernel gave up after its time limit (the affected rows are not valid).
 * Bit 2: a run length outside a replayable plan's bounds (clamped), or an
 * appended position outside its page-table row (skipped).  The workspace
 * argument is unused and may be NULL.
 */
attn_status_t attn_get_device_error(attn_plan_t plan, void *workspace, int32_t *err);

/* Static text for a status code. */
const char *attn_status_string(attn_status_t status);

/*
 * Host-side inspection of the schedule, for tests and tools (no GPU needed).
 *
 * attn_plan_host builds a plan on the host only, for a device with `num_sms`
 * SMs; it cannot be run.  attn_plan_info reports its shape:
 *   info[0] = number of row blocks, info[1] = number of work segments,
 *   info[2] = number of CTAs, info[3] = rows per block (64 or 128),
 *   info[4] = key tile (keys per tile), info[5] = multi-split blocks,
 *   info[6] = workspace bytes (low 31 bits in info[6], high bits in info[7]).
 * attn_plan_blocks copies the blocks as 8 int32 each:
 *   {b, g, row0, nrows, key_lo, key_hi, num_splits, part_row_base}
 * and attn_plan_segments copies the segments as 5 int32 each:
 *   {cta, block, tile_begin, tile_end, split}
 * where tiles are absolute (tile T holds keys [T*tile, (T+1)*tile)).
 * The destination arrays must hold info[0]*8 (resp. info[1]*5) int32.
 *
 * attn_plan_replayable_host is attn_plan_replayable on the host only (the
 * work list is that of the bounds).  attn_plan_replan_host rebuilds a
 * replayable plan's host copy of the work list for the lengths
 * seq_lens_host[B] with the device planner's arithmetic, and stores in *err
 * the error bits the device would set (4: a length clamped into its bounds).
 * attn_plan_fetch_device synchronises the plan's device and copies the work
 * list the device planner last wrote into the host copy (replayable plans
 * built by attn_plan_replayable).  All three: INVALID_ARG for other plans;
 * attn_plan_fetch_device also CUDA.
 */
attn_status_t attn_plan_host(const attn_problem_t *problem, int32_t num_sms, attn_plan_t *plan);
attn_status_t attn_plan_info(attn_plan_t plan, int32_t info[8]);
attn_status_t attn_plan_blocks(attn_plan_t plan, int32_t *blocks_host);
attn_status_t attn_plan_segments(attn_plan_t plan, int32_t *segments_host);
/*
 * attn_plan_cta_heads copies each CTA's head record, the first thing a CTA of
 * the attention kernels reads, as 20 int32 per CTA (info[2] CTAs):
 *   {seg_begin, seg_end, key tiles in all its segments, 0,
 *    its first segment {block, tile_begin, tile_end, split},
 *    that segment's block {b, g, row0, nrows, L, n, tok0, key_lo, key_hi,
 *    num_splits, part_row_base, srow}}
 * (zeros after the range for a CTA without segments), where srow places the
 * block's keys in the staging scratch (key j of its (b, g) is scratch row
 * srow + j; 0 for plans without one).  Errors: INVALID_ARG.
 */
attn_status_t attn_plan_cta_heads(attn_plan_t plan, int32_t *heads_host);
/*
 * attn_plan_stage_units reports a prefill plan's staging units, one per
 * (request, KV head) with prefill blocks: *count units (0 for plans without a
 * staging scratch) and, when units_host is not NULL, 8 int32 per unit:
 *   {b, g, j0, key_lo, key_hi, tiles, row_base, tile_off}
 * Keys [j0, j0 + 128 * tiles) (j0 a multiple of 128) occupy scratch rows
 * [row_base, row_base + 128 * tiles); keys outside [key_lo, key_hi), the
 * union of the unit's blocks' key ranges, are staged as zeros; tile_off is
 * the unit's first tile among all units'.  Errors: INVALID_ARG.
 */
attn_status_t attn_plan_stage_units(attn_plan_t plan, int32_t *count, int32_t *units_host);
/*
 * attn_plan_merge_ctas reports in *ctas how many CTAs the merge kernel of a
 * run launches (0: the run launches no merge kernel): one per 8 rows of every
 * multi-split block (of every block for a replayable plan, whose splits are
 * only known on the device).  Errors: INVALID_ARG.
 */
attn_status_t attn_plan_merge_ctas(attn_plan_t plan, int32_t *ctas);
attn_status_t attn_plan_replayable_host(const attn_problem_t *bounds, int32_t num_sms,
                                        attn_plan_t *plan);
attn_status_t attn_plan_replan_host(attn_plan_t plan, const int32_t *seq_lens_host,
                                    int32_t *err);
attn_status_t attn_plan_fetch_device(attn_plan_t plan);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_PAGED_H */
