/*
 * rk_paged.h -- C ABI of the deterministic paged-KV attention library
 * (librk_paged.so, sm_103a).
 *
 * Operation (both launch calls): batch-invariant causal attention over a
 * block-table page cache with Llama rotate-half RoPE applied in-kernel to the
 * query and to each key as it is read, one fixed ascending-KV reduction per
 * row (no split-KV), FP32 accumulation, one final BF16 round-to-nearest-even
 * write of `out`, and the FP32 attention-domain LSE.
 *   - "WS2 PR7 Fused Attention Backend Alignment", section "Current
 *     Implementation" (validate page table / positions, then run; restore
 *     out -> [B, Hq, Sq, D], lse -> [B, Hq, Sq]);
 *   - same page, "FlashInfer RoPE Fusion" (pre-RoPE Q and K cache, ROPE_LLAMA,
 *     theta 1e6, scale 1.0, rotary_dim = head_dim, rotate-half);
 *   - same page, "Split-KV Policy" (policy `disabled`) and "P2P NCCL reference
 *     and strict arithmetic provenance" (FP32 accumulation, FP32 LSE,
 *     downcast only at the final output write);
 *   - "Add FlashInfer RoPE-fused paged attention scaffold", boundary table
 *     (num_splits = 1, GQA packing from the head layout, FP32 LSE);
 *   - "flashinfer_fa2 backend for Ada (SM89)", summary and design notes
 *     (BF16, page size 16, head_dim 128, NHD; plan on host metadata, run on
 *     device metadata; no host synchronisation in the run call).
 *
 * Semantics shared by every entry point:
 *   q            bf16 [B, Hq, Sq, D], pre-RoPE, contiguous
 *   k_cache      bf16 [num_pages, page_size, Hkv, D] (NHD), pre-RoPE
 *   v_cache      bf16 [num_pages, page_size, Hkv, D]
 *   block_table  int32 [B, W]: logical page j of row b -> physical page;
 *                entries past ceil(kv_len/page_size) are -1
 *   kv_lens      int32 [B]: tokens of row b in the cache (logical 0..kv_len-1)
 *   position_ids int32 [B, Sq]: position of each query
 *   out          bf16 [B, Hq, Sq, D]
 *   lse          fp32 [B, Hq, Sq]: ln sum_t exp(score_t), scores scaled by
 *                sm_scale = 1/sqrt(D)
 * Key t of row b sits at position t; it is visible to query s iff
 * t <= position_ids[b, s] and t < kv_len[b].  Query head h reads KV head
 * h / (Hq/Hkv).  Angle of rotation pair i at position p:
 * p * theta^(-2i/D) / rope_scale, pairing element i with element i + D/2.
 * A query with no visible key gets out = 0 and lse = -inf.
 *
 * Ownership: the caller owns every buffer and the plan (plain struct).  The
 * library allocates no device memory and keeps no per-call state; launches
 * are asynchronous on the caller's stream, never synchronise and never read
 * device memory on the host, so they can be captured in a CUDA graph and
 * replayed with new metadata contents.
 *
 * Errors: every entry point returns RK_OK (0) or an RK_E_* code and sets a
 * thread-local message readable with rk_last_error().  Nothing falls back to
 * another implementation.
 */
#ifndef RK_PAGED_H
#define RK_PAGED_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RK_PAGED_ABI_VERSION 3u
#define RK_PAGED_MAX_ROPE_PAIRS 64

/* Status codes returned by the entry points. */
enum rk_status {
    RK_OK = 0,
    RK_E_ARG = 1,          /* bad argument: null/misaligned pointer, negative size, plan mismatch */
    RK_E_UNSUPPORTED = 2,  /* D != 128, page_size != 16, Hq % Hkv != 0, Hq/Hkv not in {1,2,4,8} */
    RK_E_PAGE_OOB = 3,     /* an active block-table entry outside [0, num_pages) */
    RK_E_DUP_PAGE = 4,     /* a physical page used twice among the batch's active entries */
    RK_E_PAD = 5,          /* an inactive block-table entry that is not -1 */
    RK_E_KVLEN = 6,        /* kv_len < 0 or kv_len > W * page_size */
    RK_E_POSITION = 7,     /* positions negative, not contiguous ascending, or not trailing */
    RK_E_CUDA = 8,         /* a CUDA runtime/driver call failed (message has the CUDA error) */
    RK_E_DEVICE = 9        /* current device is not a compute capability 10.3 GPU */
};

/* Bits the kernels OR into *status_d when device-side metadata is unsafe.
 * The affected row gets out = 0 and lse = NaN; no kernel ever traps. */
#define RK_STATUS_PAGE_OOB (1 << 0) /* page id read by the kernel outside [0, num_pages) */
#define RK_STATUS_KVLEN (1 << 1)    /* kv_len outside [0, W * page_size] */
#define RK_STATUS_POSITION (1 << 2) /* a negative query position */
#define RK_STATUS_TIMEOUT (1 << 3)  /* an internal pipeline wait gave up (kernel returned early) */
#define RK_STATUS_RANGE (1 << 4)    /* decode, prefill, ragged, backward: a pre-RoPE q or k element the
                                       kernel reads has |x| >= 2^15 (the FP16 score operand limit) */

/* Opaque stream handle; identical to cudaStream_t / CUstream. */
typedef struct CUstream_st *rk_stream_t;

/*
 * Validated launch plan.  Plain data, owned by the caller, filled by
 * rk_paged_plan and read by the launch calls.
 */
typedef struct rk_paged_plan {
    uint32_t abi;         /* RK_PAGED_ABI_VERSION */
    int32_t B, Sq, Hq, Hkv, D, page_size, W, num_pages;
    int32_t causal;       /* always 1 */
    int32_t max_kv_len;   /* largest kv_len seen at plan time (0 for a shape-only plan) */
    float sm_scale;       /* 1 / sqrt(D) */
    int32_t validated;    /* 1 when metadata contents were checked, 0 for a shape-only plan */
    /* Ragged batches: work units of the prefill grid (pairs of q-tiles of
     * the rows with two or more queries), counted by rk_paged_plan_ragged
     * from qo_indptr_h; -1 (rk_paged_plan, or set by the caller) sizes the
     * grid for any contents with this total_q and max_q_len. */
    int32_t pf_units;
    double rope_theta, rope_scale;
    /* Rotation rate of pair i in turns per position as a 0.64 fixed-point
     * fraction: round(2^64 * theta^(-2i/D) / (2 pi rope_scale)), i < D/2. */
    uint64_t rope_turns[RK_PAGED_MAX_ROPE_PAIRS];
    /* Fail-closed waits.  Every pipeline wait inside a kernel gives up once it
     * has waited wait_limit_ns of wall time (past its first 32 probes of the
     * barrier, each of which may sleep up to 20 us); the CTA then waits out
     * the copies it has in flight (those waits keep the 2 s limit), frees its
     * tensor memory, writes its rows as failed (out = 0, lse = NaN; NaN
     * gradients) and sets RK_STATUS_TIMEOUT.  rk_paged_plan sets 2000000000
     * (2 s); the launch calls read 0 as 2 s and clamp other values to
     * [1000, 2000000000]. */
    uint32_t wait_limit_ns;
    /* Test of that exit path, for callers that must see it work on their
     * device: when nonzero, the MMA-issuing warp of every CTA of the
     * tensor-core kernels first waits on a barrier of its CTA that nothing
     * completes, so that wait runs out after wait_limit_ns and every CTA takes
     * the timeout exit above (nothing is computed; the call returns RK_OK and
     * the status word says RK_STATUS_TIMEOUT).  rk_paged_plan sets 0. */
    int32_t timeout_drill;
} rk_paged_plan_t;

/*
 * rk_paged_plan -- validate shapes and host metadata, fill *plan.
 * Follows the validation list of "WS2 PR7 Fused Attention Backend
 * Alignment", section "Current Implementation" (page bounds, logical order,
 * duplicate pages, canonical inactive metadata, trailing query positions).
 *
 *   block_table_h [B, W], kv_lens_h [B], position_ids_h [B, Sq]: HOST memory,
 *   read only during the call.  Pass all three as NULL for a shape-only plan
 *   (contents are then checked only by the kernels' memory-safety checks).
 * Checks, in this order, returning the first failure:
 *   RK_E_ARG         plan NULL, B < 0, Sq < 1, Hq/Hkv < 1, W/num_pages < 0,
 *                    theta <= 1, rope_scale <= 0, only some metadata NULL
 *   RK_E_UNSUPPORTED D != 128, page_size != 16, Hq % Hkv, Hq/Hkv not in {1,2,4,8}
 *   RK_E_KVLEN       kv_len outside [0, W * 16]
 *   RK_E_PAGE_OOB    first ceil(kv_len/16) entries of a row outside [0, num_pages)
 *   RK_E_PAD         any later entry of the row not -1
 *   RK_E_DUP_PAGE    a physical page in two active entries (whole batch)
 *   RK_E_POSITION    a negative position, positions not contiguous ascending,
 *                    kv_len > 0 with last position not in {kv_len-1, kv_len},
 *                    kv_len == 0 with Sq > 1
 * Runs on the host only; needs no GPU.
 */
int rk_paged_plan(rk_paged_plan_t *plan, int32_t B, int32_t Sq, int32_t Hq, int32_t Hkv,
                  int32_t D, int32_t page_size, int32_t num_pages, int32_t W,
                  const int32_t *block_table_h, const int32_t *kv_lens_h,
                  const int32_t *position_ids_h, double rope_theta, double rope_scale);

/*
 * rk_paged_attn_decode -- one query per row (plan->Sq must be 1).
 * Paged decode of "flashinfer_fa2 backend for Ada (SM89)" with split-KV
 * disabled ("Split-KV is disabled" design note), RoPE fused as in
 * "WS2 PR7 ...", "FlashInfer RoPE Fusion".
 *   q [B, Hq, 1, D], out [B, Hq, 1, D], lse [B, Hq, 1]; all other buffers as
 *   in the file header.  Every pointer is DEVICE memory of the current
 *   device; q, k_cache, v_cache, out 16-byte aligned.  status_d: int32 the
 *   kernel ORs RK_STATUS_* bits into (may be NULL); never cleared here.
 * The score MMA takes the rotated q and k as FP16 (FP32 accumulation), so
 * pre-RoPE q / k elements must stay below 2^15 in magnitude: a (row, KV head)
 * whose query heads or visible keys hold a larger value is not computed; its
 * query heads get out = 0, lse = NaN and RK_STATUS_RANGE is set.
 * Returns RK_E_ARG for a null/misaligned pointer or a plan that is not a
 * decode plan, RK_E_DEVICE off sm_103, RK_E_CUDA if the launch fails.
 */
int rk_paged_attn_decode(const rk_paged_plan_t *plan, const void *q, const void *k_cache,
                         const void *v_cache, const int32_t *block_table_d,
                         const int32_t *kv_lens_d, const int32_t *position_ids_d, void *out,
                         float *lse, int32_t *status_d, rk_stream_t stream);

/*
 * rk_paged_attn_prefill -- causal chunked prefill against a paged prefix
 * (any plan->Sq >= 1; queries at position_ids, keys 0..kv_len-1 from the
 * cache, which already holds the chunk's own K/V).
 * Paged prefill of "WS2 PR7 ...", "Current Implementation"
 * (BatchPrefillWithPagedKVCacheWrapper role) with ROPE_LLAMA fused and
 * split-KV disabled.  Buffers, alignment and errors as for decode.
 * The score MMA takes the rotated q and k as FP16 (FP32 accumulation), so
 * pre-RoPE q / k elements must stay below 2^15 in magnitude: a q-tile that
 * meets a larger value (in its queries or any key it reads) is not computed;
 * its rows get out = 0, lse = NaN and RK_STATUS_RANGE is set.
 */
int rk_paged_attn_prefill(const rk_paged_plan_t *plan, const void *q, const void *k_cache,
                          const void *v_cache, const int32_t *block_table_d,
                          const int32_t *kv_lens_d, const int32_t *position_ids_d, void *out,
                          float *lse, int32_t *status_d, rk_stream_t stream);

/*
 * Fixed-split decode (a separate arithmetic policy, not bitwise equal to
 * rk_paged_attn_decode): each row's KV range is cut at fixed logical token
 * offsets s * split_tokens, every split is reduced by its own CTA in
 * ascending KV order (FP32 partial O / l and partial LSE), and the partials
 * are merged in ascending split order in FP32 before the single BF16 write.
 * The boundaries depend only on the token index, so results stay bitwise
 * identical across batch composition, table width and graph replay for a
 * given split_tokens.  Gives a long row more CTAs than its Hkv heads.
 * Follows "Add FlashInfer RoPE-fused paged attention scaffold", boundary
 * table (Split-K row: fixed num_splits, merge order fixed by the global block
 * index) and "flashinfer_fa2 backend for Ada (SM89)", the no-split vs split
 * kernel table (the cost of disabling splits on long, low-batch rows).
 *
 *   split_tokens  a positive multiple of page_size = 16 (RK_E_ARG otherwise),
 *                 as "WS2 PR7 ...", "Split-KV Policy" defines fixed:<N> in
 *                 logical tokens.  Each split's CTA sweeps 128-token tiles from
 *                 its first token, with exact RoPE angles at that token, so a
 *                 split may start and end inside a 128-token tile.
 *   n_splits      = ceil(W * page_size / split_tokens), at least 1.
 *
 * rk_paged_decode_split_scratch_bytes -- *bytes = the device scratch the
 * split entry point needs for this plan and split_tokens:
 * B * Hq * n_splits * (D + 1) * 4.  Host only.
 */
int rk_paged_decode_split_scratch_bytes(const rk_paged_plan_t *plan, int32_t split_tokens, uint64_t *bytes);

/*
 * rk_paged_attn_decode_split -- as rk_paged_attn_decode, plus:
 *   scratch        DEVICE memory owned by the caller, 16-byte aligned, at
 *                  least rk_paged_decode_split_scratch_bytes bytes; holds the
 *                  FP32 partials ([B, Hq, n_splits, D] O / l, then
 *                  [B, Hq, n_splits] log2-domain LSE).  Nothing in it needs
 *                  initialising: every partial the merge reads is written
 *                  first by the same call.  Two calls in flight at once must
 *                  not share a scratch buffer.
 *   scratch_bytes  its size.
 * Two kernel launches on `stream` (splits, then merge).  A split that meets
 * unsafe metadata or the FP16 range limit makes its row out = 0, lse = NaN
 * and sets the status bit, as in rk_paged_attn_decode.
 * Returns RK_E_ARG for a bad split_tokens or a missing / small / misaligned
 * scratch, otherwise as rk_paged_attn_decode.
 */
int rk_paged_attn_decode_split(const rk_paged_plan_t *plan, int32_t split_tokens, const void *q,
                               const void *k_cache, const void *v_cache, const int32_t *block_table_d,
                               const int32_t *kv_lens_d, const int32_t *position_ids_d, void *out,
                               float *lse, void *scratch, uint64_t scratch_bytes, int32_t *status_d,
                               rk_stream_t stream);

/*
 * rk_paged_attn_decode_split_static -- rk_paged_attn_decode_split without a
 * caller scratch buffer and without any allocation: the partials live in one
 * file-scope device array of RK_PAGED_SPLIT_STATIC_SCRATCH_BYTES inside the
 * library.  For callers that may not allocate device memory at all (a
 * process whose memory is handed out by another owner, or code that must not
 * call cudaMalloc while another stream is being captured).  The first call on
 * a device looks the array's device address up (cudaGetSymbolAddress, with
 * that device current, which may load the module): make that first call
 * before any stream capture.  The address is then kept for the life of the
 * process, which assumes the device's context is not reset (cudaDeviceReset)
 * while the library is loaded.  Arguments, results and errors as
 * rk_paged_attn_decode_split, and in addition:
 *   RK_E_ARG   rk_paged_decode_split_scratch_bytes(plan, split_tokens) is
 *              above RK_PAGED_SPLIT_STATIC_SCRATCH_BYTES (nothing launched);
 *   RK_E_CUDA  the device address of the array could not be obtained.
 * Nothing in the array needs to start at zero (each call writes every partial
 * it reads), so nothing is cleared.  The array is shared by every call on the
 * device: two calls whose kernels overlap in time (different streams, or
 * different host threads on the same device) race on it and may return wrong
 * results; serialise such calls or use rk_paged_attn_decode_split with a
 * scratch buffer per stream.
 */
#define RK_PAGED_SPLIT_STATIC_SCRATCH_BYTES (16ull << 20)
int rk_paged_attn_decode_split_static(const rk_paged_plan_t *plan, int32_t split_tokens, const void *q,
                                      const void *k_cache, const void *v_cache,
                                      const int32_t *block_table_d, const int32_t *kv_lens_d,
                                      const int32_t *position_ids_d, void *out, float *lse,
                                      int32_t *status_d, rk_stream_t stream);

/*
 * Balanced split-free decode: the same operation and the same arithmetic as
 * rk_paged_attn_decode (split-KV disabled: each (row, KV head) is reduced in
 * one ascending-KV pass, "flashinfer_fa2 backend for Ada (SM89)", "Split-KV
 * is disabled" design note), on a schedule that keeps every SM busy to the
 * end.  One CTA per SM (a cooperative launch: all resident at once), the
 * CTAs in Hkv chains, one per KV head.  The 128-token tiles of every row are
 * grouped in blocks of 1, 2, 4 or 8 tiles (the coarsest that still gives every
 * CTA of a chain work, no finer than the plan's B and W allow for a bounded
 * segment list), the rows' blocks laid end to end in row order and
 * dealt to a chain's CTAs in equal contiguous runs (the same runs for every
 * head, so the CTAs serving a row's heads read its pages together); where a
 * row crosses from one CTA's run to the next, the first CTA hands its running
 * state (running max, per-lane partial sums of l, the FP32 O accumulator) to
 * the second through the scratch buffer, and the second goes on from the next
 * tile.  The row is therefore reduced tile
 * after tile, in ascending order, by exactly the operations of the one-CTA
 * path: out and lse are bitwise identical to rk_paged_attn_decode's for every
 * row, whatever the batch, the table width or the grid.  (A CTA does the row
 * it hands on first and the row it takes over last, so a hand-off is
 * normally ready long before it is read; the read waits at most the plan's
 * wait limit and then fails closed like any other wait.)
 *
 * rk_paged_decode_balanced_scratch_bytes -- *bytes = the device scratch the
 * balanced entry point needs (RK_PAGED_BALANCED_SCRATCH_BYTES: hand-off
 * flags and states for up to 512 CTAs; independent of the plan).  Host only.
 *
 * rk_paged_attn_decode_balanced -- as rk_paged_attn_decode, plus:
 *   scratch        DEVICE memory owned by the caller, 256-byte aligned, at
 *                  least rk_paged_decode_balanced_scratch_bytes bytes, ZEROED
 *                  ONCE before its first use and then left to the library
 *                  (each launch leaves it ready for the next: a launch epoch
 *                  in its first word makes earlier hand-off flags stale, so
 *                  graph replays of one captured launch are fine).  Two
 *                  launches in flight at once must not share a scratch buffer.
 *   scratch_bytes  its size.
 * The balanced schedule is used when it can help and is safe: each chain has
 * at least two CTAs and at most as many as the batch has rows, the batch has at
 * most 12288 rows, and no CTA would hold more than 32 segments (B * ceil(W /
 * 64) blocks at most 30 per chain member); otherwise the call runs
 * rk_paged_attn_decode's one-CTA-per-(row, KV head) launch (same results;
 * scratch untouched).
 * Returns RK_E_ARG for a missing / small / misaligned scratch, otherwise as
 * rk_paged_attn_decode; RK_E_CUDA also if the cooperative launch is refused.
 */
#define RK_PAGED_BALANCED_MAX_CTAS 512
#define RK_PAGED_BALANCED_SCRATCH_BYTES (4096ull + 512ull * 3088ull * 4ull)
int rk_paged_decode_balanced_scratch_bytes(const rk_paged_plan_t *plan, uint64_t *bytes);
int rk_paged_attn_decode_balanced(const rk_paged_plan_t *plan, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *block_table_d, const int32_t *kv_lens_d,
                                  const int32_t *position_ids_d, void *out, float *lse, void *scratch,
                                  uint64_t scratch_bytes, int32_t *status_d, rk_stream_t stream);

/*
 * rk_paged_kv_append -- write new tokens' K and V into their pages, as the
 * cache holds them: pre-RoPE (the attention calls rotate K when they read
 * it; "WS2 PR7 ...", "FlashInfer RoPE Fusion").  The page walk is the one of
 * the attention calls: position t of row b is slot t % 16 of page
 * block_table_d[b, t / 16].
 *   n_new         tokens per row (>= 0; 0 is a no-op).
 *   k_new, v_new  bf16 [B, n_new, Hkv, D] DEVICE, contiguous, 16-byte aligned.
 *   kv_lens_d     [B] lengths AFTER the append: the new tokens of row b take
 *                 positions kv_len - n_new .. kv_len - 1 (a prefill chunk's
 *                 K/V is in the cache before its attention runs).  The caller
 *                 updates kv_lens and allocates the pages first; a plan built
 *                 on those host values validates them.
 *   k_cache, v_cache  bf16 [num_pages, 16, Hkv, D] DEVICE, written in place.
 *   status_d      RK_STATUS_KVLEN when kv_len < n_new or > W * 16,
 *                 RK_STATUS_PAGE_OOB when a target page id is outside
 *                 [0, num_pages): that token is not written (never out of
 *                 bounds).  May be NULL.
 * Plan: only B, Hkv, D, page_size, W, num_pages are used (Sq is ignored).
 * One launch on `stream`, no allocation, no host synchronisation.  Errors:
 * RK_E_ARG (null / misaligned pointer, n_new < 0, plan mismatch),
 * RK_E_KVLEN (tokens to append but an empty table or pool), RK_E_DEVICE,
 * RK_E_CUDA.
 */
int rk_paged_kv_append(const rk_paged_plan_t *plan, int32_t n_new, const void *k_new, const void *v_new,
                       const int32_t *block_table_d, const int32_t *kv_lens_d, void *k_cache,
                       void *v_cache, int32_t *status_d, rk_stream_t stream);

/*
 * Ragged batches: rows with different numbers of queries this step (prefill
 * chunks of any length next to single-query decode rows), queries packed
 * along one axis as in FlashInfer's ragged NHD layout (qo_indptr).  Each row
 * is computed exactly as the padded entry points compute it (the same
 * validation list, the same per-row reduction): single-query rows by the
 * decode kernel, longer rows by the prefill kernel, a choice made by the
 * row's own query count, so results stay batch-invariant.
 *   qo_indptr     int32 [B + 1]: row b's queries are packed rows
 *                 qo_indptr[b] .. qo_indptr[b + 1] - 1 (0 = no query).
 *   q, out        bf16 [total_q, Hq, D];  lse  fp32 [total_q, Hq];
 *   position_ids  int32 [total_q] (contiguous ascending per row, trailing).
 *
 * rk_paged_plan_ragged -- rk_paged_plan for a ragged batch: validates
 * qo_indptr (starts at 0, non-decreasing, ends at total_q >= 1; RK_E_ARG),
 * then shapes and, when all three metadata arrays are given, the same list
 * as rk_paged_plan per row (rows with no query are skipped by the position
 * rules).  The plan holds Sq = total_q.  *max_q_len receives the largest
 * per-row query count; plan->pf_units the number of prefill work units, a
 * pair of q-tiles (2 x 128 / (Hq / Hkv) queries) of a row with two or more
 * queries, which sizes the prefill grid exactly.  Host only.
 */
int rk_paged_plan_ragged(rk_paged_plan_t *plan, int32_t B, int32_t total_q, int32_t Hq, int32_t Hkv,
                         int32_t D, int32_t page_size, int32_t num_pages, int32_t W,
                         const int32_t *qo_indptr_h, const int32_t *block_table_h,
                         const int32_t *kv_lens_h, const int32_t *position_ids_h, double rope_theta,
                         double rope_scale, int32_t *max_q_len);

/*
 * rk_paged_attn_ragged -- causal attention for a ragged batch (plan from
 * rk_paged_plan_ragged, or a shape-only rk_paged_plan with Sq = total_q).
 *   max_q_len     1 <= max_q_len <= total_q: bound of every row's query count
 *                 this call may see (the grid is sized by it; a row above it
 *                 is not computed and sets RK_STATUS_POSITION).
 *   qo_indptr_d   DEVICE int32 [B + 1].  Other buffers as above, DEVICE,
 *                 q / out / caches 16-byte aligned.
 * Two launches on `stream` (decode rows, then prefill rows), no allocation,
 * no host synchronisation: metadata is read on the device, and each prefill
 * CTA finds its work unit from qo_indptr_d (heaviest units first).  The
 * prefill grid holds plan->pf_units units (for pf_units = -1: a bound that
 * covers every batch of this total_q and max_q_len), so a captured graph
 * replays with new contents that respect max_q_len and, unless pf_units is
 * -1, need no more units than the plan counted.  A row whose qo_indptr
 * entries are out of range or decreasing is not written and sets
 * RK_STATUS_POSITION, as does work beyond the grid.  Errors as
 * rk_paged_attn_prefill, plus RK_E_ARG for max_q_len or qo_indptr_d, and
 * RK_E_UNSUPPORTED for more than 12000 pairs of q-tiles in one row.
 */
int rk_paged_attn_ragged(const rk_paged_plan_t *plan, int32_t max_q_len, const int32_t *qo_indptr_d,
                         const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_table_d, const int32_t *kv_lens_d,
                         const int32_t *position_ids_d, void *out, float *lse, int32_t *status_d,
                         rk_stream_t stream);

/*
 * rk_paged_attn_prefill_backward -- deterministic gradient of
 * rk_paged_attn_prefill ("Add FlashInfer RoPE-fused paged attention
 * scaffold", scope table, Backward row: dropout 0, deterministic backward
 * required).  For L = sum(dout * out) it writes dL/dq and dL/d(k_cache),
 * dL/d(v_cache) (gradients of the pre-RoPE inputs; RoPE is applied to q and
 * K on the fly and undone by its transpose on dq and dk).
 *   plan, q, k_cache, v_cache, block_table_d, kv_lens_d, position_ids_d:
 *                 as for rk_paged_attn_prefill (same validation).
 *   out, lse      DEVICE bf16 [B, Hq, Sq, D] / fp32 [B, Hq, Sq]: that call's
 *                 results (P = exp(score - lse) is recomputed from them).
 *   dout          DEVICE bf16 [B, Hq, Sq, D], 16-byte aligned.
 *   dq            DEVICE fp32 [B, Hq, Sq, D], 16-byte aligned (written).
 *   dk_cache, dv_cache
 *                 DEVICE fp32 [num_pages, 16, Hkv, D], 16-byte aligned: for
 *                 every row the pages of its first ceil(kv_len / 16) table
 *                 entries are written in full (0 at slots past kv_len); no
 *                 other entry is touched.  Rows sharing a page (rejected by
 *                 rk_paged_plan) give unspecified values on it.
 *   workspace, workspace_bytes
 *                 DEVICE, 256-byte aligned, at least
 *                 rk_paged_prefill_backward_workspace_bytes bytes; caller-owned
 *                 scratch: q rotated once (FP16), the rows' keys rotated and
 *                 their values copied into logical token order (FP16 / BF16
 *                 [B, Hkv, W * 16, D]), then delta = rowsum(dout * out) (FP32
 *                 [B, Hq, Sq]).
 * Deterministic and batch-invariant: every output element is accumulated by
 * one CTA in a fixed order (dq over key tiles ascending, dk / dv over query
 * blocks ascending), no atomics.  Arithmetic: FP32 accumulation on the
 * tcgen05 tensor cores (accumulators in TMEM); rotated q / k and dS rounded
 * to FP16, P to BF16 for the dV product.  Four launches on `stream` (the
 * rotation of q and of the K pages, dq with delta, dk / dv), no allocation,
 * no host synchronisation.  Device status bits as the forward;
 * gradients a pre-RoPE element with |x| >= 2^15 or a dS beyond the FP16
 * range enters come out NaN, with RK_STATUS_RANGE.  Errors: as
 * rk_paged_attn_prefill, plus RK_E_ARG for a null or misaligned dout / dq /
 * dk_cache / dv_cache / workspace or a workspace below the required size.
 */
int rk_paged_attn_prefill_backward(const rk_paged_plan_t *plan, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_table_d,
                                   const int32_t *kv_lens_d, const int32_t *position_ids_d,
                                   const void *out, const float *lse, const void *dout, float *dq,
                                   float *dk_cache, float *dv_cache, void *workspace,
                                   uint64_t workspace_bytes, int32_t *status_d, rk_stream_t stream);

/* rk_paged_prefill_backward_workspace_bytes -- *bytes = the device workspace
 * rk_paged_attn_prefill_backward needs for this plan (2 B Hq Sq D + 2 x 2 B
 * Hkv W 16 D + 4 B Hq Sq bytes, each part rounded up to 256).  Host only;
 * RK_E_ARG for a null plan / bytes or a plan of another ABI. */
int rk_paged_prefill_backward_workspace_bytes(const rk_paged_plan_t *plan, uint64_t *bytes);

/* Message of the last failing call on this thread ("" if none).  The
 * pointer stays valid until the next library call on the same thread. */
const char *rk_last_error(void);

/*
 * Fixed arithmetic policy of this library as "key=value;..." text: split-KV,
 * accumulation and LSE types, LSE base, downcast point and rounding, KV
 * reduction order, KV tile sizes.  Provenance in the sense of "WS2 PR7 ...",
 * "P2P NCCL reference and strict arithmetic provenance" (FP32 accumulation,
 * FP32 LSE, downcast only at the final write).  Static string.
 */
const char *rk_paged_policy(void);

/* RK_PAGED_ABI_VERSION of the loaded library. */
uint32_t rk_paged_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RK_PAGED_H */
