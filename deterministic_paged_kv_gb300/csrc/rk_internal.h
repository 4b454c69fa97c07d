// rk_internal.h -- constants and kernel argument blocks shared by the host
// launch code and the kernels.  Not part of the public ABI.
#pragma once

#include <stdint.h>

#define RK_WAIT_LIMIT_NS 2000000000ull  // a pipeline wait gives up after 2 s

namespace rk {

constexpr int HEAD_DIM = 128;
constexpr int PAGE = 16;
constexpr int ROPE_PAIRS = HEAD_DIM / 2;

// ------------------------------------------------------------ decode ----
// One CTA per (row, KV head): two transform warpgroups, one softmax
// warpgroup, K and V TMA producer warps and one MMA warp (15 warps).  Tiles
// of 128 tokens.
constexpr int DEC_XFORM_THREADS = 256;
constexpr int DEC_THREADS = 16 * 32;
constexpr int DEC_BN = 128;                           // tokens per KV tile (8 pages)
constexpr int DEC_KSTAGES = 3;
constexpr int DEC_VSTAGES = 3;
constexpr int DEC_TILE_BYTES = DEC_BN * HEAD_DIM * 2;  // 32 KiB
constexpr int DEC_KAHEAD = 2;                          // K tiles a transform thread keeps in flight
constexpr int DEC_CTRL_BYTES = 2048;                   // barriers, RoPE tables, reductions
constexpr int DEC_PGT_ENTRIES = 2048;                  // page ids of a CTA's range held in shared memory
constexpr int DEC_SMEM_BYTES = (DEC_KSTAGES + DEC_VSTAGES) * DEC_TILE_BYTES + 16 * HEAD_DIM * 2 +
                               2 * 16 * DEC_BN * 2 + DEC_CTRL_BYTES + DEC_PGT_ENTRIES * 4;
// The balanced (persistent) decode: two Q^T buffers and a segment list.
constexpr int DEC_BAL_CTRL_BYTES = 4096;
constexpr int DEC_BAL_SMEM_BYTES = (DEC_KSTAGES + DEC_VSTAGES) * DEC_TILE_BYTES + 2 * 16 * HEAD_DIM * 2 +
                                   2 * 16 * DEC_BN * 2 + DEC_BAL_CTRL_BYTES + DEC_PGT_ENTRIES * 4;

struct DecodeArgs {
    const void* q;                // bf16 [B, Hq, 1, D]
    const void* k_cache;          // bf16 [num_pages, 16, Hkv, D]
    const int32_t* block_table;   // [B, W]
    const int32_t* kv_lens;       // [B]
    const int32_t* position_ids;  // [B, 1]
    void* out;                    // bf16 [B, Hq, 1, D]
    float* lse;                   // [B, Hq, 1]
    int32_t* status;              // may be null
    int32_t B, Hq, Hkv, G, W, num_pages;
    float qk_scale_log2;          // sm_scale * log2(e)
    // Fixed split of each row's KV range (0 = no split): split s covers the
    // keys [s * split_tokens, (s + 1) * split_tokens); the CTA writes its
    // partial O / l (FP32 [B, Hq, n_splits, D]) and log2-domain partial LSE
    // (FP32 [B, Hq, n_splits]; -inf when empty, NaN when unsafe) instead of out.
    int32_t split_tokens;         // a multiple of the page size
    int32_t n_splits;
    float* o_part;
    float* lse_part;
    // Ragged batch (qo_indptr != null): q / out [total_q, Hq, D], lse
    // [total_q, Hq], position_ids [total_q]; row b's queries are packed rows
    // qo_indptr[b] .. qo_indptr[b + 1] - 1 and this kernel serves the rows
    // with exactly one query.
    const int32_t* qo_indptr;
    int32_t total_q;
    int32_t max_q_len;            // rows with more queries are flagged (RK_STATUS_POSITION)
    uint32_t wait_limit_ns;       // pipeline wait limit (0: RK_WAIT_LIMIT_NS)
    int32_t timeout_drill;        // nonzero: the score MMA issuer first waits on a barrier nothing completes
    // Balanced schedule (balanced != 0; padded split-free decode only): each
    // (row, KV head)'s tiles are cut in blocks of bal_block_tiles, the blocks
    // of all of them laid end to end in (row, KV head) order and dealt to the
    // CTAs in equal contiguous runs.  A row whose blocks cross from CTA c's run
    // into CTA c + 1's hands its running softmax state (m, l, O) over through
    // bal_state slot c: the row is still reduced tile after tile in ascending
    // order, with the same operations as by a single CTA.
    int32_t balanced;
    uint32_t* bal_sync;           // [0] launch epoch, [1] CTAs done, [2 + c] hand-off flag of slot c
    float* bal_state;             // [grid - 1][DEC_BAL_STATE_FLOATS]
    int32_t bal_grid;             // CTAs of a balanced launch (all resident at once)
    int32_t bal_block_tiles;      // tiles per block of the balanced schedule (1 .. DEC_BAL_MAX_BLOCK_TILES)
    uint64_t rope_turns[ROPE_PAIRS];
};
constexpr int DEC_SPLIT_GRAIN = PAGE;  // split lengths are multiples of the page size
constexpr int DEC_BAL_MAX_BLOCK_TILES = 8;   // the largest block the host picks (tiles)
constexpr int DEC_BAL_MAX_SEGS = 32;         // segments one CTA can hold
constexpr int DEC_BAL_MAX_ROWS = 12288;      // rows whose block counts fit the set-up scratch
// Hand-off state of one row: m per head [8], info [8] (ok, range_bad), l
// partial per (token lane, head) [128][8], O^T row per output dim [128][16].
constexpr int DEC_BAL_M = 0, DEC_BAL_INFO = 8, DEC_BAL_LP = 16, DEC_BAL_O = DEC_BAL_LP + 128 * 8;
constexpr int DEC_BAL_STATE_FLOATS = DEC_BAL_O + 128 * 16;  // 3088 floats, 64-byte multiple
constexpr int DEC_BAL_SYNC_WORDS = 2;        // epoch, done; then one flag per slot

// ----------------------------------------------------------- prefill ----
// One CTA per (row, KV head, q-tile).  A q-tile is 128 accumulator rows =
// (128 / G) consecutive query positions x the G query heads of one KV head.
constexpr int PF_BM = 128;          // accumulator rows per tile
constexpr int PF_BN = 128;          // KV tokens per tile (8 pages)
constexpr int PF_PAGES_PER_TILE = PF_BN / PAGE;
constexpr int PF_TILE_BYTES = PF_BM * HEAD_DIM * 2;  // 32 KiB bf16 operand tile

struct PrefillArgs {
    const int32_t* block_table;   // [B, W]
    const int32_t* kv_lens;       // [B]
    const int32_t* position_ids;  // [B, Sq]
    void* out;                    // bf16 [B, Hq, Sq, D]
    float* lse;                   // [B, Hq, Sq]
    int32_t* status;
    int32_t B, Sq, Hq, Hkv, G, W, num_pages;
    int32_t rows_per_head;        // 128 / G positions per q-tile
    int32_t n_qtiles;             // ceil(Sq / rows_per_head) (ragged: ceil(max_q_len / rows_per_head))
    float qk_scale_log2;
    // Ragged batch (qo_indptr != null): packed q / out [total_q, Hq, D], lse
    // [total_q, Hq], position_ids [total_q]; this kernel serves the rows with
    // two or more queries (single-query rows go to the decode kernel).
    const int32_t* qo_indptr;
    int32_t total_q;
    int32_t max_q_len;            // ragged: rows with more queries are not computed
    int32_t ragged_units;         // ragged: work units of the grid (grid = ragged_units x Hkv)
    uint32_t wait_limit_ns;       // pipeline wait limit (0: RK_WAIT_LIMIT_NS)
    int32_t timeout_drill;        // nonzero: the MMA issuer first waits on a barrier nothing completes
    int32_t pad0;
    uint64_t rope_turns[ROPE_PAIRS];
};
// Ragged prefill schedule: the largest pair count of a row it handles (the
// per-CTA scan keeps 2 x levels + 1 counters in a K stage buffer).
constexpr int PF_RAGGED_MAX_LEVELS = 12000;

// ---------------------------------------------------------- backward ----
// Gradient of causal paged prefill (padded layout, q / out / dout
// [B, Hq, Sq, D] bf16, lse [B, Hq, Sq] fp32): dq [B, Hq, Sq, D] fp32, dk / dv
// in the cache layout [num_pages, 16, Hkv, D] fp32, delta [B, Hq, Sq] fp32
// (rowsum(dout * out); written by the dq launch, read by the dk/dv launch).
struct BackwardArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_table;   // [B, W]
    const int32_t* kv_lens;       // [B]
    const int32_t* position_ids;  // [B, Sq]
    const void* out;
    const float* lse;
    const void* dout;
    float* dq;
    float* dk;
    float* dv;
    float* delta;                 // workspace: [B, Hq, Sq] fp32
    void* q_rot;                  // workspace: RoPE-rotated q as FP16 [B, Hq, Sq, D]
    void* k_lin;                  // workspace: rotated K as FP16 [B, Hkv, W * 16, D], logical token order
    void* v_lin;                  // workspace: V as BF16 [B, Hkv, W * 16, D], logical token order
    int32_t* status;
    int32_t B, Sq, Hq, Hkv, G, W, num_pages;
    float sm_scale;
    float qk_scale_log2;          // sm_scale * log2(e)
    uint32_t wait_limit_ns;       // pipeline wait limit (0: RK_WAIT_LIMIT_NS)
    int32_t timeout_drill;        // nonzero: each tcgen05 kernel's MMA issuer first waits on a barrier nothing completes
    uint64_t rope_turns[ROPE_PAIRS];
};

// ------------------------------------------------------------ append ----
// Write n_new tokens per row into the page cache (kv_lens after the append).
struct AppendArgs {
    const void* k_new;            // bf16 [B, n_new, Hkv, D]
    const void* v_new;            // bf16 [B, n_new, Hkv, D]
    const int32_t* block_table;   // [B, W]
    const int32_t* kv_lens;       // [B], lengths including the new tokens
    void* k_cache;                // bf16 [num_pages, 16, Hkv, D]
    void* v_cache;
    int32_t* status;
    int32_t B, n_new, Hkv, W, num_pages;
};

}  // namespace rk
