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
// One CTA per (row, KV head, group of up to 4 query heads).  Four consumer
// warps; warp w, lane group g (8 lanes) owns token slot 4w+g of every page.
constexpr int DEC_CWARPS = 4;
constexpr int DEC_THREADS = (DEC_CWARPS + 1) * 32;  // + one TMA producer warp
constexpr int DEC_STAGES = 8;                        // pages in flight per CTA
constexpr int DEC_PAGE_BYTES = PAGE * HEAD_DIM * 2;  // one head of one page: 4 KiB
constexpr int DEC_STAGE_BYTES = 2 * DEC_PAGE_BYTES;  // K + V
constexpr int DEC_REANCHOR = 16;                     // exact RoPE angles every 16 pages
constexpr float DEC_RESCALE_THRESHOLD = 8.0f;        // log2-domain max slack
constexpr int DEC_CTRL_BYTES = 2048;                   // barriers, RoPE tables, flags
constexpr int DEC_SMEM_BYTES = DEC_STAGES * DEC_STAGE_BYTES + DEC_CTRL_BYTES;

struct DecodeArgs {
    const void* q;                // bf16 [B, Hq, 1, D]
    const int32_t* block_table;   // [B, W]
    const int32_t* kv_lens;       // [B]
    const int32_t* position_ids;  // [B, 1]
    void* out;                    // bf16 [B, Hq, 1, D]
    float* lse;                   // [B, Hq, 1]
    int32_t* status;              // may be null
    int32_t B, Hq, Hkv, G, W, num_pages;
    float qk_scale_log2;          // sm_scale * log2(e)
    int32_t pad0;
    uint64_t rope_turns[ROPE_PAIRS];
};

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
    int32_t n_qtiles;             // ceil(Sq / rows_per_head)
    float qk_scale_log2;
    uint64_t rope_turns[ROPE_PAIRS];
};

}  // namespace rk
