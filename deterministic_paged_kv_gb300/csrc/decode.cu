// decode.cu -- split-free paged decode on the 5th-gen tensor cores, RoPE
// applied to K as it is read.
//
// Operation: paged decode of "flashinfer_fa2 backend for Ada (SM89)" (BF16,
// page 16, head_dim 128, NHD; split-KV disabled so a row's reduction does not
// depend on plan width or batch), with ROPE_LLAMA fused as in "WS2 PR7 Fused
// Attention Backend Alignment", "FlashInfer RoPE Fusion", and the FP32 LSE of
// that page's "Original PR7 Requirements" table.
//
// One CTA per (row b, KV head); all G = Hq/Hkv query heads of the group are
// served by one pass over the row's pages (GQA packing: every K/V byte is
// read once).  The row's tokens are swept in ascending tiles of 128 (8 pages):
//   warp 14       V producer: V pages (3-stage ring) by TMA, one 4 KiB box
//                 per page ([64-dim half][16 tokens], 128-byte swizzled, read
//                 by the PV MMA one page per k-step); zeroes cache rows past
//                 kv_len in a partial last page;
//   warps 0-7     transform: each thread copies the K chunks it will rotate
//                 (its 4 token rows x 16 B of each 64-dim half) with 16-byte
//                 cp.async, DEC_KAHEAD tiles ahead, straight into the
//                 128-byte swizzled K-major tile of a 3-stage ring; then
//                 rotates each K row in FP32 (angles from an exact fixed-point
//                 anchor plus 32-position steps) and stores it as FP16 in
//                 place; rotates the G query rows once (FP16 Q^T).  K through
//                 the load/store path of eight warps leaves the TMA unit to V:
//                 a warp's page boxes issue at ~20 B a cycle, so K and V boxes
//                 took their producer warps ~1800-2000 cycles a tile, more than
//                 the rest of the pipeline;
//   warp 12       idle (one warp of cp.async producer could not keep enough
//                 copies in flight);
//   warp 13       score MMA issuer: S^T = K Q^T (M = 128 tokens, N = 16 >= G
//                 heads, FP16 operands, FP32 in TMEM, double-buffered);
//   warp 15       PV MMA issuer: O^T += V^T P^T (M = 128 dims, N = 16, BF16,
//                 FP32 in TMEM, P^T double-buffered in shared memory);
//   warps 8-11    softmax: thread t owns token t of the tile: masks, takes the
//                 tile max per head over the 128 tokens (xor-butterfly + fixed
//                 warp order), moves the running max only when it grows by
//                 more than 8 (log2 domain; then the O^T column is rescaled in
//                 TMEM), writes P^T as BF16 to shared memory and keeps a
//                 per-thread partial of l; epilogue reduces l in a fixed
//                 tree, writes out = O / l (BF16, once) and the LSE (FP32).
// Score precision: FP16 rotated operands (11-bit mantissa) keep the LSE
// within 1e-3 of float64 even for a single visible key; pre-RoPE q / k
// elements at or above 2^15 would overflow FP16 once rotated and are
// reported (RK_STATUS_RANGE) instead of computed.
// Every choice depends only on the row's data and logical token index, never
// on B, W, the grid or the SM.
//
// Balanced schedule (decode_bal_kernel, rk_paged_attn_decode_balanced): the
// same roles and the same arithmetic on a persistent cooperative grid, one CTA
// per SM in Hkv chains (one per KV head).  Each row's tiles are grouped in
// blocks of 1, 2, 4 or 8 tiles (the coarsest that still gives every CTA of a
// chain work) and a chain's CTAs take equal contiguous runs of the rows' blocks,
// so a batch whose
// (row, KV head) count is not a multiple of the SM count keeps every SM busy to
// the end.  A row cut between two CTAs is handed over exactly: the first CTA
// writes its running max, per-lane partial sums of l and its FP32 O^T row
// (read from TMEM) to the scratch buffer and releases a flag; the second, which
// takes that row last (the first did it first), waits (bounded) for the flag,
// loads the state (O^T back into TMEM) and goes on with the next tile.  A
// segment that starts between two RoPE anchor tiles takes the exact angles at
// the anchor before it and replays the angle steps of the tiles in between.  So
// every row is reduced tile after tile in ascending order by the operations of
// the one-CTA launch, and out / lse are bitwise identical to it.  The CTA's
// pipeline runs on across its segments: the ring phases count the CTA's tiles,
// K copies for the next segment start while the current one ends, Q^T is
// double-buffered by segment, and V pages a partial tile leaves unloaded are
// zeroed when the stage last held another segment's rows.
#include <atomic>
#include <cstring>

#include "rk_device.cuh"

namespace rk {

namespace {

constexpr int WARP_SOFTMAX0 = DEC_XFORM_THREADS / 32;  // warps 8-11
constexpr int WARP_TMA_K = WARP_SOFTMAX0 + 4;
constexpr int WARP_MMA = WARP_TMA_K + 1;
constexpr int WARP_TMA_V = WARP_TMA_K + 2;
constexpr int WARP_PV = WARP_TMA_K + 3;
constexpr int XF_ROW_STEP = DEC_XFORM_THREADS / 8;      // rows between a thread's K rows
constexpr int XF_ROWS = DEC_BN / XF_ROW_STEP;           // K rows per transform thread per tile
constexpr int XF_ANCHOR_TILES = 8;                      // tiles between exact RoPE anchors
constexpr uint32_t TMEM_COLS = 64;  // S^T buffers [0,16) [16,32), O^T [32,48)
constexpr float RESCALE_SLACK = 8.0f;
constexpr int NH = 16;  // N of both MMAs: query heads of the group, zero padded

constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + DEC_KSTAGES * DEC_TILE_BYTES;
constexpr int OFF_QT = OFF_V + DEC_VSTAGES * DEC_TILE_BYTES;  // Q^T: 16 rows x 128 dims FP16
constexpr int PT_BYTES = NH * DEC_BN * 2;                     // P^T: 16 rows x 128 tokens BF16
constexpr int OFF_PT = OFF_QT + NH * HEAD_DIM * 2;            // two P^T buffers (tile parity)
constexpr int OFF_CTRL = OFF_PT + 2 * PT_BYTES;
constexpr int OFF_PGT = OFF_CTRL + DEC_CTRL_BYTES;             // page ids of the CTA's range
static_assert(OFF_PGT + DEC_PGT_ENTRIES * 4 == DEC_SMEM_BYTES, "decode shared memory carve");

struct DecCtrl {
    uint64_t q_ready;
    uint64_t k_ready[DEC_KSTAGES], k_empty[DEC_KSTAGES];
    uint64_t v_full[DEC_VSTAGES], v_empty[DEC_VSTAGES], v_tail;
    // per tile parity b: S^T buffer (s_full, s_free), P^T buffer (p_ready) and
    // the PV that read it (pv_done); a buffer is reused two tiles later, after
    // its previous phase has been observed, so a wait never meets a later phase
    uint64_t s_full[2], s_free[2], p_ready[2], pv_done[2], o_done;
    uint64_t never;  // nothing arrives: the timeout drill's wait
    uint32_t tmem_base;
    PipeCtl pipe;
    int range_bad;
    uint64_t turns[ROPE_PAIRS];
    float2 step[ROPE_PAIRS];  // cos/sin of an XF_ROW_STEP-position turn per pair
    float red[2][4][8];  // per-warp tile maxima, double-buffered by tile parity
    float lred[4][8];    // per-warp partial l at the end
};
static_assert(sizeof(DecCtrl) <= DEC_CTRL_BYTES, "decode control block exceeds its reservation");

// out = 0 and lse = lse_val for the G heads of (b, kv head); in split mode the
// same for this split's partial (the merge turns NaN / -inf partials into the
// row's NaN / empty result).
__device__ __forceinline__ void write_empty_row(const DecodeArgs& a, int b, int tq, int h0, int split,
                                                float lse_val) {
    if (a.split_tokens > 0) {
        for (int i = threadIdx.x; i < a.G * HEAD_DIM; i += blockDim.x) {
            const int hh = i / HEAD_DIM, d = i % HEAD_DIM;
            a.o_part[(((size_t)b * a.Hq + h0 + hh) * a.n_splits + split) * HEAD_DIM + d] = 0.0f;
        }
        if (threadIdx.x < a.G) a.lse_part[((size_t)b * a.Hq + h0 + threadIdx.x) * a.n_splits + split] = lse_val;
        return;
    }
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    for (int i = threadIdx.x; i < a.G * HEAD_DIM; i += blockDim.x) {
        const int hh = i / HEAD_DIM, d = i % HEAD_DIM;
        out[((size_t)tq * a.Hq + h0 + hh) * HEAD_DIM + d] = __float2bfloat16_rn(0.0f);
    }
    if (threadIdx.x < a.G) a.lse[(size_t)tq * a.Hq + h0 + threadIdx.x] = lse_val;
}

__global__ void __launch_bounds__(DEC_THREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap vmap, const __grid_constant__ DecodeArgs a) {
    extern __shared__ __align__(1024) uint8_t sm[];
    // A launch that only reads what this grid reads (the prefill rows of a
    // ragged batch) may fill the SMs this grid's last wave leaves idle.
    griddep_launch_dependents();
    DecCtrl* ctl = reinterpret_cast<DecCtrl*>(sm + OFF_CTRL);
    const uint32_t s_base = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // work unit: (split, row, KV head), split-major; split = 0 without splitting
    const int rows_heads = a.B * a.Hkv;
    const int split = (int)(blockIdx.x / rows_heads), unit = (int)(blockIdx.x % rows_heads);
    const int kvh = unit % a.Hkv, b = unit / a.Hkv;
    const int G = a.G, h0 = kvh * G;
    if (s_base & 1023u) {  // the swizzled operand layout needs a 1024-byte aligned base
        if (tid == 0 && a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
        // Nothing was computed: padded rows (and split partials, which the merge
        // then turns into out = 0, lse = NaN) are written as failed.  A ragged
        // row's packed index is not known here; the status bit reports it.
        if (!a.qo_indptr) write_empty_row(a, b, b, h0, split, __int_as_float(0x7fc00000));
        return;
    }

    // ---- row metadata (device copy) and memory-safety checks ----
    int tq = b;  // the row's query: padded row b, or its packed row in a ragged batch
    if (a.qo_indptr) {
        const int qs = a.qo_indptr[b], qe = a.qo_indptr[b + 1];
        if (qs < 0 || qe < qs || qe > a.total_q) {  // unsafe: nowhere safe to write
            if (tid == 0 && a.status) atomicOr(a.status, RK_STATUS_POSITION);
            return;
        }
        if (qe - qs != 1) {  // no query, or a prefill row (flagged here when no prefill launch covers it)
            if (qe - qs > a.max_q_len && tid == 0 && a.status) atomicOr(a.status, RK_STATUS_POSITION);
            return;
        }
        tq = qs;
    }
    const int kv_len = a.kv_lens[b];
    const int qpos = a.position_ids[tq];
    const int32_t* bt = a.block_table + (size_t)b * a.W;
    constexpr int PPT = DEC_BN / PAGE;  // pages per tile
    // This CTA's keys start at token t_begin: 0, or split * split_tokens (a
    // multiple of the page size) for a fixed split.  Its tiles are 128 tokens
    // counted from there.
    const int t_begin = a.split_tokens > 0 ? split * a.split_tokens : 0;
    // The page ids of the CTA's part of the table are loaded before its length
    // is known (the metadata costs one round trip, not two) and judged against
    // the visible range below.
    const int pg_lo = t_begin / PAGE;
    const int pg_cap = a.split_tokens > 0 ? min(a.W, pg_lo + a.split_tokens / PAGE) : a.W;
    constexpr int PRE = 4;  // table entries per thread held from the early load
    int pre[PRE];
#pragma unroll
    for (int e = 0; e < PRE; ++e) {
        const int i = pg_lo + tid + e * DEC_THREADS;
        pre[e] = i < pg_cap ? __ldg(bt + i) : 0;
    }
    int bad = 0;
    if (kv_len < 0 || kv_len > a.W * PAGE) bad |= RK_STATUS_KVLEN;
    if (qpos < 0) bad |= RK_STATUS_POSITION;
    const int n_vis = bad ? 0 : (qpos >= kv_len ? kv_len : qpos + 1);
    // This CTA's keys [t_begin, t_end): the row's visible keys, or those of one
    // fixed split, in n_loc tiles of 128 tokens from t_begin.
    const int t_end = a.split_tokens > 0 ? min(n_vis, t_begin + a.split_tokens) : n_vis;
    const int n_loc = t_end > t_begin ? (t_end - t_begin + DEC_BN - 1) / DEC_BN : 0;
    // Last page partly filled and inside the visible range: its rows past
    // kv_len hold arbitrary bits and are zeroed in V after the copy lands
    // (by the CTA that holds the row's last key).
    const bool has_tail = n_vis == kv_len && (kv_len & (PAGE - 1)) != 0 && n_loc > 0 && t_end == n_vis;
    int oob = 0;
    const int pg_end = (t_end + PAGE - 1) / PAGE;  // the pages this CTA reads: [pg_lo, pg_end)
#pragma unroll
    for (int e = 0; e < PRE; ++e) {
        const int i = pg_lo + tid + e * DEC_THREADS;
        if (i < pg_end) oob |= (pre[e] < 0) | (pre[e] >= a.num_pages);
    }
    for (int i = pg_lo + tid + PRE * DEC_THREADS; i < pg_end; i += DEC_THREADS) {  // very wide rows
        const int pg = __ldg(bt + i);
        oob |= (pg < 0) | (pg >= a.num_pages);
    }
    // Loads take page ids from a shared-memory copy of these entries, so no
    // L2 round trip sits between consecutive tiles' copies; entries past the
    // copy (rows of more than DEC_PGT_ENTRIES pages) come from the table.
    int32_t* pgt = reinterpret_cast<int32_t*>(sm + OFF_PGT);
    static_assert(PRE * DEC_THREADS == DEC_PGT_ENTRIES, "the early table load fills the page-id copy");
#pragma unroll
    for (int e = 0; e < PRE; ++e) pgt[tid + e * DEC_THREADS] = pre[e];
    if (tid == 0) {
        ctl->pipe.abort = 0;
        ctl->pipe.limit_ns = wait_limit(a.wait_limit_ns);
        ctl->range_bad = 0;
        mbar_init(smem_u32(&ctl->never), 1);
        mbar_init(smem_u32(&ctl->q_ready), DEC_XFORM_THREADS);
        for (int k = 0; k < DEC_KSTAGES; ++k) {
            mbar_init(smem_u32(&ctl->k_ready[k]), DEC_XFORM_THREADS);
            mbar_init(smem_u32(&ctl->k_empty[k]), 1);
        }
        for (int k = 0; k < DEC_VSTAGES; ++k) {
            mbar_init(smem_u32(&ctl->v_full[k]), 1);
            mbar_init(smem_u32(&ctl->v_empty[k]), 1);
        }
        mbar_init(smem_u32(&ctl->v_tail), 1);
        for (int k = 0; k < 2; ++k) {
            mbar_init(smem_u32(&ctl->s_full[k]), 1);
            mbar_init(smem_u32(&ctl->s_free[k]), 128);
        }
        mbar_init(smem_u32(&ctl->p_ready[0]), 128);
        mbar_init(smem_u32(&ctl->p_ready[1]), 128);
        mbar_init(smem_u32(&ctl->pv_done[0]), 1);
        mbar_init(smem_u32(&ctl->pv_done[1]), 1);
        mbar_init(smem_u32(&ctl->o_done), 1);
        fence_mbar_init();
    }
    if (tid < ROPE_PAIRS) {
        ctl->turns[tid] = a.rope_turns[tid];
        float c, s;
        rope_cos_sin((uint32_t)XF_ROW_STEP, a.rope_turns[tid], c, s);
        ctl->step[tid] = make_float2(c, s);
    }
    // V stages, Q^T and P^T start as zeros (rows never written stay finite).
    for (int i = tid; i < (OFF_CTRL - OFF_V) / 16; i += DEC_THREADS)
        reinterpret_cast<uint4*>(sm + OFF_V)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (__syncthreads_or(oob)) bad |= RK_STATUS_PAGE_OOB;
    if (bad) {
        if (tid == 0 && a.status) atomicOr(a.status, bad);
        write_empty_row(a, b, tq, h0, split, __int_as_float(0x7fc00000));
        return;
    }
    if (n_loc == 0) {
        write_empty_row(a, b, tq, h0, split, -INFINITY);
        return;
    }

    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const uint32_t tO = tmem + 32;
    PipeCtl* abort = &ctl->pipe;

    if (warp == WARP_TMA_K) {
        // K arrives through the transform threads' own copies: nothing to do.
    } else if (warp == WARP_TMA_V) {
        // ============================================ V producer (TMA) ====
        if (lane == 0) prefetch_tmap(&vmap);
        int issued = 0;
        // it: the CTA's own tile count (stages, phases); i: the row's tile index
        for (int it = 0; it < n_loc; ++it) {
            const int k = it % DEC_VSTAGES;
            const uint32_t use = (uint32_t)(it / DEC_VSTAGES);
            const int np = min(PPT, pg_end - (pg_lo + it * PPT));
            const int li = it * PPT + lane;  // lane's page within the CTA's range
            const int pg = lane >= np ? 0 : li < DEC_PGT_ENTRIES ? pgt[li] : __ldg(bt + pg_lo + li);
            const uint32_t eb = smem_u32(&ctl->v_empty[k]);
            const uint32_t fb = smem_u32(&ctl->v_full[k]);
            int good = 1;
            if (lane == 0) {
                good = mbar_wait(eb, (use & 1u) ^ 1u, abort);
                if (good) mbar_arrive_expect_tx(fb, (uint32_t)np * 4096);
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) break;
            // one 4 KiB box per page: [page][half][16 rows][128 B]
            if (lane < np)
                tma_load_4d(s_base + OFF_V + k * DEC_TILE_BYTES + lane * 4096, &vmap, fb, 0, pg * PAGE, 0, kvh);
            __syncwarp();
            if (has_tail && it == n_loc - 1) {
                // this warp armed the phase it waits for: no parity aliasing
                const int landed =
                    __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(fb, use & 1u, abort) : 0, 0);
                if (landed) {
                    const int tail = kv_len - (t_begin + it * DEC_BN);
                    const int r_end = min(DEC_BN, (tail + PAGE - 1) & ~(PAGE - 1));
                    uint8_t* vt = sm + OFF_V + k * DEC_TILE_BYTES;
                    for (int idx = lane; idx < (r_end - tail) * 16; idx += 32) {
                        const int rr = tail + (idx >> 4), ch = idx & 15;
                        *reinterpret_cast<uint4*>(vt + (rr >> 4) * 4096 + (ch >> 3) * 2048 + (rr & 15) * 128 +
                                                  (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ctl->v_tail));
                }
            }
            ++issued;
        }
        if (lane == 0 && pipe_aborted(abort)) {
            for (int i = max(0, issued - DEC_VSTAGES); i < issued; ++i)
                mbar_wait_drain(smem_u32(&ctl->v_full[i % DEC_VSTAGES]), (uint32_t)((i / DEC_VSTAGES) & 1));
        }
    } else if (warp == WARP_MMA || warp == WARP_PV) {
        // ============================================ MMA issuers ====
        // Two issuing threads: warp 13 issues the score MMAs, warp 15 the PV
        // MMAs, each waiting only for its own inputs, so the barrier checks of
        // one overlap the MMAs of the other.  tcgen05.commit covers the MMAs of
        // the committing thread, which is what each completion barrier tracks.
        // Each issuer's whole warp runs its loop (converged, warp-uniform
        // operands); elect.sync picks the lane that issues MMAs and commits.
        {
            constexpr uint32_t TILE_DESC = DEC_TILE_BYTES >> 4;  // one 32 KiB tile in descriptor address units
            bool ok = true;
            if (warp == WARP_MMA) {
                const uint32_t idS = idesc_f16_f32(DEC_BN, NH);
                const uint32_t dK0 = desc_lo(s_base + OFF_K, 16), dQT = desc_lo(s_base + OFF_QT, 16);
                ok = __all_sync(0xffffffffu, (!a.timeout_drill || drill_wait(smem_u32(&ctl->never), abort)) &&
                                                 mbar_wait(smem_u32(&ctl->q_ready), 0, abort));
                for (int it = 0; it < n_loc && ok; ++it) {
                    const int k = it % DEC_KSTAGES, sb = it & 1;
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(smem_u32(&ctl->k_ready[k]), (uint32_t)((it / DEC_KSTAGES) & 1), abort) &&
                                        (it < 2 || mbar_wait(smem_u32(&ctl->s_free[sb]),
                                                             (uint32_t)(((it >> 1) - 1) & 1), abort)));
                    if (!ok) break;
                    tc_fence_after();
                    mma_ss_steps<0, 8, K_MAJOR_128, K_MAJOR_16, true>(tmem + sb * NH, dK0 + (uint32_t)k * TILE_DESC, dQT,
                                                                idS, 0u);
                    umma_commit_elect(smem_u32(&ctl->s_full[sb]));
                    umma_commit_elect(smem_u32(&ctl->k_empty[k]));
                }
            } else {
                const uint32_t idO = idesc_bf16_f32(HEAD_DIM, NH, 1, 0);
                const uint32_t dV0 = desc_lo(s_base + OFF_V, 2048), dPT = desc_lo(s_base + OFF_PT, 16);
                for (int it = 0; it < n_loc && ok; ++it) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(smem_u32(&ctl->p_ready[it & 1]), (uint32_t)((it >> 1) & 1), abort) &&
                                        mbar_wait(smem_u32(&ctl->v_full[it % DEC_VSTAGES]),
                                                  (uint32_t)((it / DEC_VSTAGES) & 1), abort) &&
                                        (!(has_tail && it == n_loc - 1) || mbar_wait(smem_u32(&ctl->v_tail), 0, abort)));
                    if (!ok) break;
                    tc_fence_after();
                    mma_ss_steps<0, 8, MN_MAJOR_PAGE, K_MAJOR_16, true>(tO, dV0 + (uint32_t)(it % DEC_VSTAGES) * TILE_DESC,
                                                             dPT + (uint32_t)(it & 1) * (PT_BYTES >> 4), idO,
                                                             it > 0 ? 1u : 0u);
                    umma_commit_elect(smem_u32(&ctl->pv_done[it & 1]));
                    umma_commit_elect(smem_u32(&ctl->v_empty[it % DEC_VSTAGES]));
                }
                if (ok) umma_commit_elect(smem_u32(&ctl->o_done));
            }
            if (!ok) {
                const uint64_t t0 = global_timer_ns();  // let issued MMAs drain before TMEM is released
                while (global_timer_ns() - t0 < 1000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp < WARP_SOFTMAX0) {
        // ============================================= transform WGs ====
        const int u = tid & 7, r0 = tid >> 3;  // rows r0 + XF_ROW_STEP * m
        // K copies: the thread's rows r0 + 32 m lie on page (r0 / 16) + 2 m of
        // a tile, row r0 % 16 of that page; chunk u of each 64-dim half.
        const size_t row_bytes = (size_t)a.Hkv * HEAD_DIM * 2;
        const char* ksrc = reinterpret_cast<const char*>(a.k_cache) +
                           ((size_t)(r0 & (PAGE - 1)) * a.Hkv + kvh) * (HEAD_DIM * 2) + u * 16;
        // Copy tile itx's chunks of this thread into ring slot itx % KSTAGES once
        // the score MMA of its previous tile has retired; one commit group per
        // tile (empty past the row's end), so group counts stay aligned.
        auto issue_k = [&](int itx) -> bool {
            bool ok_ = true;
            if (itx < n_loc) {
                const int kx = itx % DEC_KSTAGES;
                ok_ = mbar_wait(smem_u32(&ctl->k_empty[kx]), (uint32_t)(((itx / DEC_KSTAGES) & 1) ^ 1), abort);
                if (ok_) {
                    const uint32_t kt_s = s_base + OFF_K + kx * DEC_TILE_BYTES;
                    const int pages = pg_end - (pg_lo + itx * PPT);  // pages of the tile in the CTA's range
#pragma unroll
                    for (int m = 0; m < XF_ROWS; ++m) {
                        const int pit = (r0 >> 4) + 2 * m;
                        if (pit < pages) {
                            const int li = itx * PPT + pit;
                            const int pg = li < DEC_PGT_ENTRIES ? pgt[li] : __ldg(bt + pg_lo + li);
                            const char* src = ksrc + (size_t)pg * PAGE * row_bytes;
                            const uint32_t off = sw128_off(r0 + XF_ROW_STEP * m, u);
                            cp_async16(kt_s + off, src);
                            cp_async16(kt_s + 16384 + off, src + 128);
                        }
                    }
                }
            }
            cp_async_commit();
            return ok_;
        };
        bool kok = true;
#pragma unroll 1
        for (int e = 0; e < DEC_KAHEAD && kok; ++e) kok = issue_k(e);
        uint32_t range = 0;
        {
            // Q^T: thread (h, u) rotates chunk pair u of query head h at qpos.
            if (tid < G * 8) {
                const int h = tid >> 3, u = tid & 7;
                const uint4* row = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                                                  ((size_t)tq * a.Hq + h0 + h) * HEAD_DIM);
                __align__(16) uint8_t tmp[32];
                *reinterpret_cast<uint4*>(tmp) = __ldg(row + u);
                *reinterpret_cast<uint4*>(tmp + 16) = __ldg(row + 8 + u);
                float2 c[4], sn[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    rope_cos_sin((uint32_t)qpos, ctl->turns[8 * u + 2 * e], c[e].x, sn[e].x);
                    rope_cos_sin((uint32_t)qpos, ctl->turns[8 * u + 2 * e + 1], c[e].y, sn[e].y);
                }
                range = rotate_chunk_f16(tmp, tmp + 16, c, sn, range);
                const uint32_t off = sw128_off(h, u);
                *reinterpret_cast<uint4*>(sm + OFF_QT + off) = *reinterpret_cast<const uint4*>(tmp);
                *reinterpret_cast<uint4*>(sm + OFF_QT + 2048 + off) = *reinterpret_cast<const uint4*>(tmp + 16);
            }
            if (range_exceeded(range)) ctl->range_bad = 1;
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&ctl->q_ready));
        }
        float2 dcs[4], dsn[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 s0 = ctl->step[8 * u + 2 * e], s1 = ctl->step[8 * u + 2 * e + 1];
            dcs[e] = make_float2(s0.x, s1.x);
            dsn[e] = make_float2(s0.y, s1.y);
        }
        // (cos, sin) of the thread's current row: re-anchored exactly every
        // XF_ANCHOR_TILES tiles, advanced by the XF_ROW_STEP recurrence in between
        // (a thread's rows are XF_ROW_STEP apart and the next tile continues the
        // sequence), so at most XF_ANCHOR_TILES * XF_ROWS steps follow an anchor.
        float2 c[4], sn[4];
        for (int it = 0; it < n_loc && kok; ++it) {
            const int k = it % DEC_KSTAGES;
            cp_async_wait<DEC_KAHEAD - 1>();  // this thread's chunks of tile it have landed
            uint8_t* kt = sm + OFF_K + k * DEC_TILE_BYTES;
            const int t0 = t_begin + it * DEC_BN;
            if (it % XF_ANCHOR_TILES == 0) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    rope_cos_sin((uint32_t)(t0 + r0), ctl->turns[8 * u + 2 * e], c[e].x, sn[e].x);
                    rope_cos_sin((uint32_t)(t0 + r0), ctl->turns[8 * u + 2 * e + 1], c[e].y, sn[e].y);
                }
            }
            // all of the thread's rows are read before any is rotated (the
            // shared-memory latency is paid once per tile)
            uint4 lo[XF_ROWS], hi[XF_ROWS];
#pragma unroll
            for (int m = 0; m < XF_ROWS; ++m) {
                const uint32_t off = sw128_off(r0 + XF_ROW_STEP * m, u);
                lo[m] = *reinterpret_cast<const uint4*>(kt + off);
                hi[m] = *reinterpret_cast<const uint4*>(kt + 16384 + off);
            }
#pragma unroll
            for (int m = 0; m < XF_ROWS; ++m) {
                const int r = r0 + XF_ROW_STEP * m;
                if (t0 + r < t_end) {
                    range = rotate_regs_f16(lo[m], hi[m], c, sn, range);
                    const uint32_t off = sw128_off(r, u);
                    *reinterpret_cast<uint4*>(kt + off) = lo[m];
                    *reinterpret_cast<uint4*>(kt + 16384 + off) = hi[m];
                }
                rope_step(c, sn, dcs, dsn);
            }
            if (range_exceeded(range)) ctl->range_bad = 1;
            fence_proxy_async_smem();  // rotated rows, and copied rows left as they are
            mbar_arrive(smem_u32(&ctl->k_ready[k]));
            kok = issue_k(it + DEC_KAHEAD);
        }
        cp_async_wait_all();  // no copy may land after the CTA has left
        named_bar_sync(2, DEC_XFORM_THREADS + 128);  // transform done: the range flag is final
    } else if (warp < WARP_SOFTMAX0 + 4) {
        // =============================================== softmax WG ====
        const int t = tid - DEC_XFORM_THREADS;  // token of the tile == TMEM lane (S^T rows) == output dim (O^T rows)
        const int wq = warp & 3;
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        const float scl = a.qk_scale_log2;
        float m[8], lp[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            m[h] = -INFINITY;
            lp[h] = 0.0f;
        }
        // Every wait result is OR-reduced over the warpgroup at named barrier 1,
        // so the four warps leave the loop together and never strand one another
        // at a barrier; a thread whose wait gave up skips its work until then.
        bool ok = true, failed = false;
        for (int it = 0; it < n_loc; ++it) {
            const int sb = it & 1;
            const bool got = mbar_wait(smem_u32(&ctl->s_full[sb]), (uint32_t)((it >> 1) & 1), abort);
            if (named_bar_or(1, 128, failed || !got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[16];
            tmem_ld16(tmem + sb * NH + lane_addr, sr);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&ctl->s_free[sb]));
            const bool vis = t_begin + it * DEC_BN + t < t_end;
            float x[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                x[h] = (vis && h < G) ? __uint_as_float(sr[h]) * scl : -INFINITY;
                float v = x[h];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                if (lane == 0) ctl->red[sb][wq][h] = v;
            }
            // The four warps' maxima meet at named barrier 1.  red[] is indexed by
            // tile parity: a buffer is rewritten two tiles later, after every
            // thread has passed the next tile's barrier (and so read it).
            named_bar_sync(1, 128);
            float alpha[8];
            bool resc = false;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const float mt = fmaxf(fmaxf(ctl->red[sb][0][h], ctl->red[sb][1][h]),
                                       fmaxf(ctl->red[sb][2][h], ctl->red[sb][3][h]));
                alpha[h] = 1.0f;
                if (mt > m[h] + RESCALE_SLACK) {
                    alpha[h] = ex2(m[h] - mt);  // 0 when m = -inf
                    m[h] = mt;
                    resc = true;
                }
            }
            float p[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                p[h] = m[h] == -INFINITY ? 0.0f : ex2(x[h] - m[h]);
                lp[h] = lp[h] * alpha[h] + p[h];
            }
            // P^T buffer sb was last read by PV(i-2); a rescale of O^T needs PV(i-1)
            // retired (resc is uniform: every thread saw the same maxima).  One
            // barrier per buffer parity, so a wait never meets a phase of a later PV.
            bool w = true;
            if (it >= 2) w = mbar_wait(smem_u32(&ctl->pv_done[sb]), (uint32_t)(((it - 2) >> 1) & 1), abort);
            if (w && resc && it >= 1)
                w = mbar_wait(smem_u32(&ctl->pv_done[sb ^ 1]), (uint32_t)(((it - 1) >> 1) & 1), abort);
            if (!__all_sync(0xffffffffu, w)) {
                failed = true;  // leaves at the next barrier, together with the others
                continue;
            }
            tc_fence_after();
            if (resc && it >= 1) {
                uint32_t orow[16];
                tmem_ld16(tO + lane_addr, orow);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 8; ++h) orow[h] = __float_as_uint(__uint_as_float(orow[h]) * alpha[h]);
                tmem_st16(tO + lane_addr, orow);
                tmem_st_wait();
            }
            uint8_t* ptb = sm + OFF_PT + sb * PT_BYTES + (t >> 6) * 2048 + (t & 7) * 2;
#pragma unroll
            for (int h = 0; h < 8; ++h)
                if (h < G)
                    *reinterpret_cast<__nv_bfloat16*>(ptb + sw128_off(h, (t & 63) >> 3)) = __float2bfloat16_rn(p[h]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&ctl->p_ready[sb]));
        }
        if (ok && named_bar_or(1, 128, failed)) ok = false;
        named_bar_sync(2, DEC_XFORM_THREADS + 128);
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->o_done), 0, abort));
        // ---- epilogue: fixed-order reduction of l, out = O / l once, LSE ----
        float L[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            float v = lp[h];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) ctl->lred[wq][h] = v;
        }
        named_bar_sync(1, 128);
#pragma unroll
        for (int h = 0; h < 8; ++h) L[h] = ((ctl->lred[0][h] + ctl->lred[1][h]) + ctl->lred[2][h]) + ctl->lred[3][h];
        const bool range_bad = ctl->range_bad != 0;
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
        if (a.split_tokens > 0) {
            // split partial: O / l in FP32 and m + log2(l) (log2 domain); the
            // merge rescales and sums the splits in ascending order
            uint32_t orow[16];
            if (ok) {
                tc_fence_after();
                tmem_ld16(tO + lane_addr, orow);
                tmem_ld_wait();
            }
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                if (h < G) {
                    const size_t ph = ((size_t)b * a.Hq + h0 + h) * a.n_splits + split;
                    const float o = (!ok || range_bad || !(L[h] > 0.0f)) ? 0.0f : __uint_as_float(orow[h]) / L[h];
                    a.o_part[ph * HEAD_DIM + t] = o;
                    if (t == h)
                        a.lse_part[ph] = (!ok || range_bad) ? __int_as_float(0x7fc00000)
                                                            : (L[h] > 0.0f ? m[h] + log2f(L[h]) : -INFINITY);
                }
            }
            if (t == 0 && a.status && (!ok || range_bad)) atomicOr(a.status, ok ? RK_STATUS_RANGE : RK_STATUS_TIMEOUT);
        } else if (ok) {
            tc_fence_after();
            uint32_t orow[16];
            tmem_ld16(tO + lane_addr, orow);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                if (h < G) {
                    const float o = (range_bad || !(L[h] > 0.0f)) ? 0.0f : __uint_as_float(orow[h]) / L[h];
                    out[((size_t)tq * a.Hq + h0 + h) * HEAD_DIM + t] = __float2bfloat16_rn(o);
                }
            }
#pragma unroll
            for (int h = 0; h < 8; ++h)
                if (t == h && h < G)
                    a.lse[(size_t)tq * a.Hq + h0 + h] =
                        range_bad ? __int_as_float(0x7fc00000)
                                  : (L[h] > 0.0f ? (m[h] + log2f(L[h])) * 0.693147180559945309f : -INFINITY);
            if (range_bad && t == 0 && a.status) atomicOr(a.status, RK_STATUS_RANGE);
        } else {  // a wait gave up: the group's rows are written as failed
#pragma unroll
            for (int h = 0; h < 8; ++h)
                if (h < G) out[((size_t)tq * a.Hq + h0 + h) * HEAD_DIM + t] = __float2bfloat16_rn(0.0f);
            if (t < G) a.lse[(size_t)tq * a.Hq + h0 + t] = __int_as_float(0x7fc00000);
            if (t == 0 && a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
        }
    }

    // ---- teardown: all roles done; no MMA or TMEM access in flight ----
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Ordered merge of the split partials of one (row, query head); thread d owns
// output dim d.  With M the largest partial LSE (log2 domain), w_s =
// 2^(lse_s - M), out = sum_s w_s o_s / sum_s w_s and lse = M + log2(sum_s w_s),
// both sums taken in ascending split order.  A NaN partial (unsafe metadata,
// FP16 range, timeout) makes the row out = 0, lse = NaN; no visible key at
// all gives out = 0, lse = -inf.
__global__ void __launch_bounds__(HEAD_DIM) decode_merge_kernel(const __grid_constant__ DecodeArgs a) {
    // Launched after the split grid with programmatic stream serialization: the
    // CTAs may be resident early and wait here until that grid's partials are
    // complete and visible.
    griddep_wait();
    const size_t bh = blockIdx.x;  // b * Hq + h
    const int d = threadIdx.x;
    const int ns = a.n_splits;
    const float* lp = a.lse_part + bh * ns;
    const float* op = a.o_part + bh * ns * HEAD_DIM + d;
    // The partials are read MERGE_CHUNK splits at a time (independent loads in
    // flight), the arithmetic stays in split order.
    constexpr int MERGE_CHUNK = 16;
    float M = -INFINITY;
    bool bad = false;
    for (int s0 = 0; s0 < ns; s0 += MERGE_CHUNK) {
        float v[MERGE_CHUNK];
#pragma unroll
        for (int e = 0; e < MERGE_CHUNK; ++e) v[e] = s0 + e < ns ? lp[s0 + e] : -INFINITY;
#pragma unroll
        for (int e = 0; e < MERGE_CHUNK; ++e) {
            bad |= v[e] != v[e];
            M = fmaxf(M, v[e]);
        }
    }
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + bh * HEAD_DIM;
    if (bad || M == -INFINITY) {
        out[d] = __float2bfloat16_rn(0.0f);
        if (d == 0) a.lse[bh] = bad ? __int_as_float(0x7fc00000) : -INFINITY;
        return;
    }
    float wsum = 0.0f, acc = 0.0f;
    for (int s0 = 0; s0 < ns; s0 += MERGE_CHUNK) {
        float lv[MERGE_CHUNK], ov[MERGE_CHUNK];
#pragma unroll
        for (int e = 0; e < MERGE_CHUNK; ++e) {
            const bool in = s0 + e < ns;
            lv[e] = in ? lp[s0 + e] : 0.0f;
            ov[e] = in ? op[(size_t)(s0 + e) * HEAD_DIM] : 0.0f;
        }
#pragma unroll
        for (int e = 0; e < MERGE_CHUNK; ++e) {
            if (s0 + e < ns) {
                const float w = ex2(lv[e] - M);  // 0 for an empty split
                wsum += w;
                acc = fmaf(w, ov[e], acc);
            }
        }
    }
    out[d] = __float2bfloat16_rn(acc / wsum);
    if (d == 0) a.lse[bh] = (M + log2f(wsum)) * 0.693147180559945309f;
}

// ===================================================== balanced schedule ====
// The split-free decode on a persistent cooperative grid (rk_paged_attn_decode_balanced).
namespace bal {

constexpr int X_RING = 8;  // "transform done with a segment" barriers, by work segment modulo 8

constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + DEC_KSTAGES * DEC_TILE_BYTES;
constexpr int QT_BYTES = NH * HEAD_DIM * 2;                   // Q^T: 16 rows x 128 dims FP16
constexpr int OFF_QT = OFF_V + DEC_VSTAGES * DEC_TILE_BYTES;  // two Q^T buffers (work segment parity)
constexpr int PT_BYTES = NH * DEC_BN * 2;                     // P^T: 16 rows x 128 tokens BF16
constexpr int OFF_PT = OFF_QT + 2 * QT_BYTES;                 // two P^T buffers (tile parity)
constexpr int OFF_CTRL = OFF_PT + 2 * PT_BYTES;
constexpr int OFF_PGT = OFF_CTRL + DEC_BAL_CTRL_BYTES;         // page ids of the CTA's segments
static_assert(OFF_PGT + DEC_PGT_ENTRIES * 4 == DEC_BAL_SMEM_BYTES, "balanced decode shared memory carve");

constexpr int DEC_SEG_IMPORT = 1, DEC_SEG_EXPORT = 2;  // segment flags: state taken over / handed on
constexpr int DEC_SEG_TAIL = 4;                        // holds the row's partly filled last page

// One segment of one (row, KV head): its keys [t_begin, t_end) in n_loc tiles
// of 128 tokens from t_begin, the pages [pg_lo, pg_end) of row b's table (their
// ids at pgt[pg_off ...] as far as the shared copy reaches).
struct DecSeg {
    int b, kvh, tq;
    int t_begin, t_end, n_loc;
    int kv_len, qpos;
    int pg_lo, pg_end, pg_off;
    int flags;
    int bad;    // RK_STATUS_* bits of unsafe metadata (the row is written as failed)
    int range;  // nonzero: an input reached the FP16 range limit (set by the transform)
};

struct DecCtrl {
    uint64_t q_ready[2], q_empty[2];  // Q^T buffer by work segment parity
    uint64_t k_ready[DEC_KSTAGES], k_empty[DEC_KSTAGES];
    uint64_t v_full[DEC_VSTAGES], v_empty[DEC_VSTAGES], v_land;
    // per tile parity b: S^T buffer (s_full, s_free), P^T buffer (p_ready) and
    // the PV that read it (pv_done); a buffer is reused two tiles later, after
    // its previous phase has been observed, so a wait never meets a later phase
    uint64_t s_full[2], s_free[2], p_ready[2], pv_done[2];
    uint64_t o_done, o_free;    // O^T complete / read, by work segment
    uint64_t x_done[X_RING];    // the transform is done with a work segment (its range verdict is final)
    uint64_t never;             // nothing arrives: the timeout drill's wait
    uint32_t tmem_base;
    PipeCtl pipe;
    uint64_t turns[ROPE_PAIRS];
    float2 step[ROPE_PAIRS];  // cos/sin of an XF_ROW_STEP-position turn per pair
    float red[2][4][8];  // per-warp tile maxima, double-buffered by tile parity
    float lred[4][8];    // per-warp partial l at the end of a segment
    uint32_t epoch;      // balanced schedule: this launch's epoch (hand-off flags carry epoch + 1)
    int imp_ok;          // balanced schedule: the imported state arrived
    int n_seg;           // the CTA's segments, in processing order
    int n_pg;            // page ids in the shared copy
    int scan[DEC_THREADS / 32];
    DecSeg seg[DEC_BAL_MAX_SEGS];
};
static_assert(sizeof(DecCtrl) <= DEC_BAL_CTRL_BYTES, "decode control block exceeds its reservation");

__device__ __forceinline__ bool seg_work(const DecSeg& s) {
    return !s.bad && s.n_loc > 0;
}

// out = 0 and lse = lse_val for the G heads of a segment's (row, KV head), by
// the nt threads t = 0 .. nt - 1.  (Cold paths such as this one are kept out
// of line, away from the hot loops' instructions.)
__device__ __noinline__ void write_empty_row(const DecodeArgs& a, const DecSeg& s, float lse_val, int t, int nt) {
    const int h0 = s.kvh * a.G;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    for (int i = t; i < a.G * HEAD_DIM; i += nt) {
        const int hh = i / HEAD_DIM, d = i % HEAD_DIM;
        out[((size_t)s.b * a.Hq + h0 + hh) * HEAD_DIM + d] = __float2bfloat16_rn(0.0f);
    }
    if (t < a.G) a.lse[(size_t)s.b * a.Hq + h0 + t] = lse_val;
}

// ------------------------------------------------ balanced schedule ----
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until a hand-off flag holds `want`, within the launch's wait limit (then
// the CTA's pipeline is aborted and 0 returned).
__device__ __forceinline__ int bal_wait(const uint32_t* flag, uint32_t want, PipeCtl* pc) {
    if (ld_acquire_u32(flag) == want) return 1;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        __nanosleep(256);
        if (ld_acquire_u32(flag) == want) return 1;
        if (pipe_aborted(pc)) return 0;
        if (global_timer_ns() - t0 > pc->limit_ns) {
            *reinterpret_cast<volatile int*>(&pc->abort) = 1;
            return 0;
        }
    }
}

// A segment that hands its row on but could not compute it: the hand-off says
// so, and the segment that ends the row writes it as failed.  One thread.
__device__ __noinline__ void export_failed(const DecodeArgs& a, uint32_t epoch) {
    float* st = a.bal_state + (size_t)blockIdx.x * DEC_BAL_STATE_FLOATS;
    __stcg(st + DEC_BAL_INFO, 0.0f);
    __threadfence();
    st_release_u32(a.bal_sync + DEC_BAL_SYNC_WORDS + blockIdx.x, epoch + 1u);
}

// Called once by every CTA of a balanced launch as it leaves: the last one
// resets the count and advances the epoch, so the next launch's flags (epoch
// + 1 then) never match a flag this launch left.
__device__ __forceinline__ void bal_done(const DecodeArgs& a) {
    __threadfence();
    if (atomicAdd(a.bal_sync + 1, 1u) == (uint32_t)gridDim.x - 1u) {
        *reinterpret_cast<volatile uint32_t*>(a.bal_sync + 1) = 0u;
        __threadfence();
        atomicAdd(a.bal_sync, 1u);
    }
}

// This CTA's segments.  The grid is Hkv chains of grid / Hkv CTAs: CTA c
// serves KV head h = c % Hkv as member g = c / Hkv of its chain.  Every row gets
// max(1, ceil(tiles / bt)) blocks (the tiles of its visible keys, bt to a
// block), laid end to end in row order; member g takes blocks [g L, (g + 1) L),
// L = ceil(total / members), of head h.  bt is the coarsest power of two, from
// the host's finest (whose worst case keeps a CTA's segment list within
// DEC_BAL_MAX_SEGS) up to DEC_BAL_MAX_BLOCK_TILES, that still leaves the last
// member a block.  All heads of a row have the same blocks,
// so the Hkv CTAs of a member index read the same pages (the heads share them)
// at the same time.  A row cut at g L is taken over from member g - 1 (import,
// done last: by then that CTA has handed it on, having done it first); a row
// cut at (g + 1) L is handed to member g + 1 (export, done first).  The rows'
// block counts use the K ring as scratch (it is not in use yet).
__device__ __noinline__ void bal_schedule(const DecodeArgs& a, uint8_t* sm, DecCtrl* ctl) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int* nbs = reinterpret_cast<int*>(sm + OFF_K);  // blocks of row b
    int* pre = nbs + DEC_BAL_MAX_ROWS;               // blocks of the rows before b
    static_assert(2 * DEC_BAL_MAX_ROWS * 4 <= DEC_KSTAGES * DEC_TILE_BYTES, "set-up scratch exceeds the K ring");
    const int B = a.B <= DEC_BAL_MAX_ROWS ? a.B : 0;  // more rows are ruled out by the host; none taken here
    // The finest block the host allows (its worst-case bound on a CTA's
    // segments), and the coarsest power of two from there up to
    // DEC_BAL_MAX_BLOCK_TILES that still gives every member of a chain work
    // (finer cuts only pay while some member would otherwise sit idle).
    const int bt_min = (a.bal_block_tiles >= 1 && a.bal_block_tiles <= DEC_BAL_MAX_BLOCK_TILES)
                           ? a.bal_block_tiles
                           : DEC_BAL_MAX_BLOCK_TILES;
    const int per = (B + DEC_THREADS - 1) / DEC_THREADS;  // contiguous rows per thread
    const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
    // the previous launch's last CTA advanced the epoch in L2 (its load overlaps the rows')
    if (tid == DEC_THREADS - 1) ctl->epoch = __ldcg(a.bal_sync);
    int cnt[4] = {0, 0, 0, 0};  // blocks of the thread's rows at 1, 2, 4, 8 tiles a block
    for (int r = r0; r < r1; ++r) {
        const int kv = a.kv_lens[r], qp = a.position_ids[r];
        const int nv = (kv < 0 || kv > a.W * PAGE || qp < 0) ? 0 : (qp >= kv ? kv : qp + 1);
        const int nt = (nv + DEC_BN - 1) / DEC_BN;
        nbs[r] = nt;
#pragma unroll
        for (int k = 0; k < 4; ++k) cnt[k] += max(1, (nt + (1 << k) - 1) >> k);
    }
    int* wsum = reinterpret_cast<int*>(sm + OFF_V);  // [warp][4]; the V stages are zeroed afterwards
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int v = __reduce_add_sync(0xffffffffu, cnt[k]);
        if (lane == 0) wsum[warp * 4 + k] = v;
    }
    __syncthreads();
    int bt = bt_min;
    {
        // the four totals, summed over the warps by the lanes of every warp
        static_assert(DEC_THREADS / 32 <= 32, "one lane per warp partial");
        int tot[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) tot[k] = __reduce_add_sync(0xffffffffu, lane < DEC_THREADS / 32 ? wsum[lane * 4 + k] : 0);
        const int members = (int)gridDim.x / a.Hkv;
#pragma unroll
        for (int k = 3; k >= 0; --k) {
            const long long T = tot[k];
            const long long L = members > 0 ? (T + members - 1) / members : 0;
            if ((1 << k) >= bt_min && members > 0 && (long long)(members - 1) * L < T) {  // the last member gets a block
                bt = 1 << k;
                break;
            }
        }
    }
    int sum = 0;
    for (int r = r0; r < r1; ++r) {
        const int nb = max(1, (nbs[r] + bt - 1) / bt);
        nbs[r] = nb;
        sum += nb;
    }
    int inc = sum;  // inclusive scan over the warp, then over the warps
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += v;
    }
    if (lane == 31) ctl->scan[warp] = inc;
    __syncthreads();
    int wbase = 0, total = 0;
#pragma unroll 1
    for (int w = 0; w < DEC_THREADS / 32; ++w) {
        const int v = ctl->scan[w];
        if (w < warp) wbase += v;
        total += v;
    }
    int base = wbase + inc - sum;
    for (int r = r0; r < r1; ++r) {
        pre[r] = base;
        base += nbs[r];
    }
    __syncthreads();
    if (tid == 0) {
        const int Hkv = a.Hkv, members = (int)gridDim.x / Hkv;
        const int h = (int)blockIdx.x % Hkv, g = (int)blockIdx.x / Hkv;
        const long long T = total;
        const long long L = members > 0 ? (T + members - 1) / members : 0;
        const long long lo = g < members ? (long long)g * L : T, hi = min(T, lo + L);
        // the segments in row order, in shared memory (a local array would go
        // through local memory on every access); the V stages are zeroed afterwards
        int(*sg)[4] = reinterpret_cast<int(*)[4]>(sm + OFF_V + 1024);
        int n = 0;
        if (B != a.B && blockIdx.x == 0 && a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
        if (lo < hi) {
            int bl = 0, bh = B - 1;  // the last row b with pre[b] <= lo
            while (bl < bh) {
                const int mid = (bl + bh + 1) >> 1;
                if ((long long)pre[mid] <= lo) bl = mid; else bh = mid - 1;
            }
            int b = bl;
            long long P = pre[b];  // first block of row b
            while (P < hi && n < DEC_BAL_MAX_SEGS) {
                const int nb = nbs[b];
                const long long blo = P > lo ? P : lo, bhi = P + nb < hi ? P + nb : hi;
                sg[n][0] = b * Hkv + h;
                sg[n][1] = (int)(blo - P) * bt;
                sg[n][2] = (int)(bhi - P) * bt;
                sg[n][3] = (P < lo ? DEC_SEG_IMPORT : 0) | (P + nb > hi ? DEC_SEG_EXPORT : 0);
                ++n;
                P += nb;
                ++b;
            }
            if (P < hi) {  // more segments than a CTA holds: ruled out by the host; reported, not computed
                n = 0;
                if (a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
            }
        }
        // processing order: the one handed on, the whole ones, the one taken over
        int k = 0;
        const bool ex_last = n > 1 && (sg[n - 1][3] & DEC_SEG_EXPORT);
        const bool im_first = n > 1 && (sg[0][3] & DEC_SEG_IMPORT);
        auto put = [&](int i) {
            DecSeg& d = ctl->seg[k++];
            d.b = sg[i][0] / a.Hkv;
            d.kvh = sg[i][0] % a.Hkv;
            d.t_begin = sg[i][1] * DEC_BN;
            d.t_end = sg[i][2] * DEC_BN;  // a cap until the row's visible keys are known
            d.flags = sg[i][3];
        };
        if (ex_last) put(n - 1);
        for (int i = 0; i < n; ++i)
            if (!(i == n - 1 && ex_last) && !(i == 0 && im_first)) put(i);
        if (im_first) put(0);
        ctl->n_seg = n;
    }
    __syncthreads();
}


// The CTA's segments (the balanced schedule), their metadata checks and their
// page ids, once.  Every page id a segment may read is loaded in the same round
// trip as the row's length and position and judged against the visible range
// afterwards.
__device__ __noinline__ void dec_setup(const DecodeArgs& a, uint8_t* sm, DecCtrl* ctl) {
    const int tid = threadIdx.x;
    bal_schedule(a, sm, ctl);  // ends with __syncthreads
    const int n_seg = ctl->n_seg;
    if (tid == 0) {  // where each segment's page ids go in the shared copy
        int off = 0;
        for (int s = 0; s < n_seg; ++s) {
            DecSeg& d = ctl->seg[s];
            d.pg_lo = d.t_begin / PAGE;
            d.pg_off = off;
            off += max(0, min(a.W, d.t_end / PAGE) - d.pg_lo);
        }
        ctl->n_pg = off;
    }
    __syncthreads();
    // one round trip: thread s reads segment s's row metadata, every thread up
    // to PRE page ids of the concatenated ranges
    constexpr int PRE = DEC_PGT_ENTRIES / DEC_THREADS;
    int kvl = 0, qp = 0;
    if (tid < n_seg) {
        const DecSeg& d = ctl->seg[tid];
        kvl = a.kv_lens[d.b];
        qp = a.position_ids[d.b];
    }
    const int n_pg = ctl->n_pg;
    int pre[PRE], pre_s[PRE];
    int s = 0;  // the segment of entry j (entries ascend with e, so the scan resumes)
#pragma unroll
    for (int e = 0; e < PRE; ++e) {
        const int j = tid + e * DEC_THREADS;
        pre[e] = 0;
        pre_s[e] = -1;
        if (j < n_pg) {
            while (s + 1 < n_seg && ctl->seg[s + 1].pg_off <= j) ++s;
            const DecSeg& d = ctl->seg[s];
            pre_s[e] = s;
            pre[e] = __ldg(a.block_table + (size_t)d.b * a.W + d.pg_lo + (j - d.pg_off));
        }
    }
    if (tid < n_seg) {
        DecSeg& d = ctl->seg[tid];
        int bad = 0;
        const int tq = d.b;
        if (kvl < 0 || kvl > a.W * PAGE) bad |= RK_STATUS_KVLEN;
        if (qp < 0) bad |= RK_STATUS_POSITION;
        const int n_vis = bad ? 0 : (qp >= kvl ? kvl : qp + 1);
        d.tq = tq;
        d.kv_len = kvl;
        d.qpos = qp;
        d.t_end = min(n_vis, d.t_end);
        d.n_loc = d.t_end > d.t_begin ? (d.t_end - d.t_begin + DEC_BN - 1) / DEC_BN : 0;
        d.pg_end = (d.t_end + PAGE - 1) / PAGE;
        // last page partly filled and inside the visible range: its rows past
        // kv_len hold arbitrary bits and are zeroed in V after the copy lands
        if (!bad && n_vis == kvl && (kvl & (PAGE - 1)) != 0 && d.n_loc > 0 && d.t_end == n_vis)
            d.flags |= DEC_SEG_TAIL;
        d.bad = bad;
        d.range = 0;
    }
    __syncthreads();
    int32_t* pgt = reinterpret_cast<int32_t*>(sm + OFF_PGT);
#pragma unroll
    for (int e = 0; e < PRE; ++e) {
        const int j = tid + e * DEC_THREADS;
        if (pre_s[e] >= 0) {
            pgt[j] = pre[e];
            DecSeg& d = ctl->seg[pre_s[e]];
            if (d.pg_lo + (j - d.pg_off) < d.pg_end && (pre[e] < 0 || pre[e] >= a.num_pages))
                atomicOr(&d.bad, RK_STATUS_PAGE_OOB);
        }
    }
    // very wide rows (one segment): the ids past the shared copy are checked here
    // and read from the table by the loaders
    for (int s = 0; s < n_seg; ++s) {
        DecSeg& d = ctl->seg[s];
        for (int i = d.pg_lo + max(0, DEC_PGT_ENTRIES - d.pg_off) + tid; i < d.pg_end; i += DEC_THREADS) {
            const int pg = __ldg(a.block_table + (size_t)d.b * a.W + i);
            if (pg < 0 || pg >= a.num_pages) atomicOr(&d.bad, RK_STATUS_PAGE_OOB);
        }
    }
    if (tid == 0) {
        ctl->pipe.abort = 0;
        ctl->pipe.limit_ns = wait_limit(a.wait_limit_ns);
        mbar_init(smem_u32(&ctl->never), 1);
        for (int k = 0; k < 2; ++k) {
            mbar_init(smem_u32(&ctl->q_ready[k]), DEC_XFORM_THREADS);
            mbar_init(smem_u32(&ctl->q_empty[k]), 1);
            mbar_init(smem_u32(&ctl->s_full[k]), 1);
            mbar_init(smem_u32(&ctl->s_free[k]), 128);
            mbar_init(smem_u32(&ctl->p_ready[k]), 128);
            mbar_init(smem_u32(&ctl->pv_done[k]), 1);
        }
        for (int k = 0; k < DEC_KSTAGES; ++k) {
            mbar_init(smem_u32(&ctl->k_ready[k]), DEC_XFORM_THREADS);
            mbar_init(smem_u32(&ctl->k_empty[k]), 1);
        }
        for (int k = 0; k < DEC_VSTAGES; ++k) {
            mbar_init(smem_u32(&ctl->v_full[k]), 1);
            mbar_init(smem_u32(&ctl->v_empty[k]), 1);
        }
        mbar_init(smem_u32(&ctl->v_land), 1);
        mbar_init(smem_u32(&ctl->o_done), 1);
        mbar_init(smem_u32(&ctl->o_free), 128);
        for (int k = 0; k < X_RING; ++k) mbar_init(smem_u32(&ctl->x_done[k]), DEC_XFORM_THREADS);
        fence_mbar_init();
    }
    if (tid < ROPE_PAIRS) {
        ctl->turns[tid] = a.rope_turns[tid];
        float c, s;
        rope_cos_sin((uint32_t)XF_ROW_STEP, a.rope_turns[tid], c, s);
        ctl->step[tid] = make_float2(c, s);
    }
    // V stages, Q^T and P^T start as zeros (rows never written stay finite).
    for (int i = tid; i < (OFF_CTRL - OFF_V) / 16; i += DEC_THREADS)
        reinterpret_cast<uint4*>(sm + OFF_V)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    __syncthreads();
}

// Exact (cos, sin) of the 8 pairs of chunk u at position t (a RoPE anchor), out
// of line: it runs once every XF_ANCHOR_TILES tiles.
struct Angles {
    float2 c[4], s[4];
};
__device__ __noinline__ Angles anchor_angles(const DecCtrl* ctl, uint32_t t, int u) {
    Angles r;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        rope_cos_sin(t, ctl->turns[8 * u + 2 * e], r.c[e].x, r.s[e].x);
        rope_cos_sin(t, ctl->turns[8 * u + 2 * e + 1], r.c[e].y, r.s[e].y);
    }
    return r;
}

// Angles of row r0 of tile ta: exact at the last anchor tile, then the row
// steps of the tiles since (none when ta is an anchor tile).
__device__ __noinline__ Angles anchor_replay(const DecCtrl* ctl, int ta, int r0, int u) {
    const int tz = ta - ta % XF_ANCHOR_TILES;
    Angles an = anchor_angles(ctl, (uint32_t)(tz * DEC_BN + r0), u);
    float2 dcs[4], dsn[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 s0 = ctl->step[8 * u + 2 * e], s1 = ctl->step[8 * u + 2 * e + 1];
        dcs[e] = make_float2(s0.x, s1.x);
        dsn[e] = make_float2(s0.y, s1.y);
    }
#pragma unroll 1
    for (int q = 0; q < (ta - tz) * XF_ROWS; ++q) rope_step(an.c, an.s, dcs, dsn);
    return an;
}

// Q^T of a segment (thread (h, u) rotates chunk pair u of query head h at the
// row's position) into one of the two Q^T buffers; returns the thread's range
// bits.  Out of line: once per segment.
__device__ __noinline__ uint32_t rotate_q(const DecodeArgs& a, const DecCtrl* ctl, uint8_t* qt, int tq, int kvh,
                                          int qpos, int tid) {
    uint32_t range = 0;
    if (tid < a.G * 8) {
        const int h = tid >> 3, uq = tid & 7;
        const uint4* row = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                                          ((size_t)tq * a.Hq + kvh * a.G + h) * HEAD_DIM);
        __align__(16) uint8_t tmp[32];
        *reinterpret_cast<uint4*>(tmp) = __ldg(row + uq);
        *reinterpret_cast<uint4*>(tmp + 16) = __ldg(row + 8 + uq);
        const Angles an = anchor_angles(ctl, (uint32_t)qpos, uq);
        range = rotate_chunk_f16(tmp, tmp + 16, an.c, an.s, range);
        const uint32_t off = sw128_off(h, uq);
        *reinterpret_cast<uint4*>(qt + off) = *reinterpret_cast<const uint4*>(tmp);
        *reinterpret_cast<uint4*>(qt + 2048 + off) = *reinterpret_cast<const uint4*>(tmp + 16);
    }
    return range;
}

// Running softmax state of one token lane: per head the running max and this
// lane's partial sum of l.
struct LaneState {
    float m[8], lp[8];
};

// Take over a row from the previous CTA of the chain: its running state, and its
// O^T row for this output dim into TMEM.  Returns 0 (state taken), 1 (the row
// failed before: reported there) or 2 (the hand-off never came: the wait gave
// up).  The caller has set st to -inf / 0 beforehand.  Out of line (once per
// segment); the 128 softmax threads call it together (named barrier 1).
__device__ __noinline__ int import_state(const DecodeArgs& a, DecCtrl* ctl, PipeCtl* abort, LaneState& st, int t,
                                         uint32_t taddr, int s) {
    if (t == 0) ctl->imp_ok = bal_wait(a.bal_sync + DEC_BAL_SYNC_WORDS + (blockIdx.x - a.Hkv), ctl->epoch + 1u, abort);
    named_bar_sync(1, 128);
    const bool arrived = ctl->imp_ok != 0;
    const float* src = a.bal_state + (size_t)(blockIdx.x - a.Hkv) * DEC_BAL_STATE_FLOATS;
    if (arrived) (void)ld_acquire_u32(a.bal_sync + DEC_BAL_SYNC_WORDS + (blockIdx.x - a.Hkv));
    if (!arrived) return 2;
    if (__ldcg(src + DEC_BAL_INFO) == 0.0f) return 1;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        st.m[h] = __ldcg(src + DEC_BAL_M + h);
        st.lp[h] = __ldcg(src + DEC_BAL_LP + t * 8 + h);
    }
    uint32_t orow[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) orow[c] = __float_as_uint(__ldcg(src + DEC_BAL_O + t * 16 + c));
    tc_fence_after();
    tmem_st16(taddr, orow);
    tmem_st_wait();
    if (t == 0 && __ldcg(src + DEC_BAL_INFO + 1) != 0.0f) atomicOr(&ctl->seg[s].range, 1);
    return 0;
}

// Hand the running state to the next CTA of the chain, which goes on with the
// row.  The 128 softmax threads call it together (named barrier 1).
__device__ __noinline__ void export_state(const DecodeArgs& a, const DecCtrl* ctl, const LaneState& st,
                                          const uint32_t (&orow)[16], bool ok, bool range_bad, int t) {
    float* dst = a.bal_state + (size_t)blockIdx.x * DEC_BAL_STATE_FLOATS;
#pragma unroll
    for (int h = 0; h < 8; ++h) __stcg(dst + DEC_BAL_LP + t * 8 + h, st.lp[h]);
#pragma unroll
    for (int c = 0; c < 16; ++c) __stcg(dst + DEC_BAL_O + t * 16 + c, __uint_as_float(orow[c]));
    if (t == 0) {
#pragma unroll
        for (int h = 0; h < 8; ++h) __stcg(dst + DEC_BAL_M + h, st.m[h]);
        __stcg(dst + DEC_BAL_INFO, ok ? 1.0f : 0.0f);
        __stcg(dst + DEC_BAL_INFO + 1, range_bad ? 1.0f : 0.0f);
    }
    __threadfence();
    named_bar_sync(1, 128);
    if (t == 0) st_release_u32(a.bal_sync + DEC_BAL_SYNC_WORDS + blockIdx.x, ctl->epoch + 1u);
}

// Page id li (from the segment's first page) of a segment.
__device__ __forceinline__ int seg_page(const DecodeArgs& a, const int32_t* pgt, const DecSeg& d, int li) {
    const int j = d.pg_off + li;
    return j < DEC_PGT_ENTRIES ? pgt[j] : __ldg(a.block_table + (size_t)d.b * a.W + d.pg_lo + li);
}

__global__ void __launch_bounds__(DEC_THREADS, 1)
    decode_bal_kernel(const __grid_constant__ CUtensorMap vmap, const __grid_constant__ DecodeArgs a) {
    extern __shared__ __align__(1024) uint8_t sm[];
    DecCtrl* ctl = reinterpret_cast<DecCtrl*>(sm + OFF_CTRL);
    const uint32_t s_base = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.G;
    if (s_base & 1023u) {  // the swizzled operand layout needs a 1024-byte aligned base
        // nothing computed: the status bit reports it, and the rows this CTA
        // would have handed on fail the other CTAs' bounded waits
        if (tid == 0 && a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
        if (tid == 0) bal_done(a);
        return;
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    dec_setup(a, sm, ctl);  // ends with __syncthreads
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const uint32_t tO = tmem + 32;
    PipeCtl* abort = &ctl->pipe;
    const int n_seg = ctl->n_seg;
    const int32_t* pgt = reinterpret_cast<const int32_t*>(sm + OFF_PGT);
    constexpr int PPT = DEC_BN / PAGE;  // pages per tile

    if (warp == WARP_TMA_K) {
        // K arrives through the transform threads' own copies: nothing to do.
    } else if (warp == WARP_TMA_V) {
        // ============================================ V producer (TMA) ====
        // g: the CTA's tile count over its segments (stages, phases).  Pages a
        // partial tile does not load keep what the stage held: another segment's
        // rows are replaced by zeros first (every row a tile's PV reads is this
        // row's or zero).
        if (lane == 0) prefetch_tmap(&vmap);
        int g = 0, nl = 0;
        bool ok = true, land_open = false;
        int owner[DEC_VSTAGES];
#pragma unroll
        for (int k = 0; k < DEC_VSTAGES; ++k) owner[k] = -1;
        for (int s = 0; s < n_seg && ok; ++s) {
            const DecSeg d = ctl->seg[s];  // a register copy: the loops below store to shared memory
            if (!seg_work(d)) continue;
            for (int it = 0; it < d.n_loc; ++it, ++g) {
                const int k = g % DEC_VSTAGES;
                const uint32_t use = (uint32_t)(g / DEC_VSTAGES);
                const int np = min(PPT, d.pg_end - (d.pg_lo + it * PPT));
                const int pg = lane < np ? seg_page(a, pgt, d, it * PPT + lane) : 0;
                const uint32_t fb = smem_u32(&ctl->v_full[k]);
                int good = 1;
                if (lane == 0) good = mbar_wait(smem_u32(&ctl->v_empty[k]), (use & 1u) ^ 1u, abort);
                if (!(ok = __shfl_sync(0xffffffffu, good, 0) != 0)) break;
                uint8_t* vt = sm + OFF_V + k * DEC_TILE_BYTES;
                int own = 0;
#pragma unroll
                for (int q = 0; q < DEC_VSTAGES; ++q)
                    if (q == k) {
                        own = owner[q];
                        owner[q] = s;
                    }
                if (np < PPT && own != s) {
                    for (int idx = np * 256 + lane; idx < PPT * 256; idx += 32)
                        reinterpret_cast<uint4*>(vt)[idx] = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                // The row's last tile lands on v_land; its rows past kv_len are
                // zeroed and only then is v_full completed (one plain arrival).
                const bool tail = (d.flags & DEC_SEG_TAIL) && it == d.n_loc - 1;
                const uint32_t lb = tail ? smem_u32(&ctl->v_land) : fb;
                if (lane == 0) mbar_arrive_expect_tx(lb, (uint32_t)np * 4096);
                __syncwarp();
                // one 4 KiB box per page: [page][half][16 rows][128 B]
                if (lane < np)
                    tma_load_4d(s_base + OFF_V + k * DEC_TILE_BYTES + lane * 4096, &vmap, lb, 0, pg * PAGE, 0, d.kvh);
                __syncwarp();
                if (tail) {
                    // this warp is v_land's only waiter and waits each phase it armed
                    const int landed =
                        __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(lb, (uint32_t)(nl & 1), abort) : 0, 0);
                    ++nl;
                    if (!landed) {
                        land_open = true;
                        ok = false;
                        break;
                    }
                    const int tl = d.kv_len - (d.t_begin + it * DEC_BN);
                    const int r_end = min(DEC_BN, (tl + PAGE - 1) & ~(PAGE - 1));
                    for (int idx = lane; idx < (r_end - tl) * 16; idx += 32) {
                        const int rr = tl + (idx >> 4), ch = idx & 15;
                        *reinterpret_cast<uint4*>(vt + (rr >> 4) * 4096 + (ch >> 3) * 2048 + (rr & 15) * 128 +
                                                  (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(fb);
                }
            }
        }
        if (lane == 0 && pipe_aborted(abort)) {
            // the copies this warp issued land before the CTA's shared memory is released
            if (land_open) mbar_wait_drain(smem_u32(&ctl->v_land), (uint32_t)((nl - 1) & 1));
            for (int i = max(0, g - DEC_VSTAGES); i < g; ++i)
                mbar_wait_drain(smem_u32(&ctl->v_full[i % DEC_VSTAGES]), (uint32_t)((i / DEC_VSTAGES) & 1));
        }
    } else if (warp == WARP_MMA || warp == WARP_PV) {
        // ============================================ MMA issuers ====
        // Two issuing threads: warp 13 issues the score MMAs, warp 15 the PV
        // MMAs, each waiting only for its own inputs, so the barrier checks of
        // one overlap the MMAs of the other.  tcgen05.commit covers the MMAs of
        // the committing thread, which is what each completion barrier tracks.
        // Each issuer's whole warp runs its loop (converged, warp-uniform
        // operands); elect.sync picks the lane that issues MMAs and commits.
        constexpr uint32_t TILE_DESC = DEC_TILE_BYTES >> 4;  // one 32 KiB tile in descriptor address units
        bool ok = true;
        int g = 0;
        if (warp == WARP_MMA) {
            const uint32_t idS = idesc_f16_f32(DEC_BN, NH);
            const uint32_t dK0 = desc_lo(s_base + OFF_K, 16), dQT0 = desc_lo(s_base + OFF_QT, 16);
            ok = __all_sync(0xffffffffu, !a.timeout_drill || drill_wait(smem_u32(&ctl->never), abort));
            int ws = 0;  // work segments so far (Q^T buffer ws & 1)
            for (int s = 0; s < n_seg && ok; ++s) {
                const DecSeg d = ctl->seg[s];  // a register copy: the loops below store to shared memory
                if (!seg_work(d)) continue;
                if (!(ok = __all_sync(0xffffffffu,
                                      mbar_wait(smem_u32(&ctl->q_ready[ws & 1]), (uint32_t)((ws >> 1) & 1), abort))))
                    break;
                const uint32_t dQT = dQT0 + (uint32_t)(ws & 1) * (QT_BYTES >> 4);
                for (int it = 0; it < d.n_loc && ok; ++it, ++g) {
                    const int k = g % DEC_KSTAGES, sb = g & 1;
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(smem_u32(&ctl->k_ready[k]), (uint32_t)((g / DEC_KSTAGES) & 1), abort) &&
                                        (g < 2 || mbar_wait(smem_u32(&ctl->s_free[sb]),
                                                            (uint32_t)(((g >> 1) - 1) & 1), abort)));
                    if (!ok) break;
                    tc_fence_after();
                    mma_ss_steps<0, 8, K_MAJOR_128, K_MAJOR_16, true>(tmem + sb * NH, dK0 + (uint32_t)k * TILE_DESC, dQT,
                                                                idS, 0u);
                    umma_commit_elect(smem_u32(&ctl->s_full[sb]));
                    umma_commit_elect(smem_u32(&ctl->k_empty[k]));
                }
                if (!ok) break;
                umma_commit_elect(smem_u32(&ctl->q_empty[ws & 1]));  // the segment's score MMAs have read Q^T
                ++ws;
            }
            // every commit of this thread has arrived before the CTA leaves
            for (int i = max(0, g - DEC_KSTAGES); i < g && ok; ++i)
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->k_empty[i % DEC_KSTAGES]),
                                                       (uint32_t)((i / DEC_KSTAGES) & 1), abort));
            if (ok && ws > 0)
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->q_empty[(ws - 1) & 1]),
                                                       (uint32_t)(((ws - 1) >> 1) & 1), abort));
        } else {
            const uint32_t idO = idesc_bf16_f32(HEAD_DIM, NH, 1, 0);
            const uint32_t dV0 = desc_lo(s_base + OFF_V, 2048), dPT = desc_lo(s_base + OFF_PT, 16);
            int ws = 0;
            for (int s = 0; s < n_seg && ok; ++s) {
                const DecSeg d = ctl->seg[s];  // a register copy: the loops below store to shared memory
                if (!seg_work(d)) continue;
                const bool imp = (d.flags & DEC_SEG_IMPORT) != 0;
                // the previous work segment's epilogue has read O^T
                if (ws > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->o_free),
                                                                       (uint32_t)((ws - 1) & 1), abort))))
                    break;
                for (int it = 0; it < d.n_loc && ok; ++it, ++g) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(smem_u32(&ctl->p_ready[g & 1]), (uint32_t)((g >> 1) & 1), abort) &&
                                        mbar_wait(smem_u32(&ctl->v_full[g % DEC_VSTAGES]),
                                                  (uint32_t)((g / DEC_VSTAGES) & 1), abort));
                    if (!ok) break;
                    tc_fence_after();
                    mma_ss_steps<0, 8, MN_MAJOR_PAGE, K_MAJOR_16, true>(tO, dV0 + (uint32_t)(g % DEC_VSTAGES) * TILE_DESC,
                                                             dPT + (uint32_t)(g & 1) * (PT_BYTES >> 4), idO,
                                                             (it > 0 || imp) ? 1u : 0u);
                    umma_commit_elect(smem_u32(&ctl->pv_done[g & 1]));
                    umma_commit_elect(smem_u32(&ctl->v_empty[g % DEC_VSTAGES]));
                }
                if (!ok) break;
                umma_commit_elect(smem_u32(&ctl->o_done));
                ++ws;
            }
            for (int i = max(0, g - DEC_VSTAGES); i < g && ok; ++i)
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->v_empty[i % DEC_VSTAGES]),
                                                       (uint32_t)((i / DEC_VSTAGES) & 1), abort));
            for (int i = max(0, g - 2); i < g && ok; ++i)
                ok = __all_sync(0xffffffffu,
                                mbar_wait(smem_u32(&ctl->pv_done[i & 1]), (uint32_t)((i >> 1) & 1), abort));
        }
        if (!ok) {
            const uint64_t t0 = global_timer_ns();  // let issued MMAs drain before TMEM is released
            while (global_timer_ns() - t0 < 1000000ull) {
            }
        }
        __syncwarp();
    } else if (warp < WARP_SOFTMAX0) {
        // ============================================= transform WGs ====
        const int u = tid & 7, r0 = tid >> 3;  // rows r0 + XF_ROW_STEP * m
        // K copies: the thread's rows r0 + 32 m lie on page (r0 / 16) + 2 m of
        // a tile, row r0 % 16 of that page; chunk u of each 64-dim half.
        const size_t row_bytes = (size_t)a.Hkv * HEAD_DIM * 2;
        const char* kbase = reinterpret_cast<const char*>(a.k_cache) + (size_t)(r0 & (PAGE - 1)) * row_bytes + u * 16;
        // Copies run DEC_KAHEAD tiles ahead of the rotation, across segment
        // boundaries: (cs, cit) is the next tile to copy, gx its CTA tile count.
        // Each copy waits for its ring slot (the score MMA of the tile before it
        // there has retired); one commit group per tile (empty past the last),
        // so group counts stay aligned.
        int cs = 0, cit = 0, gx = 0;
        while (cs < n_seg && !seg_work(ctl->seg[cs])) ++cs;
        auto issue_k = [&]() -> bool {
            bool ok_ = true;
            if (cs < n_seg) {
                const DecSeg& d = ctl->seg[cs];  // read once per tile; few registers held across the loop
                const int kx = gx % DEC_KSTAGES;
                ok_ = mbar_wait(smem_u32(&ctl->k_empty[kx]), (uint32_t)(((gx / DEC_KSTAGES) & 1) ^ 1), abort);
                if (ok_) {
                    const uint32_t kt_s = s_base + OFF_K + kx * DEC_TILE_BYTES;
                    const int pages = d.pg_end - (d.pg_lo + cit * PPT);  // pages of the tile in the segment
                    const char* ksrc = kbase + (size_t)d.kvh * (HEAD_DIM * 2);
#pragma unroll
                    for (int m = 0; m < XF_ROWS; ++m) {
                        const int pit = (r0 >> 4) + 2 * m;
                        if (pit < pages) {
                            const int pg = seg_page(a, pgt, d, cit * PPT + pit);
                            const char* src = ksrc + (size_t)pg * PAGE * row_bytes;
                            const uint32_t off = sw128_off(r0 + XF_ROW_STEP * m, u);
                            cp_async16(kt_s + off, src);
                            cp_async16(kt_s + 16384 + off, src + 128);
                        }
                    }
                    ++gx;
                    if (++cit == d.n_loc) {
                        cit = 0;
                        do ++cs;
                        while (cs < n_seg && !seg_work(ctl->seg[cs]));
                    }
                }
            }
            cp_async_commit();
            return ok_;
        };
        bool kok = true;
#pragma unroll 1
        for (int e = 0; e < DEC_KAHEAD && kok; ++e) kok = issue_k();
        float2 dcs[4], dsn[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 s0 = ctl->step[8 * u + 2 * e], s1 = ctl->step[8 * u + 2 * e + 1];
            dcs[e] = make_float2(s0.x, s1.x);
            dsn[e] = make_float2(s0.y, s1.y);
        }
        int ws = 0;     // work segments so far
        int gcons = 0;  // the CTA tile count of the tile being rotated
        for (int s = 0; s < n_seg && kok; ++s) {
            if (!seg_work(ctl->seg[s])) continue;
            // the fields the rotation loop uses, in registers (the loop stores to
            // shared memory, so references into it would be read again and again)
            const int t_begin = ctl->seg[s].t_begin, t_end = ctl->seg[s].t_end, n_loc = ctl->seg[s].n_loc;
            uint32_t range = 0;
            {
                // Q^T into buffer ws & 1 once the score MMAs of work segment ws - 2
                // are done with it: thread (h, u) rotates chunk pair u of query
                // head h at the row's position.
                if (ws >= 2 && !(kok = mbar_wait(smem_u32(&ctl->q_empty[ws & 1]), (uint32_t)(((ws - 2) >> 1) & 1), abort)))
                    break;
                range = rotate_q(a, ctl, sm + OFF_QT + (ws & 1) * QT_BYTES, ctl->seg[s].tq, ctl->seg[s].kvh,
                                 ctl->seg[s].qpos, tid);
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&ctl->q_ready[ws & 1]));
            }
            // (cos, sin) of the thread's current row: re-anchored exactly every
            // XF_ANCHOR_TILES tiles, advanced by the XF_ROW_STEP recurrence in between
            // (a thread's rows are XF_ROW_STEP apart and the next tile continues the
            // sequence), so at most XF_ANCHOR_TILES * XF_ROWS steps follow an anchor.
            float2 c[4], sn[4];
            // Tiles are counted from the anchor tile at or before the segment's
            // first (it = aph there), so it % XF_ANCHOR_TILES == 0 marks the anchor
            // tiles; a segment that starts between anchors takes its first angles
            // from the anchor before it (out of line, once per segment).
            const int aph = (t_begin / DEC_BN) & (XF_ANCHOR_TILES - 1);
            const int t_anchor = t_begin - aph * DEC_BN;
            if (aph != 0) {
                const Angles an = anchor_replay(ctl, t_begin / DEC_BN, r0, u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    c[e] = an.c[e];
                    sn[e] = an.s[e];
                }
            }
            for (int it = aph; it < aph + n_loc && kok; ++it, ++gcons) {
                const int k = gcons % DEC_KSTAGES;
                cp_async_wait<DEC_KAHEAD - 1>();  // this thread's chunks of the tile have landed
                uint8_t* kt = sm + OFF_K + k * DEC_TILE_BYTES;
                const int t0 = t_anchor + it * DEC_BN;
                if (it % XF_ANCHOR_TILES == 0) {
                    const Angles an = anchor_angles(ctl, (uint32_t)(t0 + r0), u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        c[e] = an.c[e];
                        sn[e] = an.s[e];
                    }
                }
                // all of the thread's rows are read before any is rotated (the
                // shared-memory latency is paid once per tile)
                uint4 lo[XF_ROWS], hi[XF_ROWS];
#pragma unroll
                for (int m = 0; m < XF_ROWS; ++m) {
                    const uint32_t off = sw128_off(r0 + XF_ROW_STEP * m, u);
                    lo[m] = *reinterpret_cast<const uint4*>(kt + off);
                    hi[m] = *reinterpret_cast<const uint4*>(kt + 16384 + off);
                }
#pragma unroll
                for (int m = 0; m < XF_ROWS; ++m) {
                    const int r = r0 + XF_ROW_STEP * m;
                    if (t0 + r < t_end) {
                        range = rotate_regs_f16(lo[m], hi[m], c, sn, range);
                        const uint32_t off = sw128_off(r, u);
                        *reinterpret_cast<uint4*>(kt + off) = lo[m];
                        *reinterpret_cast<uint4*>(kt + 16384 + off) = hi[m];
                    }
                    rope_step(c, sn, dcs, dsn);
                }
                fence_proxy_async_smem();  // rotated rows, and copied rows left as they are
                mbar_arrive(smem_u32(&ctl->k_ready[k]));
                kok = issue_k();
            }
            if (!kok) break;
            // the segment's range verdict, final once every transform thread arrived
            if (range_exceeded(range)) atomicOr(&ctl->seg[s].range, 1);
            mbar_arrive(smem_u32(&ctl->x_done[ws % X_RING]));
            ++ws;
        }
        cp_async_wait_all();  // no copy may land after the CTA has left
    } else if (warp < WARP_SOFTMAX0 + 4) {
        // =============================================== softmax WG ====
        const int t = tid - DEC_XFORM_THREADS;  // token of the tile == TMEM lane (S^T rows) == output dim (O^T rows)
        const int wq = warp & 3;
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        const float scl = a.qk_scale_log2;
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
        const float nanv = __int_as_float(0x7fc00000);
        bool ok = true;      // no wait has given up
        bool stamped = false;  // RK_STATUS_TIMEOUT reported
        int g = 0, ws = 0;
        for (int s = 0; s < n_seg; ++s) {
            const DecSeg& d = ctl->seg[s];  // the epilogue's fields, read there
            const bool imp = (d.flags & DEC_SEG_IMPORT) != 0, exp_ = (d.flags & DEC_SEG_EXPORT) != 0;
            // the fields the tile loop uses, in registers (the loop stores to shared
            // memory, so references into it would be read again and again)
            const int t_begin = d.t_begin, t_end = d.t_end, n_loc = d.n_loc;
            if (!ok || !seg_work(d)) {
                // after a failure: written as failed; unsafe metadata: failed (status
                // set at set-up); no visible key: empty.  A hand-off says failed.
                if (d.bad && t == 0 && a.status) atomicOr(a.status, d.bad);
                if (exp_) {
                    if (t == 0) export_failed(a, ctl->epoch);
                } else {
                    write_empty_row(a, d, (!ok || d.bad || imp) ? nanv : -INFINITY, t, 128);
                }
                continue;
            }
            float m[8], lp[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                m[h] = -INFINITY;
                lp[h] = 0.0f;
            }
            // Every wait result is OR-reduced over the warpgroup at named barrier 1,
            // so the four warps leave the loop together and never strand one another
            // at a barrier; a thread whose wait gave up skips its work until then.
            bool failed = false, quiet = false, seg_ok = true;
            if (imp) {
                LaneState st;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    st.m[h] = -INFINITY;
                    st.lp[h] = 0.0f;
                }
                const int r = import_state(a, ctl, abort, st, t, tO + lane_addr, s);
                if (r == 0) {
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        m[h] = st.m[h];
                        lp[h] = st.lp[h];
                    }
                } else {
                    // the row failed before this segment (reported there) or its state
                    // never came (reported here): the pipeline stops at once
                    failed = true;
                    quiet = r == 1;
                    *reinterpret_cast<volatile int*>(&abort->abort) = 1;
                }
            }
            for (int it = 0; it < n_loc; ++it, ++g) {
                const int sb = g & 1;
                const bool got = mbar_wait(smem_u32(&ctl->s_full[sb]), (uint32_t)((g >> 1) & 1), abort);
                if (named_bar_or(1, 128, failed || !got)) {
                    seg_ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[16];
                tmem_ld16(tmem + sb * NH + lane_addr, sr);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(smem_u32(&ctl->s_free[sb]));
                const bool vis = t_begin + it * DEC_BN + t < t_end;
                float x[8];
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    x[h] = (vis && h < G) ? __uint_as_float(sr[h]) * scl : -INFINITY;
                    float v = x[h];
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                    if (lane == 0) ctl->red[sb][wq][h] = v;
                }
                // The four warps' maxima meet at named barrier 1.  red[] is indexed by
                // tile parity: a buffer is rewritten two tiles later, after every
                // thread has passed the next tile's barrier (and so read it).
                named_bar_sync(1, 128);
                float alpha[8];
                bool resc = false;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const float mt = fmaxf(fmaxf(ctl->red[sb][0][h], ctl->red[sb][1][h]),
                                           fmaxf(ctl->red[sb][2][h], ctl->red[sb][3][h]));
                    alpha[h] = 1.0f;
                    if (mt > m[h] + RESCALE_SLACK) {
                        alpha[h] = ex2(m[h] - mt);  // 0 when m = -inf
                        m[h] = mt;
                        resc = true;
                    }
                }
                float p[8];
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    p[h] = m[h] == -INFINITY ? 0.0f : ex2(x[h] - m[h]);
                    lp[h] = lp[h] * alpha[h] + p[h];
                }
                // P^T buffer sb was last read by the PV of the CTA's tile g - 2 (this
                // segment's or an earlier one's); a rescale of O^T needs the PV of
                // tile it - 1 of this segment retired (resc is uniform: every thread
                // saw the same maxima).  One barrier per buffer parity, so a wait
                // never meets a phase of a later PV.
                bool w = true;
                if (g >= 2) w = mbar_wait(smem_u32(&ctl->pv_done[sb]), (uint32_t)(((g - 2) >> 1) & 1), abort);
                if (w && resc && it >= 1)
                    w = mbar_wait(smem_u32(&ctl->pv_done[sb ^ 1]), (uint32_t)(((g - 1) >> 1) & 1), abort);
                if (!__all_sync(0xffffffffu, w)) {
                    failed = true;  // leaves at the next barrier, together with the others
                    continue;
                }
                tc_fence_after();
                if (resc && (it >= 1 || imp)) {  // O^T of earlier tiles (this segment's or imported)
                    uint32_t orow[16];
                    tmem_ld16(tO + lane_addr, orow);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 8; ++h) orow[h] = __float_as_uint(__uint_as_float(orow[h]) * alpha[h]);
                    tmem_st16(tO + lane_addr, orow);
                    tmem_st_wait();
                }
                uint8_t* ptb = sm + OFF_PT + sb * PT_BYTES + (t >> 6) * 2048 + (t & 7) * 2;
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    if (h < G)
                        *reinterpret_cast<__nv_bfloat16*>(ptb + sw128_off(h, (t & 63) >> 3)) = __float2bfloat16_rn(p[h]);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(smem_u32(&ctl->p_ready[sb]));
            }
            if (seg_ok && named_bar_or(1, 128, failed)) seg_ok = false;
            // the transform's verdict on the segment's inputs, then O^T complete
            if (seg_ok)
                seg_ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->x_done[ws % X_RING]),
                                                           (uint32_t)((ws / X_RING) & 1), abort));
            if (seg_ok) seg_ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->o_done), (uint32_t)(ws & 1), abort));
            if (named_bar_or(1, 128, !seg_ok)) seg_ok = false;
            // ---- epilogue: fixed-order reduction of l, out = O / l once, LSE ----
            float L[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                float v = lp[h];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0) ctl->lred[wq][h] = v;
            }
            named_bar_sync(1, 128);
#pragma unroll
            for (int h = 0; h < 8; ++h) L[h] = ((ctl->lred[0][h] + ctl->lred[1][h]) + ctl->lred[2][h]) + ctl->lred[3][h];
            const bool range_bad = ctl->seg[s].range != 0;
            const int h0 = ctl->seg[s].kvh * G, tq = ctl->seg[s].tq;
            uint32_t orow[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) orow[c] = 0u;
            if (seg_ok) {
                tc_fence_after();
                tmem_ld16(tO + lane_addr, orow);
                tmem_ld_wait();
            }
            if (exp_) {
                LaneState st;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    st.m[h] = m[h];
                    st.lp[h] = lp[h];
                }
                export_state(a, ctl, st, orow, seg_ok, range_bad, t);
            } else if (seg_ok) {
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    if (h < G) {
                        const float o = (range_bad || !(L[h] > 0.0f)) ? 0.0f : __uint_as_float(orow[h]) / L[h];
                        out[((size_t)tq * a.Hq + h0 + h) * HEAD_DIM + t] = __float2bfloat16_rn(o);
                    }
                }
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    if (t == h && h < G)
                        a.lse[(size_t)tq * a.Hq + h0 + h] =
                            range_bad ? nanv : (L[h] > 0.0f ? (m[h] + log2f(L[h])) * 0.693147180559945309f : -INFINITY);
            } else {  // a wait gave up (or the row failed earlier): the group's rows are written as failed
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    if (h < G) out[((size_t)tq * a.Hq + h0 + h) * HEAD_DIM + t] = __float2bfloat16_rn(0.0f);
                if (t < G) a.lse[(size_t)tq * a.Hq + h0 + t] = nanv;
            }
            if (t == 0 && a.status) {
                if (seg_ok && range_bad && !exp_) atomicOr(a.status, RK_STATUS_RANGE);
                if (!seg_ok && !quiet && !stamped) {
                    atomicOr(a.status, RK_STATUS_TIMEOUT);
                    stamped = true;
                }
            }
            if (!seg_ok) {
                ok = false;  // the CTA's later segments are written as failed
                continue;
            }
            // O^T has been read: the next work segment's PVs may write it
            tc_fence_before();
            mbar_arrive(smem_u32(&ctl->o_free));
            ++ws;
        }
    }

    // ---- teardown: all roles done; no MMA or TMEM access in flight ----
    tc_fence_before();
    __syncthreads();
    if (tid == 0) bal_done(a);
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace bal

}  // namespace

namespace {
// Sets a kernel's dynamic shared memory limit once per device.
template <typename K>
cudaError_t configure(std::atomic<uint64_t>& configured, K kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load() & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    return cudaSuccess;
}
std::atomic<uint64_t> g_configured{0}, g_configured_bal{0};
}  // namespace

cudaError_t decode_resident_ctas(int* ctas) {
    cudaError_t e = configure(g_configured_bal, bal::decode_bal_kernel, DEC_BAL_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, bal::decode_bal_kernel, DEC_THREADS,
                                                           DEC_BAL_SMEM_BYTES)) != cudaSuccess)
        return e;
    *ctas = sms * per;
    return cudaSuccess;
}

cudaError_t launch_decode(const CUtensorMap& vm, const DecodeArgs& a, cudaStream_t stream) {
    cudaError_t e;
    if (a.balanced) {
        if ((e = configure(g_configured_bal, bal::decode_bal_kernel, DEC_BAL_SMEM_BYTES)) != cudaSuccess) return e;
        // every CTA resident at once (a CTA may wait for its predecessor's hand-off)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)a.bal_grid);
        cfg.blockDim = dim3(DEC_THREADS);
        cfg.dynamicSmemBytes = DEC_BAL_SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeCooperative;
        at[0].val.cooperative = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, bal::decode_bal_kernel, vm, a);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    if ((e = configure(g_configured, decode_kernel, DEC_SMEM_BYTES)) != cudaSuccess) return e;
    const long long grid = (long long)a.B * a.Hkv * (a.split_tokens > 0 ? a.n_splits : 1);
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    decode_kernel<<<(unsigned)grid, DEC_THREADS, DEC_SMEM_BYTES, stream>>>(vm, a);
    e = cudaGetLastError();
    if (e != cudaSuccess || a.split_tokens <= 0) return e;
    // the merge may start while the split grid drains (it waits on the grid
    // dependency before it reads a partial)
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)((long long)a.B * a.Hq));
    cfg.blockDim = dim3(HEAD_DIM);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    std::memset(&attr, 0, sizeof attr);
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_merge_kernel, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace rk
