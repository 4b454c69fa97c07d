// prefill.cu -- causal chunked prefill over a paged prefix on the 5th-gen
// tensor cores (tcgen05 MMA into TMEM), RoPE applied in the load stage.
//
// Operation: the paged prefill of "WS2 PR7 Fused Attention Backend
// Alignment", "Current Implementation" (BatchPrefillWithPagedKVCacheWrapper
// role, ROPE_LLAMA fused on pre-RoPE Q and K, split-KV disabled, FP32 LSE),
// with the batch-invariance requirement of that page's "Batch-Invariant
// Validation" section.
//
// Work unit: two consecutive q-tiles of one (row, KV head).  A q-tile is 128
// accumulator rows = (128/G) query positions x the G query heads sharing the
// KV head (GQA packing).  A unit sweeps the row's KV tiles of 128 tokens
// (8 pages) in ascending order; every K tile is rotated once and used by both
// q-tiles.  The grid is persistent: at most one CTA per SM, each taking the
// units of the heaviest-first order (later positions see more keys) at the
// positions c, 2 G - 1 - c, 2 G + c, ... of that order (G = grid size), so
// the work per CTA is balanced and the set-up of a unit (metadata checks, Q
// load and rotation, first K tiles) overlaps the end of the one before.
// Which CTA runs a unit never changes how the unit is computed.  A ragged
// batch runs one unit per CTA (the unit found from qo_indptr).  Roles (512
// threads, registers rebalanced with setmaxnreg):
//   warp 15      scheduler: checks each unit's metadata (kv_len, positions,
//                page ids), publishes a unit descriptor (two-slot ring) and
//                loads the unit's Q tiles by TMA once the previous unit's
//                score MMAs have read the Q buffer;
//   warpgroup 0  transform: rotate both q-tiles once and each K tile in place
//                in shared memory (FP32 math; angles from an exact fixed-point
//                anchor every 4 K tiles plus 16-position angle-addition steps),
//                store FP16 in the UMMA operand layout;
//   warpgroup 1  softmax for q-tile 0, warpgroup 2 softmax for q-tile 1: one
//                thread per accumulator row reads its S row from TMEM, masks,
//                runs the online softmax in the log2 domain (the running max
//                only moves when it grows by more than 8, then the O row in
//                TMEM is rescaled), writes P as BF16 back into TMEM over S;
//                epilogue O / l -> BF16 once, LSE -> FP32;
//   warps 12/14  TMA producers: warp 12 loads each K page as two 16-token x
//                64-dim boxes (K-major tile layout), warp 14 each V page as one
//                4 KiB box ([64-dim half][16 tokens], one page per PV k-step)
//                and zeroes V rows past the last key;
//   warp 13      MMA issuer: S_j = Q_j K^T (FP16 operands, FP32 in TMEM) and
//                O_j += P_j V (P from TMEM, V from shared memory, BF16).
// Pipeline state (stage indices and barrier phases) runs on across units;
// tensor memory is allocated once per CTA.
// Score precision: rotated Q and K are rounded to FP16 (11-bit mantissa) for
// the score MMA; this keeps the LSE within 1e-3 of float64 even for rows
// that see a single key, where BF16 operands would not.  FP16 needs the
// rotated values below 65504 in magnitude: a unit whose pre-RoPE bf16 inputs
// reach 2^15 is not computed and is reported (RK_STATUS_RANGE).
// Nothing depends on B, W or the grid: tiles are fixed in logical positions
// and tokens, and the reduction order within a row is fixed.
#include <atomic>
#include <cstring>

#include "rk_device.cuh"

namespace rk {

namespace {

constexpr int PF_THREADS = 512;
constexpr int WARP_TMA_K = 12;
constexpr int WARP_MMA = 13;
constexpr int WARP_TMA_V = 14;
constexpr int WARP_SCHED = 15;
constexpr int KSTAGES = 3;
constexpr int VSTAGES = 2;
constexpr uint32_t TMEM_COLS = 512;  // S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512)
constexpr float RESCALE_SLACK = 8.0f;
// Threads that read every unit descriptor: the K and V producer warps, the MMA
// issuer, the transform and both softmax warpgroups.
constexpr uint32_t UNIT_READERS = 32 + 32 + 1 + 128 + 256;

// setmaxnreg split (sum 4 x 128 = the 512 x 128 registers the CTA launches with)
constexpr int REG_XFORM = 88;
constexpr int REG_SOFTMAX = 184;
constexpr int REG_CTRL = 56;
static_assert(REG_XFORM + 2 * REG_SOFTMAX + REG_CTRL == 4 * 128, "register split must sum to the launch budget");

// Shared memory carve (the dynamic shared memory base is 1024-byte aligned).
constexpr int OFF_Q = 0;  // Q tile j at OFF_Q + j * 32 KiB
constexpr int OFF_K = OFF_Q + 2 * PF_TILE_BYTES;
constexpr int OFF_V = OFF_K + KSTAGES * PF_TILE_BYTES;
constexpr int OFF_BAR = OFF_V + VSTAGES * PF_TILE_BYTES;
constexpr int PF_CTRL_BYTES = 3072;
constexpr int PF_SMEM_BYTES = OFF_BAR + PF_CTRL_BYTES;

// One work unit as the scheduler publishes it.
struct PfUnit {
    int end;                      // 1: the CTA has no further unit
    int b, kvh, pair, qbase, qn;  // row, KV head, pair of q-tiles, where the row's queries live
    int kv_len;
    int nt0, nt1;                 // KV tiles q-tile 0 / 1 needs
    int n_keys;                   // keys the pair reads
    int bad;                      // RK_STATUS_* bits of unsafe metadata (rows written as NaN)
};

struct PfBars {
    uint64_t q_full, q_ready, q_empty;
    uint64_t k_full[KSTAGES], k_ready[KSTAGES], k_empty[KSTAGES];
    uint64_t v_full[VSTAGES], v_empty[VSTAGES], v_land;  // v_land: the copy of a row's last V tile
    uint64_t s_full[2], p_ready[2], o_done[2], o_free[2];
    uint64_t u_full[2], u_empty[2];  // unit descriptor ring
    uint64_t r_full[2], r_empty[2];  // per-unit FP16 range verdict, transform -> softmax epilogues
    uint64_t never;                  // nothing arrives: the timeout drill's wait
    uint32_t tmem_base;
    PipeCtl pipe;
    PfUnit unit[2];
    // per transform thread (K) and softmax warp (its Q rows): did an input
    // element of the unit reach 2^15 (one byte each, so nothing is reset and
    // no barrier is needed among the writers)
    alignas(16) uint8_t r_flag[2][144];  // [0, 128) transform threads, [128, 136) softmax warps
    // positions of the rows of the unit whose Q is loaded (q-tile j row r at
    // j * rph + r; -1 past the row's queries), written with the Q load
    int qpos[2 * PF_BM];
    uint64_t turns[ROPE_PAIRS];
    float2 step16[ROPE_PAIRS];  // cos/sin of a 16-position turn per pair
    int sched[4 + PF_THREADS / 32];  // ragged schedule: level, rank, total units, row; per-warp counts
};
static_assert(sizeof(PfBars) <= PF_CTRL_BYTES, "prefill control block exceeds its reservation");
static_assert((2 * PF_RAGGED_MAX_LEVELS + 1) * 4 <= KSTAGES * PF_TILE_BYTES,
              "ragged schedule counters exceed the K stage buffers");
static_assert(PF_SMEM_BYTES <= 232448, "prefill shared memory above the 227 KiB opt-in limit");

__device__ __forceinline__ uint32_t sw_off(int row, int chunk) { return sw128_off(row, chunk); }


// Where a row's queries live: padded rows (s of row b at [b, h, s]) or a
// ragged batch (packed rows qbase .. qbase + qn - 1 at [qbase + s, h]).
struct RowMap {
    int b, qn, qbase;
    bool ragged;
    // index of (query s, head h) in lse; times HEAD_DIM in out
    __device__ __forceinline__ size_t at(const PrefillArgs& a, int h, int s) const {
        return ragged ? (size_t)(qbase + s) * a.Hq + h : ((size_t)b * a.Hq + h) * a.Sq + s;
    }
};

// Ragged batch: the rows with two or more queries are cut into pairs of
// q-tiles (2 rph queries; a row of q queries has np = ceil(q / (2 rph))
// pairs), one work unit per pair and KV head.  Units are ordered by level d,
// the pair counted back from the row's last (d = 0: every row's last pair,
// which sees the most keys), then by row, so the heaviest units start first;
// for rows of equal length this is the order of the padded grid.  Every CTA
// derives its own unit w = blockIdx.x / Hkv from qo_indptr alone: a histogram
// of np in shared memory, the level whose running count passes w, and the
// rank of the row within that level.  Rows whose indptr entries are unsafe
// or that hold more than max_q_len queries are left out; CTA 0 flags them
// and a grid too small for the units (RK_STATUS_POSITION).  All threads call
// this; it returns false when the CTA has no unit.
struct RaggedUnit {
    int b, pair, qs, qn;
};

__device__ __forceinline__ int ragged_pairs(const PrefillArgs& a, int r, int span, bool& unsafe) {
    const int qs = __ldg(a.qo_indptr + r), qe = __ldg(a.qo_indptr + r + 1);
    unsafe = !(qs >= 0 && qe >= qs && qe <= a.total_q && qe - qs <= a.max_q_len);
    return (!unsafe && qe - qs >= 2) ? (qe - qs + span - 1) / span : 0;
}

__device__ bool ragged_unit(const PrefillArgs& a, PfBars* bars, int* hist, RaggedUnit& u) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int span = 2 * a.rows_per_head;
    const int L = min((a.max_q_len + span - 1) / span, PF_RAGGED_MAX_LEVELS);
    int* cnt = hist + L + 1;  // cnt[d]: rows with more than d pairs
    const int w = (int)(blockIdx.x / a.Hkv);
    for (int i = tid; i <= L; i += PF_THREADS) hist[i] = 0;
    __syncthreads();
    int unsafe_any = 0;
    for (int r = tid; r < a.B; r += PF_THREADS) {
        bool un;
        const int np = ragged_pairs(a, r, span, un);
        unsafe_any |= un ? 1 : 0;
        if (np) atomicAdd(&hist[min(np, L)], 1);
    }
    unsafe_any = __syncthreads_or(unsafe_any);
    if (warp == 0) {
        // suffix sums of the histogram, top chunk of 32 levels first
        int carry = 0;
        for (int base = ((L - 1) >> 5) << 5; base >= 0; base -= 32) {
            const int d = base + lane;
            int v = d < L ? hist[d + 1] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_down_sync(0xffffffffu, v, o);
                if (lane + o < 32) v += t;
            }
            v += carry;
            if (d < L) cnt[d] = v;
            carry = __shfl_sync(0xffffffffu, v, 0);
        }
        __syncwarp();
        // the level whose inclusive running count first exceeds w
        int run = 0, fd = -1, fk = 0;
        for (int base = 0; base < L; base += 32) {
            const int d = base + lane;
            const int c = d < L ? cnt[d] : 0;
            int v = c;
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, run + v > w);
            if (fd < 0 && hit) {
                const int f = __ffs(hit) - 1;
                fd = base + f;
                fk = w - (run + __shfl_sync(0xffffffffu, v - c, f));
            }
            run += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) {
            bars->sched[0] = fd;
            bars->sched[1] = fk;
            bars->sched[2] = run;
            bars->sched[3] = -1;
        }
    }
    __syncthreads();
    const int d = bars->sched[0], k = bars->sched[1], total = bars->sched[2];
    if (blockIdx.x == 0 && tid == 0 && a.status && (unsafe_any || total > (int)(gridDim.x / a.Hkv)))
        atomicOr(a.status, RK_STATUS_POSITION);
    if (d < 0) return false;
    // the unit's row: the k-th row, in index order, with more than d pairs
    int offset = 0;
    for (int r0 = 0; r0 < a.B; r0 += PF_THREADS) {
        const int r = r0 + tid;
        bool un;
        const bool p = r < a.B && ragged_pairs(a, r, span, un) > d;
        const unsigned bal = __ballot_sync(0xffffffffu, p);
        if (lane == 0) bars->sched[4 + warp] = __popc(bal);
        __syncthreads();
        int pre = offset, tot = 0;
        for (int w2 = 0; w2 < PF_THREADS / 32; ++w2) {
            const int c = bars->sched[4 + w2];
            pre += w2 < warp ? c : 0;
            tot += c;
        }
        if (p && pre + __popc(bal & ((1u << lane) - 1u)) == k) bars->sched[3] = r;
        offset += tot;
        __syncthreads();
        if (bars->sched[3] >= 0) break;
    }
    const int b = bars->sched[3];
    if (b < 0) return false;  // the two passes read the same qo_indptr: not reached
    u.b = b;
    u.qs = __ldg(a.qo_indptr + b);
    u.qn = __ldg(a.qo_indptr + b + 1) - u.qs;
    u.pair = (u.qn + span - 1) / span - 1 - d;
    return true;
}


// Unit k of this CTA in the heaviest-first order (padded layout): positions
// c, 2G - 1 - c, 2G + c, 4G - 1 - c, ... (G CTAs), so a CTA that took one of
// the heaviest units next takes one of the lightest.
__device__ __forceinline__ long long cta_unit(int k, int c, int g) {
    return (k & 1) ? (long long)(k + 1) * g - 1 - c : (long long)k * g + c;
}

// (row, KV head, pair) of unit u of the padded layout: pairs from the last
// (most keys) down, rows and KV heads within a pair level.
__device__ __forceinline__ void padded_unit(const PrefillArgs& a, long long u, int& b, int& kvh, int& pair) {
    const int units = a.B * a.Hkv;
    pair = (a.n_qtiles + 1) / 2 - 1 - (int)(u / units);
    const int rem = (int)(u % units);
    b = rem / a.Hkv;
    kvh = rem % a.Hkv;
}

// Rows of q-tile j (queries s00 + j rph ..) written as out = 0, lse = lse_val
// by the 128 threads of one warpgroup (r = accumulator row).
__device__ __forceinline__ void write_qtile_rows(const PrefillArgs& a, const RowMap& rm, int kvh, int s0, int r,
                                                 float lse_val) {
    const int rph = a.rows_per_head;
    const int g = r / rph, s = s0 + r % rph;
    if (r >= a.G * rph || s >= rm.qn) return;
    const int h = kvh * a.G + g;
    uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + rm.at(a, h, s) * HEAD_DIM);
    for (int d = 0; d < HEAD_DIM / 8; ++d) o[d] = make_uint4(0, 0, 0, 0);
    a.lse[rm.at(a, h, s)] = lse_val;
}

// Unit k of this CTA and its metadata checks (one warp, all lanes): kv_len,
// the positions of both q-tiles (their largest value sets the keys each
// q-tile reads), and every page id of the row's keys (kv_len, not only the
// keys this pair sees, so all units of a row agree on unsafe pages).
__device__ __forceinline__ PfUnit unit_meta(const PrefillArgs& a, int k, int cta, int grid, long long total,
                                            const RaggedUnit& ru, int lane) {
    const bool ragged = a.qo_indptr != nullptr;
    const int rph = a.rows_per_head;
    PfUnit d;
    d.b = d.kvh = d.pair = d.qbase = d.qn = d.kv_len = d.nt0 = d.nt1 = d.n_keys = d.bad = 0;
    if (ragged) {
        d.end = k > 0;
        d.b = ru.b;
        d.kvh = cta % a.Hkv;
        d.pair = ru.pair;
        d.qbase = ru.qs;
        d.qn = ru.qn;
    } else {
        const long long u = cta_unit(k, cta, grid);
        d.end = u >= total;
        if (!d.end) padded_unit(a, u, d.b, d.kvh, d.pair);
        d.qbase = d.b * a.Sq;
        d.qn = a.Sq;
    }
    if (d.end) return d;
    const int kv_len = a.kv_lens[d.b];
    int bad = (kv_len < 0 || kv_len > a.W * PAGE) ? RK_STATUS_KVLEN : 0;
    const int32_t* pos_row = a.position_ids + d.qbase;
    const int s00 = 2 * d.pair * rph;
    int pm0 = -1, pm1 = -1, neg = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int r = lane + 32 * m;
        if (r < rph) {
            if (s00 + r < d.qn) {
                const int p = pos_row[s00 + r];
                neg |= p < 0;
                pm0 = max(pm0, p);
            }
            if (s00 + rph + r < d.qn) {
                const int p = pos_row[s00 + rph + r];
                neg |= p < 0;
                pm1 = max(pm1, p);
            }
        }
    }
    pm0 = __reduce_max_sync(0xffffffffu, pm0);
    pm1 = __reduce_max_sync(0xffffffffu, pm1);
    if (__reduce_or_sync(0xffffffffu, (unsigned)neg)) bad |= RK_STATUS_POSITION;
    const int row_pages = (bad & RK_STATUS_KVLEN) ? 0 : (kv_len + PAGE - 1) / PAGE;
    const int32_t* bt = a.block_table + (size_t)d.b * a.W;
    int oob = 0;
    for (int i = lane; i < row_pages; i += 32) {
        const int pg = __ldg(bt + i);
        oob |= (pg < 0) | (pg >= a.num_pages);
    }
    if (__reduce_or_sync(0xffffffffu, (unsigned)oob)) bad |= RK_STATUS_PAGE_OOB;
    const int nk0 = (bad || pm0 < 0) ? 0 : (pm0 >= kv_len ? kv_len : pm0 + 1);
    const int nk1 = (bad || pm1 < 0) ? 0 : (pm1 >= kv_len ? kv_len : pm1 + 1);
    d.kv_len = kv_len;
    d.nt0 = (nk0 + PF_BN - 1) / PF_BN;
    d.nt1 = (nk1 + PF_BN - 1) / PF_BN;
    d.n_keys = max(nk0, nk1);
    d.bad = bad;
    return d;
}

// Read unit descriptor k (every reader thread waits, copies, then releases
// its slot).  Returns false when the wait gave up.
__device__ __forceinline__ bool read_unit(PfBars* bars, int k, PipeCtl* abort, PfUnit& u) {
    const int slot = k & 1;
    if (!mbar_wait(smem_u32(&bars->u_full[slot]), (uint32_t)((k >> 1) & 1), abort)) return false;
    const volatile PfUnit* src = &bars->unit[slot];
    u.end = src->end;
    u.b = src->b;
    u.kvh = src->kvh;
    u.pair = src->pair;
    u.qbase = src->qbase;
    u.qn = src->qn;
    u.kv_len = src->kv_len;
    u.nt0 = src->nt0;
    u.nt1 = src->nt1;
    u.n_keys = src->n_keys;
    u.bad = src->bad;
    mbar_arrive(smem_u32(&bars->u_empty[slot]));
    return true;
}

// Launched after a ragged batch's decode launch with programmatic stream
// serialization, this grid starts while that one drains (the two write
// disjoint rows).  Its last CTA waits for that grid before it exits, so the
// grid completes after it and work ordered after this grid sees both done.
__device__ __forceinline__ void pdl_tail() {
    if (blockIdx.x == gridDim.x - 1) griddep_wait();
}

__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ PrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw;
    PfBars* bars = reinterpret_cast<PfBars*>(sm + OFF_BAR);
    const uint32_t s_base = smem_u32(sm);
    if (s_base & 1023u) {  // the swizzled operand layout needs a 1024-byte aligned base
        if (threadIdx.x == 0 && a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
        pdl_tail();
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
    const int rph = a.rows_per_head;
    const bool ragged = a.qo_indptr != nullptr;
    const int cta = (int)blockIdx.x, grid = (int)gridDim.x;
    // ---- this CTA's units: the persistent sequence, or one ragged unit ----
    const long long total = ragged ? 0 : (long long)a.B * a.Hkv * ((a.n_qtiles + 1) / 2);
    RaggedUnit ru{0, 0, 0, 0};
    if (ragged) {
        if (!ragged_unit(a, bars, reinterpret_cast<int*>(sm + OFF_K), ru)) {
            pdl_tail();
            return;
        }
    } else if (cta >= total) {
        pdl_tail();
        return;
    }
    // The scheduler warp checks its first unit's metadata while the CTA sets up
    // (the global loads overlap the barrier set-up and the stage zeroing).
    PfUnit first{};
    if (warp == WARP_SCHED) first = unit_meta(a, 0, cta, grid, total, ru, lane);
    if (tid == 0) {
        bars->pipe.abort = 0;
        bars->pipe.limit_ns = wait_limit(a.wait_limit_ns);
        mbar_init(smem_u32(&bars->never), 1);
        mbar_init(smem_u32(&bars->q_full), 1);
        mbar_init(smem_u32(&bars->q_ready), 256);
        mbar_init(smem_u32(&bars->q_empty), 1);
        for (int k = 0; k < KSTAGES; ++k) {
            mbar_init(smem_u32(&bars->k_full[k]), 1);
            mbar_init(smem_u32(&bars->k_ready[k]), 128);
            mbar_init(smem_u32(&bars->k_empty[k]), 1);
        }
        for (int k = 0; k < VSTAGES; ++k) {
            mbar_init(smem_u32(&bars->v_full[k]), 1);
            mbar_init(smem_u32(&bars->v_empty[k]), 1);
        }
        mbar_init(smem_u32(&bars->v_land), 1);
        for (int j = 0; j < 2; ++j) {
            mbar_init(smem_u32(&bars->s_full[j]), 1);
            mbar_init(smem_u32(&bars->p_ready[j]), 128);
            mbar_init(smem_u32(&bars->o_done[j]), 1);
            mbar_init(smem_u32(&bars->o_free[j]), 128);
            mbar_init(smem_u32(&bars->u_full[j]), 1);
            mbar_init(smem_u32(&bars->u_empty[j]), UNIT_READERS);
            mbar_init(smem_u32(&bars->r_full[j]), 384);
            mbar_init(smem_u32(&bars->r_empty[j]), 256);
        }
        fence_mbar_init();
    }
    // The range-verdict bytes no writer owns (the padding) stay zero.
    for (int i = tid; i < (int)sizeof(bars->r_flag) / 4; i += PF_THREADS)
        reinterpret_cast<uint32_t*>(&bars->r_flag[0][0])[i] = 0;
    // V stages start as zeros: rows of pages a tile does not load stay finite.
    for (int i = tid; i < VSTAGES * PF_TILE_BYTES / 16; i += PF_THREADS)
        reinterpret_cast<uint4*>(sm + OFF_V)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid < ROPE_PAIRS) {
        bars->turns[tid] = a.rope_turns[tid];
        float c, s;
        rope_cos_sin((uint32_t)PAGE, a.rope_turns[tid], c, s);
        bars->step16[tid] = make_float2(c, s);
    }
    // ---- TMEM allocation (warp 13 owns it, for the CTA's whole life) ----
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(&bars->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    PipeCtl* abort = &bars->pipe;

    if (wg == 3) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_CTRL));
        if (warp == WARP_SCHED) {
            // ============================================== scheduler ====
            // Unit descriptors in order, each once its slot is free; a unit's Q
            // tiles once the previous unit's score MMAs have read the buffer.
            if (lane == 0) prefetch_tmap(&qmap);
            int wq = 0;  // Q loads issued (= work units published)
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                ok = __shfl_sync(0xffffffffu,
                                 lane == 0 ? (int)mbar_wait(smem_u32(&bars->u_empty[slot]), (uint32_t)(((k >> 1) & 1) ^ 1), abort)
                                           : 0,
                                 0) != 0;
                if (!ok) break;
                const PfUnit m = k == 0 ? first : unit_meta(a, k, cta, grid, total, ru, lane);
                if (m.end) {
                    if (lane == 0) {
                        bars->unit[slot].end = 1;
                        mbar_arrive(smem_u32(&bars->u_full[slot]));
                    }
                    break;
                }
                if (lane == 0) {
                    bars->unit[slot] = m;
                    if (m.bad && a.status) atomicOr(a.status, m.bad);
                    mbar_arrive(smem_u32(&bars->u_full[slot]));
                }
                const int b = m.b, kvh = m.kvh, qbase = m.qbase, s00 = 2 * m.pair * rph;
                const bool bad = m.bad != 0;
                const int n_keys = m.n_keys;
                if (!bad && n_keys > 0) {
                    // Q of both q-tiles, once the previous unit's score MMAs are done with the
                    // buffer, and the rows' positions beside it for the Q rotation
                    int qp[8];
                    const int32_t* pos_row = a.position_ids + qbase;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int r = lane + 32 * (e & 3), s = s00 + (e >> 2) * rph + r;
                        qp[e] = (r < rph && s < m.qn) ? pos_row[s] : -1;
                    }
                    if (lane == 0) ok = mbar_wait(smem_u32(&bars->q_empty), (uint32_t)((wq & 1) ^ 1), abort);
                    ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
                    if (ok) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int r = lane + 32 * (e & 3);
                            if (r < rph) bars->qpos[(e >> 2) * rph + r] = qp[e];
                        }
                        __syncwarp();
                    }
                    if (ok && lane == 0) {
                        const uint32_t qb = smem_u32(&bars->q_full);
                        mbar_arrive_expect_tx(qb, 2 * PF_TILE_BYTES);
                        for (int j = 0; j < 2; ++j) {
                            const uint32_t dq = s_base + OFF_Q + j * PF_TILE_BYTES;
                            if (ragged) {  // packed q seen as (d, token, head): rows past the row's end are masked
                                tma_load_3d(dq, &qmap, qb, 0, qbase + s00 + j * rph, kvh * a.G);
                                tma_load_3d(dq + 16384, &qmap, qb, 64, qbase + s00 + j * rph, kvh * a.G);
                            } else {
                                tma_load_4d(dq, &qmap, qb, 0, s00 + j * rph, kvh * a.G, b);
                                tma_load_4d(dq + 16384, &qmap, qb, 64, s00 + j * rph, kvh * a.G, b);
                            }
                        }
                        ++wq;
                    }
                }
                ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
            }
            // the Q load in flight lands before the CTA's shared memory is released
            if (lane == 0 && pipe_aborted(abort) && wq > 0) mbar_wait_drain(smem_u32(&bars->q_full), (uint32_t)((wq - 1) & 1));
        } else if (warp == WARP_TMA_K || warp == WARP_TMA_V) {
            // ======================================= TMA producers ====
            // warp 12 loads the K tiles, warp 14 the V tiles; lane p issues the
            // boxes of page p of a tile.  n: tiles issued over the CTA's units.
            const bool is_k = warp == WARP_TMA_K;
            const CUtensorMap* map = is_k ? &kmap : &vmap;
            if (lane == 0) prefetch_tmap(map);
            const int nst = is_k ? KSTAGES : VSTAGES;
            int n = 0;
            int v_owner0 = -1, v_owner1 = -1;  // unit that last loaded V stage 0 / 1
            int nl = 0;                        // V tail tiles copied through v_land
            bool land_open = false;            // the last of them was not seen landing
            bool ok = true;
            for (int k = 0; ok; ++k) {
                PfUnit u;
                if (!(ok = __all_sync(0xffffffffu, read_unit(bars, k, abort, u))) || u.end) break;
                const int n_tiles = max(u.nt0, u.nt1);
                if (u.bad || n_tiles == 0) continue;
                const int32_t* bt = a.block_table + (size_t)u.b * a.W;
                const int n_pages = (u.n_keys + PAGE - 1) / PAGE;
                // The row's last page is in this unit's last tile and only partly
                // filled: its cache rows past kv_len hold arbitrary bits and are
                // zeroed in V after the copy lands (they meet P = 0, which would not
                // cancel a non-finite value).  That copy lands on v_land, and v_full
                // is completed (one plain arrival) only after the zeroing, so the
                // MMA side waits on v_full alone whatever the tile holds.
                const bool has_tail = u.n_keys == u.kv_len && (u.kv_len & (PAGE - 1)) != 0;
                for (int i = 0; i < n_tiles; ++i, ++n) {
                    const int st = n % nst;
                    const uint32_t use = (uint32_t)(n / nst);
                    const int p0 = i * PF_PAGES_PER_TILE;
                    const int np = min(PF_PAGES_PER_TILE, n_pages - p0);
                    const int pg = lane < np ? __ldg(bt + p0 + lane) : 0;
                    const uint32_t eb = smem_u32(is_k ? &bars->k_empty[st] : &bars->v_empty[st]);
                    const uint32_t fb = smem_u32(is_k ? &bars->k_full[st] : &bars->v_full[st]);
                    int good = 1;
                    if (lane == 0) good = mbar_wait(eb, (use & 1u) ^ 1u, abort);
                    if (!(ok = __shfl_sync(0xffffffffu, good, 0) != 0)) break;
                    uint8_t* vt = sm + OFF_V + st * PF_TILE_BYTES;
                    const bool other_unit = (st ? v_owner1 : v_owner0) != k;
                    if (!is_k) (st ? v_owner1 : v_owner0) = k;
                    if (!is_k && np < PF_PAGES_PER_TILE && other_unit) {
                        // pages this tile does not load hold another unit's rows: zeros
                        for (int idx = np * 256 + lane; idx < PF_PAGES_PER_TILE * 256; idx += 32)
                            reinterpret_cast<uint4*>(vt)[idx] = make_uint4(0, 0, 0, 0);
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    const bool tail_tile = !is_k && has_tail && i == n_tiles - 1;
                    const uint32_t lb = tail_tile ? smem_u32(&bars->v_land) : fb;
                    if (lane == 0) mbar_arrive_expect_tx(lb, (uint32_t)np * 2 * 2048);
                    __syncwarp();
                    if (lane < np) {
                        if (is_k) {  // two 16 x 64 boxes per page: the K-major tile layout
                            const uint32_t t = s_base + OFF_K + st * PF_TILE_BYTES + lane * 2048;
                            tma_load_3d(t, map, lb, 0, u.kvh, pg * PAGE);
                            tma_load_3d(t + 16384, map, lb, 64, u.kvh, pg * PAGE);
                        } else {     // one 4 KiB box per page: [page][half][16 rows][128 B]
                            tma_load_4d(s_base + OFF_V + st * PF_TILE_BYTES + lane * 4096, map, lb, 0, pg * PAGE, 0,
                                        u.kvh);
                        }
                    }
                    __syncwarp();
                    if (tail_tile) {
                        // this warp is v_land's only waiter and waits each phase it armed
                        const int landed =
                            __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(lb, (uint32_t)(nl & 1), abort) : 0, 0);
                        ++nl;
                        if (!landed) {
                            land_open = true;
                            ok = false;
                            break;
                        }
                        const int tail = u.kv_len - i * PF_BN;
                        const int r_end = min(PF_BN, (tail + PAGE - 1) & ~(PAGE - 1));
                        for (int idx = lane; idx < (r_end - tail) * 16; idx += 32) {
                            const int rr = tail + (idx >> 4), ch = idx & 15;
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
                if (land_open) mbar_wait_drain(smem_u32(&bars->v_land), (uint32_t)((nl - 1) & 1));
                for (int i = max(0, n - nst); i < n; ++i)
                    mbar_wait_drain(smem_u32(is_k ? &bars->k_full[i % nst] : &bars->v_full[i % nst]),
                                    (uint32_t)((i / nst) & 1));
            }
        } else if (warp == WARP_MMA && lane == 0) {
            // ============================================= MMA issuer ====
            // scores: FP16 A and B (format 0), FP32 accumulate, K-major both
            const uint32_t idS = (1u << 4) | ((uint32_t)(PF_BN >> 3) << 17) | ((uint32_t)(PF_BM >> 4) << 24);
            const uint32_t idO = idesc_bf16_f32(PF_BM, HEAD_DIM, 0, 1);
            // k-step 0 descriptors of stage 0; stages and k-steps are added to the
            // address field.  Each group of 8 MMAs is unrolled with constant offsets so
            // that the single issuing thread keeps up with the tensor pipe.
            constexpr uint32_t TILE_DESC = PF_TILE_BYTES >> 4;  // one 32 KiB tile in descriptor address units
            const uint32_t dQ0 = desc_lo(s_base + OFF_Q, 16);
            const uint32_t dK0 = desc_lo(s_base + OFF_K, 16);
            const uint32_t dV0 = desc_lo(s_base + OFF_V, 2048);
            // Phase state over the CTA's units, packed: g = KV tiles before the
            // unit (stage and phase of the K and V rings); ph bit 0 q_ready, bits
            // 2 + j s_full / p_ready of q-tile j, bits 4 + j o_free.
            int g0 = 0;
            uint32_t ph = 0;
            bool ok = !a.timeout_drill || drill_wait(smem_u32(&bars->never), abort);
            for (int kk = 0; ok; ++kk) {
                PfUnit u;
                if (!(ok = read_unit(bars, kk, abort, u)) || u.end) break;
                const int n_tiles = max(u.nt0, u.nt1);
                if (u.bad || n_tiles == 0) continue;
                const int nt0 = u.nt0, nt1 = u.nt1;
                if (!(ok = mbar_wait(smem_u32(&bars->q_ready), ph & 1u, abort))) break;
                int v_seen = -1;  // last V tile whose arrival (and tail zeroing) was observed
                // O_j += P_j(i) V(i).  implied: P_j(i) was published after K(i+1) was
                // ready, which the transform published after V(i) landed, so only
                // P_j(i) is waited for; otherwise (the q-tile's last PV) V(i) too.
                // The unit's first PV into O_j waits until the previous unit's
                // epilogue has read O_j.
                auto issue_pv = [&](int j, int i, bool implied) -> bool {
                    if (i == 0 && !mbar_wait(smem_u32(&bars->o_free[j]), ((ph >> (4 + j)) & 1u) ^ 1u, abort))
                        return false;
                    if (!mbar_wait(smem_u32(&bars->p_ready[j]), ((ph >> (2 + j)) ^ (uint32_t)i) & 1u, abort))
                        return false;
                    const int g = g0 + i;
                    if (!implied && v_seen != i) {
                        if (!mbar_wait(smem_u32(&bars->v_full[g % VSTAGES]), (uint32_t)((g / VSTAGES) & 1), abort))
                            return false;
                        v_seen = i;
                    }
                    tc_fence_after();
                    const uint32_t dv = dV0 + (uint32_t)(g % VSTAGES) * TILE_DESC;
                    const uint32_t d = tmem + 256 + j * 128, ptm = tmem + j * 128;
                    mma_ts_steps<0, 8, MN_MAJOR_PAGE>(d, ptm, dv, idO, i > 0 ? 1u : 0u);
                    return true;
                };
                for (int i = 0; i < n_tiles && ok; ++i) {
                    const int g = g0 + i, k = g % KSTAGES;
                    bool k_in = false;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (!ok) break;
                        if (i < (j ? nt1 : nt0)) {
                            // for i > 0, K(i) is implied by P_j(i-1) (see issue_pv)
                            if (i > 0 && !(ok = issue_pv(j, i - 1, true))) break;
                            if (i > 0) {
                                k_in = true;
                            } else if (!k_in) {
                                if (!(ok = mbar_wait(smem_u32(&bars->k_ready[k]), (uint32_t)((g / KSTAGES) & 1), abort)))
                                    break;
                                tc_fence_after();
                                k_in = true;
                            }
                            const uint32_t dk = dK0 + (uint32_t)k * TILE_DESC, dq = dQ0 + (uint32_t)j * TILE_DESC;
                            const uint32_t d = tmem + j * 128;
                            mma_ss_steps<0, 8, K_MAJOR_128, K_MAJOR_128>(d, dq, dk, idS, 0u);
                            umma_commit(smem_u32(&bars->s_full[j]));
                        } else if (i == (j ? nt1 : nt0) && i > 0) {
                            if (!(ok = issue_pv(j, i - 1, false))) break;
                            umma_commit(smem_u32(&bars->o_done[j]));
                        }
                    }
                    if (!ok) break;
                    umma_commit(smem_u32(&bars->k_empty[k]));                             // K(i) read by S(i)
                    if (i > 0) umma_commit(smem_u32(&bars->v_empty[(g - 1) % VSTAGES]));  // V(i-1) read by PV(i-1)
                    if (i == n_tiles - 1) umma_commit(smem_u32(&bars->q_empty));          // the unit's last S read Q
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (ok && (j ? nt1 : nt0) == n_tiles) {
                        if (!(ok = issue_pv(j, n_tiles - 1, false))) break;
                        umma_commit(smem_u32(&bars->o_done[j]));
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&bars->v_empty[(g0 + n_tiles - 1) % VSTAGES]));  // V(last) read by the last PVs
                ph ^= 1u | ((uint32_t)(nt0 & 1) << 2) | ((uint32_t)(nt1 & 1) << 3) |
                      (nt0 > 0 ? 16u : 0u) | (nt1 > 0 ? 32u : 0u);
                g0 += n_tiles;
            }
            if (!ok) {
                // let issued MMAs drain before TMEM is released
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 1000000ull) {
                }
            }
        }
        __syncwarp();
        named_bar_sync(2, PF_THREADS);
    } else if (wg == 0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_XFORM));
        // ================================================ transform WG ====
        // K tiles: thread handles pair-chunk u8 = tid % 8 of rows r0 + 16 m.
        const int u8 = tid & 7, r0 = tid >> 3;
        float2 dcs[4], dsn[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 s0 = bars->step16[8 * u8 + 2 * e], s1 = bars->step16[8 * u8 + 2 * e + 1];
            dcs[e] = make_float2(s0.x, s1.x);
            dsn[e] = make_float2(s0.y, s1.y);
        }
        // Phase state over the CTA's units: g0 = KV tiles before the unit modulo
        // 12 (stage and phase of the 3-stage K and 2-stage V rings), wu = work
        // units modulo 4 (range-verdict slot and phase).
        int g0 = 0, wu = 0;
        bool ok = true;
        for (int kk = 0; ok; ++kk) {
            PfUnit un;
            if (!(ok = read_unit(bars, kk, abort, un)) || un.end) break;
            const int n_tiles = max(un.nt0, un.nt1);
            if (un.bad || n_tiles == 0) continue;
            uint32_t range = 0;
            // Angles of the thread's next K row: an exact anchor every 4 tiles, 16-position
            // steps in between (the rows r0 + 16 m of consecutive tiles continue one
            // sequence), so at most 32 steps follow an anchor; anchoring every tile
            // spent 8 sin / cos per thread and tile (about 1% of prefill_long).
            float2 c[4], sn[4];
            for (int i = 0; i < n_tiles; ++i) {
                const int g = g0 + i, k = g % KSTAGES;
                if (!(ok = mbar_wait(smem_u32(&bars->k_full[k]), (uint32_t)((g / KSTAGES) & 1), abort))) break;
                uint8_t* kt = sm + OFF_K + k * PF_TILE_BYTES;
                const int t0 = i * PF_BN;
                if ((i & 3) == 0) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        rope_cos_sin((uint32_t)(t0 + r0), bars->turns[8 * u8 + 2 * e], c[e].x, sn[e].x);
                        rope_cos_sin((uint32_t)(t0 + r0), bars->turns[8 * u8 + 2 * e + 1], c[e].y, sn[e].y);
                    }
                }
#pragma unroll 1
                for (int m = 0; m < 8; ++m) {
                    const int r = r0 + 16 * m;
                    const uint32_t off = sw_off(r, u8);
                    if (t0 + r < un.n_keys) range = rotate_chunk_f16(kt + off, kt + 16384 + off, c, sn, range);
                    rope_step(c, sn, dcs, dsn);
                }
                fence_proxy_async_smem();
                // K(i) is published only once V(i-1) has landed, so whoever has seen
                // K(i) ready may also read V(i-1) (the MMA issuer relies on it).
                if (i > 0 && !(ok = mbar_wait(smem_u32(&bars->v_full[(g - 1) % VSTAGES]),
                                              (uint32_t)(((g - 1) / VSTAGES) & 1), abort)))
                    break;
                mbar_arrive(smem_u32(&bars->k_ready[k]));
            }
            if (!ok) break;
            // the unit's FP16 range verdict for the softmax epilogues
            const int slot = wu & 1;
            if (!(ok = mbar_wait(smem_u32(&bars->r_empty[slot]), (uint32_t)(((wu >> 1) & 1) ^ 1), abort))) break;
            bars->r_flag[slot][tid] = range_exceeded(range) ? 1 : 0;
            mbar_arrive(smem_u32(&bars->r_full[slot]));
            g0 = (g0 + n_tiles) % 12;
            wu = (wu + 1) & 3;
        }
        named_bar_sync(2, PF_THREADS);
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REG_SOFTMAX));
        // =========================================== softmax WG j ======
        const int j = wg - 1;
        const int r = tid - 128 * wg;  // accumulator row == TMEM lane
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + j * 128, tO = tmem + 256 + j * 128;
        const float scl = a.qk_scale_log2;
        const float nanv = __int_as_float(0x7fc00000);
        // Phase state over the CTA's units: g0 = KV tiles before the unit modulo 6
        // (stage and phase of the K ring), ph bit 0 s_full (this q-tile's tiles),
        // bit 1 o_done, bits 2-3 work units modulo 4 (range-verdict slot, phase).
        // The unit descriptor is read from its slot where needed and the slot
        // released after the unit's epilogue, so little stays live across the
        // tile loop.
        int g0 = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int kk = 0;; ++kk) {
            const int uslot = kk & 1;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->u_full[uslot]), (uint32_t)((kk >> 1) & 1), abort))))
                break;
            const volatile PfUnit* un = &bars->unit[uslot];
            if (un->end) break;
            const int s0 = 2 * un->pair * rph + j * rph;
            const int n_tiles = max(un->nt0, un->nt1);
            if (un->bad || n_tiles == 0) {
                write_qtile_rows(a, RowMap{un->b, un->qn, un->qbase, ragged}, un->kvh, s0, r, un->bad ? nanv : -INFINITY);
                mbar_arrive(smem_u32(&bars->u_empty[uslot]));
                continue;
            }
            int n_vis;
            {
                const int s = s0 + r % rph;
                const int p = s < un->qn ? a.position_ids[un->qbase + s] : -1;
                const int kv_len = un->kv_len;
                n_vis = p < 0 ? 0 : (p >= kv_len ? kv_len : p + 1);
            }
            const int nt = j ? un->nt1 : un->nt0;
            {
                // Q of this q-tile: thread r rotates row r at its own position (the
                // positions come with the Q load), FP16 in place; only the row's own
                // queries count for the range check (in a ragged batch the rows past
                // its end hold the next row's queries).
                uint32_t range = 0;
                const int slot = (ph >> 2) & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->q_full), (ph >> 2) & 1u, abort));
                if (ok) {
                    const int pq = bars->qpos[j * rph + r % rph];
                    const bool own = pq >= 0;
                    const int p = own ? pq : 0;
                    uint8_t* qt = sm + OFF_Q + j * PF_TILE_BYTES;
#pragma unroll 1
                    for (int u = 0; u < 8; ++u) {
                        float2 c[4], sn[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            rope_cos_sin((uint32_t)p, bars->turns[8 * u + 2 * e], c[e].x, sn[e].x);
                            rope_cos_sin((uint32_t)p, bars->turns[8 * u + 2 * e + 1], c[e].y, sn[e].y);
                        }
                        const uint32_t off = sw_off(r, u);
                        const uint32_t nr = rotate_chunk_f16(qt + off, qt + 16384 + off, c, sn, range);
                        if (own) range = nr;
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(smem_u32(&bars->q_ready));
                    // this row's verdict joins the transform's for the unit's epilogues
                    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->r_empty[slot]), ((ph >> 3) & 1u) ^ 1u, abort));
                    if (ok) {
                        const bool any_big = __any_sync(0xffffffffu, range_exceeded(range));
                        if (lane == 0) bars->r_flag[slot][128 + 4 * j + (warp & 3)] = any_big ? 1 : 0;
                        mbar_arrive(smem_u32(&bars->r_full[slot]));
                    }
                }
            }
            float m = -INFINITY, l = 0.0f;
            for (int i = 0; i < nt && ok; ++i) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[j]), (ph ^ (uint32_t)i) & 1u, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // P_j(i) is published only once K(i+1) is ready when S_j(i+1) follows,
                // so the MMA issuer need not wait for K (or V(i), see the transform).
                // Probed here, confirmed before the arrive: the latency overlaps the math.
                const bool need_k = i + 1 < nt;
                const int gn = g0 + i + 1;
                const int kn = gn % KSTAGES;
                const uint32_t kpar = (uint32_t)((gn / KSTAGES) & 1);
                const bool k_seen = !need_k || mbar_test(smem_u32(&bars->k_ready[kn]), kpar);
                uint32_t xr[128];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    tmem_ld32(tS + lane_addr + c4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&xr[c4 * 32]));
                tmem_ld_wait();
                const int lim = n_vis - i * PF_BN;  // columns < lim are visible
                // Mask only where some row of the warp ends inside this tile.
                if (__any_sync(0xffffffffu, lim < PF_BN)) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) xr[c] = c < lim ? xr[c] : 0xff800000u;  // -inf
                }
                // Row max on the raw scores (scale > 0 commutes with max), 4 chains.
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int c = 0; c < 128; c += 4) {
                    mx0 = fmaxf(mx0, __uint_as_float(xr[c]));
                    mx1 = fmaxf(mx1, __uint_as_float(xr[c + 1]));
                    mx2 = fmaxf(mx2, __uint_as_float(xr[c + 2]));
                    mx3 = fmaxf(mx3, __uint_as_float(xr[c + 3]));
                }
                const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scl;
                float alpha = 1.0f;
                bool resc = false;
                if (mt > m + RESCALE_SLACK) {
                    alpha = ex2(m - mt);  // 0 when m = -inf
                    m = mt;
                    resc = true;
                }
                // p = 2^(x * scale - m): one packed FMA per pair, packed row sum.  A row
                // with nothing visible yet (m = -inf, every x = -inf) gives 2^-inf = 0.
                const float nm = (m == -INFINITY) ? 0.0f : -m;
                const float2 sc2 = make_float2(scl, scl), nm2 = make_float2(nm, nm);
                float2 acc2 = make_float2(0.0f, 0.0f);
                // P packed as BF16 pairs into xr[0..63] (each slot is rewritten only
                // after both of its sources have been read).
#pragma unroll
                for (int c = 0; c < 128; c += 2) {
                    const float2 t = ffma2(make_float2(__uint_as_float(xr[c]), __uint_as_float(xr[c + 1])), sc2, nm2);
                    const float2 e = make_float2(ex2(t.x), ex2(t.y));
                    acc2 = fadd2(acc2, e);
                    xr[c >> 1] = pack_bf16x2(e.x, e.y);
                }
                const float rs = acc2.x + acc2.y;
                l = l * alpha + rs;
                // S_j(i) complete implies PV_j(i-1) complete (MMAs of one issuer
                // retire in order), so O_j is stable and S_j's columns may take P_j(i).
                if (i > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t rr[32];
                        tmem_ld32(tO + lane_addr + c4 * 32, rr);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 32; ++q) rr[q] = __float_as_uint(__uint_as_float(rr[q]) * alpha);
                        tmem_st32(tO + lane_addr + c4 * 32, rr);
                    }
                }
                tmem_st32(tS + lane_addr, *reinterpret_cast<uint32_t(*)[32]>(&xr[0]));
                tmem_st32(tS + lane_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&xr[32]));
                tmem_st_wait();
                if (!__all_sync(0xffffffffu, k_seen || mbar_wait(smem_u32(&bars->k_ready[kn]), kpar, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&bars->p_ready[j]));
            }
            // ---- epilogue ----
            if (ok && nt > 0) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->o_done[j]), (ph >> 1) & 1u, abort));
            bool range_bad = false;
            if (ok) {  // the transform's verdict on this unit's inputs
                const int slot = (ph >> 2) & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->r_full[slot]), (ph >> 3) & 1u, abort));
                if (ok) {
                    const uint4* f = reinterpret_cast<const uint4*>(bars->r_flag[slot]);
                    uint32_t any = 0;
#pragma unroll
                    for (int q = 0; q < 9; ++q) {
                        const uint4 x = f[q];
                        any |= x.x | x.y | x.z | x.w;
                    }
                    range_bad = any != 0;
                    mbar_arrive(smem_u32(&bars->r_empty[slot]));
                }
            }
            const RowMap rm{un->b, un->qn, un->qbase, ragged};
            const int kvh = un->kvh;
            if (!ok) {  // a wait gave up: this unit's rows and the CTA's later units are written as failed
                write_qtile_rows(a, rm, kvh, s0, r, nanv);
                for (int k2 = kk + 1; !ragged; ++k2) {
                    const long long u2 = cta_unit(k2, cta, grid);
                    if (u2 >= total) break;
                    int b2, kvh2, pair2;
                    padded_unit(a, u2, b2, kvh2, pair2);
                    write_qtile_rows(a, RowMap{b2, a.Sq, b2 * a.Sq, false}, kvh2, 2 * pair2 * rph + j * rph, r, nanv);
                }
                if (r == 0 && a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
                break;
            }
            const int g = r / rph, s = s0 + r % rph;
            const bool valid = s < rm.qn;
            const int h = kvh * a.G + g;
            uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + rm.at(a, h, valid ? s : 0) * HEAD_DIM);
            if (nt > 0) {
                tc_fence_after();
                const bool zero = range_bad || !(l > 0.0f);
                const float inv_l = zero ? 0.0f : 1.0f / l;
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t rr[32];
                    tmem_ld32(tO + lane_addr + c4 * 32, rr);
                    tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int q = 0; q < 32; q += 8) {
                            float f[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(rr[q + e]) * inv_l;
                            o[(c4 * 32 + q) / 8] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                                              pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                        }
                    }
                }
                // O_j has been read: the next unit's first PV may overwrite it
                tc_fence_before();
                mbar_arrive(smem_u32(&bars->o_free[j]));
                if (valid)
                    a.lse[rm.at(a, h, s)] =
                        range_bad ? nanv : (l > 0.0f ? (m + log2f(l)) * 0.693147180559945309f : -INFINITY);
                if (range_bad && r == 0 && a.status) atomicOr(a.status, RK_STATUS_RANGE);
            } else if (valid) {
                for (int d = 0; d < HEAD_DIM / 8; ++d) o[d] = make_uint4(0, 0, 0, 0);
                a.lse[rm.at(a, h, s)] = range_bad ? nanv : -INFINITY;
            }
            mbar_arrive(smem_u32(&bars->u_empty[uslot]));
            g0 = (g0 + n_tiles) % 6;
            ph ^= (uint32_t)(nt & 1) | (nt > 0 ? 2u : 0u);
            ph = (ph & 3u) | ((((ph >> 2) + 1u) & 3u) << 2);
        }
        named_bar_sync(2, PF_THREADS);
    }

    // ---- teardown: every role has passed barrier 2; no MMA or TMEM access is in flight ----
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    pdl_tail();
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                           const PrefillArgs& a, cudaStream_t stream, bool overlap_previous) {
    static std::atomic<uint64_t> configured{0};
    static std::atomic<int> sm_count[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load() & bit)) {
        e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    int nsm = dev < 64 ? sm_count[dev].load() : 0;
    if (nsm <= 0) {
        e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (dev < 64) sm_count[dev].store(nsm);
    }
    // padded: a persistent grid of at most one CTA per SM over the units;
    // ragged: one CTA per unit and KV head
    const long long units = (long long)a.B * a.Hkv * ((a.n_qtiles + 1) / 2);
    const long long grid = a.qo_indptr ? (long long)a.ragged_units * a.Hkv : (units < nsm ? units : nsm);
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (!overlap_previous) {
        prefill_kernel<<<(unsigned)grid, PF_THREADS, PF_SMEM_BYTES, stream>>>(qm, km, vm, a);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(PF_THREADS);
    cfg.dynamicSmemBytes = PF_SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    std::memset(&attr, 0, sizeof attr);
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_kernel, qm, km, vm, a);
}

}  // namespace rk
