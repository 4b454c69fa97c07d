// backward_tc.cu -- dk / dv of the deterministic prefill backward on the
// 5th-gen tensor cores (tcgen05 MMA into TMEM, TMA operand staging).
//
// Same operation and determinism contract as backward.cu ("Add FlashInfer
// RoPE-fused paged attention scaffold", scope table, Backward row): for a tile
// of 128 keys of one (row, KV head), over the query blocks that see it in
// ascending order,
//   S^T = K' Q'^T,  dP^T = V dout^T,
//   P^T = exp(S^T - lse),  dS^T = P^T (dP^T - delta)        (per query column)
//   dV += P^T dout,  dK' += scale dS^T Q',
// and at the end dk = R(t)^T dK' is written into the page layout.  One CTA
// owns its 128 keys for the whole walk, so every dk / dv element is summed in
// one fixed order (no atomics, no split).
//
// A query block is 128 accumulator columns = (128 / G) positions x the G
// query heads of the KV head, laid out like the forward's q-tile.  TMEM
// (512 columns): S^T [0,128), dP^T [128,256), dV [256,384), dK' [384,512).
// The same shared tiles serve both operand orientations: Q' and dout are
// K-major B operands of the score products and MN-major B operands of the
// dV / dK' products; K' and V are K-major A operands.  Roles (512 threads):
//   warpgroup 0   transform: rotates the key tile once and each query block in
//                 place (FP32 math, FP16 out), stages the block's lse / delta /
//                 positions;
//   warpgroups 1, 2  gradient of the softmax on query columns 0..63 / 64..127
//                 (thread = key row = TMEM lane): P^T (BF16) and dS^T (FP16)
//                 written back over S^T / dP^T; at the end warpgroup 1 writes
//                 dk, warpgroup 2 dv;
//   warp 12       TMA producer (the key and value tiles once, query / dout
//                 blocks double-buffered); warp 13 MMA issuer.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "rk_device.cuh"

namespace rk {

namespace {

constexpr int BT_THREADS = 512;
constexpr int BT_KEYS = 128;  // keys per CTA (MMA M)
constexpr int BT_QB = 128;    // query columns per block (MMA N)
constexpr int WARP_TMA = 12;
constexpr int WARP_MMA = 13;
constexpr uint32_t BT_TMEM_COLS = 512;
constexpr int BT_TILE = BT_KEYS * HEAD_DIM * 2;  // 32 KiB 16-bit tile

// setmaxnreg split (sum 4 x 128 = the 512 x 128 registers the CTA launches with)
constexpr int BT_REG_XFORM = 104;
constexpr int BT_REG_GRAD = 184;
constexpr int BT_REG_CTRL = 40;
static_assert(BT_REG_XFORM + 2 * BT_REG_GRAD + BT_REG_CTRL == 4 * 128, "register split must sum to the launch budget");

// Shared memory carve (1024-byte aligned base).
constexpr int BT_OFF_K = 0;
constexpr int BT_OFF_V = BT_OFF_K + BT_TILE;
constexpr int BT_OFF_Q = BT_OFF_V + BT_TILE;      // two stages
constexpr int BT_OFF_DO = BT_OFF_Q + 2 * BT_TILE;  // two stages
constexpr int BT_OFF_LD = BT_OFF_DO + 2 * BT_TILE; // two stages of [lse2 | delta | position] x 128
constexpr int BT_LD_BYTES = 3 * BT_QB * 4 + 16;  // + the smallest position of each 32-column quarter
constexpr int BT_OFF_BAR = BT_OFF_LD + 2 * BT_LD_BYTES;
constexpr int BT_CTRL_BYTES = 2048;
constexpr int BT_SMEM = BT_OFF_BAR + BT_CTRL_BYTES;
static_assert(BT_SMEM <= 232448, "shared memory above the 227 KiB opt-in limit");

struct BtBars {
    uint64_t k_full, v_full;
    uint64_t q_full[2], q_ready[2], q_empty[2];
    uint64_t s_full, p_ready, done;
    uint64_t never;  // nothing arrives: the timeout drill's wait
    uint32_t tmem_base;
    PipeCtl pipe;
    int range_bad;
    int first_block;
    uint64_t turns[ROPE_PAIRS];
    float2 step16[ROPE_PAIRS];
};
static_assert(sizeof(BtBars) <= BT_CTRL_BYTES, "control block exceeds its reservation");

// D[tmem] (+)= A[tmem] * B[smem] over 8 k-steps of 16 query rows whose packed
// A columns sit at 8 ks (ks < 4, written by warpgroup 1) and 32 + 8 ks
// (ks >= 4, warpgroup 2): each warpgroup packs its 64 columns into the first
// half of the 64 TMEM columns it read.
template <int KS, int LB>
__device__ __forceinline__ void mma_ts_split(uint32_t d, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                             uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 at, bl;\n\t.reg .b64 db;\n\t"
        "add.u32 at, %1, %5;\n\tadd.u32 bl, %2, %6;\n\t"
        "mov.b64 db, {bl, %4};\n\t"
        "setp.ne.b32 p, %7, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(DESC_HI), "n"(KS < 4 ? KS * 8 : 32 + KS * 8),
        "n"(kstep_off(LB, KS)), "r"(KS > 0 ? 1u : acc0)
        : "memory");
    if constexpr (KS + 1 < 8) mma_ts_split<KS + 1, LB>(d, a_tmem, b_lo, idesc, acc0);
}


// ---------------------------------------------------------- rotation ----
// The backward reads every query block once per key tile and every key tile
// once per query tile, so RoPE is applied once per call instead: q and each
// row's keys are rotated (FP32 math, exact angles from the fixed-point rates)
// and stored as FP16 in the caller's workspace, the keys (and a copy of V)
// gathered from their pages into logical token order [B, Hkv, W * 16, D], so
// that a 128-key tile is two 16 KiB copies instead of 16 page-sized ones.  A
// pre-RoPE element with |x| >= 2^15 (whose rotation may leave the FP16 range)
// is stored as infinity: the gradients it enters come out non-finite and are
// reported as RK_STATUS_RANGE by the kernels below.
__device__ __forceinline__ void rotate_store(const uint4* src, uint4* dst, int c, int pos, const uint64_t* turns) {
    uint4 lo = __ldg(src + c), hi = __ldg(src + c + 8);
    const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w}, hw[4] = {hi.x, hi.y, hi.z, hi.w};
    uint32_t big = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) big |= (uint32_t)range_exceeded(__vmaxu2(lw[k] & 0x7fff7fffu, hw[k] & 0x7fff7fffu));
    float2 cs[4], sn[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        rope_cos_sin((uint32_t)pos, turns[8 * c + 2 * e], cs[e].x, sn[e].x);
        rope_cos_sin((uint32_t)pos, turns[8 * c + 2 * e + 1], cs[e].y, sn[e].y);
    }
    rotate_regs_f16(lo, hi, cs, sn, 0u);
    if (big) lo = hi = make_uint4(0x7c007c00u, 0x7c007c00u, 0x7c007c00u, 0x7c007c00u);
    dst[c] = lo;
    dst[c + 8] = hi;
}

// one thread per (query row, chunk pair): q_rot[b, h, s] = R(position) q[b, h, s]
__global__ void __launch_bounds__(256) rotate_q_kernel(const __grid_constant__ BackwardArgs a) {
    const long long n = (long long)a.B * a.Hq * a.Sq * 8;
    for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < n; it += (long long)gridDim.x * blockDim.x) {
        const long long row = it >> 3;  // (b * Hq + h) * Sq + s
        const int c = (int)(it & 7), s = (int)(row % a.Sq), b = (int)(row / ((long long)a.Hq * a.Sq));
        const int p = a.position_ids[(size_t)b * a.Sq + s];
        rotate_store(reinterpret_cast<const uint4*>(a.q) + row * 16, reinterpret_cast<uint4*>(a.q_rot) + row * 16, c,
                     max(p, 0), a.rope_turns);
    }
}

// one thread per (row, KV head, token, chunk pair): k_lin[b, kvh, t] = R(t) K(b, t),
// v_lin[b, kvh, t] = V(b, t) for t < kv_len, zeros up to W * 16; unsafe lengths
// or page ids are skipped (the kernels report them)
__global__ void __launch_bounds__(256) rotate_k_kernel(const __grid_constant__ BackwardArgs a) {
    const int T = a.W * PAGE;
    const long long per_row = (long long)a.Hkv * T * 8;
    const long long n = (long long)a.B * per_row;
    for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < n; it += (long long)gridDim.x * blockDim.x) {
        const int b = (int)(it / per_row);
        const long long rem = it % per_row;
        const int c = (int)(rem & 7), t = (int)((rem >> 3) % T), kvh = (int)((rem >> 3) / T);
        const int kv_len = a.kv_lens[b];
        if (kv_len < 0 || kv_len > T) continue;
        const size_t l = ((size_t)b * a.Hkv + kvh) * T + t;  // 256-byte linear row
        uint4* kd = reinterpret_cast<uint4*>(a.k_lin) + l * 16;
        uint4* vd = reinterpret_cast<uint4*>(a.v_lin) + l * 16;
        if (t >= kv_len) {  // zeros: tiles read whole rows of 128 tokens, and 0 * NaN would not vanish
            kd[c] = kd[c + 8] = vd[c] = vd[c + 8] = make_uint4(0, 0, 0, 0);
            continue;
        }
        const int pg = __ldg(a.block_table + (size_t)b * a.W + t / PAGE);
        if (pg < 0 || pg >= a.num_pages) continue;
        const size_t e = ((size_t)pg * PAGE + t % PAGE) * a.Hkv + kvh;  // 256-byte cache row
        rotate_store(reinterpret_cast<const uint4*>(a.k_cache) + e * 16, kd, c, t, a.rope_turns);
        const uint4* vs = reinterpret_cast<const uint4*>(a.v_cache) + e * 16;
        vd[c] = __ldg(vs + c);
        vd[c + 8] = __ldg(vs + c + 8);
    }
}

// Write rows [0, n_rows) of a key tile's dk and dv as zeros (no query sees it).
__device__ __forceinline__ void write_zero_tile(const BackwardArgs& a, const int32_t* bt, int t0, int n_rows,
                                                int kvh) {
    const size_t kstride = (size_t)a.Hkv * HEAD_DIM;
    for (int i = threadIdx.x; i < n_rows * (HEAD_DIM / 4); i += blockDim.x) {
        const int r = i / (HEAD_DIM / 4), c = i % (HEAD_DIM / 4), t = t0 + r;
        const size_t off = ((size_t)__ldg(bt + t / PAGE) * PAGE + t % PAGE) * kstride + (size_t)kvh * HEAD_DIM;
        reinterpret_cast<float4*>(a.dk + off)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4*>(a.dv + off)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

__global__ void __launch_bounds__(BT_THREADS, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                            const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                            const __grid_constant__ BackwardArgs a) {
    extern __shared__ __align__(1024) uint8_t sm[];
    BtBars* bars = reinterpret_cast<BtBars*>(sm + BT_OFF_BAR);
    const uint32_t s_base = smem_u32(sm);
    if (s_base & 1023u) {  // the swizzled operand layout needs a 1024-byte aligned base
        if (threadIdx.x == 0 && a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
    const int G = a.G, rph = BT_QB / G;
    const int units = a.B * a.Hkv;
    const int kt = (int)(blockIdx.x / units);  // first key tiles first: they are seen by the most queries
    const int b = (int)(blockIdx.x % units) / a.Hkv, kvh = (int)(blockIdx.x % units) % a.Hkv;
    const int t0 = kt * BT_KEYS;
    const int kv_len = a.kv_lens[b];
    if (kv_len < 0 || kv_len > a.W * PAGE) {  // nothing is known about the row's pages
        if (tid == 0 && kt == 0 && a.status) atomicOr(a.status, RK_STATUS_KVLEN);
        return;
    }
    const int n_rows = min(BT_KEYS, (kv_len + PAGE - 1) / PAGE * PAGE - t0);  // keys of the tile on the row's pages
    if (n_rows <= 0) return;
    const int n_pg = (n_rows + PAGE - 1) / PAGE;
    const int32_t* bt = a.block_table + (size_t)b * a.W + t0 / PAGE;  // this tile's table entries
    if (tid == 0) {
        bars->pipe.abort = 0;
        bars->pipe.limit_ns = wait_limit(a.wait_limit_ns);
        bars->range_bad = 0;
        mbar_init(smem_u32(&bars->never), 1);
        mbar_init(smem_u32(&bars->k_full), 1);
        mbar_init(smem_u32(&bars->v_full), 1);
        for (int j = 0; j < 2; ++j) {
            mbar_init(smem_u32(&bars->q_full[j]), 1);
            mbar_init(smem_u32(&bars->q_ready[j]), 128);
            mbar_init(smem_u32(&bars->q_empty[j]), 1);
        }
        mbar_init(smem_u32(&bars->s_full), 1);
        mbar_init(smem_u32(&bars->p_ready), 256);
        mbar_init(smem_u32(&bars->done), 1);
        fence_mbar_init();
        // first query position >= t0 (positions ascend along the row): its block
        int lo = 0, hi = a.Sq;
        const int32_t* pr = a.position_ids + (size_t)b * a.Sq;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (pr[mid] >= t0) hi = mid; else lo = mid + 1;
        }
        bars->first_block = lo / rph;
    }
    if (tid < ROPE_PAIRS) {
        bars->turns[tid] = a.rope_turns[tid];
        float c, s;
        rope_cos_sin((uint32_t)PAGE, a.rope_turns[tid], c, s);
        bars->step16[tid] = make_float2(c, s);
    }
    int pg_bad = 0;
    if (tid < n_pg) {
        const int pg = __ldg(bt + tid);
        pg_bad = (pg < 0) | (pg >= a.num_pages);
    }
    if (__syncthreads_or(pg_bad)) {  // the tile's pages are not safe to write
        if (tid == 0 && a.status) atomicOr(a.status, RK_STATUS_PAGE_OOB);
        return;
    }
    const int j0 = bars->first_block, nblk = max(0, (a.Sq + rph - 1) / rph - j0);
    if (nblk == 0) {
        write_zero_tile(a, bt - t0 / PAGE, t0, n_rows, kvh);
        return;
    }

    // ---- TMEM allocation (warp 13 owns it) ----
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(&bars->tmem_base), BT_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    PipeCtl* abort = &bars->pipe;
    const float nanv = __int_as_float(0x7fc00000);

    if (wg == 3) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BT_REG_CTRL));
        if (warp == WARP_TMA && lane == 0) {
            // ================================================ TMA producer ====
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
            prefetch_tmap(&qmap);
            prefetch_tmap(&omap);
            // key and value tiles from the linear workspace: two 128-token x 64-dim boxes each
            const uint32_t kb = smem_u32(&bars->k_full), vb = smem_u32(&bars->v_full);
            const int lrow = b * a.Hkv + kvh;
            mbar_arrive_expect_tx(kb, 2 * 16384);
            mbar_arrive_expect_tx(vb, 2 * 16384);
            tma_load_3d(s_base + BT_OFF_K, &kmap, kb, 0, t0, lrow);
            tma_load_3d(s_base + BT_OFF_K + 16384, &kmap, kb, 64, t0, lrow);
            tma_load_3d(s_base + BT_OFF_V, &vmap, vb, 0, t0, lrow);
            tma_load_3d(s_base + BT_OFF_V + 16384, &vmap, vb, 64, t0, lrow);
            // query / dout blocks, two stages
            int issued = 0;
            const int h0 = kvh * G;
            int s0 = j0 * rph;
            for (int jj = 0; jj < nblk; ++jj, s0 += rph) {
                const int st = jj & 1;
                const uint32_t q_empty = smem_u32(&bars->q_empty[0]) + 8 * st, fb = smem_u32(&bars->q_full[0]) + 8 * st;
                if (!mbar_wait(q_empty, (((uint32_t)jj >> 1) & 1u) ^ 1u, abort)) break;
                mbar_arrive_expect_tx(fb, 4 * 16384);
                const uint32_t dq = s_base + BT_OFF_Q + st * BT_TILE;
                tma_load_4d(dq, &qmap, fb, 0, s0, h0, b);
                tma_load_4d(dq + 16384, &qmap, fb, 64, s0, h0, b);
                tma_load_4d(dq + 2 * BT_TILE, &omap, fb, 0, s0, h0, b);
                tma_load_4d(dq + 2 * BT_TILE + 16384, &omap, fb, 64, s0, h0, b);
                ++issued;
            }
            if (pipe_aborted(abort)) {  // let the copies in flight land before the CTA's shared memory is released
                mbar_wait_drain(kb, 0);
                mbar_wait_drain(vb, 0);
                for (int jj = max(0, issued - 2); jj < issued; ++jj)
                    mbar_wait_drain(smem_u32(&bars->q_full[jj & 1]), (uint32_t)((jj >> 1) & 1));
            }
        } else if (warp == WARP_MMA && lane == 0) {
            // ================================================= MMA issuer ====
            // FP16 scores (format 0) and BF16 dout products; K-major A operands; B
            // K-major for the score products, MN-major (LBO 16 KiB) for dV / dK'.
            const uint32_t idS = (1u << 4) | ((uint32_t)(BT_QB >> 3) << 17) | ((uint32_t)(BT_KEYS >> 4) << 24);
            const uint32_t idP = idesc_bf16_f32(BT_KEYS, BT_QB, 0, 0);
            const uint32_t idV = idesc_bf16_f32(BT_KEYS, HEAD_DIM, 0, 1);
            const uint32_t idK = (1u << 4) | (1u << 16) | ((uint32_t)(HEAD_DIM >> 3) << 17) |
                                 ((uint32_t)(BT_KEYS >> 4) << 24);
            const uint32_t dK = desc_lo(s_base + BT_OFF_K, 16), dV = desc_lo(s_base + BT_OFF_V, 16);
            bool ok = (!a.timeout_drill || drill_wait(smem_u32(&bars->never), abort)) &&
                      mbar_wait(smem_u32(&bars->k_full), 0, abort) && mbar_wait(smem_u32(&bars->v_full), 0, abort);
            for (int jj = 0; jj < nblk && ok; ++jj) {
                const int st = jj & 1;
                if (!(ok = mbar_wait(smem_u32(&bars->q_ready[st]), (uint32_t)((jj >> 1) & 1), abort))) break;
                tc_fence_after();
                const uint32_t qa = s_base + BT_OFF_Q + st * BT_TILE, oa = s_base + BT_OFF_DO + st * BT_TILE;
                mma_ss_steps<0, 8, K_MAJOR_128, K_MAJOR_128>(tmem, dK, desc_lo(qa, 16), idS, 0u);
                mma_ss_steps<0, 8, K_MAJOR_128, K_MAJOR_128>(tmem + 128, dV, desc_lo(oa, 16), idP, 0u);
                umma_commit(smem_u32(&bars->s_full));
                if (!(ok = mbar_wait(smem_u32(&bars->p_ready), (uint32_t)(jj & 1), abort))) break;
                tc_fence_after();
                mma_ts_split<0, MN_MAJOR>(tmem + 256, tmem, desc_lo(oa, 16384), idV, jj > 0 ? 1u : 0u);
                mma_ts_split<0, MN_MAJOR>(tmem + 384, tmem + 128, desc_lo(qa, 16384), idK, jj > 0 ? 1u : 0u);
                umma_commit(smem_u32(&bars->q_empty[st]));  // Q'(jj) and dout(jj) read
            }
            if (ok) {
                umma_commit(smem_u32(&bars->done));
            } else {  // let issued MMAs drain before TMEM is released
                const uint64_t ts = global_timer_ns();
                while (global_timer_ns() - ts < 1000000ull) {
                }
            }
        }
        __syncwarp();
        named_bar_sync(2, BT_THREADS);
    } else if (wg == 0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BT_REG_XFORM));
        // ================================================= staging WG ====
        // q and K arrive rotated (FP16, workspace); this warpgroup stages each
        // block's lse (log2 domain), delta and positions for the gradient warps
        bool ok = true;
        for (int jj = 0; jj < nblk && ok; ++jj) {
            const int st = jj & 1;
            if (!(ok = mbar_wait(smem_u32(&bars->q_full[st]), (uint32_t)((jj >> 1) & 1), abort))) break;
            const int s0 = (j0 + jj) * rph;
            {  // lse (log2 domain), delta and position of column tid
                const int g = tid / rph, s = s0 + tid % rph;
                const bool valid = s < a.Sq;
                const size_t o = ((size_t)b * a.Hq + kvh * G + g) * a.Sq + s;
                float* ld = reinterpret_cast<float*>(sm + BT_OFF_LD + st * BT_LD_BYTES);
                ld[tid] = valid ? a.lse[o] * 1.4426950408889634074f : 0.0f;
                ld[BT_QB + tid] = valid ? a.delta[o] : 0.0f;
                const int pq = valid ? a.position_ids[(size_t)b * a.Sq + s] : -1;
                reinterpret_cast<int*>(ld)[2 * BT_QB + tid] = pq;
                const int pmin = __reduce_min_sync(0xffffffffu, pq);  // warp w holds columns 32 w .. 32 w + 31
                if (lane == 0) reinterpret_cast<int*>(ld)[3 * BT_QB + warp] = pmin;
            }
            mbar_arrive(smem_u32(&bars->q_ready[st]));
        }
        named_bar_sync(1, 384);

        named_bar_sync(2, BT_THREADS);
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(BT_REG_GRAD));
        // ================================================ softmax gradient ====
        const int hsel = wg - 1, c0 = 64 * hsel;  // query columns c0 .. c0 + 63
        const int r = tid - 128 * wg;             // key row == TMEM lane
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const int t = t0 + r;
        const bool key_ok = t < kv_len;
        const float scl = a.qk_scale_log2;
        bool over = false, ok = true;
        for (int jj = 0; jj < nblk; ++jj) {
            const int st = jj & 1;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full), (uint32_t)(jj & 1), abort)))) break;
            // the block's staged lse / delta / positions: q_ready(jj) is already
            // complete (S^T(jj) was issued after it); waiting orders their reads
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->q_ready[st]), (uint32_t)((jj >> 1) & 1), abort))))
                break;
            tc_fence_after();
            const float* ld = reinterpret_cast<const float*>(sm + BT_OFF_LD + st * BT_LD_BYTES);
            const int* lp = reinterpret_cast<const int*>(ld) + 2 * BT_QB;
            // 32 columns at a time; the packed pairs of columns c0 + 2i, 2i + 1 go
            // to TMEM column c0 + i, which this warpgroup has already read
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int cb = c0 + 32 * h;
                uint32_t xs[32], xd[32];  // packed results overwrite slots already read
                tmem_ld32(tmem + lane_addr + cb, xs);
                tmem_ld32(tmem + lane_addr + 128 + cb, xd);
                tmem_ld_wait();
                // every column (valid, position >= this key) sees every key row of the warp: no masks
                if (__all_sync(0xffffffffu, key_ok && t <= lp[BT_QB + (cb >> 5)])) {
                    const float2 sc2 = make_float2(scl, scl);
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 l4 = *reinterpret_cast<const float4*>(ld + cb + c);
                        const float4 d4 = *reinterpret_cast<const float4*>(ld + BT_QB + cb + c);
#pragma unroll
                        for (int e = 0; e < 4; e += 2) {
                            const float2 nl = e ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
                            const float2 nd = e ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
                            const float2 t2 =
                                ffma2(make_float2(__uint_as_float(xs[c + e]), __uint_as_float(xs[c + e + 1])), sc2, nl);
                            const float2 pp = make_float2(ex2(t2.x), ex2(t2.y));
                            const float2 ds = fmul2(
                                pp, fadd2(make_float2(__uint_as_float(xd[c + e]), __uint_as_float(xd[c + e + 1])), nd));
                            xs[(c + e) >> 1] = pack_bf16x2(pp.x, pp.y);
                            xd[(c + e) >> 1] = pack_f16x2(ds.x, ds.y);
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 l4 = *reinterpret_cast<const float4*>(ld + cb + c);
                        const float4 d4 = *reinterpret_cast<const float4*>(ld + BT_QB + cb + c);
                        const int4 p4 = *reinterpret_cast<const int4*>(lp + cb + c);
                        const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
                        const int pv[4] = {p4.x, p4.y, p4.z, p4.w};
                        float pp[4], ds[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const bool vis = key_ok && t <= pv[e];
                            pp[e] = vis ? ex2(__uint_as_float(xs[c + e]) * scl - lv[e]) : 0.0f;
                            ds[e] = vis ? pp[e] * (__uint_as_float(xd[c + e]) - dv[e]) : 0.0f;
                        }
                        xs[c >> 1] = pack_bf16x2(pp[0], pp[1]);
                        xs[(c >> 1) + 1] = pack_bf16x2(pp[2], pp[3]);
                        xd[c >> 1] = pack_f16x2(ds[0], ds[1]);
                        xd[(c >> 1) + 1] = pack_f16x2(ds[2], ds[3]);
                    }
                }
                tmem_st16(tmem + lane_addr + c0 + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(&xs[0]));
                tmem_st16(tmem + lane_addr + 128 + c0 + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(&xd[0]));
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars->p_ready));
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->done), 0, abort));
        tc_fence_after();
        if (ok) {  // an operand or dS beyond the FP16 range (infinity) leaves dK' / dV non-finite
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_addr + (hsel ? 256 : 384) + 32 * c4, v);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; ++k) over |= !isfinite(__uint_as_float(v[k]));
            }
        }
        if (over) bars->range_bad = 1;
        named_bar_sync(1, 384);  // every range flag is set
        const bool bad_out = bars->range_bad != 0 || !ok;
        if (tid == 128 && bad_out && a.status) atomicOr(a.status, ok ? RK_STATUS_RANGE : RK_STATUS_TIMEOUT);
        // epilogue: warpgroup 1 writes dk = R(t)^T (scale dK'), warpgroup 2 writes dv;
        // dims i and i + 64 (a rotation pair) are loaded together, 32 of each at a
        // time.  The TMEM loads are warp-collective: every lane issues them, only
        // rows on the row's pages (r < n_rows) are written.
        const bool write_row = r < n_rows;
        const size_t off = write_row ? ((size_t)__ldg(bt + r / PAGE) * PAGE + t % PAGE) * ((size_t)a.Hkv * HEAD_DIM) +
                                           (size_t)kvh * HEAD_DIM
                                     : 0;
        float* dst = (hsel ? a.dv : a.dk) + off;
        const uint32_t col = tmem + lane_addr + (hsel ? 256 : 384);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            uint32_t lo[32], hi[32];
            if (ok) {  // warp-uniform
                tmem_ld32(col + 32 * h, lo);
                tmem_ld32(col + 64 + 32 * h, hi);
                tmem_ld_wait();
            }
            if (!write_row) continue;
            if (hsel == 0 && !bad_out) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float cth, sth;
                    rope_cos_sin((uint32_t)t, bars->turns[32 * h + i], cth, sth);
                    const float x = __uint_as_float(lo[i]) * a.sm_scale, y = __uint_as_float(hi[i]) * a.sm_scale;
                    lo[i] = __float_as_uint(x * cth + y * sth);
                    hi[i] = __float_as_uint(y * cth - x * sth);
                }
            }
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                float4 v = make_float4(__uint_as_float(lo[c]), __uint_as_float(lo[c + 1]), __uint_as_float(lo[c + 2]),
                                       __uint_as_float(lo[c + 3]));
                float4 w = make_float4(__uint_as_float(hi[c]), __uint_as_float(hi[c + 1]), __uint_as_float(hi[c + 2]),
                                       __uint_as_float(hi[c + 3]));
                if (bad_out) v = w = make_float4(nanv, nanv, nanv, nanv);
                *reinterpret_cast<float4*>(dst + 32 * h + c) = v;
                *reinterpret_cast<float4*>(dst + 64 + 32 * h + c) = w;
            }
        }
        named_bar_sync(2, BT_THREADS);
    }
    // ---- teardown: every role has passed barrier 2; no MMA or TMEM access is in flight ----
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, BT_TMEM_COLS);
    }
}


// ---------------------------------------------------------------- dq ----
// One CTA per (row b, KV head, query tile of 128 rows = 128 / G positions x
// the G query heads), latest tiles first (they see the most keys).  Q' and
// dout are loaded once; the key / value tiles of 128 keys stream through two
// stages in ascending order:
//   S = Q' K'^T,  dP = dout V^T,  P = exp(S - lse),  dS = P (dP - delta),
//   dQ' += dS K'   (dS written back over S as the A operand, K' read MN-major),
// and at the end dq = R(p)^T (scale dQ').  delta = rowsum(dout * out) of the
// tile's rows is formed first (from the staged dout tile and out) and written
// for the dk / dv kernel.  TMEM: S0 [0,128), S1 [128,256), dP [256,384),
// dQ' [384,512): S(i + 1) goes into the other S buffer while the gradient of
// tile i runs, so the tensor pipe does not wait for it.  Three K stages (K(i)
// is read by S(i) and dQ'(i), K(i + 1) by S(i + 1) meanwhile), two V stages.
constexpr int DT_KST = 3, DT_VST = 2;
constexpr int DT_OFF_Q = 0;
constexpr int DT_OFF_DO = DT_OFF_Q + BT_TILE;
constexpr int DT_OFF_K = DT_OFF_DO + BT_TILE;
constexpr int DT_OFF_V = DT_OFF_K + DT_KST * BT_TILE;
constexpr int DT_OFF_BAR = DT_OFF_V + DT_VST * BT_TILE;
constexpr int DT_SMEM = DT_OFF_BAR + BT_CTRL_BYTES;
static_assert(DT_SMEM <= 232448, "shared memory above the 227 KiB opt-in limit");

struct DqBars {
    uint64_t q_full;
    uint64_t k_full[DT_KST], k_empty[DT_KST], v_full[DT_VST], v_empty[DT_VST];
    uint64_t s_full, p_ready, done;
    uint64_t never;  // nothing arrives: the timeout drill's wait
    uint32_t tmem_base;
    PipeCtl pipe;
    int range_bad;
    int n_keys;
    int flags;
    uint64_t turns[ROPE_PAIRS];
    float2 step16[ROPE_PAIRS];
    float dpart[BT_QB];  // delta over dims 0..63 of each row (added to the other half's)
};
static_assert(sizeof(DqBars) <= BT_CTRL_BYTES, "control block exceeds its reservation");

__global__ void __launch_bounds__(BT_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                          const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const __grid_constant__ BackwardArgs a) {
    extern __shared__ __align__(1024) uint8_t sm[];
    DqBars* bars = reinterpret_cast<DqBars*>(sm + DT_OFF_BAR);
    const uint32_t s_base = smem_u32(sm);
    if (s_base & 1023u) {
        if (threadIdx.x == 0 && a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
    const int G = a.G, rph = BT_QB / G;
    const int units = a.B * a.Hkv;
    const int nqt = (a.Sq + rph - 1) / rph;
    const int qt = nqt - 1 - (int)(blockIdx.x / units);
    const int b = (int)(blockIdx.x % units) / a.Hkv, kvh = (int)(blockIdx.x % units) % a.Hkv;
    const int s0 = qt * rph;
    const int kv_len = a.kv_lens[b];
    const int32_t* bt = a.block_table + (size_t)b * a.W;
    const int32_t* pos_row = a.position_ids + (size_t)b * a.Sq;
    if (tid == 0) {
        bars->pipe.abort = 0;
        bars->pipe.limit_ns = wait_limit(a.wait_limit_ns);
        bars->range_bad = 0;
        mbar_init(smem_u32(&bars->never), 1);
        mbar_init(smem_u32(&bars->q_full), 1);
        for (int j = 0; j < DT_KST; ++j) {
            mbar_init(smem_u32(&bars->k_full[j]), 1);
            mbar_init(smem_u32(&bars->k_empty[j]), 1);
        }
        for (int j = 0; j < DT_VST; ++j) {
            mbar_init(smem_u32(&bars->v_full[j]), 1);
            mbar_init(smem_u32(&bars->v_empty[j]), 1);
        }
        mbar_init(smem_u32(&bars->s_full), 1);
        mbar_init(smem_u32(&bars->p_ready), 256);
        mbar_init(smem_u32(&bars->done), 1);
        fence_mbar_init();
        // keys the tile sees: up to its last position (positions ascend along the row)
        int fl = (kv_len < 0 || kv_len > a.W * PAGE) ? RK_STATUS_KVLEN : 0;
        const int p_last = pos_row[min(s0 + rph, a.Sq) - 1];
        const int p_first = pos_row[s0];
        if (p_first < 0) fl |= RK_STATUS_POSITION;
        bars->flags = fl;
        bars->n_keys = fl ? 0 : min(p_last + 1, kv_len);
    }
    if (tid < ROPE_PAIRS) {
        bars->turns[tid] = a.rope_turns[tid];
        float c, s;
        rope_cos_sin((uint32_t)PAGE, a.rope_turns[tid], c, s);
        bars->step16[tid] = make_float2(c, s);
    }
    __syncthreads();
    const int n_keys = bars->n_keys;
    {  // page ids of every key the tile reads
        int bad = 0;
        for (int i = tid; i < (n_keys + PAGE - 1) / PAGE; i += BT_THREADS) {
            const int pg = __ldg(bt + i);
            bad |= (pg < 0) | (pg >= a.num_pages);
        }
        if (__syncthreads_or(bad) && tid == 0) bars->flags |= RK_STATUS_PAGE_OOB;
        __syncthreads();
    }
    const int flags = bars->flags;
    const int n_tiles = (n_keys + BT_KEYS - 1) / BT_KEYS;
    const float nanv = __int_as_float(0x7fc00000);
    if (flags || n_tiles == 0) {  // unsafe metadata (NaN, status) or no visible key (dq = 0, delta = 0)
        if (flags && tid == 0 && a.status) atomicOr(a.status, flags);
        for (int i = tid; i < BT_QB * (HEAD_DIM / 4); i += BT_THREADS) {
            const int r = i / (HEAD_DIM / 4), c = i % (HEAD_DIM / 4), s = s0 + r % rph;
            if (s >= a.Sq) continue;
            const size_t o = ((size_t)b * a.Hq + kvh * G + r / rph) * a.Sq + s;
            const float v = flags ? nanv : 0.0f;
            reinterpret_cast<float4*>(a.dq + o * HEAD_DIM)[c] = make_float4(v, v, v, v);
            if (c == 0) a.delta[o] = v;
        }
        return;
    }

    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(&bars->tmem_base), BT_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    PipeCtl* abort = &bars->pipe;

    if (wg == 3) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BT_REG_CTRL));
        if (warp == WARP_TMA && lane == 0) {
            // ================================================ TMA producer ====
            prefetch_tmap(&qmap);
            prefetch_tmap(&omap);
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
            const uint32_t qb = smem_u32(&bars->q_full);
            mbar_arrive_expect_tx(qb, 4 * 16384);
            tma_load_4d(s_base + DT_OFF_Q, &qmap, qb, 0, s0, kvh * G, b);
            tma_load_4d(s_base + DT_OFF_Q + 16384, &qmap, qb, 64, s0, kvh * G, b);
            tma_load_4d(s_base + DT_OFF_DO, &omap, qb, 0, s0, kvh * G, b);
            tma_load_4d(s_base + DT_OFF_DO + 16384, &omap, qb, 64, s0, kvh * G, b);
            int issued = 0;
            const int lrow = b * a.Hkv + kvh;
            for (int i = 0; i < n_tiles; ++i) {
                const int ks = i % DT_KST, vs = i % DT_VST;
                if (!mbar_wait(smem_u32(&bars->k_empty[ks]), (((uint32_t)(i / DT_KST)) & 1u) ^ 1u, abort)) break;
                if (!mbar_wait(smem_u32(&bars->v_empty[vs]), (((uint32_t)(i / DT_VST)) & 1u) ^ 1u, abort)) break;
                const uint32_t kb = smem_u32(&bars->k_full[ks]), vb = smem_u32(&bars->v_full[vs]);
                mbar_arrive_expect_tx(kb, 2 * 16384);
                mbar_arrive_expect_tx(vb, 2 * 16384);
                const uint32_t kt = s_base + DT_OFF_K + ks * BT_TILE, vt = s_base + DT_OFF_V + vs * BT_TILE;
                // two 128-token x 64-dim boxes each from the linear workspace (tokens past the
                // row's pages are zeros there; past the table, zero fill)
                tma_load_3d(kt, &kmap, kb, 0, i * BT_KEYS, lrow);
                tma_load_3d(kt + 16384, &kmap, kb, 64, i * BT_KEYS, lrow);
                tma_load_3d(vt, &vmap, vb, 0, i * BT_KEYS, lrow);
                tma_load_3d(vt + 16384, &vmap, vb, 64, i * BT_KEYS, lrow);
                ++issued;
            }
            if (pipe_aborted(abort)) {  // let the copies in flight land before the CTA's shared memory is released
                mbar_wait_drain(qb, 0);
                for (int i = max(0, issued - DT_KST); i < issued; ++i)
                    mbar_wait_drain(smem_u32(&bars->k_full[i % DT_KST]), (uint32_t)((i / DT_KST) & 1));
                for (int i = max(0, issued - DT_VST); i < issued; ++i)
                    mbar_wait_drain(smem_u32(&bars->v_full[i % DT_VST]), (uint32_t)((i / DT_VST) & 1));
            }
        } else if (warp == WARP_MMA && lane == 0) {
            // ================================================= MMA issuer ====
            const uint32_t idS = (1u << 4) | ((uint32_t)(BT_KEYS >> 3) << 17) | ((uint32_t)(BT_QB >> 4) << 24);
            const uint32_t idP = idesc_bf16_f32(BT_QB, BT_KEYS, 0, 0);
            const uint32_t idQ = (1u << 4) | (1u << 16) | ((uint32_t)(HEAD_DIM >> 3) << 17) |
                                 ((uint32_t)(BT_QB >> 4) << 24);
            const uint32_t dQa = desc_lo(s_base + DT_OFF_Q, 16), dOa = desc_lo(s_base + DT_OFF_DO, 16);
            // pipe order: S(0), dP(0), S(1), dQ'(0), dP(1), S(2), dQ'(1), ...
            bool ok = (!a.timeout_drill || drill_wait(smem_u32(&bars->never), abort)) &&
                      mbar_wait(smem_u32(&bars->q_full), 0, abort) && mbar_wait(smem_u32(&bars->k_full[0]), 0, abort);
            if (ok) {
                tc_fence_after();
                mma_ss_steps<0, 8, K_MAJOR_128, K_MAJOR_128>(tmem, dQa, desc_lo(s_base + DT_OFF_K, 16), idS, 0u);
            }
            for (int i = 0; i < n_tiles && ok; ++i) {
                const int ks = i % DT_KST, vs = i % DT_VST;
                if (!(ok = mbar_wait(smem_u32(&bars->v_full[vs]), (uint32_t)((i / DT_VST) & 1), abort))) break;
                tc_fence_after();
                mma_ss_steps<0, 8, K_MAJOR_128, K_MAJOR_128>(tmem + 256, dOa, desc_lo(s_base + DT_OFF_V + vs * BT_TILE, 16),
                                                             idP, 0u);
                umma_commit(smem_u32(&bars->s_full));        // S(i) and dP(i)
                umma_commit(smem_u32(&bars->v_empty[vs]));   // V(i) read
                if (i + 1 < n_tiles) {  // S(i + 1) into the other S buffer while the gradient of tile i runs
                    const int k1 = (i + 1) % DT_KST;
                    if (!(ok = mbar_wait(smem_u32(&bars->k_full[k1]), (uint32_t)(((i + 1) / DT_KST) & 1), abort))) break;
                    tc_fence_after();
                    mma_ss_steps<0, 8, K_MAJOR_128, K_MAJOR_128>(tmem + 128 * ((i + 1) & 1), dQa,
                                                                 desc_lo(s_base + DT_OFF_K + k1 * BT_TILE, 16), idS, 0u);
                }
                if (!(ok = mbar_wait(smem_u32(&bars->p_ready), (uint32_t)(i & 1), abort))) break;
                tc_fence_after();
                mma_ts_split<0, MN_MAJOR>(tmem + 384, tmem + 128 * (i & 1),
                                          desc_lo(s_base + DT_OFF_K + ks * BT_TILE, 16384), idQ, i > 0 ? 1u : 0u);
                umma_commit(smem_u32(&bars->k_empty[ks]));  // K'(i) read by S(i) and dQ'(i)
            }
            if (ok) {
                umma_commit(smem_u32(&bars->done));
            } else {
                const uint64_t ts = global_timer_ns();
                while (global_timer_ns() - ts < 1000000ull) {
                }
            }
        }
        __syncwarp();
        named_bar_sync(2, BT_THREADS);
    } else if (wg == 0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BT_REG_XFORM));
        // q and K arrive rotated (FP16, workspace): this warpgroup has no work
        named_bar_sync(1, 384);
        named_bar_sync(2, BT_THREADS);
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(BT_REG_GRAD));
        // ================================================ softmax gradient ====
        const int hsel = wg - 1, c0 = 64 * hsel;  // key columns c0 .. c0 + 63 of each tile
        const int r = tid - 128 * wg;             // query row == TMEM lane
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const int g = r / rph, s = s0 + r % rph;
        const bool valid = s < a.Sq;
        const size_t o = ((size_t)b * a.Hq + kvh * G + g) * a.Sq + (valid ? s : 0);
        const int p = valid ? pos_row[s] : -1;
        const float l2 = valid ? a.lse[o] * 1.4426950408889634074f : 0.0f;
        const float scl = a.qk_scale_log2;
        bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->q_full), 0, abort));
        // delta = rowsum(dout * out): this warpgroup's half of the dims (dout from the staged tile)
        float dsum = 0.0f;
        if (ok && valid) {
            const uint8_t* dh = sm + DT_OFF_DO + hsel * 16384;
            const uint4* ov = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.out) + o * HEAD_DIM) +
                              8 * hsel;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const uint4 x = *reinterpret_cast<const uint4*>(dh + sw128_off(r, ch)), y = __ldg(ov + ch);
                const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    dsum = fmaf(bf16lo(xw[k]), bf16lo(yw[k]), dsum);
                    dsum = fmaf(bf16hi(xw[k]), bf16hi(yw[k]), dsum);
                }
            }
        }
        if (hsel == 0) bars->dpart[r] = dsum;
        named_bar_sync(3, 256);
        const float dl = hsel ? bars->dpart[r] + dsum : dsum;  // (dims 0..63) + (dims 64..127)
        named_bar_sync(3, 256);
        if (hsel == 1) bars->dpart[r] = dl;
        named_bar_sync(3, 256);
        const float delta = bars->dpart[r];
        // (without the staged dout tile delta is unknown: NaN, so the dk / dv
        // kernel's gradients that use it come out NaN too)
        if (hsel == 1 && valid) a.delta[o] = ok ? delta : nanv;
        bool over = false;
        for (int i = 0; i < n_tiles && ok; ++i) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full), (uint32_t)(i & 1), abort)))) break;
            tc_fence_after();
            const int tb = i * BT_KEYS;
            const uint32_t sbuf = 128u * (uint32_t)(i & 1);  // this tile's S buffer
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int cb = c0 + 32 * h;
                uint32_t xs[32], xd[32];
                tmem_ld32(tmem + lane_addr + sbuf + cb, xs);
                tmem_ld32(tmem + lane_addr + 256 + cb, xd);
                tmem_ld_wait();
                // every key of these 32 columns visible to every row of the warp: no masks
                if (__all_sync(0xffffffffu, tb + cb + 31 <= p && tb + cb + 31 < kv_len)) {
                    const float2 sc2 = make_float2(scl, scl), nl2 = make_float2(-l2, -l2), nd2 = make_float2(-delta, -delta);
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float2 t2 = ffma2(make_float2(__uint_as_float(xs[c]), __uint_as_float(xs[c + 1])), sc2, nl2);
                        const float2 pp = make_float2(ex2(t2.x), ex2(t2.y));
                        const float2 ds = fmul2(pp, fadd2(make_float2(__uint_as_float(xd[c]), __uint_as_float(xd[c + 1])), nd2));
                        xs[c >> 1] = pack_f16x2(ds.x, ds.y);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        float ds[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int t = tb + cb + c + e;
                            const bool vis = t <= p && t < kv_len;
                            const float pp = vis ? ex2(__uint_as_float(xs[c + e]) * scl - l2) : 0.0f;
                            ds[e] = vis ? pp * (__uint_as_float(xd[c + e]) - delta) : 0.0f;
                        }
                        xs[c >> 1] = pack_f16x2(ds[0], ds[1]);
                    }
                }
                tmem_st16(tmem + lane_addr + sbuf + c0 + 16 * h, *reinterpret_cast<uint32_t(*)[16]>(&xs[0]));
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars->p_ready));
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->done), 0, abort));
        tc_fence_after();
        // epilogue: dq = R(p)^T (scale dQ'); warpgroup 1 takes rotation pairs 0..31
        // (dims 0..31 and 64..95), warpgroup 2 pairs 32..63 (dims 32..63 and 96..127).
        // A dS beyond the FP16 range (rounded to infinity) leaves dQ' non-finite.
        uint32_t lo[32], hi[32];
        if (ok) {  // warp-uniform; every lane loads
            tmem_ld32(tmem + lane_addr + 384 + 32 * hsel, lo);
            tmem_ld32(tmem + lane_addr + 384 + 64 + 32 * hsel, hi);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) over |= !isfinite(__uint_as_float(lo[k])) || !isfinite(__uint_as_float(hi[k]));
        }
        if (over && valid) bars->range_bad = 1;
        named_bar_sync(1, 384);
        const bool bad_out = bars->range_bad != 0 || !ok;
        if (tid == 128 && bad_out && a.status) atomicOr(a.status, ok ? RK_STATUS_RANGE : RK_STATUS_TIMEOUT);
        if (valid) {
            float* dst = a.dq + o * HEAD_DIM;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                float cth, sth;
                rope_cos_sin((uint32_t)max(p, 0), bars->turns[32 * hsel + k], cth, sth);
                const float x = __uint_as_float(lo[k]) * a.sm_scale, y = __uint_as_float(hi[k]) * a.sm_scale;
                lo[k] = __float_as_uint(bad_out ? nanv : x * cth + y * sth);
                hi[k] = __float_as_uint(bad_out ? nanv : y * cth - x * sth);
            }
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                *reinterpret_cast<float4*>(dst + 32 * hsel + c) =
                    make_float4(__uint_as_float(lo[c]), __uint_as_float(lo[c + 1]), __uint_as_float(lo[c + 2]),
                                __uint_as_float(lo[c + 3]));
                *reinterpret_cast<float4*>(dst + 64 + 32 * hsel + c) =
                    make_float4(__uint_as_float(hi[c]), __uint_as_float(hi[c + 1]), __uint_as_float(hi[c + 2]),
                                __uint_as_float(hi[c + 3]));
            }
        }
        named_bar_sync(2, BT_THREADS);
    }
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, BT_TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_backward_dkdv_tc(const CUtensorMap& qm, const CUtensorMap& om, const CUtensorMap& km,
                                    const CUtensorMap& vm, const BackwardArgs& a, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load() & bit)) {
        e = cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BT_SMEM);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    const long long tiles = ((long long)a.W * PAGE + BT_KEYS - 1) / BT_KEYS;
    const long long grid = (long long)a.B * a.Hkv * tiles;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    attn_bwd_dkdv_tc_kernel<<<(unsigned)grid, BT_THREADS, BT_SMEM, stream>>>(qm, om, km, vm, a);
    return cudaGetLastError();
}

}  // namespace rk

namespace rk {

cudaError_t launch_backward_dq_tc(const CUtensorMap& qm, const CUtensorMap& om, const CUtensorMap& km,
                                  const CUtensorMap& vm, const BackwardArgs& a, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load() & bit)) {
        e = cudaFuncSetAttribute(attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DT_SMEM);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    const long long rph = BT_QB / a.G;
    const long long grid = (long long)a.B * a.Hkv * ((a.Sq + rph - 1) / rph);
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    attn_bwd_dq_tc_kernel<<<(unsigned)grid, BT_THREADS, DT_SMEM, stream>>>(qm, om, km, vm, a);
    return cudaGetLastError();
}

}  // namespace rk

namespace rk {

cudaError_t launch_backward_rotate(const BackwardArgs& a, cudaStream_t stream) {
    const long long nq = (long long)a.B * a.Hq * a.Sq * 8, nk = (long long)a.B * a.Hkv * a.W * PAGE * 8;
    const int grid_q = (int)std::min<long long>((nq + 255) / 256, 152 * 16);
    const int grid_k = (int)std::min<long long>((nk + 255) / 256, 152 * 16);
    if (grid_q > 0) rotate_q_kernel<<<grid_q, 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (grid_k > 0 && a.num_pages > 0) rotate_k_kernel<<<grid_k, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace rk
