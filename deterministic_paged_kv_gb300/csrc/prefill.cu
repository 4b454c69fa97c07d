// prefill.cu -- causal chunked prefill over a paged prefix on the 5th-gen
// tensor cores (tcgen05 MMA into TMEM), RoPE applied in the load stage.
//
// Operation: the paged prefill of "WS2 PR7 Fused Attention Backend
// Alignment", "Current Implementation" (BatchPrefillWithPagedKVCacheWrapper
// role, ROPE_LLAMA fused on pre-RoPE Q and K, split-KV disabled, FP32 LSE),
// with the batch-invariance requirement of that page's "Batch-Invariant
// Validation" section.
//
// One CTA owns one q-tile: 128 accumulator rows = (128/G) consecutive query
// positions x the G query heads that share one KV head (GQA packing), so each
// K/V tile is read once per head group.  It sweeps the row's KV tiles of 128
// tokens (8 pages) in ascending order:
//   warp 8      TMA producer: Q once, then per KV tile the 8 pages of K and V
//               (4 boxes of 16 tokens x 64 dims each, 128-byte swizzle) into a
//               two-stage ring;
//   warps 0-3   transform: rotate Q once and each K tile in place in shared
//               memory (FP32 math, angles from the exact fixed-point anchor
//               plus a 16-position angle-addition step), round to BF16 in the
//               UMMA operand layout; zero V rows past the last visible key;
//   warp 9      MMA issuer: S = Q K^T into TMEM (128 columns), then
//               O += P V into TMEM (128 columns), tcgen05.commit to mbarriers;
//   warps 4-7   softmax: one thread per accumulator row, reads its S row from
//               TMEM, causal mask, online softmax in the log2 domain with a
//               slack of 8 before the running max moves (rescale of the O row
//               in TMEM only then), P rounded to BF16 into shared memory;
//               epilogue O / l -> BF16 once, LSE -> FP32.
// Score precision: the rotated Q is kept as two BF16 terms (hi + lo) and the
// score MMA is Q_hi K^T + Q_lo K^T, so only K's BF16 rounding remains (its
// error is independent per key and averages out in the LSE; a single BF16 Q
// rounding shifts every score of a row the same way and does not).  q-tiles
// whose first position is below PF_PRECISE_POS also split K (adding
// Q_hi K_lo^T), so rows that see few keys keep an FP32-grade LSE.  Both
// choices depend on the logical position only.  Nothing depends on B, W or
// the grid.
#include <atomic>

#include "rk_device.cuh"

namespace rk {

namespace {

constexpr int PF_THREADS = 320;
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr uint32_t TMEM_COLS = 256;  // S: [0,128), O: [128,256)
constexpr float RESCALE_SLACK = 8.0f;

// Shared memory carve (offsets from a 1024-byte aligned base).
constexpr int OFF_Q = 0;                        // Q hi  [2 blocks][128 rows][128 B]
constexpr int OFF_QLO = OFF_Q + PF_TILE_BYTES;  // Q lo: rotated Q minus its BF16 rounding
constexpr int OFF_K = OFF_QLO + PF_TILE_BYTES;  // K stage 0, K stage 1 (= K lo when precise)
constexpr int OFF_V = OFF_K + 2 * PF_TILE_BYTES;
constexpr int OFF_P = OFF_V + 2 * PF_TILE_BYTES;
constexpr int OFF_BAR = OFF_P + PF_TILE_BYTES;
constexpr int PF_SMEM_BYTES = OFF_BAR + 1024 + 1024;  // barriers + alignment slack

struct PfBars {
    uint64_t q_full, q_ready;
    uint64_t kv_full[2], kv_ready[2], kv_empty[2];
    uint64_t s_full, s_free, p_ready, pv_done;
    uint32_t tmem_base;
    int abort;
    float2 step16[ROPE_PAIRS];  // cos/sin of a 16-position turn per pair
};
static_assert(sizeof(PfBars) <= 1024, "prefill control block exceeds its reservation");
static_assert(PF_SMEM_BYTES <= 232448, "prefill shared memory above the 227 KiB opt-in limit");

__device__ __forceinline__ uint32_t sw_off(int row, int chunk) {
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int ks) {
    return smem_desc(tile + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, 2);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int ks) {
    return smem_desc(tile + ks * 2048, 16384, 1024, 2);
}

// Rotate one 16-byte chunk pair (8 rotate-half pairs) in place; optionally
// write the BF16 residual (lo part) to a second tile at the same offsets.
__device__ __forceinline__ void rotate_chunk(uint8_t* lo_ptr, uint8_t* hi_ptr, const float (&c)[8],
                                             const float (&s)[8], uint8_t* res_lo, uint8_t* res_hi) {
    uint4 a = *reinterpret_cast<const uint4*>(lo_ptr);
    uint4 b = *reinterpret_cast<const uint4*>(hi_ptr);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
    uint32_t ow[4], pw[4], rl[4], rh[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int e0 = 2 * k, e1 = 2 * k + 1;
        const float l0 = bf16lo(aw[k]), l1 = bf16hi(aw[k]);
        const float u0 = bf16lo(bw[k]), u1 = bf16hi(bw[k]);
        const float x0 = l0 * c[e0] - u0 * s[e0], y0 = u0 * c[e0] + l0 * s[e0];
        const float x1 = l1 * c[e1] - u1 * s[e1], y1 = u1 * c[e1] + l1 * s[e1];
        ow[k] = pack_bf16x2(x0, x1);
        pw[k] = pack_bf16x2(y0, y1);
        if (res_lo) {
            rl[k] = pack_bf16x2(x0 - bf16lo(ow[k]), x1 - bf16hi(ow[k]));
            rh[k] = pack_bf16x2(y0 - bf16lo(pw[k]), y1 - bf16hi(pw[k]));
        }
    }
    *reinterpret_cast<uint4*>(lo_ptr) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    *reinterpret_cast<uint4*>(hi_ptr) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
    if (res_lo) {
        *reinterpret_cast<uint4*>(res_lo) = make_uint4(rl[0], rl[1], rl[2], rl[3]);
        *reinterpret_cast<uint4*>(res_hi) = make_uint4(rh[0], rh[1], rh[2], rh[3]);
    }
}

__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    PfBars* bars = reinterpret_cast<PfBars*>(sm + OFF_BAR);
    const uint32_t s_base = smem_u32(sm);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- work unit: longest q-tiles first (later positions see more keys) --
    const int units_per_qt = a.B * a.Hkv;
    const int qt = a.n_qtiles - 1 - (int)(blockIdx.x / units_per_qt);
    const int rem = (int)(blockIdx.x % units_per_qt);
    const int b = rem / a.Hkv, kvh = rem % a.Hkv;
    const int rph = a.rows_per_head;
    const int s0 = qt * rph;
    const int s_last = min(s0 + rph, a.Sq) - 1;

    // ---- row metadata (device copy) and memory-safety checks ----
    const int kv_len = a.kv_lens[b];
    const int32_t* pos_row = a.position_ids + (size_t)b * a.Sq;
    const int pos_first = pos_row[s0];
    const int pos_last = pos_row[s_last];
    int bad = 0;
    if (kv_len < 0 || kv_len > a.W * PAGE) bad |= RK_STATUS_KVLEN;
    if (pos_first < 0 || pos_last < 0) bad |= RK_STATUS_POSITION;
    int n_keys = 0;  // keys any row of this tile may see
    if (!bad) {
        // the largest position of the tile (positions need not be ascending for safety)
        int pmax = -1;
        for (int s = s0; s <= s_last; ++s) pmax = max(pmax, pos_row[s]);
        n_keys = pmax >= kv_len ? kv_len : pmax + 1;
    }
    const int n_pages = (n_keys + PAGE - 1) / PAGE;
    const int n_tiles = (n_keys + PF_BN - 1) / PF_BN;
    const int32_t* bt = a.block_table + (size_t)b * a.W;
    int oob = 0;
    for (int i = tid; i < n_pages; i += PF_THREADS) {
        const int pg = __ldg(bt + i);
        oob |= (pg < 0) | (pg >= a.num_pages);
    }
    const bool precise = pos_first < PF_PRECISE_POS;

    if (tid == 0) {
        bars->abort = 0;
        mbar_init(smem_u32(&bars->q_full), 1);
        mbar_init(smem_u32(&bars->q_ready), 128);
        for (int k = 0; k < 2; ++k) {
            mbar_init(smem_u32(&bars->kv_full[k]), 1);
            mbar_init(smem_u32(&bars->kv_ready[k]), 128);
            mbar_init(smem_u32(&bars->kv_empty[k]), 1);
        }
        mbar_init(smem_u32(&bars->s_full), 1);
        mbar_init(smem_u32(&bars->s_free), 128);
        mbar_init(smem_u32(&bars->p_ready), 128);
        mbar_init(smem_u32(&bars->pv_done), 1);
        fence_mbar_init();
    }
    if (tid < ROPE_PAIRS) {
        float c, s;
        rope_cos_sin((uint32_t)PAGE, a.rope_turns[tid], c, s);
        bars->step16[tid] = make_float2(c, s);
    }
    if (__syncthreads_or(oob)) bad |= RK_STATUS_PAGE_OOB;

    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    if (bad || n_tiles == 0) {
        // Whole tile: zero output; LSE NaN for unsafe metadata, -inf for no keys.
        if (bad && tid == 0 && a.status) atomicOr(a.status, bad);
        const float lv = bad ? __int_as_float(0x7fc00000) : -INFINITY;
        for (int r = tid; r < PF_BM; r += PF_THREADS) {
            const int g = r / rph, j = r % rph, s = s0 + j;
            if (s >= a.Sq) continue;
            const int h = kvh * a.G + g;
            __nv_bfloat16* o = out + (((size_t)b * a.Hq + h) * a.Sq + s) * HEAD_DIM;
            for (int d = 0; d < HEAD_DIM; ++d) o[d] = __float2bfloat16_rn(0.0f);
            a.lse[((size_t)b * a.Hq + h) * a.Sq + s] = lv;
        }
        return;
    }

    // ---- TMEM allocation (warp 9) ----
    if (warp == WARP_MMA) {
        tmem_alloc(smem_u32(&bars->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tS = tmem, tO = tmem + 128;
    volatile int* abort = &bars->abort;

    auto stage_of = [&](int i) { return precise ? 0 : (i & 1); };
    auto use_of = [&](int i) { return precise ? i : (i >> 1); };

    if (warp == WARP_TMA) {
        // ================================================ TMA producer ====
        if (lane == 0) {
            prefetch_tmap(&qmap);
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
            const uint32_t qb = smem_u32(&bars->q_full);
            mbar_arrive_expect_tx(qb, PF_TILE_BYTES);
            tma_load_4d(s_base + OFF_Q, &qmap, qb, 0, s0, kvh * a.G, b);
            tma_load_4d(s_base + OFF_Q + 16384, &qmap, qb, 64, s0, kvh * a.G, b);
        }
        int issued = 0;
        for (int i = 0; i < n_tiles; ++i) {
            const int k = stage_of(i);
            const uint32_t par = (uint32_t)(use_of(i) & 1);
            const int p0 = i * PF_PAGES_PER_TILE;
            const int np = min(PF_PAGES_PER_TILE, n_pages - p0);
            const int pg = lane < np ? __ldg(bt + p0 + lane) : 0;
            int good = 1;
            if (lane == 0) good = mbar_wait(smem_u32(&bars->kv_empty[k]), par ^ 1u, abort);
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) break;
            if (lane == 0) mbar_arrive_expect_tx(smem_u32(&bars->kv_full[k]), (uint32_t)np * 4 * 2048);
            // Lane p holds the page id of page p of the tile; lane 0 issues.
            for (int p = 0; p < np; ++p) {
                const int page = __shfl_sync(0xffffffffu, pg, p);
                if (lane == 0) {
                    const uint32_t fb = smem_u32(&bars->kv_full[k]);
                    const uint32_t kt = s_base + OFF_K + k * PF_TILE_BYTES + p * 2048;
                    const uint32_t vt = s_base + OFF_V + k * PF_TILE_BYTES + p * 2048;
                    tma_load_3d(kt, &kmap, fb, 0, kvh, page * PAGE);
                    tma_load_3d(kt + 16384, &kmap, fb, 64, kvh, page * PAGE);
                    tma_load_3d(vt, &vmap, fb, 0, kvh, page * PAGE);
                    tma_load_3d(vt + 16384, &vmap, fb, 64, kvh, page * PAGE);
                }
            }
            ++issued;
        }
        if (lane == 0 && *abort) {
            for (int i = max(0, issued - 2); i < issued; ++i)
                mbar_wait_drain(smem_u32(&bars->kv_full[stage_of(i)]), (uint32_t)(use_of(i) & 1));
        }
    } else if (warp < 4) {
        // ================================================ transform WG ====
        // Q: thread r rotates accumulator row r at its own query position.
        {
            const int r = tid;
            const int g = r / rph, j = r % rph, s = s0 + j;
            const int p = s < a.Sq ? pos_row[s] : 0;
            if (mbar_wait(smem_u32(&bars->q_full), 0, abort)) {
                uint8_t* q0 = sm + OFF_Q;
                for (int u = 0; u < 8; ++u) {
                    float c[8], sn[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) rope_cos_sin((uint32_t)p, a.rope_turns[8 * u + e], c[e], sn[e]);
                    const uint32_t off = sw_off(r, u);
                    rotate_chunk(q0 + off, q0 + 16384 + off, c, sn, sm + OFF_QLO + off,
                                 sm + OFF_QLO + 16384 + off);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bars->q_ready));
        }
        // K tiles: thread handles pair-chunk u = tid % 8 of rows r0 + 16 m.
        const int u = tid & 7, r0 = tid >> 3;
        float dcs[8], dsn[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 st = bars->step16[8 * u + e];
            dcs[e] = st.x;
            dsn[e] = st.y;
        }
        for (int i = 0; i < n_tiles; ++i) {
            const int k = stage_of(i);
            if (!mbar_wait(smem_u32(&bars->kv_full[k]), (uint32_t)(use_of(i) & 1), abort)) break;
            uint8_t* kt = sm + OFF_K + k * PF_TILE_BYTES;
            uint8_t* klo = sm + OFF_K + PF_TILE_BYTES;  // stage 1 holds lo parts when precise
            const int t0 = i * PF_BN;
            float c[8], sn[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) rope_cos_sin((uint32_t)(t0 + r0), a.rope_turns[8 * u + e], c[e], sn[e]);
#pragma unroll 1
            for (int m = 0; m < 8; ++m) {
                const int r = r0 + 16 * m;
                const uint32_t off = sw_off(r, u);
                if (t0 + r < n_keys)
                    rotate_chunk(kt + off, kt + 16384 + off, c, sn, precise ? klo + off : nullptr,
                                 precise ? klo + 16384 + off : nullptr);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float cn = c[e] * dcs[e] - sn[e] * dsn[e];
                    const float snn = sn[e] * dcs[e] + c[e] * dsn[e];
                    c[e] = cn;
                    sn[e] = snn;
                }
            }
            // V rows past the last key this tile may use: zero (they meet P = 0
            // and must not carry stale or non-finite bits into the MMA).
            if (t0 + PF_BN > n_keys) {
                uint8_t* vt = sm + OFF_V + k * PF_TILE_BYTES;
                for (int idx = tid; idx < PF_BN * 16; idx += 128) {
                    const int r = idx >> 4, ch = idx & 15;
                    if (t0 + r >= n_keys)
                        *reinterpret_cast<uint4*>(vt + (ch >> 3) * 16384 + r * 128 + (ch & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bars->kv_ready[k]));
        }
    } else if (warp == WARP_MMA) {
        // ================================================= MMA issuer ====
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(PF_BM, PF_BN, 0, 0);
            const uint32_t idO = idesc_bf16_f32(PF_BM, HEAD_DIM, 0, 1);
            const uint32_t q = s_base + OFF_Q, qlo = s_base + OFF_QLO, p_t = s_base + OFF_P;
            bool ok = mbar_wait(smem_u32(&bars->q_ready), 0, abort);
            auto issue_s = [&](int i) -> bool {
                const int k = stage_of(i);
                if (!mbar_wait(smem_u32(&bars->kv_ready[k]), (uint32_t)(use_of(i) & 1), abort)) return false;
                if (i > 0 && !mbar_wait(smem_u32(&bars->s_free), (uint32_t)((i - 1) & 1), abort)) return false;
                tc_fence_after();
                const uint32_t kt = s_base + OFF_K + k * PF_TILE_BYTES;
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks) umma_ss(tS, kmajor_desc(q, ks), kmajor_desc(kt, ks), idS, ks > 0);
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks) umma_ss(tS, kmajor_desc(qlo, ks), kmajor_desc(kt, ks), idS, 1);
                if (precise) {
                    const uint32_t klo = s_base + OFF_K + PF_TILE_BYTES;
#pragma unroll 1
                    for (int ks = 0; ks < 8; ++ks) umma_ss(tS, kmajor_desc(q, ks), kmajor_desc(klo, ks), idS, 1);
                }
                umma_commit(smem_u32(&bars->s_full));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int i = 0; i < n_tiles && ok; ++i) {
                if (i + 1 < n_tiles && !precise) ok = issue_s(i + 1);
                if (!ok) break;
                if (!mbar_wait(smem_u32(&bars->p_ready), (uint32_t)(i & 1), abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t vt = s_base + OFF_V + stage_of(i) * PF_TILE_BYTES;
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks)
                    umma_ss(tO, kmajor_desc(p_t, ks), mnmajor_desc(vt, ks), idO, (i > 0 || ks > 0) ? 1u : 0u);
                umma_commit(smem_u32(&bars->pv_done));
                umma_commit(smem_u32(&bars->kv_empty[stage_of(i)]));
                // precise tiles use one stage: the next score MMA needs this
                // tile's K buffers released and refilled first.
                if (precise && i + 1 < n_tiles) ok = issue_s(i + 1);
            }
            if (!ok) {
                // let issued MMAs finish before TMEM is released
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 1000000ull) {
                }
            }
        }
    } else {
        // ================================================ softmax WG =====
        const int r = tid - 128;  // accumulator row == TMEM lane
        const int wq = warp - 4;  // lane quarter of this warp
        const int g = r / rph, j = r % rph, s = s0 + j;
        const bool valid = s < a.Sq;
        const int p = valid ? pos_row[s] : -1;
        const int n_vis = valid ? (p >= kv_len ? kv_len : p + 1) : 0;
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        const float scl = a.qk_scale_log2;
        float m = -INFINITY, l = 0.0f;
        bool ok = true;
        uint8_t* pt = sm + OFF_P;
        for (int i = 0; i < n_tiles; ++i) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full), (uint32_t)(i & 1), abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t xr[128];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
                tmem_ld32(tS + lane_addr + c4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&xr[c4 * 32]));
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars->s_free));
            const int t0 = i * PF_BN;
            const int lim = n_vis - t0;  // columns < lim are visible
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                const float v = c < lim ? __uint_as_float(xr[c]) * scl : -INFINITY;
                xr[c] = __float_as_uint(v);
                mt = fmaxf(mt, v);
            }
            float alpha = 1.0f;
            bool resc = false;
            if (mt > m + RESCALE_SLACK) {
                alpha = ex2(m - mt);  // 0 when m = -inf
                m = mt;
                resc = true;
            }
            l *= alpha;
            float rs = 0.0f;
            const bool none = (m == -INFINITY);
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                const float e = none ? 0.0f : ex2(__uint_as_float(xr[c]) - m);
                xr[c] = __float_as_uint(e);
                rs += e;
            }
            l += rs;
            if (i > 0) {
                // P buffer and O are free once the previous PV finished.
                if (!__all_sync(0xffffffffu,
                                mbar_wait(smem_u32(&bars->pv_done), (uint32_t)((i - 1) & 1), abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
                const int c = cc * 8;
                const uint4 v = make_uint4(
                    pack_bf16x2(__uint_as_float(xr[c]), __uint_as_float(xr[c + 1])),
                    pack_bf16x2(__uint_as_float(xr[c + 2]), __uint_as_float(xr[c + 3])),
                    pack_bf16x2(__uint_as_float(xr[c + 4]), __uint_as_float(xr[c + 5])),
                    pack_bf16x2(__uint_as_float(xr[c + 6]), __uint_as_float(xr[c + 7])));
                *reinterpret_cast<uint4*>(pt + (cc >> 3) * 16384 + sw_off(r, cc & 7)) = v;
            }
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
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars->p_ready));
        }
        // ---- epilogue ----
        if (ok) ok = __all_sync(0xffffffffu,
                                mbar_wait(smem_u32(&bars->pv_done), (uint32_t)((n_tiles - 1) & 1), abort));
        if (ok) {
            tc_fence_after();
            const int h = kvh * a.G + g;
            __nv_bfloat16* o = out + (((size_t)b * a.Hq + h) * a.Sq + (valid ? s : 0)) * HEAD_DIM;
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
                        for (int e = 0; e < 8; ++e) f[e] = l > 0.0f ? __uint_as_float(rr[q + e]) / l : 0.0f;
                        *reinterpret_cast<uint4*>(o + c4 * 32 + q) =
                            make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                       pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                    }
                }
            }
            if (valid)
                a.lse[((size_t)b * a.Hq + h) * a.Sq + s] =
                    l > 0.0f ? (m + log2f(l)) * 0.693147180559945309f : -INFINITY;
        } else if (tid == 128 && a.status) {
            atomicOr(a.status, RK_STATUS_TIMEOUT);
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                           const PrefillArgs& a, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load() & bit)) {
        e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    const long long grid = (long long)a.B * a.Hkv * a.n_qtiles;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prefill_kernel<<<(unsigned)grid, PF_THREADS, PF_SMEM_BYTES, stream>>>(qm, km, vm, a);
    return cudaGetLastError();
}

}  // namespace rk
