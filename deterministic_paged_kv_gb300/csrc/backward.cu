// backward.cu -- deterministic gradient of causal paged prefill with fused
// RoPE (dq, and dk / dv scattered back into the page layout).
//
// Operation: the training lane of "Add FlashInfer RoPE-fused paged attention
// scaffold", scope table, Backward row (dropout 0, deterministic backward
// required), for the attention the forward kernels compute: q and the K cache
// pre-RoPE, rotate-half RoPE at each token's own position, causal visibility
// t <= position and t < kv_len, GQA head h -> KV head h / G, FP32 LSE.  With
// P = exp(s - lse) from the forward's LSE, for L = sum(dout * out):
//   delta = rowsum(dout * out),  dP = dout V^T,  dS = P (dP - delta),
//   dV = P^T dout,  dK' = scale dS^T Q',  dQ' = scale dS K',
// and the rotation is undone by its transpose: dq = R(p)^T dQ', dk = R(t)^T dK'.
//
// Determinism: every output element is accumulated by exactly one CTA in a
// fixed order that depends only on its own row -- dq by the CTA of its 64
// query rows over key tiles in ascending order, dk / dv by the CTA of their 64
// keys over query blocks in ascending order.  No atomics, no split.
//
// Tensor cores: warp-level mma.sync m16n8k16 with FP32 accumulation.  Scores
// and the dS products use FP16 operands (rotated q / k rounded to FP16 as in
// the forward's score MMA, dS rounded to FP16), the dout products BF16 (P
// rounded to BF16 for dV).  Shared-memory rows of 128 16-bit elements are
// stored with their 16-byte chunks XOR-swizzled by (row & 7), so the eight
// row addresses of every ldmatrix hit distinct banks.
#include <atomic>

#include "rk_device.cuh"

namespace rk {

namespace {

constexpr float LOG2E = 1.4426950408889634074f;
constexpr float F16_MAX = 65504.0f;

// byte offset of 16-byte chunk `chunk` (0..15) of 256-byte row `row`
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)row * 256u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Lane addresses of the three ldmatrix patterns (rows of 128 16-bit elements):
// A fragment (16 rows x k16 at chunk pair kc): rows base + (lane & 15), chunk kc + (lane >> 4).
__device__ __forceinline__ uint32_t a_addr(uint32_t base, int row0, int kc, int lane) {
    return base + swz(row0 + (lane & 15), kc + (lane >> 4));
}
// B fragments of two n8 tiles from an [n][k] matrix (n = rows): rows row0 + (lane & 7) + 8 (lane >> 4),
// chunk kc + ((lane >> 3) & 1)  ->  {b0, b1} of tile 0, {b0, b1} of tile 1.
__device__ __forceinline__ uint32_t b_addr(uint32_t base, int row0, int kc, int lane) {
    return base + swz(row0 + (lane & 7) + ((lane >> 4) << 3), kc + ((lane >> 3) & 1));
}
// B fragments of two n8 tiles from a [k][n] matrix (k = rows, .trans): rows row0 + (lane & 7) +
// 8 ((lane >> 3) & 1), chunk nc + (lane >> 4)  ->  {b0, b1} of tile nc, {b0, b1} of tile nc + 1.
__device__ __forceinline__ uint32_t bt_addr(uint32_t base, int row0, int nc, int lane) {
    return base + swz(row0 + (lane & 7) + (((lane >> 3) & 1) << 3), nc + (lane >> 4));
}

// Rotate rows of 128 bf16 into swizzled FP16 rows: row r of `rows` comes from
// src(r) (nullptr: a zero row) at position pos(r).  One work item is a chunk
// pair (dims 8c..8c+7 and 64+8c..64+8c+7) of one row.  Returns the running
// maximum of the |input| bf16 patterns (FP16 range check).
template <class Src, class Pos>
__device__ __forceinline__ uint32_t load_rotated(uint8_t* dst, int rows, Src src, Pos pos, const uint64_t* turns,
                                                 uint32_t range) {
    for (int it = threadIdx.x; it < rows * 8; it += BW_THREADS) {
        const int r = it >> 3, c = it & 7;
        const uint4* p = src(r);
        uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
        int ps = 0;
        if (p) {
            lo = __ldg(p + c);
            hi = __ldg(p + c + 8);
            ps = pos(r);
        }
        float2 cs[4], sn[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            rope_cos_sin((uint32_t)ps, turns[8 * c + 2 * e], cs[e].x, sn[e].x);
            rope_cos_sin((uint32_t)ps, turns[8 * c + 2 * e + 1], cs[e].y, sn[e].y);
        }
        range = rotate_regs_f16(lo, hi, cs, sn, range);
        *reinterpret_cast<uint4*>(dst + swz(r, c)) = lo;
        *reinterpret_cast<uint4*>(dst + swz(r, c + 8)) = hi;
    }
    return range;
}

// Copy rows of 128 bf16 unchanged into swizzled rows (nullptr: a zero row).
template <class Src>
__device__ __forceinline__ void load_plain(uint8_t* dst, int rows, Src src) {
    for (int it = threadIdx.x; it < rows * 16; it += BW_THREADS) {
        const int r = it >> 4, c = it & 15;
        const uint4* p = src(r);
        *reinterpret_cast<uint4*>(dst + swz(r, c)) = p ? __ldg(p + c) : make_uint4(0, 0, 0, 0);
    }
}

// Asynchronous 16-byte global -> shared copy (zero fill when !valid: nothing is read).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Start copying rows of 128 bf16 into swizzled rows: row r from src(r)
// (nullptr: zeros).  Completion: cp_async_wait_all by the issuing threads,
// then a barrier.
template <class Src>
__device__ __forceinline__ void copy_rows_async(uint32_t dst, int rows, Src src, const void* any_valid) {
    for (int it = threadIdx.x; it < rows * 16; it += BW_THREADS) {
        const int r = it >> 4, c = it & 15;
        const uint4* p = src(r);
        cp_async16(dst + swz(r, c), p ? static_cast<const void*>(p + c) : any_valid, p != nullptr);
    }
}

// Rotate in place 64 swizzled bf16 rows at positions t0 + r into FP16: thread
// handles chunk pair c = tid & 7 of rows r0 + 16 m (r0 = tid >> 3), with exact
// angles at r0 and 16-position angle-addition steps (step16) after it.
static_assert(BW_THREADS == 128 && BW_KT == 64, "rotate_tile_inplace: 16 row groups of 8 chunk pairs, 4 rows each");
__device__ __forceinline__ uint32_t rotate_tile_inplace(uint8_t* buf, int t0, const uint64_t* turns,
                                                        const float2* step16, uint32_t range) {
    const int c = threadIdx.x & 7, r0 = threadIdx.x >> 3;
    float2 cs[4], sn[4], dcs[4], dsn[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        rope_cos_sin((uint32_t)(t0 + r0), turns[8 * c + 2 * e], cs[e].x, sn[e].x);
        rope_cos_sin((uint32_t)(t0 + r0), turns[8 * c + 2 * e + 1], cs[e].y, sn[e].y);
        const float2 a = step16[8 * c + 2 * e], b = step16[8 * c + 2 * e + 1];
        dcs[e] = make_float2(a.x, b.x);
        dsn[e] = make_float2(a.y, b.y);
    }
#pragma unroll
    for (int m = 0; m < BW_KT / 16; ++m) {
        const int r = r0 + 16 * m;
        uint4* lo = reinterpret_cast<uint4*>(buf + swz(r, c));
        uint4* hi = reinterpret_cast<uint4*>(buf + swz(r, c + 8));
        uint4 x = *lo, y = *hi;
        range = rotate_regs_f16(x, y, cs, sn, range);
        *lo = x;
        *hi = y;
        rope_step(cs, sn, dcs, dsn);
    }
    return range;
}

// Rotate in place `rows` swizzled bf16 rows into FP16, row r at position pos(r)
// (exact angles per row).
template <class Pos>
__device__ __forceinline__ uint32_t rotate_rows_inplace(uint8_t* buf, int rows, Pos pos, const uint64_t* turns,
                                                        uint32_t range) {
    for (int it = threadIdx.x; it < rows * 8; it += BW_THREADS) {
        const int r = it >> 3, c = it & 7;
        const int ps = pos(r);
        float2 cs[4], sn[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            rope_cos_sin((uint32_t)ps, turns[8 * c + 2 * e], cs[e].x, sn[e].x);
            rope_cos_sin((uint32_t)ps, turns[8 * c + 2 * e + 1], cs[e].y, sn[e].y);
        }
        uint4* lo = reinterpret_cast<uint4*>(buf + swz(r, c));
        uint4* hi = reinterpret_cast<uint4*>(buf + swz(r, c + 8));
        uint4 x = *lo, y = *hi;
        range = rotate_regs_f16(x, y, cs, sn, range);
        *lo = x;
        *hi = y;
    }
    return range;
}

// dS -> FP16 pair; flags a value outside the FP16 range.
__device__ __forceinline__ uint32_t pack_ds(float a, float b, bool& over) {
    over |= !(fabsf(a) < F16_MAX) || !(fabsf(b) < F16_MAX);
    return pack_f16x2(a, b);
}

// Undo the rotation of one row's gradient held as C fragments acc[16][4]
// (tile j covers dims 8j..8j+7; this lane holds dims 8j + 2 (lane & 3) + e
// in acc[j][e] (row g) and acc[j][2 + e] (row g + 8)): dim i < 64 pairs with
// i + 64 in tile j + 8.  R(p)^T: lo' = lo c + hi s, hi' = hi c - lo s.
__device__ __forceinline__ void unrotate_row(float (&acc)[16][4], int half_sel, int p, const uint64_t* turns,
                                             int lane) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = 8 * j + 2 * (lane & 3) + e;
            float c, s;
            rope_cos_sin((uint32_t)p, turns[i], c, s);
            const float lo = acc[j][2 * half_sel + e], hi = acc[j + 8][2 * half_sel + e];
            acc[j][2 * half_sel + e] = lo * c + hi * s;
            acc[j + 8][2 * half_sel + e] = hi * c - lo * s;
        }
    }
}

// Shared memory of the dq kernel: Q' / dout of the CTA's 64 query rows, K' / V
// of one key tile, per-row lse (log2 domain), delta and position, RoPE rates.
constexpr int DQ_OFF_Q = 0;
constexpr int DQ_OFF_DO = DQ_OFF_Q + BW_QB * 256;
constexpr int DQ_OFF_K = DQ_OFF_DO + BW_QB * 256;  // two K stages (copied raw, rotated in place)
constexpr int DQ_OFF_V = DQ_OFF_K + 2 * BW_KT * 256;  // two V stages
constexpr int DQ_OFF_S = DQ_OFF_V + 2 * BW_KT * 256;  // cos / sin of a 16-position step per pair
constexpr int DQ_OFF_L = DQ_OFF_S + ROPE_PAIRS * 8;
constexpr int DQ_OFF_D = DQ_OFF_L + BW_QB * 4;
constexpr int DQ_OFF_P = DQ_OFF_D + BW_QB * 4;
constexpr int DQ_OFF_T = DQ_OFF_P + BW_QB * 4;
constexpr int DQ_OFF_F = DQ_OFF_T + ROPE_PAIRS * 8;
constexpr int DQ_SMEM = DQ_OFF_F + 16;

// One CTA per (row b, KV head, block of 64 query rows), latest blocks first
// (they see the most keys).  Query row r of the block is position s = r / G
// of head g = r % G.  Also writes delta for its rows (read by the dk/dv kernel).
__global__ void __launch_bounds__(BW_THREADS) attn_bwd_dq_kernel(const __grid_constant__ BackwardArgs a) {
    extern __shared__ __align__(128) uint8_t sm[];
    float* sL = reinterpret_cast<float*>(sm + DQ_OFF_L);
    float* sD = reinterpret_cast<float*>(sm + DQ_OFF_D);
    int* sP = reinterpret_cast<int*>(sm + DQ_OFF_P);
    uint64_t* sT = reinterpret_cast<uint64_t*>(sm + DQ_OFF_T);
    int* sF = reinterpret_cast<int*>(sm + DQ_OFF_F);  // [0] status bits, [1] largest visible key count
    float2* sS = reinterpret_cast<float2*>(sm + DQ_OFF_S);
    const uint32_t base = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.G, nrows = a.Sq * G;
    const int nqb = (nrows + BW_QB - 1) / BW_QB;
    const int units = a.B * a.Hkv;
    const int qb = nqb - 1 - (int)(blockIdx.x / units);
    const int b = (int)(blockIdx.x % units) / a.Hkv, kvh = (int)(blockIdx.x % units) % a.Hkv;
    const int kv_len = a.kv_lens[b];
    const int32_t* bt = a.block_table + (size_t)b * a.W;
    auto qrow_off = [&](int r) -> size_t {  // element offset of query row r in [B, Hq, Sq, D]
        const int qr = qb * BW_QB + r;
        return (((size_t)b * a.Hq + kvh * G + qr % G) * a.Sq + qr / G) * HEAD_DIM;
    };
    auto row_ok = [&](int r) { return qb * BW_QB + r < nrows; };

    if (tid == 0) {
        sF[0] = (kv_len < 0 || kv_len > a.W * PAGE) ? RK_STATUS_KVLEN : 0;
        sF[1] = 0;
    }
    if (tid < ROPE_PAIRS) {
        sT[tid] = a.rope_turns[tid];
        float c, sn;
        rope_cos_sin(16u, a.rope_turns[tid], c, sn);  // the row step of rotate_tile_inplace
        sS[tid] = make_float2(c, sn);
    }
    __syncthreads();
    if (tid < BW_QB) {
        int p = -1;
        float l2 = 0.0f;
        if (row_ok(tid)) {
            const int qr = qb * BW_QB + tid;
            p = a.position_ids[(size_t)b * a.Sq + qr / G];
            if (p < 0) atomicOr(&sF[0], RK_STATUS_POSITION);
            l2 = a.lse[((size_t)b * a.Hq + kvh * G + qr % G) * a.Sq + qr / G] * LOG2E;
        }
        sP[tid] = p;
        sL[tid] = l2;
        const int nv = (p < 0 || sF[0]) ? 0 : min(p + 1, kv_len);
        atomicMax(&sF[1], nv);
    }
    __syncthreads();
    const int n_keys = sF[1];
    for (int i = tid; i < (n_keys + PAGE - 1) / PAGE; i += BW_THREADS) {
        const int pg = __ldg(bt + i);
        if (pg < 0 || pg >= a.num_pages) atomicOr(&sF[0], RK_STATUS_PAGE_OOB);
    }
    // delta = rowsum(dout * out): two threads per row, 64 dims each, halves added in a fixed order
    {
        const int r = tid >> 1, hf = tid & 1;
        float acc = 0.0f;
        if (row_ok(r)) {
            const uint4* go = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.dout) + qrow_off(r)) + 8 * hf;
            const uint4* ov = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.out) + qrow_off(r)) + 8 * hf;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 x = __ldg(go + c), y = __ldg(ov + c);
                const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc = fmaf(bf16lo(xw[k]), bf16lo(yw[k]), acc);
                    acc = fmaf(bf16hi(xw[k]), bf16hi(yw[k]), acc);
                }
            }
        }
        const float other = __shfl_xor_sync(0xffffffffu, acc, 1);
        const float dsum = hf ? other + acc : acc + other;  // (low half) + (high half) on both threads
        if (hf == 0) {
            sD[r] = dsum;
            if (row_ok(r)) a.delta[((size_t)b * a.Hq + kvh * G + (qb * BW_QB + r) % G) * a.Sq + (qb * BW_QB + r) / G] = dsum;
        }
    }
    __syncthreads();
    const int bad = sF[0];
    uint32_t range = 0;
    if (!bad) {
        range = load_rotated(
            sm + DQ_OFF_Q, BW_QB,
            [&](int r) -> const uint4* {
                return row_ok(r) ? reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + qrow_off(r))
                                 : nullptr;
            },
            [&](int r) { return sP[r]; }, sT, range);
        load_plain(sm + DQ_OFF_DO, BW_QB, [&](int r) -> const uint4* {
            return row_ok(r) ? reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.dout) + qrow_off(r))
                             : nullptr;
        });
    }

    float acc[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
    const int ra = 16 * warp + (lane >> 2), rb = ra + 8;  // this lane's two accumulator rows
    const int n_tiles = bad ? 0 : (n_keys + BW_KT - 1) / BW_KT;
    bool over = false;
    const size_t kstride = (size_t)a.Hkv * HEAD_DIM;
    // K / V tiles of 64 keys, double-buffered: tile kt + 1 is copied (cp.async)
    // while tile kt is rotated and used; keys no row of the block sees are
    // zero-filled (their pages were not checked).
    auto key_ptr = [&](const void* cache, int t) -> const uint4* {
        if (t >= n_keys) return nullptr;
        const int pg = __ldg(bt + t / PAGE);
        return reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(cache) +
                                              ((size_t)pg * PAGE + t % PAGE) * kstride + (size_t)kvh * HEAD_DIM);
    };
    auto issue_tile = [&](int kt) {
        const int t0 = kt * BW_KT, st = kt & 1;
        copy_rows_async(base + DQ_OFF_K + st * BW_KT * 256, BW_KT, [&](int r) { return key_ptr(a.k_cache, t0 + r); },
                        a.k_cache);
        copy_rows_async(base + DQ_OFF_V + st * BW_KT * 256, BW_KT, [&](int r) { return key_ptr(a.v_cache, t0 + r); },
                        a.v_cache);
        cp_async_commit();
    };
    if (n_tiles > 0) issue_tile(0);
    for (int kt = 0; kt < n_tiles; ++kt) {
        const int t0 = kt * BW_KT, st = kt & 1;
        const uint32_t offK = DQ_OFF_K + st * BW_KT * 256, offV = DQ_OFF_V + st * BW_KT * 256;
        cp_async_wait_all();
        __syncthreads();  // tile kt landed everywhere; tile kt - 1 is no longer read
        if (kt + 1 < n_tiles) issue_tile(kt + 1);
        range = rotate_tile_inplace(sm + offK, t0, sT, sS, range);
        __syncthreads();
        // S = Q' K'^T and dP = dout V^T for this warp's 16 rows x 64 keys
        float s[8][4], dp[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = dp[j][0] = dp[j][1] = dp[j][2] = dp[j][3] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t aq[4], ao[4];
            ldsm_x4(aq, a_addr(base + DQ_OFF_Q, 16 * warp, 2 * kk, lane));
            ldsm_x4(ao, a_addr(base + DQ_OFF_DO, 16 * warp, 2 * kk, lane));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bk[4], bv[4];
                ldsm_x4(bk, b_addr(base + offK, 16 * np, 2 * kk, lane));
                ldsm_x4(bv, b_addr(base + offV, 16 * np, 2 * kk, lane));
                mma_f16(s[2 * np], aq, bk[0], bk[1]);
                mma_f16(s[2 * np + 1], aq, bk[2], bk[3]);
                mma_bf16(dp[2 * np], ao, bv[0], bv[1]);
                mma_bf16(dp[2 * np + 1], ao, bv[2], bv[3]);
            }
        }
        // P = exp(s - lse) on visible keys, dS = P (dP - delta)
        const int pa = sP[ra], pb = sP[rb];
        const float la = sL[ra], lb = sL[rb], da = sD[ra], db = sD[rb];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = t0 + 8 * j + 2 * (lane & 3) + e;
                const bool vis_a = t <= pa && t < kv_len, vis_b = t <= pb && t < kv_len;
                const float p0 = vis_a ? ex2(s[j][e] * a.qk_scale_log2 - la) : 0.0f;
                const float p1 = vis_b ? ex2(s[j][2 + e] * a.qk_scale_log2 - lb) : 0.0f;
                s[j][e] = p0 * (dp[j][e] - da);
                s[j][2 + e] = p1 * (dp[j][2 + e] - db);
            }
        }
        // dQ' += dS K' (k = keys, 4 steps of 16)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t sa[4];
            sa[0] = pack_ds(s[2 * ks][0], s[2 * ks][1], over);
            sa[1] = pack_ds(s[2 * ks][2], s[2 * ks][3], over);
            sa[2] = pack_ds(s[2 * ks + 1][0], s[2 * ks + 1][1], over);
            sa[3] = pack_ds(s[2 * ks + 1][2], s[2 * ks + 1][3], over);
#pragma unroll
            for (int nd = 0; nd < 8; ++nd) {
                uint32_t bk[4];
                ldsm_x4_t(bk, bt_addr(base + offK, 16 * ks, 2 * nd, lane));
                mma_f16(acc[2 * nd], sa, bk[0], bk[1]);
                mma_f16(acc[2 * nd + 1], sa, bk[2], bk[3]);
            }
        }
    }
    // status: unsafe metadata, FP16 range of rotated operands or of dS
    const bool rng_bad = __syncthreads_or((int)(range_exceeded(range) || over)) != 0;
    if (tid == 0 && a.status && (bad || rng_bad)) atomicOr(a.status, bad | (rng_bad ? RK_STATUS_RANGE : 0));
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] *= a.sm_scale;
    if (!bad) {
        unrotate_row(acc, 0, max(sP[ra], 0), sT, lane);
        unrotate_row(acc, 1, max(sP[rb], 0), sT, lane);
    }
    const float nanv = __int_as_float(0x7fc00000);
#pragma unroll
    for (int hsel = 0; hsel < 2; ++hsel) {
        const int r = hsel ? rb : ra;
        if (!row_ok(r)) continue;
        float* dst = a.dq + qrow_off(r);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int d = 8 * j + 2 * (lane & 3);
            float2 v = make_float2(acc[j][2 * hsel], acc[j][2 * hsel + 1]);
            if (bad || rng_bad) v = make_float2(nanv, nanv);
            *reinterpret_cast<float2*>(dst + d) = v;
        }
    }
}

// Shared memory of the dk/dv kernel: K' / V of the CTA's 64 keys, Q' / dout of
// one block of 64 query rows, per-row lse (natural log), delta, position.
constexpr int KV_OFF_K = 0;
constexpr int KV_OFF_V = KV_OFF_K + BW_KT * 256;
constexpr int KV_OFF_Q = KV_OFF_V + BW_KT * 256;          // two query blocks (copied raw, rotated in place)
constexpr int KV_OFF_DO = KV_OFF_Q + 2 * BW_QB_KV * 256;   // two dout blocks
constexpr int KV_OFF_L = KV_OFF_DO + 2 * BW_QB_KV * 256;   // [2][64] lse (natural log)
constexpr int KV_OFF_D = KV_OFF_L + 2 * BW_QB_KV * 4;      // [2][64] delta
constexpr int KV_OFF_P = KV_OFF_D + 2 * BW_QB_KV * 4;      // [2][64] positions
constexpr int KV_OFF_T = KV_OFF_P + 2 * BW_QB_KV * 4;
constexpr int KV_OFF_F = KV_OFF_T + ROPE_PAIRS * 8;
constexpr int KV_SMEM = KV_OFF_F + 16;

// One CTA per (row b, KV head, tile of 64 keys), first tiles first (they are
// seen by the most queries).  Walks the query rows that can see the tile (the
// first position >= the tile's first key, found by bisection of the ascending
// positions) in blocks of 64, ascending, and writes the tile's pages of dk / dv
// (slots past kv_len get 0).  Reads delta from the dq launch.
__global__ void __launch_bounds__(BW_THREADS) attn_bwd_dkdv_kernel(const __grid_constant__ BackwardArgs a) {
    extern __shared__ __align__(128) uint8_t sm[];
    float* sL = reinterpret_cast<float*>(sm + KV_OFF_L);
    float* sD = reinterpret_cast<float*>(sm + KV_OFF_D);
    int* sP = reinterpret_cast<int*>(sm + KV_OFF_P);
    uint64_t* sT = reinterpret_cast<uint64_t*>(sm + KV_OFF_T);
    int* sF = reinterpret_cast<int*>(sm + KV_OFF_F);  // [0] status bits, [1] first query position index
    const uint32_t base = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.G, nrows = a.Sq * G;
    const int units = a.B * a.Hkv;
    const int kt = (int)(blockIdx.x / units);
    const int b = (int)(blockIdx.x % units) / a.Hkv, kvh = (int)(blockIdx.x % units) % a.Hkv;
    const int t0 = kt * BW_KT;
    const int kv_len = a.kv_lens[b];
    if (kv_len < 0 || kv_len > a.W * PAGE) {  // nothing is known about the row's pages
        if (tid == 0 && kt == 0 && a.status) atomicOr(a.status, RK_STATUS_KVLEN);
        return;
    }
    const int n_rows = min(BW_KT, (kv_len + PAGE - 1) / PAGE * PAGE - t0);  // keys of this tile on the row's pages
    if (n_rows <= 0) return;
    const int32_t* bt = a.block_table + (size_t)b * a.W;
    if (tid == 0) {
        sF[0] = 0;
        // first s with position >= t0 (positions ascend along the row)
        int lo = 0, hi = a.Sq;
        const int32_t* pr = a.position_ids + (size_t)b * a.Sq;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (pr[mid] >= t0) hi = mid; else lo = mid + 1;
        }
        sF[1] = lo;
    }
    if (tid < ROPE_PAIRS) sT[tid] = a.rope_turns[tid];
    __syncthreads();
    if (tid < (n_rows + PAGE - 1) / PAGE) {
        const int pg = __ldg(bt + t0 / PAGE + tid);
        if (pg < 0 || pg >= a.num_pages) atomicOr(&sF[0], RK_STATUS_PAGE_OOB);
    }
    __syncthreads();
    const int bad = sF[0];
    if (bad) {  // the tile's pages are not safe to write
        if (tid == 0 && a.status) atomicOr(a.status, bad);
        return;
    }
    const size_t kstride = (size_t)a.Hkv * HEAD_DIM;
    auto key_src = [&](const void* cache, int r) -> const uint4* {
        const int t = t0 + r;
        if (t >= kv_len) return nullptr;
        const int pg = __ldg(bt + t / PAGE);
        return reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(cache) +
                                              ((size_t)pg * PAGE + t % PAGE) * kstride + (size_t)kvh * HEAD_DIM);
    };
    uint32_t range = load_rotated(
        sm + KV_OFF_K, BW_KT, [&](int r) { return key_src(a.k_cache, r); }, [&](int r) { return t0 + r; }, sT, 0u);
    load_plain(sm + KV_OFF_V, BW_KT, [&](int r) { return key_src(a.v_cache, r); });

    float dv[16][4], dk[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) dv[j][e] = dk[j][e] = 0.0f;
    const int ka = t0 + 16 * warp + (lane >> 2), kb = ka + 8;  // this lane's two key rows
    bool over = false;
    const int qb0 = sF[1] * G / BW_QB_KV, nqb = (nrows + BW_QB_KV - 1) / BW_QB_KV;
    // Query blocks of 64 rows, double-buffered: block qb + 1 (q, dout, lse,
    // delta, positions) is copied (cp.async) while block qb is rotated and used.
    auto q_off = [&](int qr) -> size_t {  // element offset / HEAD_DIM of query row qr in [B, Hq, Sq]
        return (((size_t)b * a.Hq + kvh * G + qr % G) * a.Sq + qr / G);
    };
    auto issue_block = [&](int qb) {
        const int sb = qb & 1, r0 = qb * BW_QB_KV;
        copy_rows_async(base + KV_OFF_Q + sb * BW_QB_KV * 256, BW_QB_KV, [&](int r) -> const uint4* {
            return r0 + r < nrows ? reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                                   q_off(r0 + r) * HEAD_DIM)
                                  : nullptr;
        }, a.q);
        copy_rows_async(base + KV_OFF_DO + sb * BW_QB_KV * 256, BW_QB_KV, [&](int r) -> const uint4* {
            return r0 + r < nrows ? reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.dout) +
                                                                   q_off(r0 + r) * HEAD_DIM)
                                  : nullptr;
        }, a.dout);
        if (tid < BW_QB_KV) {
            const bool ok = r0 + tid < nrows;
            const size_t o = ok ? q_off(r0 + tid) : 0;
            cp_async4(base + KV_OFF_P + (sb * BW_QB_KV + tid) * 4,
                      a.position_ids + (size_t)b * a.Sq + (ok ? (r0 + tid) / G : 0), ok);
            cp_async4(base + KV_OFF_L + (sb * BW_QB_KV + tid) * 4, a.lse + o, ok);
            cp_async4(base + KV_OFF_D + (sb * BW_QB_KV + tid) * 4, a.delta + o, ok);
        }
        cp_async_commit();
    };
    if (qb0 < nqb) issue_block(qb0);
    for (int qb = qb0; qb < nqb; ++qb) {
        const int sb = qb & 1;
        const int nvalid = nrows - qb * BW_QB_KV;  // rows of this block that exist
        const uint32_t offQ = KV_OFF_Q + sb * BW_QB_KV * 256, offO = KV_OFF_DO + sb * BW_QB_KV * 256;
        const int* bP = sP + sb * BW_QB_KV;
        const float* bL = sL + sb * BW_QB_KV;
        const float* bD = sD + sb * BW_QB_KV;
        cp_async_wait_all();
        __syncthreads();  // block qb landed everywhere; block qb - 1 is no longer read
        if (qb + 1 < nqb) issue_block(qb + 1);
        range = rotate_rows_inplace(sm + offQ, BW_QB_KV, [&](int r) { return max(bP[r], 0); }, sT, range);
        __syncthreads();
        // S^T = K' Q'^T and dP^T = V dout^T: this warp's 16 keys x 64 query rows
        float st[8][4], dpt[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) st[j][0] = st[j][1] = st[j][2] = st[j][3] = dpt[j][0] = dpt[j][1] = dpt[j][2] = dpt[j][3] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t ak[4], av[4];
            ldsm_x4(ak, a_addr(base + KV_OFF_K, 16 * warp, 2 * kk, lane));
            ldsm_x4(av, a_addr(base + KV_OFF_V, 16 * warp, 2 * kk, lane));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bq[4], bo[4];
                ldsm_x4(bq, b_addr(base + offQ, 16 * np, 2 * kk, lane));
                ldsm_x4(bo, b_addr(base + offO, 16 * np, 2 * kk, lane));
                mma_f16(st[2 * np], ak, bq[0], bq[1]);
                mma_f16(st[2 * np + 1], ak, bq[2], bq[3]);
                mma_bf16(dpt[2 * np], av, bo[0], bo[1]);
                mma_bf16(dpt[2 * np + 1], av, bo[2], bo[3]);
            }
        }
        // P^T (BF16, for dV) and dS^T (FP16, for dK') packed straight into the A
        // fragments of the k = query-row steps: score tile j is half j & 1 of step j >> 1
        uint32_t pa[4][4], sa[4][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float pv[4], dv4[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int qc = 8 * j + 2 * (lane & 3) + e;
                const int p = qc < nvalid ? bP[qc] : -1;
                const float l2 = bL[qc] * LOG2E, dl = bD[qc];
                pv[e] = (ka <= p && ka < kv_len) ? ex2(st[j][e] * a.qk_scale_log2 - l2) : 0.0f;
                pv[2 + e] = (kb <= p && kb < kv_len) ? ex2(st[j][2 + e] * a.qk_scale_log2 - l2) : 0.0f;
                dv4[e] = pv[e] * (dpt[j][e] - dl);
                dv4[2 + e] = pv[2 + e] * (dpt[j][2 + e] - dl);
            }
            const int ks = j >> 1, h = j & 1;
            pa[ks][2 * h] = pack_bf16x2(pv[0], pv[1]);
            pa[ks][2 * h + 1] = pack_bf16x2(pv[2], pv[3]);
            sa[ks][2 * h] = pack_ds(dv4[0], dv4[1], over);
            sa[ks][2 * h + 1] = pack_ds(dv4[2], dv4[3], over);
        }
        // dV += P^T dout and dK' += dS^T Q' (k = query rows, 4 steps of 16)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int nd = 0; nd < 8; ++nd) {
                uint32_t bo[4], bq[4];
                ldsm_x4_t(bo, bt_addr(base + offO, 16 * ks, 2 * nd, lane));
                ldsm_x4_t(bq, bt_addr(base + offQ, 16 * ks, 2 * nd, lane));
                mma_bf16(dv[2 * nd], pa[ks], bo[0], bo[1]);
                mma_bf16(dv[2 * nd + 1], pa[ks], bo[2], bo[3]);
                mma_f16(dk[2 * nd], sa[ks], bq[0], bq[1]);
                mma_f16(dk[2 * nd + 1], sa[ks], bq[2], bq[3]);
            }
        }
    }
    const bool rng_bad = __syncthreads_or((int)(range_exceeded(range) || over)) != 0;
    if (tid == 0 && a.status && rng_bad) atomicOr(a.status, RK_STATUS_RANGE);
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) dk[j][e] *= a.sm_scale;
    unrotate_row(dk, 0, ka, sT, lane);
    unrotate_row(dk, 1, kb, sT, lane);
    const float nanv = __int_as_float(0x7fc00000);
#pragma unroll
    for (int hsel = 0; hsel < 2; ++hsel) {
        const int t = hsel ? kb : ka;
        if (t - t0 >= n_rows) continue;
        const int pg = __ldg(bt + t / PAGE);
        const size_t off = ((size_t)pg * PAGE + t % PAGE) * kstride + (size_t)kvh * HEAD_DIM;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int d = 8 * j + 2 * (lane & 3);
            float2 x = make_float2(dk[j][2 * hsel], dk[j][2 * hsel + 1]);
            float2 y = make_float2(dv[j][2 * hsel], dv[j][2 * hsel + 1]);
            if (rng_bad) x = y = make_float2(nanv, nanv);
            *reinterpret_cast<float2*>(a.dk + off + d) = x;
            *reinterpret_cast<float2*>(a.dv + off + d) = y;
        }
    }
}

}  // namespace

cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load() & bit)) {
        e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KV_SMEM);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    const long long units = (long long)a.B * a.Hkv;
    const long long nqb = ((long long)a.Sq * a.G + BW_QB - 1) / BW_QB;
    const long long g_dq = units * nqb, g_kv = units * a.n_key_tiles;
    if (g_dq > 0x7fffffffLL || g_kv > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (g_dq > 0) {
        attn_bwd_dq_kernel<<<(unsigned)g_dq, BW_THREADS, DQ_SMEM, stream>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (g_kv > 0) {
        attn_bwd_dkdv_kernel<<<(unsigned)g_kv, BW_THREADS, KV_SMEM, stream>>>(a);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace rk
