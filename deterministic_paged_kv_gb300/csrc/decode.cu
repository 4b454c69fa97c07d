// decode.cu -- split-free paged decode with fused RoPE and GQA packing.
//
// Operation: paged decode of "flashinfer_fa2 backend for Ada (SM89)" (BF16,
// page 16, head_dim 128, NHD, split-KV disabled so a row's reduction does not
// depend on plan width or batch), with ROPE_LLAMA fused as in "WS2 PR7 Fused
// Attention Backend Alignment", "FlashInfer RoPE Fusion", and the FP32 LSE of
// the same page's "Original PR7 Requirements" table.
//
// Design (bandwidth-bound: 512 B of K+V per token and KV head):
//   * one CTA per (row b, KV head, up to 4 query heads); the CTA streams the
//     row's pages in ascending logical order, one page (16 tokens x 256 B for
//     K, the same for V) per pipeline stage, fetched by a dedicated producer
//     warp with TMA into an 8-deep shared-memory ring;
//   * four consumer warps; the 8-lane group g of warp w owns token slot
//     4w+g of every page, each lane 16 of the 128 dimensions laid out so a
//     lane holds both members of its 8 rotate-half pairs (dims 8j..8j+7 and
//     64+8j..64+8j+7): K is rotated in registers in FP32 as it is read;
//   * the rotation angles come from an exact fixed-point anchor every 16
//     pages and an angle-addition step of 16 positions in between;
//   * scores are reduced over the group with an xor butterfly (bitwise
//     identical in all 8 lanes), online softmax in the log2 domain with a
//     slack of 8 before the running maximum is moved (exact result, fewer
//     rescales), PV accumulated in FP32 registers;
//   * the 16 slot partial states are merged in fixed slot order 0..15, then
//     out is rounded to BF16 once (RNE) and the LSE written in FP32.
// Every choice above depends only on the row's own data and logical token
// index, never on B, W, grid size or which SM runs the CTA.
#include <atomic>

#include "rk_device.cuh"

namespace rk {

namespace {

constexpr uint32_t FULL = 0xffffffffu;

struct DecShared {
    uint64_t full_bar[DEC_STAGES];
    uint64_t empty_bar[DEC_STAGES];
    uint64_t turns[ROPE_PAIRS];
    float4 step[ROPE_PAIRS / 2];  // (cos, sin) of a 16-position turn, two pairs per entry
    int abort;
};
static_assert(sizeof(DecShared) <= DEC_CTRL_BYTES, "decode control block exceeds its reservation");
static_assert(16 * 4 * HEAD_DIM * 4 + 16 * 4 * 2 * 4 <= DEC_STAGES * DEC_STAGE_BYTES,
              "merge scratch must fit in the stage ring");

template <int GH>
__device__ __forceinline__ void write_empty_row(const DecodeArgs& a, int b, int h0, float lse_val) {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    for (int i = threadIdx.x; i < GH * HEAD_DIM; i += blockDim.x) {
        const int hh = i / HEAD_DIM, d = i % HEAD_DIM;
        out[((size_t)b * a.Hq + h0 + hh) * HEAD_DIM + d] = __float2bfloat16_rn(0.0f);
    }
    if (threadIdx.x < GH) a.lse[(size_t)b * a.Hq + h0 + threadIdx.x] = lse_val;
}

// 16 bf16 (two 16-byte chunks: dims 8j.. and 64+8j..) -> rotated floats.
__device__ __forceinline__ void load_rotate16(const uint4& lo4, const uint4& hi4, const float (&c)[8],
                                              const float (&s)[8], float (&x)[16]) {
    const uint32_t lw[4] = {lo4.x, lo4.y, lo4.z, lo4.w};
    const uint32_t hw[4] = {hi4.x, hi4.y, hi4.z, hi4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float l0 = bf16lo(lw[k]), l1 = bf16hi(lw[k]);
        const float u0 = bf16lo(hw[k]), u1 = bf16hi(hw[k]);
        const int e0 = 2 * k, e1 = 2 * k + 1;
        x[e0] = l0 * c[e0] - u0 * s[e0];
        x[8 + e0] = u0 * c[e0] + l0 * s[e0];
        x[e1] = l1 * c[e1] - u1 * s[e1];
        x[8 + e1] = u1 * c[e1] + l1 * s[e1];
    }
}

template <int GH>
__global__ void __launch_bounds__(DEC_THREADS, 2)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const __grid_constant__ DecodeArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* stages = smem;
    DecShared* sh = reinterpret_cast<DecShared*>(smem + DEC_STAGES * DEC_STAGE_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_hg = a.G / GH;
    int unit = blockIdx.x;
    const int hg = unit % n_hg;
    unit /= n_hg;
    const int kvh = unit % a.Hkv;
    const int b = unit / a.Hkv;
    const int h0 = kvh * a.G + hg * GH;

    // ---- row metadata and memory-safety checks (device copy of metadata) --
    const int kv_len = a.kv_lens[b];
    const int qpos = a.position_ids[b];
    int bad = 0;
    if (kv_len < 0 || kv_len > a.W * PAGE) bad |= RK_STATUS_KVLEN;
    if (qpos < 0) bad |= RK_STATUS_POSITION;
    const int n_vis = bad ? 0 : (qpos >= kv_len ? kv_len : qpos + 1);
    const int n_pages = (n_vis + PAGE - 1) / PAGE;
    const int32_t* bt = a.block_table + (size_t)b * a.W;
    int oob = 0;
    for (int i = threadIdx.x; i < n_pages; i += blockDim.x) {
        const int pg = __ldg(bt + i);
        oob |= (pg < 0) | (pg >= a.num_pages);
    }
    if (threadIdx.x < ROPE_PAIRS) sh->turns[threadIdx.x] = a.rope_turns[threadIdx.x];
    if (threadIdx.x < ROPE_PAIRS / 2) {
        float c0, s0, c1, s1;
        rope_cos_sin((uint32_t)PAGE, a.rope_turns[2 * threadIdx.x], c0, s0);
        rope_cos_sin((uint32_t)PAGE, a.rope_turns[2 * threadIdx.x + 1], c1, s1);
        sh->step[threadIdx.x] = make_float4(c0, s0, c1, s1);
    }
    if (threadIdx.x == 0) {
        sh->abort = 0;
        for (int s = 0; s < DEC_STAGES; ++s) {
            mbar_init(smem_u32(&sh->full_bar[s]), 1);
            mbar_init(smem_u32(&sh->empty_bar[s]), DEC_CWARPS);
        }
        fence_mbar_init();
    }
    if (__syncthreads_or(oob)) bad |= RK_STATUS_PAGE_OOB;
    if (bad) {
        if (threadIdx.x == 0 && a.status) atomicOr(a.status, bad);
        write_empty_row<GH>(a, b, h0, __int_as_float(0x7fc00000));
        return;
    }
    if (n_vis == 0) {
        write_empty_row<GH>(a, b, h0, -INFINITY);
        return;
    }

    if (warp == DEC_CWARPS) {
        // ------------------------------------------------ TMA producer ----
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
        bool ok = true;
        int issued = 0;
        for (int base = 0; base < n_pages && ok; base += 32) {
            const int idx = base + lane;
            const int pg = idx < n_pages ? __ldg(bt + idx) : 0;
            const int cnt = min(32, n_pages - base);
            for (int jj = 0; jj < cnt; ++jj) {
                const int page = __shfl_sync(FULL, pg, jj);
                const int it = base + jj;
                const int st = it % DEC_STAGES;
                const uint32_t ph = (uint32_t)(it / DEC_STAGES) & 1u;
                int good = 1;
                if (lane == 0) {
                    good = mbar_wait(smem_u32(&sh->empty_bar[st]), ph ^ 1u, &sh->abort);
                    if (good) {
                        const uint32_t fb = smem_u32(&sh->full_bar[st]);
                        mbar_arrive_expect_tx(fb, DEC_STAGE_BYTES);
                        const uint32_t dst = smem_u32(stages + st * DEC_STAGE_BYTES);
                        tma_load_3d(dst, &kmap, fb, 0, kvh, page * PAGE);
                        tma_load_3d(dst + DEC_PAGE_BYTES, &vmap, fb, 0, kvh, page * PAGE);
                    }
                }
                ok = __shfl_sync(FULL, good, 0) != 0;
                if (!ok) break;
                ++issued;
            }
        }
        if (!ok && lane == 0) {
            // Let copies already issued land before the CTA exits.
            for (int it = max(0, issued - DEC_STAGES); it < issued; ++it)
                mbar_wait_drain(smem_u32(&sh->full_bar[it % DEC_STAGES]),
                                (uint32_t)(it / DEC_STAGES) & 1u);
            if (a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
        }
        return;
    }

    // ---------------------------------------------------------- consumers --
    const int g = lane >> 3, j = lane & 7;
    const int slot = warp * 4 + g;
    const uint32_t gmask = 0xffu << (8 * g);

    // Query: rotate at its position, pre-scale by sm_scale * log2(e).
    float qv[GH][16];
    {
        float c[8], s[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) rope_cos_sin((uint32_t)qpos, sh->turns[8 * j + e], c[e], s[e]);
        const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
        for (int hh = 0; hh < GH; ++hh) {
            const uint4* row =
                reinterpret_cast<const uint4*>(qb + ((size_t)b * a.Hq + h0 + hh) * HEAD_DIM);
            load_rotate16(__ldg(row + j), __ldg(row + 8 + j), c, s, qv[hh]);
#pragma unroll
            for (int e = 0; e < 16; ++e) qv[hh][e] *= a.qk_scale_log2;
        }
    }

    // Key rotation state for this lane's 8 pairs at token t = 16*it + slot.
    float kc[8], ks[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) rope_cos_sin((uint32_t)slot, sh->turns[8 * j + e], kc[e], ks[e]);

    float m[GH], l[GH], acc[GH][16];
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
        m[hh] = -INFINITY;
        l[hh] = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[hh][e] = 0.0f;
    }

    bool ok = true;
    for (int it = 0; it < n_pages; ++it) {
        const int st = it % DEC_STAGES;
        const uint32_t ph = (uint32_t)(it / DEC_STAGES) & 1u;
        if (!mbar_wait(smem_u32(&sh->full_bar[st]), ph, &sh->abort)) {
            ok = false;
            break;
        }
        const int t = it * PAGE + slot;
        if (t < n_vis) {
            const uint8_t* kbase = stages + st * DEC_STAGE_BYTES + slot * (HEAD_DIM * 2);
            const uint4* krow = reinterpret_cast<const uint4*>(kbase);
            float kf[16];
            load_rotate16(krow[j], krow[8 + j], kc, ks, kf);
            float sc[GH];
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) {
                float p0 = 0.f, p1 = 0.f;
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    p0 = fmaf(qv[hh][e], kf[e], p0);
                    p1 = fmaf(qv[hh][e + 1], kf[e + 1], p1);
                }
                sc[hh] = p0 + p1;
            }
#pragma unroll
            for (int off = 4; off >= 1; off >>= 1) {
#pragma unroll
                for (int hh = 0; hh < GH; ++hh) sc[hh] += __shfl_xor_sync(gmask, sc[hh], off);
            }
            float p[GH];
#pragma unroll
            for (int hh = 0; hh < GH; ++hh) {
                if (sc[hh] > m[hh] + DEC_RESCALE_THRESHOLD) {
                    const float alpha = ex2(m[hh] - sc[hh]);
                    m[hh] = sc[hh];
                    l[hh] *= alpha;
#pragma unroll
                    for (int e = 0; e < 16; ++e) acc[hh][e] *= alpha;
                }
                p[hh] = ex2(sc[hh] - m[hh]);
                l[hh] += p[hh];
            }
            const uint4* vrow = reinterpret_cast<const uint4*>(kbase + DEC_PAGE_BYTES);
            const uint4 vlo = vrow[j], vhi = vrow[8 + j];
            const uint32_t lw[4] = {vlo.x, vlo.y, vlo.z, vlo.w};
            const uint32_t hw[4] = {vhi.x, vhi.y, vhi.z, vhi.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float v0 = bf16lo(lw[k]), v1 = bf16hi(lw[k]);
                const float w0 = bf16lo(hw[k]), w1 = bf16hi(hw[k]);
#pragma unroll
                for (int hh = 0; hh < GH; ++hh) {
                    acc[hh][2 * k] = fmaf(p[hh], v0, acc[hh][2 * k]);
                    acc[hh][2 * k + 1] = fmaf(p[hh], v1, acc[hh][2 * k + 1]);
                    acc[hh][8 + 2 * k] = fmaf(p[hh], w0, acc[hh][8 + 2 * k]);
                    acc[hh][8 + 2 * k + 1] = fmaf(p[hh], w1, acc[hh][8 + 2 * k + 1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh->empty_bar[st]));
        // Advance this lane's angles by one page (16 positions).
        if ((it + 1) % DEC_REANCHOR == 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                rope_cos_sin((uint32_t)(t + PAGE), sh->turns[8 * j + e], kc[e], ks[e]);
        } else {
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                const float4 st4 = sh->step[4 * j + e2];
                const float d0c = st4.x, d0s = st4.y, d1c = st4.z, d1s = st4.w;
                const int e0 = 2 * e2, e1 = 2 * e2 + 1;
                const float c0 = kc[e0] * d0c - ks[e0] * d0s, s0 = ks[e0] * d0c + kc[e0] * d0s;
                const float c1 = kc[e1] * d1c - ks[e1] * d1s, s1 = ks[e1] * d1c + kc[e1] * d1s;
                kc[e0] = c0; ks[e0] = s0; kc[e1] = c1; ks[e1] = s1;
            }
        }
    }

    // ------------------------------------ fixed-order merge of 16 slots ----
    named_bar_sync(1, DEC_CWARPS * 32);
    if (!ok || sh->abort) {
        if (threadIdx.x == 0 && a.status) atomicOr(a.status, RK_STATUS_TIMEOUT);
        return;
    }
    float* part = reinterpret_cast<float*>(stages);  // [16][GH][128]
    float* ml = part + 16 * GH * HEAD_DIM;           // [16][GH][2]
#pragma unroll
    for (int hh = 0; hh < GH; ++hh) {
        float* dst = part + (slot * GH + hh) * HEAD_DIM;
        *reinterpret_cast<float4*>(dst + 8 * j) = make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
        *reinterpret_cast<float4*>(dst + 8 * j + 4) =
            make_float4(acc[hh][4], acc[hh][5], acc[hh][6], acc[hh][7]);
        *reinterpret_cast<float4*>(dst + 64 + 8 * j) =
            make_float4(acc[hh][8], acc[hh][9], acc[hh][10], acc[hh][11]);
        *reinterpret_cast<float4*>(dst + 64 + 8 * j + 4) =
            make_float4(acc[hh][12], acc[hh][13], acc[hh][14], acc[hh][15]);
        if (j == 0) {
            ml[(slot * GH + hh) * 2 + 0] = m[hh];
            ml[(slot * GH + hh) * 2 + 1] = l[hh];
        }
    }
    named_bar_sync(1, DEC_CWARPS * 32);
    const int d = threadIdx.x;  // 0..127: one output dimension per thread
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
#pragma unroll 1
    for (int hh = 0; hh < GH; ++hh) {
        float M = -INFINITY;
#pragma unroll
        for (int sl = 0; sl < 16; ++sl) M = fmaxf(M, ml[(sl * GH + hh) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int sl = 0; sl < 16; ++sl) {
            const float w = ex2(ml[(sl * GH + hh) * 2] - M);
            L = fmaf(ml[(sl * GH + hh) * 2 + 1], w, L);
            O = fmaf(part[(sl * GH + hh) * HEAD_DIM + d], w, O);
        }
        out[((size_t)b * a.Hq + h0 + hh) * HEAD_DIM + d] = __float2bfloat16_rn(O / L);
        if (d == 0) a.lse[(size_t)b * a.Hq + h0 + hh] = (M + log2f(L)) * 0.693147180559945309f;
    }
}

}  // namespace

template <int GH>
static cudaError_t launch_decode_gh(const CUtensorMap& km, const CUtensorMap& vm, const DecodeArgs& a,
                                    cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load() & bit)) {
        e = cudaFuncSetAttribute(decode_kernel<GH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 DEC_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    const int grid = a.B * a.Hkv * (a.G / GH);
    decode_kernel<GH><<<grid, DEC_THREADS, DEC_SMEM_BYTES, stream>>>(km, vm, a);
    return cudaGetLastError();
}

cudaError_t launch_decode(const CUtensorMap& km, const CUtensorMap& vm, const DecodeArgs& a,
                          cudaStream_t stream) {
    switch (a.G) {
        case 1: return launch_decode_gh<1>(km, vm, a, stream);
        case 2: return launch_decode_gh<2>(km, vm, a, stream);
        default: return launch_decode_gh<4>(km, vm, a, stream);  // G = 4, or 8 as two CTAs
    }
}

}  // namespace rk
