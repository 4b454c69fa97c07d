// append.cu -- write new tokens' K and V (pre-RoPE, as the cache holds them)
// into their pages.
//
// The cache layout and the page walk are those of the attention kernels: the
// token at logical position t of row b lives in page block_table[b, t / 16],
// slot t % 16, as [Hkv, D] BF16 (NHD; "flashinfer_fa2 backend for Ada
// (SM89)", summary; "WS2 PR7 Fused Attention Backend Alignment", "FlashInfer
// RoPE Fusion": the K cache stays pre-RoPE and RoPE is applied when K is read).
// kv_lens are the lengths after the append: the n_new tokens of row b take
// positions kv_len - n_new .. kv_len - 1 (the chunk's own K/V is in the cache
// before its attention runs, "Current Implementation", trailing positions).
//
// One warp per (row, new token): a token is Hkv * D * 2 bytes of K and the same
// of V, copied with 16-byte loads and stores, its first loads issued before its
// page id is read.  Memory-safe: a token whose position or page is out of range
// is not written and flags the status word.
#include <atomic>

#include "rk_device.cuh"

namespace rk {

namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(const __grid_constant__ AppendArgs a) {
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (warp >= a.B * a.n_new) return;
    const int b = warp / a.n_new, j = warp % a.n_new;
    const size_t row16 = (size_t)a.Hkv * HEAD_DIM / 8;  // 16-byte chunks per token
    const uint4* ks = reinterpret_cast<const uint4*>(a.k_new) + ((size_t)b * a.n_new + j) * row16;
    const uint4* vs = reinterpret_cast<const uint4*>(a.v_new) + ((size_t)b * a.n_new + j) * row16;
    // The token's first chunks are loaded before its page is known (their
    // addresses need no metadata), so the data and the metadata round trips
    // overlap; every load of a pass is issued before its stores, a lane keeping
    // 2 x APPEND_UNROLL 16-byte loads in flight (the whole token for Hkv = 8).
    constexpr int APPEND_UNROLL = 4;
    uint4 kx[APPEND_UNROLL], vx[APPEND_UNROLL];
#pragma unroll
    for (int u = 0; u < APPEND_UNROLL; ++u) {
        const size_t c = lane + 32 * u;
        if (c < row16) {
            kx[u] = __ldcs(ks + c);  // the new tokens are read once: streaming loads
            vx[u] = __ldcs(vs + c);
        }
    }
    const int kv_len = a.kv_lens[b];
    int bad = 0;
    if (kv_len < a.n_new || kv_len > a.W * PAGE) bad |= RK_STATUS_KVLEN;
    const int t = kv_len - a.n_new + j;
    int pg = -1;
    if (!bad) {
        pg = a.block_table[(size_t)b * a.W + t / PAGE];
        if (pg < 0 || pg >= a.num_pages) bad |= RK_STATUS_PAGE_OOB;
    }
    if (bad) {
        if (lane == 0 && a.status) atomicOr(a.status, bad);
        return;
    }
    uint4* kd = reinterpret_cast<uint4*>(a.k_cache) + ((size_t)pg * PAGE + t % PAGE) * row16;
    uint4* vd = reinterpret_cast<uint4*>(a.v_cache) + ((size_t)pg * PAGE + t % PAGE) * row16;
    for (size_t c0 = lane;; c0 += 32 * APPEND_UNROLL) {
#pragma unroll
        for (int u = 0; u < APPEND_UNROLL; ++u) {
            const size_t c = c0 + 32 * u;
            if (c < row16) {
                kd[c] = kx[u];
                vd[c] = vx[u];
            }
        }
        if (c0 + 32 * APPEND_UNROLL >= row16) break;
#pragma unroll
        for (int u = 0; u < APPEND_UNROLL; ++u) {  // the next pass (Hkv > 8)
            const size_t c = c0 + 32 * APPEND_UNROLL + 32 * u;
            if (c < row16) {
                kx[u] = __ldcs(ks + c);
                vx[u] = __ldcs(vs + c);
            }
        }
    }
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream) {
    const long long warps = (long long)a.B * a.n_new;
    if (warps <= 0) return cudaSuccess;
    const long long blocks = (warps + 7) / 8;  // 8 warps per block
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kv_append_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace rk
