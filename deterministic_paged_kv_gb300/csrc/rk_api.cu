// rk_api.cu -- the C ABI: host-side validation (rk_paged_plan), tensor-map
// construction and the two asynchronous launch calls.  No device memory is
// allocated and no call synchronises or reads device memory on the host.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "rk_internal.h"
#include "rk_paged.h"

namespace rk {
cudaError_t launch_decode(const CUtensorMap& vm, const DecodeArgs& a, cudaStream_t stream);
cudaError_t decode_resident_ctas(int* ctas);
cudaError_t launch_prefill(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                           const PrefillArgs& a, cudaStream_t stream, bool overlap_previous = false);
cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream);
cudaError_t launch_backward_dkdv_tc(const CUtensorMap& qm, const CUtensorMap& om, const CUtensorMap& km,
                                    const CUtensorMap& vm, const BackwardArgs& a, cudaStream_t stream);
cudaError_t launch_backward_dq_tc(const CUtensorMap& qm, const CUtensorMap& om, const CUtensorMap& km,
                                  const CUtensorMap& vm, const BackwardArgs& a, cudaStream_t stream);
cudaError_t launch_backward_rotate(const BackwardArgs& a, cudaStream_t stream);
}  // namespace rk

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

const double kTwoPi = 6.283185307179586476925286766559;

// -------------------------------------------------------------- plan ----

int check_shape(int32_t B, int32_t Sq, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                int32_t num_pages, int32_t W, double theta, double scale) {
    if (B < 0 || Sq < 1 || Hq < 1 || Hkv < 1 || W < 0 || num_pages < 0)
        return fail(RK_E_ARG, "bad sizes: B=%d Sq=%d Hq=%d Hkv=%d W=%d num_pages=%d", B, Sq, Hq, Hkv,
                    W, num_pages);
    if (!(theta > 1.0) || !std::isfinite(theta))
        return fail(RK_E_ARG, "rope_theta must be a finite value > 1 (got %g)", theta);
    if (!(scale > 0.0) || !std::isfinite(scale))
        return fail(RK_E_ARG, "rope_scale must be a finite value > 0 (got %g)", scale);
    if (D != rk::HEAD_DIM) return fail(RK_E_UNSUPPORTED, "head_dim %d unsupported (only 128)", D);
    if (page_size != rk::PAGE)
        return fail(RK_E_UNSUPPORTED, "page_size %d unsupported (only 16)", page_size);
    if (Hq % Hkv) return fail(RK_E_UNSUPPORTED, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
    const int G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(RK_E_UNSUPPORTED, "GQA group size %d unsupported (1, 2, 4 or 8)", G);
    if ((int64_t)W * rk::PAGE > INT32_MAX / 2) return fail(RK_E_ARG, "table width %d too large", W);
    if ((int64_t)num_pages * rk::PAGE > INT32_MAX / 2)
        return fail(RK_E_ARG, "num_pages %d too large", num_pages);
    if ((int64_t)B * Hq * Sq > INT32_MAX) return fail(RK_E_ARG, "B * Hq * Sq too large");
    return RK_OK;
}

// Row b's queries are pos[b * Sq .. b * Sq + Sq) (qo == nullptr), or the
// packed range pos[qo[b] .. qo[b + 1]) of a ragged batch (rows may be empty).
int check_metadata(int32_t B, int32_t Sq, int32_t num_pages, int32_t W, const int32_t* bt,
                   const int32_t* kv, const int32_t* pos, int32_t* max_kv, const int32_t* qo = nullptr) {
    *max_kv = 0;
    for (int b = 0; b < B; ++b) {
        const int n = kv[b];
        if (n < 0 || (int64_t)n > (int64_t)W * rk::PAGE)
            return fail(RK_E_KVLEN, "row %d: kv_len %d outside [0, %d]", b, n, W * rk::PAGE);
        if (n > *max_kv) *max_kv = n;
    }
    for (int b = 0; b < B; ++b) {
        const int n = kv[b];
        const int npg = (n + rk::PAGE - 1) / rk::PAGE;
        const int32_t* row = bt + (size_t)b * W;
        for (int j = 0; j < npg; ++j)
            if (row[j] < 0 || row[j] >= num_pages)
                return fail(RK_E_PAGE_OOB, "row %d: block_table[%d] = %d outside [0, %d)", b, j,
                            row[j], num_pages);
        for (int j = npg; j < W; ++j)
            if (row[j] != -1)
                return fail(RK_E_PAD, "row %d: inactive block_table[%d] = %d (must be -1)", b, j,
                            row[j]);
    }
    std::vector<uint8_t> used((size_t)num_pages, 0);
    for (int b = 0; b < B; ++b) {
        const int npg = (kv[b] + rk::PAGE - 1) / rk::PAGE;
        const int32_t* row = bt + (size_t)b * W;
        for (int j = 0; j < npg; ++j) {
            if (used[row[j]])
                return fail(RK_E_DUP_PAGE, "physical page %d appears twice (row %d, entry %d)",
                            row[j], b, j);
            used[row[j]] = 1;
        }
    }
    for (int b = 0; b < B; ++b) {
        const int32_t* p = qo ? pos + qo[b] : pos + (size_t)b * Sq;
        const int nq = qo ? qo[b + 1] - qo[b] : Sq;
        if (nq == 0) continue;  // a ragged row with no query this step
        for (int s = 0; s < nq; ++s) {
            if (p[s] < 0) return fail(RK_E_POSITION, "row %d: position_ids[%d] = %d < 0", b, s, p[s]);
            if (s > 0 && p[s] != p[s - 1] + 1)
                return fail(RK_E_POSITION, "row %d: positions not contiguous ascending at %d", b, s);
        }
        const int n = kv[b];
        const int last = p[nq - 1];
        if (n == 0) {
            if (nq > 1)
                return fail(RK_E_POSITION,
                            "row %d: empty row with %d queries (only decode rows may be empty)", b, nq);
        } else if (last != n - 1 && last != n) {
            return fail(RK_E_POSITION,
                        "row %d: last query position %d is neither kv_len-1 = %d nor kv_len = %d", b,
                        last, n - 1, n);
        }
    }
    return RK_OK;
}

// ----------------------------------------------------------- device -----

std::atomic<uint64_t> g_dev_ok{0}, g_dev_bad{0};

int check_device() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(RK_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 64) {
        const uint64_t bit = 1ull << dev;
        if (g_dev_ok.load() & bit) return RK_OK;
        if (g_dev_bad.load() & bit)
            return fail(RK_E_DEVICE, "device %d is not compute capability 10.3 (sm_103)", dev);
    }
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return fail(RK_E_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    const bool ok = (major == 10 && minor == 3);
    if (dev < 64) (ok ? g_dev_ok : g_dev_bad).fetch_or(1ull << dev);
    if (!ok)
        return fail(RK_E_DEVICE, "device %d is compute capability %d.%d; this library is built for sm_103a",
                    dev, major, minor);
    return RK_OK;
}

// ------------------------------------------------------- tensor maps ----

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
             const cuuint64_t* strides_bytes, const cuuint32_t* box, CUtensorMapSwizzle swz,
             const char* what) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(RK_E_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims,
                    strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(RK_E_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
    return RK_OK;
}

// Page cache [num_pages, 16, Hkv, 128] seen as 3-D (d, head, token row).
int make_cache_map(CUtensorMap* m, const void* cache, int num_pages, int Hkv, int box_d,
                   CUtensorMapSwizzle swz, const char* what) {
    const cuuint64_t dims[3] = {(cuuint64_t)rk::HEAD_DIM, (cuuint64_t)Hkv,
                                (cuuint64_t)(num_pages > 0 ? num_pages : 1) * rk::PAGE};
    const cuuint64_t strides[2] = {(cuuint64_t)rk::HEAD_DIM * 2, (cuuint64_t)Hkv * rk::HEAD_DIM * 2};
    const cuuint32_t box[3] = {(cuuint32_t)box_d, 1, (cuuint32_t)rk::PAGE};
    return make_map(m, cache, 3, dims, strides, box, swz, what);
}

// The same cache seen as 4-D (64 dims, token row, 64-dim half, head): one box
// of (64, 16, 2, 1) copies a whole page of one head (4 KiB) and lands as
// [half][16 rows][128 B], 128-byte swizzled.
int make_page_map(CUtensorMap* m, const void* cache, int num_pages, int Hkv, const char* what) {
    const cuuint64_t dims[4] = {64, (cuuint64_t)(num_pages > 0 ? num_pages : 1) * rk::PAGE, 2, (cuuint64_t)Hkv};
    const cuuint64_t strides[3] = {(cuuint64_t)Hkv * rk::HEAD_DIM * 2, 128, (cuuint64_t)rk::HEAD_DIM * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)rk::PAGE, 2, 1};
    return make_map(m, cache, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, what);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_launch_common(const rk_paged_plan_t* plan, const void* q, const void* kc, const void* vc,
                        const int32_t* bt, const int32_t* kl, const int32_t* pos, const void* out,
                        const float* lse) {
    if (!plan) return fail(RK_E_ARG, "plan is NULL");
    if (plan->abi != RK_PAGED_ABI_VERSION)
        return fail(RK_E_ARG, "plan ABI %u does not match library ABI %u (plan not filled by rk_paged_plan?)",
                    plan->abi, RK_PAGED_ABI_VERSION);
    int rc = check_shape(plan->B, plan->Sq, plan->Hq, plan->Hkv, plan->D, plan->page_size,
                         plan->num_pages, plan->W, plan->rope_theta, plan->rope_scale);
    if (rc) return rc;
    if (plan->B == 0) return RK_OK;
    if (!q || !out || !lse || !kl || !pos) return fail(RK_E_ARG, "null device pointer");
    if (plan->W > 0 && !bt) return fail(RK_E_ARG, "block_table is NULL");
    if (plan->num_pages > 0 && (!kc || !vc)) return fail(RK_E_ARG, "k_cache / v_cache is NULL");
    if (!aligned(q, 16) || !aligned(out, 16) || (kc && !aligned(kc, 16)) || (vc && !aligned(vc, 16)))
        return fail(RK_E_ARG, "q, k_cache, v_cache and out must be 16-byte aligned");
    if (!aligned(lse, 4) || !aligned(kl, 4) || !aligned(pos, 4) || (bt && !aligned(bt, 4)))
        return fail(RK_E_ARG, "lse and metadata must be 4-byte aligned");
    return check_device();
}

}  // namespace

extern "C" {

const char* rk_last_error(void) { return g_err.c_str(); }

uint32_t rk_paged_abi_version(void) { return RK_PAGED_ABI_VERSION; }

const char* rk_paged_policy(void) {
    return "split_kv=disabled;acc=fp32;lse=fp32,natural,scaled_scores;softmax_scale=1/sqrt(head_dim);"
           "downcast=final_write,bf16,rne;order=ascending_kv;rope=llama_rotate_half,fused_q_and_k,"
           "rotary_dim=head_dim;gqa=contiguous_groups;decode_tile=kv128,score_mma=fp16_operands_fp32_acc,"
           "pv_mma=bf16_operands_fp32_acc,l_merge=fixed_tree;"
           "prefill_tile=2xq128xkv128,score_mma=fp16_operands_fp32_acc,pv_mma=bf16_operands_fp32_acc;"
           "batch_invariant=1;page_size=16;head_dim=128;"
           "decode_split_entry=fixed_splits_of_16k_tokens,ordered_fp32_merge,separate_policy";
}

int rk_paged_plan(rk_paged_plan_t* plan, int32_t B, int32_t Sq, int32_t Hq, int32_t Hkv, int32_t D,
                  int32_t page_size, int32_t num_pages, int32_t W, const int32_t* block_table_h,
                  const int32_t* kv_lens_h, const int32_t* position_ids_h, double rope_theta,
                  double rope_scale) {
    g_err.clear();
    if (!plan) return fail(RK_E_ARG, "plan is NULL");
    std::memset(plan, 0, sizeof *plan);
    int rc = check_shape(B, Sq, Hq, Hkv, D, page_size, num_pages, W, rope_theta, rope_scale);
    if (rc) return rc;
    const bool any = block_table_h || kv_lens_h || position_ids_h;
    const bool check = kv_lens_h && position_ids_h && (block_table_h || W == 0);
    if (any && !check)
        return fail(RK_E_ARG, "pass all three host metadata arrays, or none for a shape-only plan");
    int32_t max_kv = 0;
    if (check && B > 0) {
        static const int32_t kEmpty = -1;
        rc = check_metadata(B, Sq, num_pages, W, block_table_h ? block_table_h : &kEmpty, kv_lens_h,
                            position_ids_h, &max_kv);
        if (rc) return rc;
    }
    plan->abi = RK_PAGED_ABI_VERSION;
    plan->B = B;
    plan->Sq = Sq;
    plan->Hq = Hq;
    plan->Hkv = Hkv;
    plan->D = D;
    plan->page_size = page_size;
    plan->W = W;
    plan->num_pages = num_pages;
    plan->causal = 1;
    plan->max_kv_len = max_kv;
    plan->pf_units = -1;
    plan->sm_scale = (float)(1.0 / std::sqrt((double)D));
    plan->validated = check ? 1 : 0;
    plan->rope_theta = rope_theta;
    plan->rope_scale = rope_scale;
    plan->wait_limit_ns = (uint32_t)RK_WAIT_LIMIT_NS;
    plan->timeout_drill = 0;
    for (int i = 0; i < D / 2; ++i) {
        // Turns per position of pair i: theta^(-2i/D) / (2 pi scale), in [0, 1/(2 pi)].
        const double w = std::pow(rope_theta, -2.0 * (double)i / (double)D) / (kTwoPi * rope_scale);
        const double fx = std::ldexp(w, 64);
        plan->rope_turns[i] = fx >= 18446744073709551615.0 ? ~0ull : (uint64_t)fx;
    }
    return RK_OK;
}

int rk_paged_plan_ragged(rk_paged_plan_t* plan, int32_t B, int32_t total_q, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t page_size, int32_t num_pages, int32_t W, const int32_t* qo_indptr_h,
                         const int32_t* block_table_h, const int32_t* kv_lens_h, const int32_t* position_ids_h,
                         double rope_theta, double rope_scale, int32_t* max_q_len) {
    g_err.clear();
    if (!plan || !qo_indptr_h || !max_q_len) return fail(RK_E_ARG, "plan, qo_indptr and max_q_len must be non-null");
    std::memset(plan, 0, sizeof *plan);
    if (B < 0 || total_q < 1) return fail(RK_E_ARG, "bad sizes: B=%d total_q=%d (need B >= 0, total_q >= 1)", B, total_q);
    if (qo_indptr_h[0] != 0 || qo_indptr_h[B] != total_q)
        return fail(RK_E_ARG, "qo_indptr must start at 0 and end at total_q = %d (got %d .. %d)", total_q,
                    qo_indptr_h[0], qo_indptr_h[B]);
    int32_t mq = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t n = qo_indptr_h[b + 1] - qo_indptr_h[b];
        if (n < 0) return fail(RK_E_ARG, "qo_indptr decreases at row %d", b);
        mq = n > mq ? n : mq;
    }
    // shapes as a padded plan of Sq = total_q (the packed q has total_q tokens)
    int rc = rk_paged_plan(plan, B, total_q, Hq, Hkv, D, page_size, num_pages, W, nullptr, nullptr, nullptr,
                           rope_theta, rope_scale);
    if (rc) return rc;
    const bool any = block_table_h || kv_lens_h || position_ids_h;
    const bool check = kv_lens_h && position_ids_h && (block_table_h || W == 0);
    if (any && !check) {
        std::memset(plan, 0, sizeof *plan);
        return fail(RK_E_ARG, "pass all three host metadata arrays, or none for a shape-only plan");
    }
    if (check && B > 0) {
        static const int32_t kEmpty = -1;
        int32_t max_kv = 0;
        rc = check_metadata(B, total_q, num_pages, W, block_table_h ? block_table_h : &kEmpty, kv_lens_h,
                            position_ids_h, &max_kv, qo_indptr_h);
        if (rc) {
            std::memset(plan, 0, sizeof *plan);
            return rc;
        }
        plan->max_kv_len = max_kv;
        plan->validated = 1;
    }
    const int32_t span = 2 * (rk::PF_BM / (Hq / Hkv));
    int64_t units = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t n = qo_indptr_h[b + 1] - qo_indptr_h[b];
        if (n >= 2) units += (n + span - 1) / span;
    }
    plan->pf_units = (int32_t)units;  // at most total_q / 2
    *max_q_len = mq;
    return RK_OK;
}

namespace {

// Splits of a row's KV range for split_tokens per split: enough for the
// widest row the table allows (W pages), at least one.
int64_t split_count(const rk_paged_plan_t* plan, int32_t split_tokens) {
    const int64_t cap = (int64_t)plan->W * rk::PAGE;
    return cap > 0 ? (cap + split_tokens - 1) / split_tokens : 1;
}

int64_t split_scratch_need(const rk_paged_plan_t* plan, int32_t split_tokens) {
    const int64_t n = (int64_t)plan->B * plan->Hq * split_count(plan, split_tokens);
    return n * rk::HEAD_DIM * 4 + n * 4;  // o_part then lse_part
}

// Shared by the split-free and the split entry points (split_tokens = 0: none).
int decode_common(const rk_paged_plan_t* plan, int32_t split_tokens, const void* q, const void* k_cache,
                  const void* v_cache, const int32_t* block_table_d, const int32_t* kv_lens_d,
                  const int32_t* position_ids_d, void* out, float* lse, void* scratch, uint64_t scratch_bytes,
                  int32_t* status_d, rk_stream_t stream, bool balanced = false) {
    g_err.clear();
    int rc = check_launch_common(plan, q, k_cache, v_cache, block_table_d, kv_lens_d, position_ids_d,
                                 out, lse);
    if (rc) return rc;
    if (plan->Sq != 1) return fail(RK_E_ARG, "decode needs a plan with Sq == 1 (got %d)", plan->Sq);
    if (split_tokens < 0 || (split_tokens > 0 && split_tokens % rk::DEC_SPLIT_GRAIN != 0))
        return fail(RK_E_ARG, "split_tokens must be a positive multiple of %d (got %d)", rk::DEC_SPLIT_GRAIN,
                    split_tokens);
    if (split_tokens > 0) {
        const int64_t need = split_scratch_need(plan, split_tokens);
        if (!scratch || !aligned(scratch, 16))
            return fail(RK_E_ARG, "split decode scratch must be a non-null 16-byte aligned device pointer");
        if ((uint64_t)need > scratch_bytes)
            return fail(RK_E_ARG, "split decode scratch too small: %lld bytes needed, %llu given", (long long)need,
                        (unsigned long long)scratch_bytes);
        if (split_count(plan, split_tokens) > 0x7fffffffLL) return fail(RK_E_ARG, "too many splits");
    }
    if (balanced) {
        if (!scratch || !aligned(scratch, 256))
            return fail(RK_E_ARG, "balanced decode scratch must be a non-null 256-byte aligned device pointer");
        if (scratch_bytes < RK_PAGED_BALANCED_SCRATCH_BYTES)
            return fail(RK_E_ARG, "balanced decode scratch too small: %llu bytes needed, %llu given",
                        (unsigned long long)RK_PAGED_BALANCED_SCRATCH_BYTES, (unsigned long long)scratch_bytes);
    }
    if (plan->B == 0) return RK_OK;
    const bool have = plan->num_pages > 0;
    CUtensorMap vm;
    if ((rc = make_page_map(&vm, have ? v_cache : q, have ? plan->num_pages : 1, have ? plan->Hkv : 1, "v_cache")))
        return rc;
    rk::DecodeArgs a;
    std::memset(&a, 0, sizeof a);
    a.q = q;
    a.k_cache = k_cache;
    a.block_table = block_table_d;
    a.kv_lens = kv_lens_d;
    a.position_ids = position_ids_d;
    a.out = out;
    a.lse = lse;
    a.status = status_d;
    a.B = plan->B;
    a.Hq = plan->Hq;
    a.Hkv = plan->Hkv;
    a.G = plan->Hq / plan->Hkv;
    a.W = plan->W;
    a.num_pages = plan->num_pages;
    a.qk_scale_log2 = (float)((1.0 / std::sqrt((double)plan->D)) * 1.4426950408889634074);
    a.wait_limit_ns = plan->wait_limit_ns;
    a.timeout_drill = plan->timeout_drill;
    if (split_tokens > 0) {
        const int64_t n = (int64_t)plan->B * plan->Hq * split_count(plan, split_tokens);
        a.split_tokens = split_tokens;
        a.n_splits = (int32_t)split_count(plan, split_tokens);
        a.o_part = static_cast<float*>(scratch);
        a.lse_part = static_cast<float*>(scratch) + n * rk::HEAD_DIM;
    }
    std::memcpy(a.rope_turns, plan->rope_turns, sizeof a.rope_turns);
    if (balanced) {
        int ctas = 0;
        cudaError_t e = rk::decode_resident_ctas(&ctas);
        if (e != cudaSuccess) return fail(RK_E_CUDA, "decode occupancy: %s", cudaGetErrorString(e));
        // Hkv chains of `members` CTAs (one per KV head)
        const int members = std::min(ctas, RK_PAGED_BALANCED_MAX_CTAS) / plan->Hkv;
        // the finest block (tiles, a power of two up to 8) for which the most
        // blocks one CTA could get (every row as wide as the table) still fit its
        // segment list; finer blocks balance the chains more evenly
        int block_tiles = 0;
        for (int bt = 1; members > 0 && bt <= rk::DEC_BAL_MAX_BLOCK_TILES && !block_tiles; bt *= 2) {
            const int64_t row_blocks =
                std::max<int64_t>(1, ((int64_t)plan->W * rk::PAGE + bt * rk::DEC_BN - 1) / (bt * rk::DEC_BN));
            const int64_t per_cta = ((int64_t)plan->B * row_blocks + members - 1) / members;
            if (per_cta + 2 <= rk::DEC_BAL_MAX_SEGS) block_tiles = bt;
        }
        if (members >= 2 && plan->B >= members && plan->B <= rk::DEC_BAL_MAX_ROWS && block_tiles > 0) {
            a.balanced = 1;
            a.bal_block_tiles = block_tiles;
            a.bal_grid = members * plan->Hkv;
            a.bal_sync = static_cast<uint32_t*>(scratch);
            a.bal_state = reinterpret_cast<float*>(static_cast<char*>(scratch) + 4096);
        }
    }
    cudaError_t e = rk::launch_decode(vm, a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(RK_E_CUDA, "decode launch: %s", cudaGetErrorString(e));
    return RK_OK;
}

}  // namespace

int rk_paged_attn_decode(const rk_paged_plan_t* plan, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_table_d, const int32_t* kv_lens_d,
                         const int32_t* position_ids_d, void* out, float* lse, int32_t* status_d,
                         rk_stream_t stream) {
    return decode_common(plan, 0, q, k_cache, v_cache, block_table_d, kv_lens_d, position_ids_d, out, lse,
                         nullptr, 0, status_d, stream);
}

static_assert((rk::DEC_BAL_SYNC_WORDS + RK_PAGED_BALANCED_MAX_CTAS) * 4 <= 4096 &&
                  RK_PAGED_BALANCED_SCRATCH_BYTES ==
                      4096ull + (uint64_t)RK_PAGED_BALANCED_MAX_CTAS * rk::DEC_BAL_STATE_FLOATS * 4,
              "balanced scratch layout: 4 KiB of flags, then one hand-off state per CTA");

int rk_paged_decode_balanced_scratch_bytes(const rk_paged_plan_t* plan, uint64_t* bytes) {
    g_err.clear();
    if (!plan || !bytes) return fail(RK_E_ARG, "plan and bytes must be non-null");
    if (plan->abi != RK_PAGED_ABI_VERSION) return fail(RK_E_ARG, "plan ABI %u != %u", plan->abi, RK_PAGED_ABI_VERSION);
    *bytes = RK_PAGED_BALANCED_SCRATCH_BYTES;
    return RK_OK;
}

int rk_paged_attn_decode_balanced(const rk_paged_plan_t* plan, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_table_d, const int32_t* kv_lens_d,
                                  const int32_t* position_ids_d, void* out, float* lse, void* scratch,
                                  uint64_t scratch_bytes, int32_t* status_d, rk_stream_t stream) {
    return decode_common(plan, 0, q, k_cache, v_cache, block_table_d, kv_lens_d, position_ids_d, out, lse,
                         scratch, scratch_bytes, status_d, stream, true);
}

int rk_paged_decode_split_scratch_bytes(const rk_paged_plan_t* plan, int32_t split_tokens, uint64_t* bytes) {
    g_err.clear();
    if (!plan || !bytes) return fail(RK_E_ARG, "plan and bytes must be non-null");
    if (plan->abi != RK_PAGED_ABI_VERSION) return fail(RK_E_ARG, "plan ABI %u != %u", plan->abi, RK_PAGED_ABI_VERSION);
    if (split_tokens <= 0 || split_tokens % rk::DEC_SPLIT_GRAIN != 0)
        return fail(RK_E_ARG, "split_tokens must be a positive multiple of %d (got %d)", rk::DEC_SPLIT_GRAIN,
                    split_tokens);
    *bytes = (uint64_t)split_scratch_need(plan, split_tokens);
    return RK_OK;
}

int rk_paged_attn_decode_split(const rk_paged_plan_t* plan, int32_t split_tokens, const void* q,
                               const void* k_cache, const void* v_cache, const int32_t* block_table_d,
                               const int32_t* kv_lens_d, const int32_t* position_ids_d, void* out, float* lse,
                               void* scratch, uint64_t scratch_bytes, int32_t* status_d, rk_stream_t stream) {
    if (split_tokens <= 0) {
        g_err.clear();
        return fail(RK_E_ARG, "split_tokens must be a positive multiple of %d (got %d)", rk::DEC_SPLIT_GRAIN,
                    split_tokens);
    }
    return decode_common(plan, split_tokens, q, k_cache, v_cache, block_table_d, kv_lens_d, position_ids_d, out,
                         lse, scratch, scratch_bytes, status_d, stream);
}

namespace {

// Scratch of rk_paged_attn_decode_split_static: one file-scope device array
// shared by every call on a device (the library allocates nothing).
static __device__ __align__(256) unsigned char g_split_scratch[RK_PAGED_SPLIT_STATIC_SCRATCH_BYTES];

// Its device address, looked up once per device (with that device current).
std::atomic<uintptr_t> g_split_scratch_addr[64];

int split_static_scratch(void** p) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(RK_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < 64) {
        const uintptr_t a = g_split_scratch_addr[dev].load();
        if (a) {
            *p = reinterpret_cast<void*>(a);
            return RK_OK;
        }
    }
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_split_scratch);
    if (e != cudaSuccess || !a)
        return fail(RK_E_CUDA, "cudaGetSymbolAddress(split scratch): %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < 64) g_split_scratch_addr[dev].store(reinterpret_cast<uintptr_t>(a));
    *p = a;
    return RK_OK;
}

}  // namespace

int rk_paged_attn_decode_split_static(const rk_paged_plan_t* plan, int32_t split_tokens, const void* q,
                                      const void* k_cache, const void* v_cache, const int32_t* block_table_d,
                                      const int32_t* kv_lens_d, const int32_t* position_ids_d, void* out,
                                      float* lse, int32_t* status_d, rk_stream_t stream) {
    g_err.clear();
    if (!plan) return fail(RK_E_ARG, "plan must be non-null");
    if (split_tokens <= 0 || split_tokens % rk::DEC_SPLIT_GRAIN != 0)
        return fail(RK_E_ARG, "split_tokens must be a positive multiple of %d (got %d)", rk::DEC_SPLIT_GRAIN,
                    split_tokens);
    if (plan->abi != RK_PAGED_ABI_VERSION) return fail(RK_E_ARG, "plan ABI %u != %u", plan->abi, RK_PAGED_ABI_VERSION);
    const int64_t need = split_scratch_need(plan, split_tokens);
    if (need > (int64_t)RK_PAGED_SPLIT_STATIC_SCRATCH_BYTES)
        return fail(RK_E_ARG, "split partials need %lld bytes, above the %llu-byte static scratch", (long long)need,
                    (unsigned long long)RK_PAGED_SPLIT_STATIC_SCRATCH_BYTES);
    void* scratch = nullptr;
    int rc = split_static_scratch(&scratch);
    if (rc) return rc;
    // Nothing in the scratch has to start at zero: the split kernel writes every
    // partial the merge reads, in the same call, so nothing is cleared here.
    return decode_common(plan, split_tokens, q, k_cache, v_cache, block_table_d, kv_lens_d, position_ids_d, out,
                         lse, scratch, RK_PAGED_SPLIT_STATIC_SCRATCH_BYTES, status_d, stream);
}

int rk_paged_kv_append(const rk_paged_plan_t* plan, int32_t n_new, const void* k_new, const void* v_new,
                       const int32_t* block_table_d, const int32_t* kv_lens_d, void* k_cache, void* v_cache,
                       int32_t* status_d, rk_stream_t stream) {
    g_err.clear();
    if (!plan) return fail(RK_E_ARG, "plan is NULL");
    if (plan->abi != RK_PAGED_ABI_VERSION)
        return fail(RK_E_ARG, "plan ABI %u does not match library ABI %u (plan not filled by rk_paged_plan?)",
                    plan->abi, RK_PAGED_ABI_VERSION);
    int rc = check_shape(plan->B, plan->Sq, plan->Hq, plan->Hkv, plan->D, plan->page_size, plan->num_pages,
                         plan->W, plan->rope_theta, plan->rope_scale);
    if (rc) return rc;
    if (n_new < 0) return fail(RK_E_ARG, "n_new must be >= 0 (got %d)", n_new);
    if (plan->B == 0 || n_new == 0) return RK_OK;
    if (plan->W == 0 || plan->num_pages == 0)
        return fail(RK_E_KVLEN, "appending %d tokens needs a non-empty block table and page pool", n_new);
    if (!k_new || !v_new || !block_table_d || !kv_lens_d || !k_cache || !v_cache)
        return fail(RK_E_ARG, "null device pointer");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return fail(RK_E_ARG, "k_new, v_new, k_cache and v_cache must be 16-byte aligned");
    if (!aligned(block_table_d, 4) || !aligned(kv_lens_d, 4)) return fail(RK_E_ARG, "metadata must be 4-byte aligned");
    if ((rc = check_device())) return rc;
    rk::AppendArgs a;
    std::memset(&a, 0, sizeof a);
    a.k_new = k_new;
    a.v_new = v_new;
    a.block_table = block_table_d;
    a.kv_lens = kv_lens_d;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.status = status_d;
    a.B = plan->B;
    a.n_new = n_new;
    a.Hkv = plan->Hkv;
    a.W = plan->W;
    a.num_pages = plan->num_pages;
    cudaError_t e = rk::launch_kv_append(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(RK_E_CUDA, "append launch: %s", cudaGetErrorString(e));
    return RK_OK;
}

int rk_paged_attn_prefill(const rk_paged_plan_t* plan, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* block_table_d, const int32_t* kv_lens_d,
                          const int32_t* position_ids_d, void* out, float* lse, int32_t* status_d,
                          rk_stream_t stream) {
    g_err.clear();
    int rc = check_launch_common(plan, q, k_cache, v_cache, block_table_d, kv_lens_d, position_ids_d,
                                 out, lse);
    if (rc) return rc;
    if (plan->B == 0) return RK_OK;
    const int G = plan->Hq / plan->Hkv;
    const int rph = rk::PF_BM / G;
    // Q [B, Hq, Sq, D] as 4-D (d, position, head, row); box = one 64-column
    // half of a q-tile: (64, 128/G positions, G heads, 1 row), 128-byte swizzle.
    CUtensorMap qm, km, vm;
    {
        const cuuint64_t dims[4] = {(cuuint64_t)rk::HEAD_DIM, (cuuint64_t)plan->Sq, (cuuint64_t)plan->Hq,
                                    (cuuint64_t)plan->B};
        const cuuint64_t strides[3] = {(cuuint64_t)rk::HEAD_DIM * 2,
                                       (cuuint64_t)plan->Sq * rk::HEAD_DIM * 2,
                                       (cuuint64_t)plan->Hq * plan->Sq * rk::HEAD_DIM * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)rph, (cuuint32_t)G, 1};
        if ((rc = make_map(&qm, q, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "q"))) return rc;
    }
    const bool have = plan->num_pages > 0;
    if ((rc = make_cache_map(&km, have ? k_cache : q, have ? plan->num_pages : 1, have ? plan->Hkv : 1, 64,
                             CU_TENSOR_MAP_SWIZZLE_128B, "k_cache")))
        return rc;
    if ((rc = make_page_map(&vm, have ? v_cache : q, have ? plan->num_pages : 1, have ? plan->Hkv : 1, "v_cache")))
        return rc;
    rk::PrefillArgs a;
    std::memset(&a, 0, sizeof a);
    a.block_table = block_table_d;
    a.kv_lens = kv_lens_d;
    a.position_ids = position_ids_d;
    a.out = out;
    a.lse = lse;
    a.status = status_d;
    a.B = plan->B;
    a.Sq = plan->Sq;
    a.Hq = plan->Hq;
    a.Hkv = plan->Hkv;
    a.G = G;
    a.W = plan->W;
    a.num_pages = plan->num_pages;
    a.rows_per_head = rph;
    a.n_qtiles = (plan->Sq + rph - 1) / rph;
    a.qk_scale_log2 = (float)((1.0 / std::sqrt((double)plan->D)) * 1.4426950408889634074);
    a.wait_limit_ns = plan->wait_limit_ns;
    a.timeout_drill = plan->timeout_drill;
    std::memcpy(a.rope_turns, plan->rope_turns, sizeof a.rope_turns);
    cudaError_t e = rk::launch_prefill(qm, km, vm, a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(RK_E_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return RK_OK;
}

}  // extern "C"

namespace {

// Workspace of the prefill backward, each part 256-byte aligned: RoPE-rotated
// q (FP16), rotated K and a copy of V in logical token order (FP16 / BF16
// [B, Hkv, W * 16, D]), delta (FP32 [B, Hq, Sq]).
int64_t backward_ws_q(const rk_paged_plan_t* p) { return (int64_t)p->B * p->Hq * p->Sq * rk::HEAD_DIM * 2; }
int64_t backward_ws_k(const rk_paged_plan_t* p) {
    return (int64_t)p->B * p->Hkv * p->W * rk::PAGE * rk::HEAD_DIM * 2;
}
int64_t align256(int64_t x) { return (x + 255) & ~(int64_t)255; }
int64_t backward_ws_need(const rk_paged_plan_t* p) {
    return align256(backward_ws_q(p)) + 2 * align256(backward_ws_k(p)) + align256((int64_t)p->B * p->Hq * p->Sq * 4);
}

}  // namespace

extern "C" {

int rk_paged_prefill_backward_workspace_bytes(const rk_paged_plan_t* plan, uint64_t* bytes) {
    g_err.clear();
    if (!plan || !bytes) return fail(RK_E_ARG, "plan and bytes must be non-null");
    if (plan->abi != RK_PAGED_ABI_VERSION) return fail(RK_E_ARG, "plan ABI %u != %u", plan->abi, RK_PAGED_ABI_VERSION);
    *bytes = (uint64_t)backward_ws_need(plan);
    return RK_OK;
}

int rk_paged_attn_prefill_backward(const rk_paged_plan_t* plan, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_table_d, const int32_t* kv_lens_d,
                                   const int32_t* position_ids_d, const void* out, const float* lse,
                                   const void* dout, float* dq, float* dk_cache, float* dv_cache, void* workspace,
                                   uint64_t workspace_bytes, int32_t* status_d, rk_stream_t stream) {
    g_err.clear();
    int rc = check_launch_common(plan, q, k_cache, v_cache, block_table_d, kv_lens_d, position_ids_d, out, lse);
    if (rc) return rc;
    if (plan->B == 0) return RK_OK;
    if (!dout || !dq || !workspace) return fail(RK_E_ARG, "dout, dq and workspace must be non-null device pointers");
    if (plan->num_pages > 0 && (!dk_cache || !dv_cache)) return fail(RK_E_ARG, "dk_cache / dv_cache is NULL");
    if (!aligned(dout, 16) || !aligned(dq, 16) || (dk_cache && !aligned(dk_cache, 16)) ||
        (dv_cache && !aligned(dv_cache, 16)) || !aligned(workspace, 256))
        return fail(RK_E_ARG, "dout, dq, dk_cache and dv_cache must be 16-byte aligned, workspace 256-byte aligned");
    if ((uint64_t)backward_ws_need(plan) > workspace_bytes)
        return fail(RK_E_ARG, "backward workspace too small: %lld bytes needed, %llu given",
                    (long long)backward_ws_need(plan), (unsigned long long)workspace_bytes);
    rk::BackwardArgs a;
    std::memset(&a, 0, sizeof a);
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table_d;
    a.kv_lens = kv_lens_d;
    a.position_ids = position_ids_d;
    a.out = out;
    a.lse = lse;
    a.dout = dout;
    a.dq = dq;
    a.dk = dk_cache;
    a.dv = dv_cache;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.q_rot = ws;
    a.k_lin = ws + align256(backward_ws_q(plan));
    a.v_lin = ws + align256(backward_ws_q(plan)) + align256(backward_ws_k(plan));
    a.delta = reinterpret_cast<float*>(ws + align256(backward_ws_q(plan)) + 2 * align256(backward_ws_k(plan)));
    a.status = status_d;
    a.B = plan->B;
    a.Sq = plan->Sq;
    a.Hq = plan->Hq;
    a.Hkv = plan->Hkv;
    a.G = plan->Hq / plan->Hkv;
    a.W = plan->W;
    a.num_pages = plan->num_pages;
    a.sm_scale = (float)(1.0 / std::sqrt((double)plan->D));
    a.qk_scale_log2 = (float)((1.0 / std::sqrt((double)plan->D)) * 1.4426950408889634074);
    a.wait_limit_ns = plan->wait_limit_ns;
    a.timeout_drill = plan->timeout_drill;
    std::memcpy(a.rope_turns, plan->rope_turns, sizeof a.rope_turns);
    // tensor maps of the dk / dv kernel: q and dout [B, Hq, Sq, D] as 4-D (d, position, head, row) with
    // a box of one 64-column half of a query block (64, 128/G positions, G heads, 1 row); both caches
    // in 16-token x 64-dim page boxes (the K-major tile layout of both A operands)
    CUtensorMap qm, om, km, vm;
    {
        const int G = plan->Hq / plan->Hkv;
        const cuuint64_t dims[4] = {(cuuint64_t)rk::HEAD_DIM, (cuuint64_t)plan->Sq, (cuuint64_t)plan->Hq,
                                    (cuuint64_t)plan->B};
        const cuuint64_t strides[3] = {(cuuint64_t)rk::HEAD_DIM * 2, (cuuint64_t)plan->Sq * rk::HEAD_DIM * 2,
                                       (cuuint64_t)plan->Hq * plan->Sq * rk::HEAD_DIM * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)(rk::PF_BM / G), (cuuint32_t)G, 1};
        if ((rc = make_map(&qm, a.q_rot, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "rotated q"))) return rc;
        if ((rc = make_map(&om, dout, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "dout"))) return rc;
    }
    {  // rotated K and V in logical order: (d, token, row x KV head), box of 128 tokens x 64 dims
        const int64_t T = (int64_t)plan->W * rk::PAGE;
        const cuuint64_t dims[3] = {(cuuint64_t)rk::HEAD_DIM, (cuuint64_t)(T > 0 ? T : 1),
                                    (cuuint64_t)plan->B * plan->Hkv};
        const cuuint64_t strides[2] = {(cuuint64_t)rk::HEAD_DIM * 2, (cuuint64_t)(T > 0 ? T : 1) * rk::HEAD_DIM * 2};
        const cuuint32_t box[3] = {64, 128, 1};
        if ((rc = make_map(&km, a.k_lin, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "rotated k"))) return rc;
        if ((rc = make_map(&vm, a.v_lin, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "linear v"))) return rc;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = rk::launch_backward_rotate(a, st);                 // q and K rotated once
    if (e == cudaSuccess) e = rk::launch_backward_dq_tc(qm, om, km, vm, a, st);  // dq and delta
    if (e == cudaSuccess) e = rk::launch_backward_dkdv_tc(qm, om, km, vm, a, st);
    if (e != cudaSuccess) return fail(RK_E_CUDA, "backward launch: %s", cudaGetErrorString(e));
    return RK_OK;
}

int rk_paged_attn_ragged(const rk_paged_plan_t* plan, int32_t max_q_len, const int32_t* qo_indptr_d, const void* q,
                         const void* k_cache, const void* v_cache, const int32_t* block_table_d,
                         const int32_t* kv_lens_d, const int32_t* position_ids_d, void* out, float* lse,
                         int32_t* status_d, rk_stream_t stream) {
    g_err.clear();
    int rc = check_launch_common(plan, q, k_cache, v_cache, block_table_d, kv_lens_d, position_ids_d, out, lse);
    if (rc) return rc;
    if (plan->B == 0) return RK_OK;
    const int32_t total_q = plan->Sq;
    if (max_q_len < 1 || max_q_len > total_q)
        return fail(RK_E_ARG, "max_q_len %d outside [1, total_q = %d]", max_q_len, total_q);
    if (!qo_indptr_d || !aligned(qo_indptr_d, 4)) return fail(RK_E_ARG, "qo_indptr must be a 4-byte aligned device pointer");
    const int G = plan->Hq / plan->Hkv;
    const int rph = rk::PF_BM / G;
    const bool have = plan->num_pages > 0;
    const float qk = (float)((1.0 / std::sqrt((double)plan->D)) * 1.4426950408889634074);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // single-query rows: the decode kernel
    {
        CUtensorMap vm;
        if ((rc = make_page_map(&vm, have ? v_cache : q, have ? plan->num_pages : 1, have ? plan->Hkv : 1,
                                "v_cache")))
            return rc;
        rk::DecodeArgs a;
        std::memset(&a, 0, sizeof a);
        a.q = q;
        a.k_cache = k_cache;
        a.block_table = block_table_d;
        a.kv_lens = kv_lens_d;
        a.position_ids = position_ids_d;
        a.out = out;
        a.lse = lse;
        a.status = status_d;
        a.B = plan->B;
        a.Hq = plan->Hq;
        a.Hkv = plan->Hkv;
        a.G = G;
        a.W = plan->W;
        a.num_pages = plan->num_pages;
        a.qk_scale_log2 = qk;
        a.qo_indptr = qo_indptr_d;
        a.total_q = total_q;
        a.max_q_len = max_q_len;
        a.wait_limit_ns = plan->wait_limit_ns;
        a.timeout_drill = plan->timeout_drill;
        std::memcpy(a.rope_turns, plan->rope_turns, sizeof a.rope_turns);
        cudaError_t e = rk::launch_decode(vm, a, st);
        if (e != cudaSuccess) return fail(RK_E_CUDA, "ragged decode launch: %s", cudaGetErrorString(e));
    }
    if (max_q_len < 2) return RK_OK;
    // rows of two or more queries: the prefill kernel, one CTA per work unit
    // (pair of q-tiles) and KV head.  Without a count from the plan, bound the
    // units over every batch of this shape: at most m = min(B, total_q / 2)
    // rows hold two or more queries, each row at most levels pairs, and all
    // of them together at most (total_q + (span - 1) m) / span.
    const int64_t span = 2 * rph;
    const int64_t levels = (max_q_len + span - 1) / span;
    if (levels > rk::PF_RAGGED_MAX_LEVELS)
        return fail(RK_E_UNSUPPORTED, "max_q_len %d needs %lld pairs of q-tiles per row (at most %d)", max_q_len,
                    (long long)levels, rk::PF_RAGGED_MAX_LEVELS);
    int64_t units = plan->pf_units;
    if (units < 0) {
        const int64_t m = std::min<int64_t>(plan->B, total_q / 2);
        units = std::min<int64_t>(m * levels, ((int64_t)total_q + (span - 1) * m) / span);
    }
    units = std::max<int64_t>(units, 1);  // one CTA still checks the device indptr
    // packed q [total_q, Hq, D]
    // seen as (d, token, head) so that a box (64, 128/G tokens, G heads) lands
    // head-major like the padded layout's q-tile
    CUtensorMap qm, km, vm;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)rk::HEAD_DIM, (cuuint64_t)total_q, (cuuint64_t)plan->Hq};
        const cuuint64_t strides[2] = {(cuuint64_t)plan->Hq * rk::HEAD_DIM * 2, (cuuint64_t)rk::HEAD_DIM * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)rph, (cuuint32_t)G};
        if ((rc = make_map(&qm, q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "q (packed)"))) return rc;
    }
    if ((rc = make_cache_map(&km, have ? k_cache : q, have ? plan->num_pages : 1, have ? plan->Hkv : 1, 64,
                             CU_TENSOR_MAP_SWIZZLE_128B, "k_cache")))
        return rc;
    if ((rc = make_page_map(&vm, have ? v_cache : q, have ? plan->num_pages : 1, have ? plan->Hkv : 1, "v_cache")))
        return rc;
    rk::PrefillArgs a;
    std::memset(&a, 0, sizeof a);
    a.block_table = block_table_d;
    a.kv_lens = kv_lens_d;
    a.position_ids = position_ids_d;
    a.out = out;
    a.lse = lse;
    a.status = status_d;
    a.B = plan->B;
    a.Sq = total_q;
    a.Hq = plan->Hq;
    a.Hkv = plan->Hkv;
    a.G = G;
    a.W = plan->W;
    a.num_pages = plan->num_pages;
    a.rows_per_head = rph;
    a.n_qtiles = (max_q_len + rph - 1) / rph;
    a.qk_scale_log2 = qk;
    a.qo_indptr = qo_indptr_d;
    a.total_q = total_q;
    a.max_q_len = max_q_len;
    a.ragged_units = (int32_t)units;
    a.wait_limit_ns = plan->wait_limit_ns;
    a.timeout_drill = plan->timeout_drill;
    std::memcpy(a.rope_turns, plan->rope_turns, sizeof a.rope_turns);
    // started while the decode launch drains: the two write disjoint rows
    cudaError_t e = rk::launch_prefill(qm, km, vm, a, st, true);
    if (e != cudaSuccess) return fail(RK_E_CUDA, "ragged prefill launch: %s", cudaGetErrorString(e));
    return RK_OK;
}

}  // extern "C"
