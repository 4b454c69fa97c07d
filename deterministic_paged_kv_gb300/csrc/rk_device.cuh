// rk_device.cuh -- inline-PTX building blocks for the sm_103a kernels:
// mbarriers with bounded waits, TMA tensor loads, tcgen05 (TMEM alloc, MMA,
// commit, loads), bf16 packing, RoPE angle generation.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "rk_internal.h"
#include "rk_paged.h"

namespace rk {

// ------------------------------------------------------------- basics ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two bf16 (low half = element 2k, high half = element 2k+1) -> two floats.
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two floats -> packed bf16x2, round-to-nearest-even (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------- mbarriers ----

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// A waiting thread is suspended until the phase completes or the hint time
// passes, so waiting warps leave the issue slots to the working ones.
constexpr uint32_t RK_SUSPEND_HINT_NS = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(RK_SUSPEND_HINT_NS)
        : "memory");
    return ok != 0;
}

// Non-blocking test of whether phase `parity` of an mbarrier has completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared state of one CTA's pipeline waits: the abort flag every wait
// watches, and the wall time after which a wait gives up (the launch's wait
// limit, at most RK_WAIT_LIMIT_NS).
struct PipeCtl {
    int abort;
    uint32_t limit_ns;
};
__device__ __forceinline__ bool pipe_aborted(PipeCtl* pc) { return *reinterpret_cast<volatile int*>(&pc->abort) != 0; }

// Wait for phase `parity` of an mbarrier to complete.  Gives up (returns
// false) once it has waited limit_ns of wall time past its first 32 probes,
// or as soon as another warp has set the abort flag, so that a pipeline that
// lost a participant cannot hang.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, PipeCtl* pc) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    const uint64_t lim = pc->limit_ns;
#pragma unroll 1
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (pipe_aborted(pc)) return false;
        if (global_timer_ns() - t0 > lim) {
            *reinterpret_cast<volatile int*>(&pc->abort) = 1;
            return false;
        }
    }
}

// Launch wait limit as the kernels use it: 0 means the default, and nothing
// above the default or below 1 us.
__device__ __forceinline__ uint32_t wait_limit(uint32_t ns) {
    return ns == 0 ? (uint32_t)RK_WAIT_LIMIT_NS : (ns < 1000u ? 1000u : (ns > (uint32_t)RK_WAIT_LIMIT_NS ? (uint32_t)RK_WAIT_LIMIT_NS : ns));
}

// Test of the timeout exit (a launch's timeout_drill flag): the calling thread
// waits on an mbarrier of its CTA that nothing arrives at, so the wait runs
// out after the launch's limit, sets the abort flag and returns false; every
// other wait of the CTA then gives up and the CTA takes its drain-and-exit
// path.  `never` must be initialised with an arrival count of 1.
__device__ __forceinline__ bool drill_wait(uint32_t never, PipeCtl* pc) { return mbar_wait(never, 0, pc); }

// Wait with a time limit only (used on the way out after an abort).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < RK_WAIT_LIMIT_NS) {
    }
}

// Named barrier among `nthreads` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier over nthreads threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- TMA ----

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// 16-byte asynchronous copy global -> shared through the load/store path,
// cached in L2 only.  Completion is tracked per thread in commit groups; the
// data lands in the generic proxy (fence before the tensor core reads it).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor core operand reads, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------- programmatic launch ----
// A grid launched next on the stream with programmatic stream serialization
// may start its CTAs once every CTA of this grid has executed this or exited.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the grids this one depends on programmatically have completed
// and their writes are visible (at once for a launch without that dependency).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------ tcgen05 ----

// Allocate `ncols` TMEM columns (power of two >= 32); whole warp executes.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]; kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on an mbarrier once every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Unrolled MMA groups.  Every operand of these kernels is a 128-byte-swizzled
// tile in the CTA's shared memory whose descriptor has SBO = 1024 B, version
// bit 46 and swizzle mode 2, so descriptors differ only in their low word
// (start address >> 4 in bits 0..13, leading byte offset >> 4 in bits 16..29).
// The k-step offset of each MMA is an immediate added inside the asm: the
// issuing thread keeps two base words live and issues one MMA after another
// without recomputing descriptors, which a single thread must do to keep up
// with the tensor pipe.
constexpr uint32_t DESC_HI = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
    return ((saddr & 0x3FFFFu) >> 4) | ((lbo_bytes >> 4) << 16);
}
// Operand layouts and their k-step (16 elements) offsets in descriptor units
// (no carry into bit 14: all operands lie below 256 KiB of shared memory).
enum OperandLayout : int {
    K_MAJOR_128 = 0,  // [128 rows][2 x 64 elements] K-major: 64-element blocks 16 KiB apart
    K_MAJOR_16 = 1,   // [16 rows][2 x 64 elements] K-major: blocks 2 KiB apart
    MN_MAJOR = 2,     // [2 x 64 MN elements][K rows]: a k-step is 16 rows = 2 KiB
    MN_MAJOR_PAGE = 3 // [page][2 x 64 MN elements][16 rows] (LBO 2 KiB): a k-step is one 4 KiB page
};
__host__ __device__ constexpr uint32_t kstep_off(int layout, int ks) {
    return layout == K_MAJOR_128 ? (uint32_t)(((ks >> 2) * 16384 + (ks & 3) * 32) >> 4)
           : layout == K_MAJOR_16 ? (uint32_t)(((ks >> 2) * 2048 + (ks & 3) * 32) >> 4)
           : layout == MN_MAJOR   ? (uint32_t)(ks * (2048 >> 4))
                                  : (uint32_t)(ks * (4096 >> 4));
}
// D[tmem] (+)= A[smem] * B[smem], k-steps KS..END-1 of operands with the given
// layouts; accumulates from k-step 1 on, and at k-step 0 iff acc0.
// ELECT = false: called by the single issuing thread.  ELECT = true: called by
// a whole converged warp (operands stay warp-uniform) and the lane chosen by
// elect.sync (the lowest active lane, the same every time) issues; that lane
// must also issue the tcgen05.commit tracking the MMAs (umma_commit_elect).
template <int KS, int END, int LA, int LB, bool ELECT = false>
__device__ __forceinline__ void mma_ss_steps(uint32_t d, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                             uint32_t acc0) {
    if constexpr (ELECT) {
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 al, bl;\n\t.reg .b64 da, db;\n\t"
            "add.u32 al, %1, %5;\n\tadd.u32 bl, %2, %6;\n\t"
            "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
            "setp.ne.b32 p, %7, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d),
            "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(DESC_HI), "n"(kstep_off(LA, KS)), "n"(kstep_off(LB, KS)),
            "r"(KS > 0 ? 1u : acc0)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t.reg .b32 al, bl;\n\t.reg .b64 da, db;\n\t"
            "add.u32 al, %1, %5;\n\tadd.u32 bl, %2, %6;\n\t"
            "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
            "setp.ne.b32 p, %7, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d),
            "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(DESC_HI), "n"(kstep_off(LA, KS)), "n"(kstep_off(LB, KS)),
            "r"(KS > 0 ? 1u : acc0)
            : "memory");
    }
    if constexpr (KS + 1 < END) mma_ss_steps<KS + 1, END, LA, LB, ELECT>(d, a_lo, b_lo, idesc, acc0);
}
// D[tmem] (+)= A[tmem] * B[smem], k-steps KS..END-1; A holds 8 columns of
// packed 16-bit pairs per k-step.  ELECT as above.
template <int KS, int END, int LB, bool ELECT = false>
__device__ __forceinline__ void mma_ts_steps(uint32_t d, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                             uint32_t acc0) {
    if constexpr (ELECT) {
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t.reg .b32 at, bl;\n\t.reg .b64 db;\n\t"
            "add.u32 at, %1, %5;\n\tadd.u32 bl, %2, %6;\n\t"
            "mov.b64 db, {bl, %4};\n\t"
            "setp.ne.b32 p, %7, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, p;\n\t}" ::"r"(d),
            "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(DESC_HI), "n"(KS * 8), "n"(kstep_off(LB, KS)),
            "r"(KS > 0 ? 1u : acc0)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t.reg .b32 at, bl;\n\t.reg .b64 db;\n\t"
            "add.u32 at, %1, %5;\n\tadd.u32 bl, %2, %6;\n\t"
            "mov.b64 db, {bl, %4};\n\t"
            "setp.ne.b32 p, %7, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, p;\n\t}" ::"r"(d),
            "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(DESC_HI), "n"(KS * 8), "n"(kstep_off(LB, KS)),
            "r"(KS > 0 ? 1u : acc0)
            : "memory");
    }
    if constexpr (KS + 1 < END) mma_ts_steps<KS + 1, END, LB, ELECT>(d, a_tmem, b_lo, idesc, acc0);
}
// tcgen05.commit by the elected lane of a converged warp (the lane that
// issued the MMAs it tracks with ELECT = true).
__device__ __forceinline__ void umma_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets, fixed version bits 46..48 = 0b001, swizzle mode in
// bits 61..63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle_mode) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(swizzle_mode & 7u) << 61;
    return d;
}

// Instruction descriptor for kind::f16: bf16 A and B, fp32 D, dense.
// a_mn_major / b_mn_major select MN-major (transposed) operand layouts.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn_major, int b_mn_major) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | ((uint32_t)a_mn_major << 15)  // A major-ness
           | ((uint32_t)b_mn_major << 16)  // B major-ness
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets row
// (warp's lane quarter + i), columns col..col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Store 32 consecutive 32-bit columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]; A is 16-bit, two elements per 32-bit column.
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                        uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// Instruction descriptor for kind::f16 with FP16 A and B, FP32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Two floats -> packed f16x2, round-to-nearest-even (lo in the low half).
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 128-byte swizzle: byte offset of 16-byte chunk `chunk` (0..7) of 128-byte row `row`
// inside a 1024-byte aligned swizzle atom sequence.
__device__ __forceinline__ uint32_t sw128_off(int row, int chunk) {
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Packed FP32 pair arithmetic (sm_100+): two lanes of a*b+c / a*b in one instruction.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Rotate one chunk pair (8 rotate-half pairs: 16 bf16 at lo_ptr / hi_ptr) in FP32
// and write FP16 in place.  c2 / s2 hold the cos / sin of pairs (2k, 2k+1).
// Returns the running max of the |input| bf16 bit patterns (FP16 range check).
__device__ __forceinline__ uint32_t rotate_regs_f16(uint4& a, uint4& b, const float2 (&c2)[4], const float2 (&s2)[4],
                                                    uint32_t range) {
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
    uint32_t ow[4], pw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        range = __vmaxu2(range, aw[k] & 0x7fff7fffu);
        range = __vmaxu2(range, bw[k] & 0x7fff7fffu);
        const float2 lo = make_float2(bf16lo(aw[k]), bf16hi(aw[k]));
        const float2 hi = make_float2(bf16lo(bw[k]), bf16hi(bw[k]));
        const float2 nhi = make_float2(-hi.x, -hi.y);
        const float2 x = ffma2(nhi, s2[k], fmul2(lo, c2[k]));  // lo*c - hi*s
        const float2 y = ffma2(lo, s2[k], fmul2(hi, c2[k]));   // hi*c + lo*s
        ow[k] = pack_f16x2(x.x, x.y);
        pw[k] = pack_f16x2(y.x, y.y);
    }
    a = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    b = make_uint4(pw[0], pw[1], pw[2], pw[3]);
    return range;
}
__device__ __forceinline__ uint32_t rotate_chunk_f16(uint8_t* lo_ptr, uint8_t* hi_ptr, const float2 (&c2)[4],
                                                     const float2 (&s2)[4], uint32_t range) {
    uint4 a = *reinterpret_cast<const uint4*>(lo_ptr);
    uint4 b = *reinterpret_cast<const uint4*>(hi_ptr);
    range = rotate_regs_f16(a, b, c2, s2, range);
    *reinterpret_cast<uint4*>(lo_ptr) = a;
    *reinterpret_cast<uint4*>(hi_ptr) = b;
    return range;
}

// Advance 8 pairs' (cos, sin) by a fixed angle step (cos, sin) = (dc, ds):
// c' = c dc - s ds, s' = s dc + c ds.
__device__ __forceinline__ void rope_step(float2 (&c2)[4], float2 (&s2)[4], const float2 (&dc2)[4],
                                          const float2 (&ds2)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 ns = make_float2(-s2[k].x, -s2[k].y);
        const float2 cn = ffma2(ns, ds2[k], fmul2(c2[k], dc2[k]));
        const float2 sn = ffma2(c2[k], ds2[k], fmul2(s2[k], dc2[k]));
        c2[k] = cn;
        s2[k] = sn;
    }
}

// bf16 bit pattern of 2^15: pre-RoPE inputs at or above it may overflow FP16
// once rotated (|rotated| <= sqrt(2) * max |input|).
constexpr uint32_t RANGE_LIMIT_BF16 = 0x4700u;
__device__ __forceinline__ bool range_exceeded(uint32_t r) {
    return (r & 0xffffu) >= RANGE_LIMIT_BF16 || (r >> 16) >= RANGE_LIMIT_BF16;
}

// -------------------------------------------------------------- RoPE -----

// cos / sin of the rotation angle of one pair at integer position t.
// `turns` is the pair's rate in turns per position as a 0.64 fixed-point
// fraction; t * turns mod 1 is formed exactly in integer arithmetic (top 32
// bits), so the angle handed to the sine/cosine lies in [-pi, pi) with an
// error of at most 2 pi * 2^-32 from the fixed-point quantisation, for any t.
__device__ __forceinline__ void rope_cos_sin(uint32_t t, uint64_t turns, float& c, float& s) {
    const uint32_t lo = (uint32_t)turns, hi = (uint32_t)(turns >> 32);
    const uint32_t frac = t * hi + __umulhi(t, lo);
    const float ang = (float)(int32_t)frac * 1.46291807926715968e-09f;  // 2 pi / 2^32
    __sincosf(ang, &s, &c);
}

}  // namespace rk
