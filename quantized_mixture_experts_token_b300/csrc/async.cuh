// async.cuh -- asynchronous-copy, mbarrier and programmatic-dependent-launch
// helpers (inline PTX for sm_103a) shared by the kernels of libmoeq.
#pragma once

#include "common.cuh"

namespace moeq {

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- mbarriers

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes initialised mbarriers visible to the async proxy (bulk copies, MMA commits).
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

// One arrival that also announces `bytes` of asynchronous copies into this phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bound of a pipeline wait (moe_set_wait_limit; 2 s by default).  Each kernel
// reads it once at entry (wait_limit()) and passes it to its waits.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s
__device__ uint64_t g_wait_limit_ns = kDefaultWaitLimitNs;
// Bound of the waits that drain a CTA's own copies and MMAs before it exits
// after an abort: fixed, so that a short pipeline limit never lets a CTA leave
// with asynchronous copies still landing in its shared memory.
constexpr uint64_t kDrainLimitNs = 2000000000ull;
// Limits below this poll the barrier without suspending (so that they run out
// on time); longer ones use the hardware-suspended try_wait.
constexpr uint64_t kPollBelowNs = 1000000ull;  // 1 ms

__device__ __forceinline__ uint64_t wait_limit() { return *(volatile uint64_t *)&g_wait_limit_ns; }

__device__ __forceinline__ bool wait_give_up(volatile int *abort_flag) {
    set_status(MOEQ_STATUS_WAIT_TIMEOUT);
    *abort_flag = 1;
    return false;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// (and raises the CTA's abort flag and MOEQ_STATUS_WAIT_TIMEOUT) if it did not
// within `limit` ns, or (honour_abort) if another thread of the CTA aborted.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              bool honour_abort, uint64_t limit) {
    if (limit >= kPollBelowNs) {
        if (mbar_try(bar, parity)) return true;
        const uint64_t t0 = globaltimer();
        for (uint32_t it = 1;; ++it) {
            if (mbar_try(bar, parity)) return true;
            if ((it & 15u) == 0u) {
                if (honour_abort && *abort_flag) return false;
                if (globaltimer() - t0 > limit) return wait_give_up(abort_flag);
            }
        }
    }
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_test(bar, parity)) return true;
        if (honour_abort && *abort_flag) return false;
        if (globaltimer() - t0 > limit) return wait_give_up(abort_flag);
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, uint64_t limit) {
    return mbar_wait_for(bar, parity, abort_flag, true, limit);
}

// Wait for copies or MMAs this CTA issued itself (after an abort, before it
// exits); ignores the abort flag, fixed bound.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    return mbar_wait_for(bar, parity, abort_flag, false, kDrainLimitNs);
}

// --------------------------------------------------------- bulk copies

// L2 policy for data read once per call (expert and router weights): evict first,
// so activations and routing state stay resident.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global -> shared bulk copy completing on `bar` (transaction bytes).  dst, src
// 16-byte aligned; bytes a multiple of 16.  pol: an L2 policy, or 0 for none.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    if (pol)
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
                "r"(dst),
            "l"(src), "r"(bytes), "r"(bar), "l"(pol)
            : "memory");
    else
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                     "l"(src), "r"(bytes), "r"(bar)
                     : "memory");
}

// 2-D tiled tensor copy global -> shared (TMA) completing on `bar`.  `tmap` is
// the address of a CUtensorMap in kernel-parameter or global memory; (x, y)
// the box origin in elements (x * element size a multiple of 16 bytes).
// pol: an L2 policy, or 0 for none.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint32_t bar, uint64_t pol) {
    if (pol)
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
            " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(pol)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
            : "memory");
}

// ------------------------------------------------------------- timeline
// Compile-time tracing (build with -DMOEQ_TIMELINE): thread 0 of a CTA records
// (global time, clock, SM, kernel, phase, CTA) at phase boundaries into a
// device ring that moe_timeline_read() copies out.  Compiled out otherwise.
#ifdef MOEQ_TIMELINE
constexpr unsigned kTlEntries = 1u << 20;
__device__ unsigned long long g_tl[2 * kTlEntries];
__device__ unsigned g_tl_n;
__device__ __forceinline__ void tl_stamp(int kernel, int phase) {
    if (threadIdx.x != 0) return;
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const unsigned i = atomicAdd(&g_tl_n, 1u) & (kTlEntries - 1u);
    g_tl[2 * i] = globaltimer();
    g_tl[2 * i + 1] = ((unsigned long long)(clock64() & 0xFFFFFFu) << 40) | ((unsigned long long)(smid & 0xFF) << 32) |
                      ((unsigned long long)(kernel & 0xFF) << 24) | ((unsigned long long)(phase & 0xFF) << 16) |
                      (unsigned long long)(blockIdx.x & 0xFFFF);
}
// Stamp from the calling thread, with `tag` in place of the CTA index.
__device__ __forceinline__ void tl_stamp_tag(int kernel, int phase, unsigned tag) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const unsigned i = atomicAdd(&g_tl_n, 1u) & (kTlEntries - 1u);
    g_tl[2 * i] = globaltimer();
    g_tl[2 * i + 1] = ((unsigned long long)(clock64() & 0xFFFFFFu) << 40) | ((unsigned long long)(smid & 0xFF) << 32) |
                      ((unsigned long long)(kernel & 0xFF) << 24) | ((unsigned long long)(phase & 0xFF) << 16) |
                      (unsigned long long)(tag & 0xFFFF);
}
#define MOEQ_TL(k, p) ::moeq::tl_stamp((k), (p))
#define MOEQ_TL_TAG(k, p, tag) ::moeq::tl_stamp_tag((k), (p), (tag))
#else
#define MOEQ_TL_TAG(k, p, tag) \
    do {                       \
    } while (0)
#define MOEQ_TL(k, p) \
    do {              \
    } while (0)
#endif

// --------------------------------------------- programmatic dependent launch

// Blocks until every grid this one depends on (the previous kernel on the
// stream, when launched with programmatic stream serialisation) has completed
// and its memory is visible.  A no-op for kernels launched without it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel on the stream begin launching (its blocks still wait in
// pdl_wait for this grid to finish before touching its results).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace moeq
