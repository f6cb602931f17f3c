// peaks.cu -- libmoeq_peaks: a microbenchmark of the legacy warp-level int8
// tensor path (mma.sync m16n8k32 s8 x s8 -> s32) on this GPU, the denominator
// that a prompt-expert GEMM on int8 MMAs would be measured against.  The pages'
// fused prompt-expert kernels use the int8 tensor cores of consumer cards
// ("Strata - the details", "Speed (measured)", engine 0.1.36); sm_103a has no
// int8 tcgen05 MMA, so this is the only int8 tensor path here.  Not part of
// the layer: bench.py loads it to report the prefill GEMMs against it.  It also
// measures what one tcgen05.mma costs its issuing thread at small N, the limit
// of a grouped GEMM whose groups are small.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moeq_peaks.h"

namespace {

constexpr int kAcc = 8;  // independent accumulator tiles per warp (hides the MMA latency)
__device__ int g_sink;

__global__ void __launch_bounds__(256) mma_s8_loop(int iters, int seed) {
    uint32_t a[4], b[2];
    int c[kAcc][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = 0x01010101u * (uint32_t)(threadIdx.x + i + seed);
    b[0] = 0x02020202u * (uint32_t)(threadIdx.x + seed);
    b[1] = 0x03030303u * (uint32_t)(threadIdx.x + 1);
#pragma unroll
    for (int t = 0; t < kAcc; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[t][i] = 0;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int t = 0; t < kAcc; ++t)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                "{%0, %1, %2, %3};"
                : "+r"(c[t][0]), "+r"(c[t][1]), "+r"(c[t][2]), "+r"(c[t][3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    }
    int s = 0;
#pragma unroll
    for (int t = 0; t < kAcc; ++t) s += c[t][0] ^ c[t][1] ^ c[t][2] ^ c[t][3];
    if (s == 0x7fffffff) g_sink = s;  // keeps the loop alive; practically never taken
}

// ---- tcgen05.mma issue cost: M = 128, K = 16, fp16, one issuing thread.
__device__ long long g_umma_cycles;
constexpr int kUmmaBytes = 2 * 16384 + 2 * 32768;  // two 128 x 64 A blocks, two 256 x 64 B images (fp16)

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t a) {  // 128-byte swizzle, 8-row groups 1 KB apart
    return (uint64_t)((a & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
           ((uint64_t)2 << 61);
}

__device__ __forceinline__ bool mbar_try_once(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Thread 0 issues `stages` groups of PER_STAGE MMAs (N = n) from resident
// operands in the order the grouped GEMM uses: for each K = 16 step, both
// M = 128 blocks (two accumulators), and with PER_STAGE = 16 a second B image
// (the lo half of a split operand).  WITH_SYNC adds what a pipelined GEMM does
// per stage: two tests of (already completed) mbarriers, a tcgen05 fence and a
// commit.  Both are compile-time, so no conditional branch separates the MMAs
// (one per MMA was measured to double their cost to the issuing thread).
template <int PER_STAGE, bool WITH_SYNC>
__global__ void __launch_bounds__(128, 1) umma_issue_loop(int n, int stages) {
    extern __shared__ unsigned char raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t full, slot_free, fin;
    __shared__ uint32_t tslot;
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < kUmmaBytes / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(sm)[i] = 0x3C003C00u * ((i & 7) == 0);
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&full)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&slot_free)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&fin)));
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(&full)) : "memory");  // phase 0 done
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&tslot)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tm = tslot;
    if (tid == 0) {
        const uint64_t da = sw128_kmajor_desc(su32(sm)), db = sw128_kmajor_desc(su32(sm + 2 * 16384));
        constexpr uint64_t kA = 16384 >> 4, kB = 32768 >> 4;  // descriptor strides of an A block and a B image
        const uint32_t idesc = (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
        const long long t0 = clock64();
        uint32_t seen = 1;
        for (int g = 0; g < stages; ++g) {
            if (WITH_SYNC) {
                seen &= (uint32_t)mbar_try_once(su32(&full), 0);
                seen &= (uint32_t)mbar_try_once(su32(&full), 0);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int h = 0; h < PER_STAGE / 8; ++h)
                        asm volatile(
                            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tm + (uint32_t)(m * n)),
                            "l"(da + m * kA + 2 * kk), "l"(db + h * kB + 2 * kk), "r"(idesc), "r"(1)
                            : "memory");
            if (WITH_SYNC)
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(&slot_free))
                             : "memory");
        }
        if (!seen) g_umma_cycles = -2;  // the completed phase was not observed (never expected)
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(&fin)) : "memory");
        bool ok = false;  // the MMAs end within a few milliseconds; give up after about two seconds
        for (const long long tw = clock64(); !ok && clock64() - tw < 4000000000ll;) ok = mbar_try_once(su32(&fin), 0);
        if (blockIdx.x == 0 && seen) g_umma_cycles = ok ? clock64() - t0 : -1;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tm) : "memory");
    }
}

}  // namespace

extern "C" int moe_peak_umma_issue(int n, int per_stage, int with_sync, double *cycles_per_mma) {
    if (!cycles_per_mma || n < 16 || n > 256 || n % 16 || (per_stage != 8 && per_stage != 16)) return -1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -5;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -5;
    const int smem = 1024 + kUmmaBytes + 24 * 1024;  // the spare 24 KB keeps one CTA on each SM
    const int stages = 4096 / per_stage + 1;
    auto launch = [&](auto kernel) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return false;
        kernel<<<sms, 128, smem>>>(n, stages);
        return true;
    };
    const bool launched = per_stage == 8 ? (with_sync ? launch(umma_issue_loop<8, true>) : launch(umma_issue_loop<8, false>))
                                         : (with_sync ? launch(umma_issue_loop<16, true>) : launch(umma_issue_loop<16, false>));
    if (!launched) return -5;
    long long cyc = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return -5;
    if (cudaMemcpyFromSymbol(&cyc, g_umma_cycles, sizeof cyc) != cudaSuccess || cyc <= 0) return -5;
    *cycles_per_mma = (double)cyc / ((double)stages * per_stage);
    return 0;
}

extern "C" int moe_peak_mma_s8(int iters, int blocks_per_sm, double *tops_out) {
    if (!tops_out || iters < 1 || blocks_per_sm < 1) return -1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -5;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -5;
    const int blocks = sms * blocks_per_sm;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    mma_s8_loop<<<blocks, 256>>>(iters / 8 + 1, 1);  // warm-up
    cudaEventRecord(e0);
    mma_s8_loop<<<blocks, 256>>>(iters, 2);
    cudaEventRecord(e1);
    cudaError_t err = cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (err != cudaSuccess || ms <= 0.f) return -5;
    const double ops = 2.0 * 16 * 8 * 32 * (double)kAcc * iters * (double)blocks * (256 / 32);
    *tops_out = ops / (ms * 1e-3) / 1e12;
    return 0;
}
