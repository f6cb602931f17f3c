// peaks.cu -- libmoeq_peaks: a microbenchmark of the legacy warp-level int8
// tensor path (mma.sync m16n8k32 s8 x s8 -> s32) on this GPU, the denominator
// that a prompt-expert GEMM on int8 MMAs would be measured against.  The pages'
// fused prompt-expert kernels use the int8 tensor cores of consumer cards
// ("Strata - the details", "Speed (measured)", engine 0.1.36); sm_103a has no
// int8 tcgen05 MMA, so this is the only int8 tensor path here.  Not part of
// the layer: bench.py loads it to report the prefill GEMMs against it.
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

}  // namespace

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
