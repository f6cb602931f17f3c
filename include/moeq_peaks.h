/*
 * moeq_peaks.h -- C ABI of libmoeq_peaks, the measurement companion of libmoeq
 * (not part of the layer).
 *
 * The pages' prompt experts run on the int8 tensor cores of consumer cards
 * ("Strata - the details", "Speed (measured)", engine 0.1.36 fused int8
 * tensor-core kernels).  sm_103a has no int8 tcgen05 MMA; the legacy warp-level
 * mma.sync s8 path is the only int8 tensor path, and its measured rate is the
 * int8 roofline the prefill GEMMs are reported against beside the fp16 one.
 */
#ifndef MOEQ_PEAKS_H
#define MOEQ_PEAKS_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Dense int8 tensor throughput of mma.sync.m16n8k32.s8.s8.s32 on the current
 * device: blocks_per_sm x (SM count) CTAs of 8 warps, each warp issuing
 * `iters` rounds of 8 independent MMAs from registers.  Writes tera-ops per
 * second (2 ops per multiply-add) to *tops_out.  Synchronises the device.
 * Returns 0, -1 on a bad argument, -5 on a CUDA error.  Allocates nothing.
 */
int moe_peak_mma_s8(int iters, int blocks_per_sm, double *tops_out);

/*
 * Cycles per tcgen05.mma (kind::f16, M = 128, N = n, K = 16) issued by one
 * thread from operands resident in shared memory, one CTA per SM, in the order
 * the grouped prefill GEMMs of libmoeq issue them: per K = 16 step both
 * M = 128 blocks (two TMEM accumulators of n columns), times two B images when
 * per_stage = 16 (the hi and lo halves of a split operand); 8 or 16 MMAs per
 * K = 64 stage.  with_sync != 0 adds what a pipelined GEMM does per stage (two
 * mbarrier tests, a tcgen05 fence, a commit).  n a multiple of 16 in [16, 256],
 * per_stage 8 or 16.  Synchronises the device; returns 0, -1 on a bad argument,
 * -5 on a CUDA error.  Allocates no device memory.
 */
int moe_peak_umma_issue(int n, int per_stage, int with_sync, double *cycles_per_mma);

#ifdef __cplusplus
}
#endif

#endif /* MOEQ_PEAKS_H */
