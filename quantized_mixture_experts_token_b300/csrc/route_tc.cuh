// route_tc.cuh -- router logits for prompt chunks on the tensor cores: a
// 3xTF32 GEMM L[T,E] = x[T,H] Wr[E,H]^T + b (tcgen05 kind::tf32, TMEM
// accumulator) whose error stays at the level of an fp32 dot product.
//
// The pages run the routers on the GPU ("Strata - the details", "How it
// works"); a 4,096-token chunk needs 8.6 GFLOP of router work.  Splitting each
// fp32 operand v into hi = v with its 13 low mantissa bits cleared (exactly a
// tf32 value) and lo = v - hi (exact in fp32, itself read as tf32), the product
// is formed as x_hi W_hi + x_hi W_lo + x_lo W_hi; the dropped x_lo W_lo term
// and the tf32 reading of lo are ~2^-21 of |x||W|, below fp32 accumulation
// error over H = 2048 terms.
//
// The tensor core's fp32 accumulator rounds each addition toward zero, so a
// single accumulator over all 768 MMAs of H = 2048 drifts by ~768 ulps; the
// K loop is therefore cut into chunks of kRtChunk stages, each accumulated
// afresh in one of two TMEM buffers and added into fp32 registers (round to
// nearest) by the accumulator warps while the next chunk runs.
//
// One CTA per (128-token, 128-expert) tile, 320 threads:
//   warp 0     producer: TMA loads of the raw fp32 x and Wr tiles (K = 32
//              values = one 128-byte swizzled row per stage) into a 3-slot ring
//   warp 1     TMEM owner; lane 0 issues the MMAs (3 per K = 8 step)
//   warps 2-5  split each stage in place (hi) and into a lo copy at the same
//              swizzled offsets
//   warps 6-9  drain each chunk's accumulator into registers; the epilogue
//              (bias add, fp32 stores)
// Every wait is bounded; a wait that gives up raises the CTA's abort flag and
// a device status bit, copies and MMAs are drained and TMEM is freed.
#pragma once

#include "async.cuh"

namespace moeq {

constexpr int kRtM = 128;      // tokens per tile (MMA M)
constexpr int kRtN = 128;      // experts per tile (MMA N)
constexpr int kRtK = 32;       // fp32 values per stage (one 128-byte row)
constexpr int kRtStages = 3;
constexpr int kRtChunk = 1;  // stages per accumulator chunk (K = 32, 12 MMAs)
constexpr int kRtTile = kRtM * kRtK * 4;  // 16 KB: one operand tile of one stage (x or Wr; hi or lo)
constexpr int kRtSlot = 4 * kRtTile;      // x hi, Wr hi, x lo, Wr lo
constexpr size_t kRtSmem = 1024 + (size_t)kRtStages * kRtSlot + 256;

struct RouteTcArgs {
    int T, H, E;
    const float *bias;
    float *logits;
    CUtensorMap tm_x, tm_w;  // [T][H] and [E][H] fp32, box {32, 128}, 128-byte swizzle
};

__device__ __forceinline__ uint64_t rt_desc(uint32_t saddr) {  // K-major, 128-byte swizzle, 8-row groups 1 KB apart
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::tf32 instruction descriptor: fp32 accumulator, A and B tf32 (format
// 2), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__device__ __forceinline__ uint32_t tf32_idesc(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void rt_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void rt_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "{\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "}"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// hi = v with the 13 low mantissa bits cleared, lo = v - hi (exact).
__device__ __forceinline__ void tf32_split(uint32_t v, uint32_t &hi, uint32_t &lo) {
    hi = v & 0xFFFFE000u;
    lo = __float_as_uint(__uint_as_float(v) - __uint_as_float(hi));
}

__global__ void __launch_bounds__(320, 1) route_tc_kernel(const __grid_constant__ RouteTcArgs a) {
    constexpr int S = kRtStages;
    extern __shared__ unsigned char rt_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(rt_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)S * kRtSlot);
    uint64_t *full = bars, *conv = bars + S, *empty = bars + 2 * S, *acc_full = bars + 3 * S,
             *acc_empty = acc_full + 2, *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t wl = wait_limit();
    const int m0 = blockIdx.y * kRtM, n0 = blockIdx.x * kRtN;
    const int nk = a.H / kRtK;
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&conv[i]), 128);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&acc_full[i]), 1);
            mbar_init(smem_u32(&acc_empty[i]), 128);
        }
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(2 * kRtN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_x)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_w)) : "memory");
            int issued = 0;  // (both operands are re-read by other CTAs: default L2 policy)
            for (int g = 0; g < nk; ++g) {
                const int s = g % S;
                if (!mbar_wait(smem_u32(&empty[s]), ((g / S) & 1) ^ 1, abort_flag, wl)) break;
                unsigned char *slot = smem + (size_t)s * kRtSlot;
                const uint32_t bar = smem_u32(&full[s]);
                mbar_arrive_expect_tx(bar, 2 * kRtTile);
                tma_load_2d(smem_u32(slot), &a.tm_x, g * kRtK, m0, bar, 0);
                tma_load_2d(smem_u32(slot + kRtTile), &a.tm_w, g * kRtK, n0, bar, 0);
                issued = g + 1;
            }
            for (int g = max(0, issued - S); g < issued; ++g)  // copies in flight land before the CTA can leave
                mbar_drain(smem_u32(&full[g % S]), (g / S) & 1, abort_flag);
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idesc = tf32_idesc(kRtM, kRtN);
            const uint64_t d0 = rt_desc(smem_u32(smem));
            bool ok = true;
            for (int g = 0; g < nk && ok; ++g) {
                const int s = g % S, c = g / kRtChunk, buf = c & 1, first = g % kRtChunk == 0;
                if (first && !mbar_wait(smem_u32(&acc_empty[buf]), ((c >> 1) & 1) ^ 1, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(smem_u32(&conv[s]), (g / S) & 1, abort_flag, wl)) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t acc = tmem + (uint32_t)(buf * kRtN);
                const uint64_t ds = d0 + (uint64_t)((s * kRtSlot) >> 4);
                const uint64_t xh = ds, wh = ds + (kRtTile >> 4), xl = ds + (2 * kRtTile >> 4),
                               wl_ = ds + (3 * kRtTile >> 4);
#pragma unroll
                for (int kk = 0; kk < kRtK / 8; ++kk) {  // K = 8 tf32 = 32 bytes per MMA
                    mma_tf32(acc, xh + 2 * kk, wh + 2 * kk, idesc, !(first && kk == 0));
                    mma_tf32(acc, xh + 2 * kk, wl_ + 2 * kk, idesc, 1u);
                    mma_tf32(acc, xl + 2 * kk, wh + 2 * kk, idesc, 1u);
                }
                rt_commit(smem_u32(&empty[s]));
                if (g % kRtChunk == kRtChunk - 1 || g == nk - 1) rt_commit(smem_u32(&acc_full[buf]));
            }
            rt_commit(smem_u32(drain));  // every MMA issued above is complete once this lands
            mbar_drain(smem_u32(drain), 0, abort_flag);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ split
        const int r = tid - 64;  // operand row of this thread (token row of x, expert row of Wr)
        for (int g = 0; g < nk; ++g) {
            const int s = g % S;
            if (!mbar_wait(smem_u32(&full[s]), (g / S) & 1, abort_flag, wl)) break;
            unsigned char *slot = smem + (size_t)s * kRtSlot;
#pragma unroll
            for (int op = 0; op < 2; ++op) {  // x, Wr
                uint4 *hi = reinterpret_cast<uint4 *>(slot + op * kRtTile + r * 128);
                uint4 *lo = reinterpret_cast<uint4 *>(slot + (2 + op) * kRtTile + r * 128);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    // visit the row's 16-byte chunks in swizzled order, so that the 8
                    // rows a quarter-warp touches hit 8 different bank groups
                    const int c = c8 ^ (r & 7);
                    const uint4 v = hi[c];
                    uint4 h, l;
                    tf32_split(v.x, h.x, l.x);
                    tf32_split(v.y, h.y, l.y);
                    tf32_split(v.z, h.z, l.z);
                    tf32_split(v.w, h.w, l.w);
                    hi[c] = h;
                    lo[c] = l;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(smem_u32(&conv[s]));
        }
    } else {
        // ------------------------------------- chunk accumulation, epilogue
        // lane quadrant of TMEM = warp % 4; thread = token row
        const int q = warp & 3, row = 32 * q + lane, t = m0 + row;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
        float sum[kRtN];
#pragma unroll
        for (int i = 0; i < kRtN; ++i) sum[i] = 0.f;
        const int nch = (nk + kRtChunk - 1) / kRtChunk;
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int buf = c & 1;
            if (!mbar_wait(smem_u32(&acc_full[buf]), (c >> 1) & 1, abort_flag, wl)) {
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
            for (int c0 = 0; c0 < kRtN; c0 += 16) {
                float v[16];
                rt_ld16(tl + (uint32_t)(buf * kRtN + c0), v);
#pragma unroll
                for (int i = 0; i < 16; ++i) sum[c0 + i] += v[i];
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(smem_u32(&acc_empty[buf]));
        }
        if (ok && t < a.T) {
            float *dst = a.logits + (size_t)t * a.E + n0;
            if (n0 + kRtN <= a.E) {
#pragma unroll
                for (int i = 0; i < kRtN; i += 4) {
                    float4 o;
                    o.x = sum[i] + (a.bias ? a.bias[n0 + i] : 0.f);
                    o.y = sum[i + 1] + (a.bias ? a.bias[n0 + i + 1] : 0.f);
                    o.z = sum[i + 2] + (a.bias ? a.bias[n0 + i + 2] : 0.f);
                    o.w = sum[i + 3] + (a.bias ? a.bias[n0 + i + 3] : 0.f);
                    *reinterpret_cast<float4 *>(dst + i) = o;
                }
            } else {
#pragma unroll
                for (int i = 0; i < kRtN; ++i)
                    if (n0 + i < a.E) dst[i] = sum[i] + (a.bias ? a.bias[n0 + i] : 0.f);
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kRtN) : "memory");
    }
}

}  // namespace moeq
