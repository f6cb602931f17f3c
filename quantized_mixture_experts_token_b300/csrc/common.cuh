// common.cuh -- shared device helpers of libmoeq (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moeq.h"

namespace moeq {

// Per-device status word (MOEQ_STATUS_* bits); read and cleared by
// moe_get_device_status().
__device__ int g_status;

__device__ __forceinline__ void set_status(int bits) { atomicOr(&g_status, bits); }

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;

// One active expert's work record for the decode expert kernel: the expert,
// the first sorted position of its (token, slot) pairs, their count, and the
// first kUnitTok tokens with their routing weights (the rest are read from
// the permutation arrays).
constexpr int kUnitTok = 8;
struct __align__(16) UnitRec {
    int e, pb, ne, pad;
    int tok[kUnitTok];
    float w[kUnitTok];
};

// Byte position of element i of a 32-block in the order the 2-bit block dot
// consumes activations: word m (m < 4) holds elements {m, 4+m, 8+m, 12+m},
// word 4+m the same for elements 16..31 (what masking the packed 2-bit codes
// with 0x03030303 after a shift by 2m lines up against).
__host__ __device__ __forceinline__ int pack_pos2(int i) { return (4 * (i >> 4) + (i & 3)) * 4 + ((i & 15) >> 2); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_int(int v) { return __reduce_add_sync(0xffffffffu, v); }

// max |v| over the warp; non-negative floats order like their bit patterns.
__device__ __forceinline__ float warp_absmax(float v) {
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
}

// The per-32-block int8 rule: s = amax / 127 in IEEE fp32, q = rint(v / s)
// (round half to even), clamped to +-127; s == 0 gives q = 0.
__device__ __forceinline__ float block_scale(float amax) { return __fdiv_rn(amax, 127.0f); }

__device__ __forceinline__ int block_code(float v, float s) {
    if (s == 0.0f) return 0;
    float r = rintf(__fdiv_rn(v, s));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return (int)r;
}

// Power-of-two normaliser for the fp16 hi/lo operand split: with the largest
// block scale smax of a row, values q*s*2^-e stay below 2^14.
__device__ __forceinline__ int row_exponent(float smax) {
    if (!(smax > 0.0f)) return 0;
    return min(120, max(-120, ilogbf(smax) - 6));
}

__device__ __forceinline__ float exp2i(int e) {  // 2^e for e in [-126, 127]
    return __int_as_float((127 + e) << 23);
}

// Split v into fp16 hi + lo with hi + lo == v to about 2^-22 relative.
__device__ __forceinline__ void split_hi_lo(float v, __half &hi, __half &lo) {
    hi = __float2half_rn(v);
    lo = __float2half_rn(v - __half2float(hi));
}

// Exclusive scan of n <= 4 * blockDim.x ints held in shared memory, in place.
// Returns the total.  All threads of the block must call it.
__device__ int block_exclusive_scan(int *data, int n, int *scratch /* >= 33 ints */) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (n + nt - 1) / nt;
    int local[4];
    int sum = 0;
    for (int i = 0; i < per; ++i) {
        int idx = tid * per + i;
        int v = idx < n ? data[idx] : 0;
        local[i] = sum;
        sum += v;
    }
    // inclusive warp scan of per-thread sums
    const int lane = tid & 31, warp = tid >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int nw = nt >> 5;
        int v = lane < nw ? scratch[lane] : 0;
        int iv = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, iv, o);
            if (lane >= o) iv += u;
        }
        if (lane < nw) scratch[lane] = iv - v;  // exclusive warp offsets
        if (lane == nw - 1) scratch[32] = iv;   // total
    }
    __syncthreads();
    const int base = scratch[warp] + incl - sum;
    for (int i = 0; i < per; ++i) {
        int idx = tid * per + i;
        if (idx < n) data[idx] = base + local[i];
    }
    const int total = scratch[32];
    __syncthreads();
    return total;
}

// Loads that bypass L1 (data written earlier in the same kernel by other CTAs).
__device__ __forceinline__ float ld_cg(const float *p) { return __ldcg(p); }

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

}  // namespace moeq
