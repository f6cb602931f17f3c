// quant.cuh -- per-32-block int8 activation quantisation (the quantised
// activations of the pages' MMQ / fused int8 prompt-expert kernels, "Strata -
// the details", "Speed (measured)"), plus the fp16 hi/lo operand split the
// tensor-core expert GEMM consumes.
#pragma once

#include "common.cuh"

namespace moeq {

// One CTA (256 threads) per row of n values (n multiple of 32).  Warp w
// quantises blocks w, w+8, ...; lane i holds element i of the block.
// Optional outputs: hi/lo fp16 rows of q*s*2^-e with e = row_exponent(max s);
// sum_out[row][b] = the sum of the block's codes.  pack2: q is stored in the
// 2-bit block dot's order (pack_pos2) instead of the natural order (no hi/lo).
// `src_q`/`src_s` non-null: the row is already quantised (only the split runs).
__global__ void __launch_bounds__(256) quant_rows_kernel(const float *__restrict__ v, int n, int8_t *q_out,
                                                         float *s_out, __half *hi, __half *lo, int *e_out,
                                                         const int8_t *__restrict__ src_q,
                                                         const float *__restrict__ src_s,
                                                         const int32_t *__restrict__ row_map,
                                                         int *sum_out, int pack2) {
    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = n / 32;
    __shared__ float s_max[8];
    const int8_t *qrow;
    const float *srow;
    float smax = 0.f;
    if (src_q) {
        qrow = src_q + (size_t)row * n;
        srow = src_s + (size_t)row * nb;
        for (int b = tid; b < nb; b += blockDim.x) smax = fmaxf(smax, srow[b]);
    } else {
        const size_t src_row = row_map ? (size_t)row_map[row] : (size_t)row;
        const float *vr = v + src_row * n;
        int8_t *qr = q_out + (size_t)row * n;
        float *sr = s_out + (size_t)row * nb;
        for (int b = warp; b < nb; b += 8) {
            const float val = vr[32 * b + lane];
            const float s = block_scale(warp_absmax(val));
            const int q = block_code(val, s);
            qr[32 * b + (pack2 ? pack_pos2(lane) : lane)] = (int8_t)q;
            if (sum_out) {
                const int qs = warp_sum_int(q);
                if (lane == 0) sum_out[(size_t)row * nb + b] = qs;
            }
            if (lane == 0) sr[b] = s;
            smax = fmaxf(smax, s);
        }
        qrow = qr;
        srow = sr;
    }
    if (!hi) return;
    // row maximum of the block scales -> exponent
    for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
    if (lane == 0) s_max[warp] = smax;
    __syncthreads();  // also orders this CTA's q/s stores before the re-reads below
    float m = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) m = fmaxf(m, s_max[w]);
    const int e = row_exponent(m);
    if (tid == 0 && e_out) e_out[row] = e;
    const float inv = exp2i(-e);
    __half *hr = hi + (size_t)row * n;
    __half *lr = lo + (size_t)row * n;
    for (int i = 2 * tid; i < n; i += 2 * blockDim.x) {
        const float s = srow[i / 32] * inv;
        const float v0 = (float)qrow[i] * s, v1 = (float)qrow[i + 1] * s;
        __half h0, l0, h1, l1;
        split_hi_lo(v0, h0, l0);
        split_hi_lo(v1, h1, l1);
        *reinterpret_cast<__half2 *>(hr + i) = __halves2half2(h0, h1);
        *reinterpret_cast<__half2 *>(lr + i) = __halves2half2(l0, l1);
    }
}

// fp16 hi/lo operand image for the tensor-core GEMM.  Output row r (a sorted
// pair position) is input row row_map[r] (or r) of q [*, n] int8 with block
// scales s [*, n/32]; its values q*s*2^-e are split into hi + lo with
// e = row_exponent(max block scale of the row), e_out[r] = e.
//
// The image is laid out so that a GEMM tile's operand for one K stage is one
// contiguous run of rows that lands in shared memory already in the 128-byte
// swizzled K-major form the MMA descriptors expect:
//   img[st][half][row][64]  (st = K stage of 64 values, half 0 = hi, 1 = lo,
//                            rows = img_rows >= rows + kTileMax per (st, half))
// and the 16-byte chunk c of a 128-byte stage row is stored at chunk
// c ^ ((r - t0) & 7), t0 = the first row of r's tile.  Tiles start at every
// tile_n-th position of each expert's segment [offsets[e], offsets[e+1]),
// tile_n a multiple of 16, so the phase is (r - offsets[e]) & 7.  One warp per output row, one 16-byte chunk
// of each half per lane per step.
__global__ void __launch_bounds__(256) split_rows_kernel(const int8_t *__restrict__ q, const float *__restrict__ s,
                                                         int n, const int32_t *__restrict__ row_map, int rows,
                                                         int src_rows,
                                                         const int32_t *__restrict__ offsets, int E,
                                                         __half *__restrict__ img, long long img_rows,
                                                         int *__restrict__ e_out) {
    const int lane = threadIdx.x & 31;
    const int nb = n / 32;
    const size_t half_stride = (size_t)img_rows * 64;  // elements of one (stage, half) plane
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += (gridDim.x * blockDim.x) >> 5) {
        // expert segment of r: the last e with offsets[e] <= r
        int lo_e = 0, hi_e = E;  // invariant offsets[lo_e] <= r < offsets[hi_e]
        while (hi_e - lo_e > 1) {
            const int mid = (lo_e + hi_e) >> 1;
            if (offsets[mid] <= r) lo_e = mid;
            else hi_e = mid;
        }
        const uint32_t phase = (uint32_t)(r - offsets[lo_e]) & 7u;
        int srow = row_map ? row_map[r] : r;
        if (srow < 0 || srow >= src_rows) {  // a caller's bad permutation: read row 0 instead
            if (lane == 0) set_status(MOEQ_STATUS_BAD_INDEX);
            srow = 0;
        }
        const size_t src = (size_t)srow;
        const float *sr = s + src * nb;
        float m = 0.f;
        for (int b = lane; b < nb; b += 32) m = fmaxf(m, sr[b]);
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int e = row_exponent(m);
        if (lane == 0) e_out[r] = e;
        const float inv = exp2i(-e);
        const int8_t *qr = q + src * n;
        for (int c = lane; c < n / 8; c += 32) {
            const uint2 qv = *reinterpret_cast<const uint2 *>(qr + 8 * c);
            const float sc = sr[(8 * c) / 32] * inv;
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t word = i < 2 ? qv.x : qv.y;
                const float v0 = (float)(int8_t)(word >> (16 * (i & 1))) * sc;
                const float v1 = (float)(int8_t)(word >> (16 * (i & 1) + 8)) * sc;
                __half h0, l0, h1, l1;
                split_hi_lo(v0, h0, l0);
                split_hi_lo(v1, h1, l1);
                hw[i] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
                lw[i] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
            }
            const size_t st = (size_t)(c >> 3);
            const size_t off = (size_t)r * 64 + ((((uint32_t)c & 7u) ^ phase) << 3);
            *reinterpret_cast<uint4 *>(img + (2 * st) * half_stride + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(img + (2 * st + 1) * half_stride + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
    }
}

// The x operand image of the grouped GEMM straight from x: for every token t
// (one warp), its row is quantised per 32-block by the rule of
// quant_rows_kernel and the resulting q*s*2^-e values, split into fp16 hi +
// lo, are written to the image rows inv[t*k + j] of all its k pairs (rows
// that split_rows_kernel would write from q and s, bit for bit), with
// e_out[row] = e.  Two passes over the row: the block scales and their
// maximum (the row exponent e), then the codes and the image.  Lane l holds
// values 4l .. 4l + 3 of each 128-value group, so eight lanes make a block
// and two lanes one 16-byte chunk (each stores its 8 bytes).  inv < 0: a
// pair the permutation rejected (not written).
__global__ void __launch_bounds__(256) quant_split_kernel(const float *__restrict__ x, int T, int H, int k,
                                                          const int32_t *__restrict__ inv,
                                                          const int32_t *__restrict__ offsets, int E,
                                                          __half *__restrict__ img, long long img_rows,
                                                          int *__restrict__ e_out) {
    const int lane = threadIdx.x & 31;
    const size_t half_stride = (size_t)img_rows * 64;  // elements of one (stage, half) plane
    const int NG = H / 128;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
        const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)t * H) + lane;
        // pass 1: the row's largest block scale
        float smax = 0.f;
        for (int g = 0; g < NG; ++g) {
            const float4 v = xr[32 * g];
            float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            smax = fmaxf(smax, block_scale(a));
        }
        smax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(smax)));
        const int e = row_exponent(smax);
        const float inv2 = exp2i(-e);
        // the image row of pair j (lane j) and its swizzle phase: (row - first row of its expert) & 7
        int prow = -1;
        uint32_t phase = 0;
        if (lane < k) {
            prow = inv[(size_t)t * k + lane];
            if (prow >= 0) {
                int lo_e = 0, hi_e = E;  // the last e with offsets[e] <= prow
                while (hi_e - lo_e > 1) {
                    const int mid = (lo_e + hi_e) >> 1;
                    if (offsets[mid] <= prow) lo_e = mid;
                    else hi_e = mid;
                }
                phase = (uint32_t)(prow - offsets[lo_e]) & 7u;
                e_out[prow] = e;
            }
        }
        // pass 2: codes, the hi/lo split, and the stores to every pair row
        for (int g = 0; g < NG; ++g) {
            const float4 v = xr[32 * g];
            float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            const float s = block_scale(a);
            const float sc = s * inv2;
            const float vals[4] = {v.x, v.y, v.z, v.w};
            uint32_t hw[2], lw[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                __half h0, l0, h1, l1;
                split_hi_lo((float)block_code(vals[2 * i], s) * sc, h0, l0);
                split_hi_lo((float)block_code(vals[2 * i + 1], s) * sc, h1, l1);
                hw[i] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
                lw[i] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
            }
            const int c = 16 * g + (lane >> 1);  // 16-byte chunk of the row
            const size_t st = (size_t)(c >> 3);
            const uint32_t cc = (uint32_t)c & 7u;
            for (int j = 0; j < k; ++j) {
                const int r = __shfl_sync(0xffffffffu, prow, j);
                const uint32_t ph = __shfl_sync(0xffffffffu, phase, j);
                if (r < 0) continue;
                const size_t off = (size_t)r * 64 + ((cc ^ ph) << 3) + 4 * (lane & 1);
                *reinterpret_cast<uint2 *>(img + (2 * st) * half_stride + off) = make_uint2(hw[0], hw[1]);
                *reinterpret_cast<uint2 *>(img + (2 * st + 1) * half_stride + off) = make_uint2(lw[0], lw[1]);
            }
        }
    }
}

// inv[t*k + j] = the sorted position of pair (t, j), from the permutation's
// perm_tok / perm_slot (inv filled with -1 beforehand: rejected pairs stay so).
__global__ void __launch_bounds__(256) pair_rows_kernel(const int32_t *__restrict__ perm_tok,
                                                        const int32_t *__restrict__ perm_slot, int P, int T, int k,
                                                        int32_t *__restrict__ inv) {
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < P; r += gridDim.x * blockDim.x) {
        const int t = perm_tok[r], j = perm_slot[r];
        if (t >= 0 && t < T && j >= 0 && j < k) inv[(size_t)t * k + j] = r;
    }
}

// The x image rows of sorted positions that no pair's inverse points back to
// (a caller's permutation with out-of-range or repeated entries): zeroed, with
// exponent 0, so that the GEMMs only ever read defined operand rows.  One warp
// per sorted position; a no-op for a consistent permutation.
__global__ void __launch_bounds__(256) orphan_rows_kernel(const int32_t *__restrict__ perm_tok,
                                                          const int32_t *__restrict__ perm_slot, int P, int T, int k,
                                                          const int32_t *__restrict__ inv, int H,
                                                          __half *__restrict__ img, long long img_rows,
                                                          int *__restrict__ e_out) {
    const int lane = threadIdx.x & 31;
    const size_t half_stride = (size_t)img_rows * 64;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < P; r += (gridDim.x * blockDim.x) >> 5) {
        const int t = perm_tok[r], j = perm_slot[r];
        const bool claimed = t >= 0 && t < T && j >= 0 && j < k && inv[(size_t)t * k + j] == r;
        if (claimed) continue;  // uniform over the warp
        if (lane == 0) e_out[r] = 0;
        for (int c = lane; c < 2 * (H / 64) * 8; c += 32)  // (stage, half) plane c / 8, 16-byte chunk c % 8
            *reinterpret_cast<uint4 *>(img + (size_t)(c >> 3) * half_stride + (size_t)r * 64 + (c & 7) * 8) =
                make_uint4(0u, 0u, 0u, 0u);
    }
}

}  // namespace moeq
