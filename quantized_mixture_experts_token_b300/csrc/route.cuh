// route.cuh -- router logits, top-k + renormalised softmax, and the decode
// fast path that also builds the token-to-expert permutation.
//
// Routers run on the GPU and pick 10 of 512 experts per token ("Strata - the
// details", sections "How it works" and "Which model?").
#pragma once

#include "common.cuh"

namespace moeq {

// ---------------------------------------------------------------- top-k

// One warp ranks one token's E logits (E <= 1024): k rounds of a warp-wide
// argmax; ties resolve to the lower expert index.  Lane l holds logits
// l, l+32, l+64, ... in registers.
template <int PER>  // ceil(E / 32), <= 32
__device__ __forceinline__ void warp_topk(const float *row, int E, int k, int32_t *idx_out, float *w_out,
                                          int *sel_idx /* smem [k] or null */) {
    const int lane = threadIdx.x & 31;
    float v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        int e = lane + 32 * i;
        v[i] = e < E ? ld_cg(row + e) : -INFINITY;
    }
    unsigned taken = 0;  // bit i: register slot i already selected
    float top0 = 0.f, my_w = 0.f;
    int my_idx = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            int e = lane + 32 * i;
            bool ok = e < E && !((taken >> i) & 1u);
            if (ok && (v[i] > bv || be == 0x7fffffff)) { bv = v[i]; be = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (j == 0) top0 = bv;
        if (lane == j) { my_idx = be; my_w = bv; }
    }
    // softmax over the k selected logits, relative to the largest
    float ex = lane < k ? expf(my_w - top0) : 0.0f;
    float den = warp_sum(ex);
    if (lane < k) {
        idx_out[lane] = my_idx;
        w_out[lane] = __fdiv_rn(ex, den);
        if (sel_idx) sel_idx[lane] = my_idx;
    }
}

template <int PER>
__global__ void __launch_bounds__(256) topk_kernel(const float *logits, int T, int E, int k, int32_t *idx,
                                                   float *w) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= T) return;
    warp_topk<PER>(logits + (size_t)warp * E, E, k, idx + (size_t)warp * k, w + (size_t)warp * k, nullptr);
}

// ------------------------------------------------- router logits, small T

// CTA = 8 warps over 4 experts; warp w covers the H-slice [w*H/8, (w+1)*H/8)
// for all 4 experts, so every x value loaded is used 4 times.  Each lane keeps
// REXP x TOKC accumulators; the H-slice partials are summed over the 8 warps
// in a fixed order (deterministic).
constexpr int kRouteRows = 4;
constexpr int kRouteTok = 16;

struct DecodeTail {  // outputs of the fused decode routing tail
    int k;
    int32_t *idx;
    float *w;
    int32_t *counts, *offsets, *perm_tok, *perm_slot, *inv, *active;
    int *ctrl;  // [0] arrival counter, [1] active experts
    float *y;
    int residual;
};

template <int PER>
__global__ void __launch_bounds__(256) route_gemv_kernel(const float *__restrict__ x, int T, int H,
                                                         const float *__restrict__ Wr,
                                                         const float *__restrict__ bias, int E,
                                                         float *logits, int fuse, DecodeTail tail) {
    __shared__ float part[8][kRouteRows][kRouteTok];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int e0 = blockIdx.x * kRouteRows;
    const int hs = H / 8;  // multiple of 16 (H multiple of 128)
    const int h0 = warp * hs;

    if (fuse) {  // y = residual ? x : 0, before any expert adds into it
        const size_t n = (size_t)T * H;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + tid; i < n; i += (size_t)gridDim.x * blockDim.x)
            tail.y[i] = tail.residual ? x[i] : 0.0f;
    }

    for (int t0 = 0; t0 < T; t0 += kRouteTok) {
        const int nt = min(kRouteTok, T - t0);
        float acc[kRouteRows][kRouteTok];
#pragma unroll
        for (int r = 0; r < kRouteRows; ++r)
#pragma unroll
            for (int t = 0; t < kRouteTok; ++t) acc[r][t] = 0.f;
        for (int h = h0 + 4 * lane; h < h0 + hs; h += 128) {
            float4 wv[kRouteRows];
#pragma unroll
            for (int r = 0; r < kRouteRows; ++r)
                wv[r] = (e0 + r < E) ? __ldg(reinterpret_cast<const float4 *>(Wr + (size_t)(e0 + r) * H + h))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int t = 0; t < kRouteTok; ++t) {
                if (t < nt) {
                    float4 xv = __ldg(reinterpret_cast<const float4 *>(x + (size_t)(t0 + t) * H + h));
#pragma unroll
                    for (int r = 0; r < kRouteRows; ++r)
                        acc[r][t] = fmaf(wv[r].x, xv.x, fmaf(wv[r].y, xv.y, fmaf(wv[r].z, xv.z, fmaf(wv[r].w, xv.w, acc[r][t]))));
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRouteRows; ++r)
#pragma unroll
            for (int t = 0; t < kRouteTok; ++t) {
                float s = warp_sum(acc[r][t]);
                if (lane == 0) part[warp][r][t] = s;
            }
        __syncthreads();
        if (tid < kRouteRows * kRouteTok) {
            const int r = tid / kRouteTok, t = tid % kRouteTok;
            if (t < nt && e0 + r < E) {
                float s = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) s += part[w8][r][t];
                s += bias ? bias[e0 + r] : 0.f;
                logits[(size_t)(t0 + t) * E + e0 + r] = s;
            }
        }
        __syncthreads();
    }
    if (!fuse) return;

    // ---- last CTA to finish ranks every token and builds the permutation
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        int prev = atomicAdd(&tail.ctrl[0], 1);
        s_last = (prev == (int)gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    __shared__ int s_sel[kRouteTok][kMaxK];
    __shared__ unsigned s_mask[kMaxE];  // bit t: token t picked expert e (T <= 32)
    __shared__ int s_cnt[kMaxE];
    __shared__ int s_act[kMaxE];
    __shared__ int s_scan[33];
    const int k = tail.k;
    for (int t = warp; t < T; t += 8)
        warp_topk<PER>(logits + (size_t)t * E, E, k, tail.idx + (size_t)t * k, tail.w + (size_t)t * k, s_sel[t]);
    for (int e = tid; e < E; e += blockDim.x) s_mask[e] = 0u;
    __syncthreads();
    for (int p = tid; p < T * k; p += blockDim.x) atomicOr(&s_mask[s_sel[p / k][p % k]], 1u << (p / k));
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        int c = __popc(s_mask[e]);
        s_cnt[e] = c;
        s_act[e] = c > 0;
        tail.counts[e] = c;
    }
    __syncthreads();
    const int total = block_exclusive_scan(s_cnt, E, s_scan);
    const int n_active = block_exclusive_scan(s_act, E, s_scan);
    for (int e = tid; e < E; e += blockDim.x) {
        tail.offsets[e] = s_cnt[e];
        if (s_mask[e]) tail.active[s_act[e]] = e;
    }
    if (tid == 0) {
        tail.offsets[E] = total;
        tail.ctrl[1] = n_active;
        tail.ctrl[0] = 0;  // re-arm the arrival counter for the next call
    }
    for (int p = tid; p < T * k; p += blockDim.x) {
        const int t = p / k, j = p % k, e = s_sel[t][j];
        const int pos = s_cnt[e] + __popc(s_mask[e] & ((1u << t) - 1u));
        tail.perm_tok[pos] = t;
        tail.perm_slot[pos] = j;
        tail.inv[p] = pos;
    }
}

// ------------------------------------------------- router logits, large T

// Plain SIMT SGEMM  L[T,E] = x[T,H] Wr[E,H]^T + b: 128x64 tile per CTA, 256
// threads with 8x4 outputs each, K-slabs of 16 staged transposed in shared
// memory.
constexpr int kSgBM = 128, kSgBN = 64, kSgBK = 16;

__global__ void __launch_bounds__(256) route_sgemm_kernel(const float *__restrict__ x, int T, int H,
                                                          const float *__restrict__ Wr,
                                                          const float *__restrict__ bias, int E,
                                                          float *__restrict__ logits) {
    __shared__ float As[2][kSgBK][kSgBM + 4];
    __shared__ float Bs[2][kSgBK][kSgBN + 4];
    const int tid = threadIdx.x;
    const int m0 = blockIdx.y * kSgBM, n0 = blockIdx.x * kSgBN;
    const int tx = tid % 16, ty = tid / 16;  // 16 x 16 threads; thread owns rows ty*8.., cols tx*4..
    float acc[8][4] = {};
    // loaders: A tile 128x16 = 512 float4 (2 per thread), B tile 64x16 = 256 float4 (1 per thread)
    auto load = [&](int buf, int k0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            int f = tid + 256 * i;
            int r = f / 4, c = (f % 4) * 4;
            int gr = m0 + r;
            float4 v = gr < T ? __ldg(reinterpret_cast<const float4 *>(x + (size_t)gr * H + k0 + c))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            As[buf][c + 0][r] = v.x;
            As[buf][c + 1][r] = v.y;
            As[buf][c + 2][r] = v.z;
            As[buf][c + 3][r] = v.w;
        }
        {
            int r = tid / 4, c = (tid % 4) * 4;
            int gr = n0 + r;
            float4 v = gr < E ? __ldg(reinterpret_cast<const float4 *>(Wr + (size_t)gr * H + k0 + c))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            Bs[buf][c + 0][r] = v.x;
            Bs[buf][c + 1][r] = v.y;
            Bs[buf][c + 2][r] = v.z;
            Bs[buf][c + 3][r] = v.w;
        }
    };
    load(0, 0);
    __syncthreads();
    const int nk = H / kSgBK;
    for (int kt = 0; kt < nk; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < nk) load(buf ^ 1, (kt + 1) * kSgBK);
#pragma unroll
        for (int kk = 0; kk < kSgBK; ++kk) {
            float a[8], b[4];
            float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][kk][ty * 8]);
            float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][kk][ty * 8 + 4]);
            float4 b0 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][tx * 4]);
            a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
            a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
            b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int r = m0 + ty * 8 + i;
        if (r >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int c = n0 + tx * 4 + j;
            if (c < E) logits[(size_t)r * E + c] = acc[i][j] + (bias ? bias[c] : 0.f);
        }
    }
}

}  // namespace moeq
