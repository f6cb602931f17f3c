// ffn_gemv.cuh -- the experts for few tokens per expert (decode): one CTA per
// (active expert, 32-row block of the intermediate dimension).
//
// The pages run the experts a decode step selects on the GPU when they are
// cached ("Strata - the details", "How it works"); here all are resident and
// the step is bound by reading the selected experts' bytes once.
//
// CTA work, for the tokens routed to expert e (in chunks of kGvTok):
//   1. quantise each token's x per 32-block (int8 + fp32 scale) into shared
//      memory, packed for __dp4a;
//   2. gate/up rows i in [32*ib, 32*ib+32): warp w handles matrix w/4 and a
//      quarter of the K-blocks, lane = row; each 32-block product is an exact
//      integer (__dp4a) scaled by s_w * s_x in fp32;
//   3. warp s = token s: h = silu(G) * U for the 32 rows (one quantisation
//      block), amax by warp reduction, int8 re-quantisation;
//   4. down projection of that single I-block for all H outputs (exact block
//      dots again) and the routing-weighted add into y (red.global.add.v4).
// The I-blocks of one expert land in y through fp32 atomics, so their
// summation order is not fixed.
#pragma once

#include "common.cuh"

namespace moeq {

constexpr int kGvTok = 8;

struct GemvArgs {
    const float *x;
    int T, H, I, E, k;
    const uint8_t *codes[3];
    const uint16_t *scales[3];
    const int32_t *offsets, *perm_tok, *perm_slot;
    const float *w;
    const int32_t *active;
    const int *ctrl;  // ctrl[1] = number of active experts
    float *y, *out_sorted;
    int8_t *qh_out;
    float *sh_out;
};

// Byte position of block element i in the 8 packed words the block dot uses.
// 2-bit: word m (m < 4) holds elements {m, 4+m, 8+m, 12+m}, word 4+m the same
// for elements 16..31 -- the order that masking the code words with
// 0x03030303 after a shift by 2m produces.  3-bit: natural order.
template <int BITS>
__device__ __forceinline__ int pack_pos(int i) {
    if (BITS == 2) return (4 * (i >> 4) + (i & 3)) * 4 + ((i & 15) >> 2);
    return i;
}

template <int BITS>
struct BlockCodes {
    uint32_t w[BITS];  // 8 (2-bit) or 12 (3-bit) bytes of one 32-block
};

template <int BITS>
__device__ __forceinline__ BlockCodes<BITS> load_block(const uint8_t *p) {
    BlockCodes<BITS> c;
    if (BITS == 2) {
        uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
        c.w[0] = v.x;
        c.w[1] = v.y;
    } else {
        const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
#pragma unroll
        for (int i = 0; i < BITS; ++i) c.w[i] = __ldg(q + i);
    }
    return c;
}

// Exact sum_i code_i * a_i over the block (codes unsigned, before the level
// offset), with a packed as pack_pos<BITS> orders it.
template <int BITS>
__device__ __forceinline__ int block_dot_raw(const BlockCodes<BITS> &c, const int4 a0, const int4 a1) {
    int d = 0;
    if (BITS == 2) {
        d = __dp4a((int)(c.w[0] & 0x03030303u), a0.x, d);
        d = __dp4a((int)((c.w[0] >> 2) & 0x03030303u), a0.y, d);
        d = __dp4a((int)((c.w[0] >> 4) & 0x03030303u), a0.z, d);
        d = __dp4a((int)((c.w[0] >> 6) & 0x03030303u), a0.w, d);
        d = __dp4a((int)(c.w[1] & 0x03030303u), a1.x, d);
        d = __dp4a((int)((c.w[1] >> 2) & 0x03030303u), a1.y, d);
        d = __dp4a((int)((c.w[1] >> 4) & 0x03030303u), a1.z, d);
        d = __dp4a((int)((c.w[1] >> 6) & 0x03030303u), a1.w, d);
    } else {
        const int av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t packed = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int i = 4 * j + b, off = 3 * i, wi = off >> 5, sh = off & 31;
                const uint32_t hiw = (wi + 1 < BITS) ? c.w[wi + 1] : 0u;
                const uint32_t f = __funnelshift_r(c.w[wi], hiw, sh) & 7u;
                packed |= f << (8 * b);
            }
            d = __dp4a((int)packed, av[j], d);
        }
    }
    return d;
}

template <int BITS>
__global__ void __launch_bounds__(256) ffn_gemv_kernel(GemvArgs a) {
    constexpr int BPB = 4 * BITS;
    constexpr int OFF = 1 << (BITS - 1);
    const int nIB = a.I / 32, KBH = a.H / 32;
    const int u = blockIdx.x / nIB, ib = blockIdx.x % nIB;
    if (u >= a.ctrl[1]) return;
    const int e = a.active[u];
    if (e < 0 || e >= a.E) {
        set_status(MOEQ_STATUS_BAD_INDEX);
        return;
    }
    const int pb = a.offsets[e], ne = a.offsets[e + 1] - pb;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    extern __shared__ __align__(16) unsigned char smem[];
    int4 *xpack = reinterpret_cast<int4 *>(smem);                         // [kGvTok][KBH][2]
    float *xs = reinterpret_cast<float *>(xpack + kGvTok * KBH * 2);      // [kGvTok][KBH]
    int *xsum = reinterpret_cast<int *>(xs + kGvTok * KBH);              // [kGvTok][KBH]
    float *part = reinterpret_cast<float *>(xsum + kGvTok * KBH);        // [2][4][kGvTok][32]
    int4 *hpack = reinterpret_cast<int4 *>(part + 2 * 4 * kGvTok * 32);  // [kGvTok][2]
    float *hs = reinterpret_cast<float *>(hpack + kGvTok * 2);           // [kGvTok]
    int *hsum = reinterpret_cast<int *>(hs + kGvTok);                    // [kGvTok]
    int *tok = hsum + kGvTok;                                            // [kGvTok]
    float *wt = reinterpret_cast<float *>(tok + kGvTok);                 // [kGvTok]

    const uint8_t *cgu = warp < 4 ? a.codes[0] : a.codes[1];
    const uint16_t *sgu = warp < 4 ? a.scales[0] : a.scales[1];
    const int mat = warp >> 2, quarter = warp & 3;
    const int i_row = 32 * ib + lane;
    const int kbq = KBH / 4;  // H multiple of 128
    const uint8_t *cbase = cgu + (size_t)e * KBH * a.I * BPB;
    const uint16_t *sbase = sgu + (size_t)e * KBH * a.I;
    const uint8_t *dbase = a.codes[2] + ((size_t)e * nIB + ib) * a.H * BPB;
    const uint16_t *dsbase = a.scales[2] + ((size_t)e * nIB + ib) * a.H;

    for (int c0 = 0; c0 < ne; c0 += kGvTok) {
        const int nt = min(kGvTok, ne - c0);
        if (tid < nt) {
            const int p = pb + c0 + tid;
            const int t = a.perm_tok[p];
            tok[tid] = t;
            wt[tid] = a.w ? a.w[(size_t)t * a.k + a.perm_slot[p]] : 0.f;
        }
        __syncthreads();
        // 1. quantise the chunk's activations into packed shared memory
        for (int job = warp; job < nt * KBH; job += 8) {
            const int s = job / KBH, b = job - s * KBH;
            const float v = a.x[(size_t)tok[s] * a.H + 32 * b + lane];
            const float sc = block_scale(warp_absmax(v));
            const int q = block_code(v, sc);
            reinterpret_cast<int8_t *>(xpack + (s * KBH + b) * 2)[pack_pos<BITS>(lane)] = (int8_t)q;
            const int qs = warp_sum_int(q);
            if (lane == 0) {
                xs[s * KBH + b] = sc;
                xsum[s * KBH + b] = qs;
            }
        }
        __syncthreads();
        // 2. gate / up partial sums over this warp's quarter of the K-blocks
        float acc[kGvTok];
#pragma unroll
        for (int s = 0; s < kGvTok; ++s) acc[s] = 0.f;
#pragma unroll 4
        for (int kb = quarter * kbq; kb < (quarter + 1) * kbq; ++kb) {
            const BlockCodes<BITS> c = load_block<BITS>(cbase + ((size_t)kb * a.I + i_row) * BPB);
            const float sw = __half2float(__ushort_as_half(__ldg(sbase + (size_t)kb * a.I + i_row)));
#pragma unroll
            for (int s = 0; s < kGvTok; ++s) {
                if (s < nt) {
                    const int4 *ap = xpack + (s * KBH + kb) * 2;
                    const int d = block_dot_raw<BITS>(c, ap[0], ap[1]) - OFF * xsum[s * KBH + kb];
                    acc[s] = fmaf(sw * xs[s * KBH + kb], (float)d, acc[s]);
                }
            }
        }
#pragma unroll
        for (int s = 0; s < kGvTok; ++s) part[((mat * 4 + quarter) * kGvTok + s) * 32 + lane] = acc[s];
        __syncthreads();
        // 3. SwiGLU and re-quantisation of this I-block, one warp per token
        if (warp < nt) {
            const int s = warp;
            float G = 0.f, U = 0.f;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                G += part[((0 * 4 + qq) * kGvTok + s) * 32 + lane];
                U += part[((1 * 4 + qq) * kGvTok + s) * 32 + lane];
            }
            const float h = __fdiv_rn(G, 1.0f + expf(-G)) * U;
            const float sh = block_scale(warp_absmax(h));
            const int q = block_code(h, sh);
            reinterpret_cast<int8_t *>(hpack + s * 2)[pack_pos<BITS>(lane)] = (int8_t)q;
            const int qs = warp_sum_int(q);
            if (lane == 0) {
                hs[s] = sh;
                hsum[s] = qs;
            }
            const size_t p = (size_t)(pb + c0 + s);
            if (a.qh_out) a.qh_out[p * a.I + i_row] = (int8_t)q;
            if (a.sh_out && lane == 0) a.sh_out[p * nIB + ib] = sh;
        }
        __syncthreads();
        // 4. down projection of I-block ib for every output row, 4 rows per thread
        for (int g = tid; g < a.H / 4; g += blockDim.x) {
            const int n0 = 4 * g;
            BlockCodes<BITS> c[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) c[r] = load_block<BITS>(dbase + (size_t)(n0 + r) * BPB);
            const uint2 sv = __ldg(reinterpret_cast<const uint2 *>(dsbase + n0));
            const float sd[4] = {__half2float(__ushort_as_half((unsigned short)(sv.x & 0xffff))),
                                 __half2float(__ushort_as_half((unsigned short)(sv.x >> 16))),
                                 __half2float(__ushort_as_half((unsigned short)(sv.y & 0xffff))),
                                 __half2float(__ushort_as_half((unsigned short)(sv.y >> 16)))};
            for (int s = 0; s < nt; ++s) {
                const int4 h0 = hpack[s * 2], h1 = hpack[s * 2 + 1];
                float D[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int d = block_dot_raw<BITS>(c[r], h0, h1) - OFF * hsum[s];
                    D[r] = sd[r] * hs[s] * (float)d;
                }
                if (a.y) {
                    const float ws = wt[s];
                    red_add_v4(a.y + (size_t)tok[s] * a.H + n0, ws * D[0], ws * D[1], ws * D[2], ws * D[3]);
                }
                if (a.out_sorted)
                    red_add_v4(a.out_sorted + (size_t)(pb + c0 + s) * a.H + n0, D[0], D[1], D[2], D[3]);
            }
        }
        __syncthreads();
    }
}

inline size_t gemv_smem_bytes(int H) {
    const int KBH = H / 32;
    return (size_t)kGvTok * KBH * 32 + 2 * (size_t)kGvTok * KBH * 4 + 2 * 4 * kGvTok * 32 * 4 +
           kGvTok * 32 + 4 * kGvTok * 4;
}

}  // namespace moeq
