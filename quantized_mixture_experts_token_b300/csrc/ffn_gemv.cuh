// ffn_gemv.cuh -- the experts for few tokens per expert (decode): one CTA per
// (active expert, 32-row block of the intermediate dimension).
//
// The pages run the experts a decode step selects on the GPU when they are
// cached ("Strata - the details", "How it works"); here all are resident and
// the step is bound by reading the selected experts' bytes once.
//
// A CTA owns rows i in [32*ib, 32*ib+32) of gate and up and the matching
// 32-column slice of down -- one quantisation block of the SwiGLU activation,
// so the whole gate/up -> SwiGLU -> int8 -> down chain stays inside the CTA.
//   0. right after the routing of this call is visible, one warp issues bulk
//      asynchronous copies (cp.async.bulk, one mbarrier per matrix group) of
//      the CTA's whole weight slice into shared memory: 32 rows x H of gate
//      and of up, H rows x 32 of down -- 60 KB at H = 2048 (2-bit), all in
//      flight at once;
//   1. meanwhile bulk copies stage its tokens' activations, quantised per
//      32-block by the routing kernel (int8 codes already in the __dp4a
//      order, fp32 scales, code sums), in shared memory;
//   2. gate/up: warp w handles matrix w/4 and every fourth K-block, lane = row;
//      each 32-block product is an exact integer (__dp4a) scaled by s_w * s_x;
//   3. warp s = token s: h = silu(G) * U for the 32 rows, amax by warp
//      reduction, int8 re-quantisation;
//   4. down projection of that I-block for all H outputs (exact block dots)
//      and the routing-weighted add into y (red.global.add.v4.f32).
// The weights stay in shared memory for every token of the expert.  Shapes
// whose slice exceeds the buffers (H > 2048) stream it through them in pieces.
// The I-blocks of one expert land in y through fp32 atomics, so their
// summation order is not fixed.
#pragma once

#include <cuda.h>

#include "async.cuh"
#include "route.cuh"

namespace moeq {

constexpr int kGvTok = 8;        // tokens per pass (register accumulators)
constexpr int kGvMaxKB = 64;     // gate/up K-blocks held in shared memory at once
constexpr int kGvMaxRows = 2048; // down rows held in shared memory at once

struct GemvArgs {
    const float *x;
    const int8_t *qx;     // x quantised per 32-block [T][H] (natural order), written by the previous kernel
    const float *sx;      // block scales [T][H/32]
    const int *xsum;      // block sums of the codes [T][H/32]
    int T, H, I, E, k;
    const uint8_t *codes[3];
    const uint16_t *scales[3];
    const int32_t *perm_tok, *perm_slot;  // sorted pairs (tokens past a unit's first kUnitTok)
    const float *w;                       // routing weights [T][k]
    const UnitRec *units;                 // route_mode 0: one record per active expert
    const int *ctrl;                      // route_mode 0: ctrl[1] = number of records
    int route_mode;                       // 1: rank the router logits in every CTA (T <= kGvTok)
    const float *logits;                  // route_mode 1: [T][E] router logits
    int32_t *idx_out;                     // route_mode 1: routing outputs written by CTA 0 (or NULL)
    float *w_out;
    float *y, *out_sorted;
    int8_t *qh_out;
    float *sh_out;
    int kc, rc, tc;  // K-blocks of gate/up and rows of down held at once; tokens per pass (<= kGvTok)
    // TMA maps of gate/up: [0..1] codes viewed as uint32 [E*H/32][I*bits] with
    // box {32*bits, kc} (32 rows x kc K-blocks), [2..3] scales uint16 [E*H/32][I]
    // with box {32, kc}
    CUtensorMap tm[4];  // 64-byte aligned by its declaration
};

// Shared-memory carve-up of ffn_gemv_kernel (byte offsets, all 128-aligned).
struct GemvSmem {
    int bars, gu_codes, gu_scales, d_codes, d_scales, xpack, xs, xsum, part, hpack, hs, hsum, tok, wt, xrow, abort,
        total;
};

__host__ __device__ inline GemvSmem gemv_smem(int H, int bits, int kc, int rc, int tc) {
    const int bpb = 4 * bits, KBH = H / 32;
    GemvSmem L;
    int off = 0;
    auto take = [&](int bytes) {  // 128-byte aligned pieces (TMA destinations)
        const int o = off;
        off += (bytes + 127) & ~127;
        return o;
    };
    L.bars = take(32);
    L.abort = take(16);
    L.gu_codes = take(2 * kc * 32 * bpb);
    L.gu_scales = take(2 * kc * 32 * 2);
    L.d_codes = take(rc * bpb);
    L.d_scales = take(rc * 2);
    L.xpack = take(tc * KBH * 32);
    L.xs = take(tc * KBH * 4);
    L.xsum = take(tc * KBH * 4);
    L.part = take(2 * 4 * kGvTok * 32 * 4);
    L.hpack = take(kGvTok * 32);
    L.hs = take(kGvTok * 4);
    L.hsum = take(kGvTok * 4);
    L.tok = take(kGvTok * 4);
    L.wt = take(kGvTok * 4);
    L.xrow = take(kGvTok * 4);
    L.total = off;
    return L;
}

// Byte position of block element i in the activation words the block dot
// uses: pack_pos2 for 2-bit, natural order for 3-bit.
template <int BITS>
__device__ __forceinline__ int pack_pos(int i) {
    return BITS == 2 ? pack_pos2(i) : i;
}

template <int BITS>
struct BlockCodes {
    uint32_t w[BITS];  // 8 (2-bit) or 12 (3-bit) bytes of one 32-block
};

// One block's codes from shared memory (8-byte aligned for 2-bit, 4 for 3-bit).
template <int BITS>
__device__ __forceinline__ BlockCodes<BITS> smem_block(const unsigned char *p) {
    BlockCodes<BITS> c;
    if (BITS == 2) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        c.w[0] = v.x;
        c.w[1] = v.y;
    } else {
        const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
#pragma unroll
        for (int i = 0; i < BITS; ++i) c.w[i] = q[i];
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

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half((unsigned short)bits16));
}

// Gate/up partial sums over this warp's K-blocks (kl = q4, q4+4, ...) of one
// shared-memory chunk for NT tokens.  NT is a compile-time count so that no
// issue slot is spent on absent tokens.
template <int BITS, int NT, int AT>
__device__ __forceinline__ void gu_accumulate(float (&acc)[AT], const unsigned char *gu_codes,
                                              const uint16_t *gu_scales, const int4 *xpack, const float *xs,
                                              const int *xsum, const int *xrow, int m, int q4, int kc, int kb0,
                                              int nkb, int KBH, int lane) {
    constexpr int BPB = 4 * BITS, OFF = 1 << (BITS - 1);
    int rb[NT];  // staged activation row of each token, in K-blocks
#pragma unroll
    for (int s = 0; s < NT; ++s) rb[s] = xrow[s] * KBH;
#pragma unroll 4
    for (int kl = q4; kl < nkb; kl += 4) {
        const BlockCodes<BITS> c = smem_block<BITS>(gu_codes + (size_t)((m * kc + kl) * 32 + lane) * BPB);
        const float sw = half_bits_to_float(gu_scales[(m * kc + kl) * 32 + lane]);
        const int kb = kb0 + kl;
#pragma unroll
        for (int s = 0; s < NT; ++s) {
            const int4 *ap = xpack + (rb[s] + kb) * 2;
            const int d = block_dot_raw<BITS>(c, ap[0], ap[1]) - OFF * xsum[rb[s] + kb];
            acc[s] = fmaf(sw * xs[rb[s] + kb], (float)d, acc[s]);
        }
    }
}

// Work assignment of one CTA: expert e, its pair base pb and pair count ne;
// the first pass's tokens and routing weights are placed in tok / wt.
//
// route_mode 1 (T <= kGvTok, fused decode): every CTA ranks the T tokens'
// router logits itself (one warp per token, written by the router kernel just
// before) instead of waiting for a separate routing step.  Unit u is the u-th
// distinct expert in (token, slot) order of first selection; CTA 0 also
// writes the idx / w outputs.
// route_mode 0: unit u's record was written by the routing tail or the plan
// kernel.
template <int PER>
__device__ __forceinline__ bool gemv_unit(const GemvArgs &a, int u, int *tok, float *wt, int &e, int &pb, int &ne) {
    __shared__ int s_sel[kGvTok][kMaxK];
    __shared__ float s_w[kGvTok][kMaxK];
    __shared__ uint32_t s_mask[kMaxE];
    __shared__ int s_e, s_n;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (a.route_mode == 1) {
        const int T = a.T, k = a.k, E = a.E;
        MOEQ_TL(2, 10);
        if (warp < T) {
            const bool out = blockIdx.x == 0;  // the routing outputs are optional (NULL: not written)
            warp_topk<PER>(a.logits + (size_t)warp * E, E, k, out && a.idx_out ? a.idx_out + (size_t)warp * k : nullptr,
                           out && a.w_out ? a.w_out + (size_t)warp * k : nullptr, s_sel[warp], s_w[warp]);
        }
        MOEQ_TL(2, 11);
        __syncthreads();
        MOEQ_TL(2, 12);
        pb = 0;
        if (T == 1) {
            if (u >= k) return false;
            e = s_sel[0][u];
            ne = 1;
            if (tid == 0) {
                tok[0] = 0;
                wt[0] = s_w[0][u];
            }
            return true;
        }
        const int P = T * k;
        for (int p = tid; p < P; p += blockDim.x) s_mask[s_sel[p / k][p % k]] = 0u;
        __syncthreads();
        for (int p = tid; p < P; p += blockDim.x) atomicOr(&s_mask[s_sel[p / k][p % k]], 1u << (p / k));
        __syncthreads();
        if (warp == 0) {  // units in order of first selection
            int base = 0;
            for (int p0 = 0; p0 < P; p0 += 32) {
                const int p = p0 + lane;
                int ee = -1;
                bool first = false;
                if (p < P) {
                    const int t = p / k;
                    ee = s_sel[t][p - t * k];
                    first = (__ffs(s_mask[ee]) - 1) == t;
                }
                const unsigned bal = __ballot_sync(0xffffffffu, first);
                if (first && base + __popc(bal & ((1u << lane) - 1u)) == u) s_e = ee;
                base += __popc(bal);
            }
            if (lane == 0) s_n = base;
        }
        __syncthreads();
        if (u >= s_n) return false;
        e = s_e;
        const uint32_t m = s_mask[e];
        ne = __popc(m);
        if (tid < ne) {
            const int t = __fns(m, 0, tid + 1);
            tok[tid] = t;
            float wv = 0.f;
            for (int j = 0; j < k; ++j)
                if (s_sel[t][j] == e) wv = s_w[t][j];
            wt[tid] = wv;
        }
        return true;
    }
    const int nunits = __ldcg(a.ctrl + 1);
    const int4 head = __ldcg(reinterpret_cast<const int4 *>(a.units + u));
    if (u >= nunits) return false;
    e = head.x;
    pb = head.y;
    ne = head.z;
    if (tid < min(ne, kUnitTok)) {
        tok[tid] = __ldcg(&a.units[u].tok[tid]);
        wt[tid] = a.y ? __ldcg(&a.units[u].w[tid]) : 0.f;
    }
    return true;
}

// MAXNT: the most tokens a pass holds (a.tc <= MAXNT).  The single-token
// instantiation carries one block-dot loop instead of eight; B = 1 decode
// launches run it, and its smaller code takes fewer instruction-cache misses
// in CTAs that each run the body once.
template <int BITS, int PER, int MAXNT>
__global__ void __launch_bounds__(256) ffn_gemv_kernel(const __grid_constant__ GemvArgs a) {
    constexpr int BPB = 4 * BITS;
    constexpr int OFF = 1 << (BITS - 1);
    const int nIB = a.I / 32, KBH = a.H / 32;
    const int u = blockIdx.x / nIB, ib = blockIdx.x % nIB;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t wl = wait_limit();

    extern __shared__ __align__(128) unsigned char smem[];
    const GemvSmem L = gemv_smem(a.H, BITS, a.kc, a.rc, a.tc);
    const uint32_t bar_gu = smem_u32(smem + L.bars), bar_d = bar_gu + 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.abort);
    unsigned char *gu_codes = smem + L.gu_codes, *d_codes = smem + L.d_codes;
    const uint16_t *gu_scales = reinterpret_cast<const uint16_t *>(smem + L.gu_scales);
    const uint16_t *d_scales = reinterpret_cast<const uint16_t *>(smem + L.d_scales);
    int4 *xpack = reinterpret_cast<int4 *>(smem + L.xpack);  // [tc][KBH][2]
    float *xs = reinterpret_cast<float *>(smem + L.xs);      // [tc][KBH]
    int *xsum = reinterpret_cast<int *>(smem + L.xsum);      // [tc][KBH]
    float *part = reinterpret_cast<float *>(smem + L.part);  // [2][4][kGvTok][32]
    int4 *hpack = reinterpret_cast<int4 *>(smem + L.hpack);  // [kGvTok][2]
    float *hs = reinterpret_cast<float *>(smem + L.hs);
    int *hsum = reinterpret_cast<int *>(smem + L.hsum);
    int *tok = reinterpret_cast<int *>(smem + L.tok);
    float *wt = reinterpret_cast<float *>(smem + L.wt);
    int *xrow = reinterpret_cast<int *>(smem + L.xrow);  // staged activation row of each pass slot
    const uint32_t bar_x = bar_gu + 16;

    // set-up that needs nothing from earlier kernels runs before the dependency wait
    if (tid == 0) {
        mbar_init(bar_gu, 1);
        mbar_init(bar_d, 1);
        mbar_init(bar_x, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane < 4) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm[lane])) : "memory");
    __syncthreads();

    MOEQ_TL(2, 0);
    pdl_wait();  // the router logits (or routing records) and quantised x of this call are complete
    pdl_trigger();
    MOEQ_TL(2, 1);
    // quantised activation rows (codes already in the block dot's order, block
    // scales, block code sums) of the given tokens into staging rows 0, 1, ...
    // of shared memory, one bulk copy each (thread 0)
    auto issue_x = [&](bool by_token, int n) {  // row r holds token r (by_token) or tok[r]
        mbar_arrive_expect_tx(bar_x, (uint32_t)(n * (a.H + 8 * KBH)));
        for (int r = 0; r < n; ++r) {
            const size_t t = by_token ? (size_t)r : (size_t)tok[r];
            bulk_g2s(smem_u32(smem + L.xpack + (size_t)r * a.H), a.qx + t * a.H, (uint32_t)a.H, bar_x, 0);
            bulk_g2s(smem_u32(xs + r * KBH), a.sx + t * KBH, (uint32_t)(4 * KBH), bar_x, 0);
            bulk_g2s(smem_u32(xsum + r * KBH), a.xsum + t * KBH, (uint32_t)(4 * KBH), bar_x, 0);
        }
    };
    bool x_staged = false;   // route_mode 1: every token staged once, row = token
    bool x_pending = false;  // a copy into the staging rows is in flight (not yet waited for)
    if (a.route_mode == 1) {
        if (tid == 0) issue_x(true, a.T);
        x_staged = true;
        x_pending = true;
    }
    int e = 0, pb = 0, ne = 0;
    const bool have = gemv_unit<PER>(a, u, tok, wt, e, pb, ne);  // uniform over the CTA
    MOEQ_TL(2, 2);
    const bool bad = have && (e < 0 || e >= a.E);
    if (!have || bad || ne <= 0) {
        if (bad && tid == 0) set_status(MOEQ_STATUS_BAD_INDEX);
        // the CTA's shared memory must not be released while the staging copy lands
        if (x_pending && tid == 0) mbar_drain(bar_x, 0, abort_flag);
        return;
    }

    const int ngc = (KBH + a.kc - 1) / a.kc, ndc = (a.H + a.rc - 1) / a.rc;
    const uint64_t pol = l2_evict_first();
    // gate/up rows of this I-block for K-blocks [c*kc, c*kc + kc): one TMA box
    // of codes and one of scales per matrix (a box running past the expert's
    // last block reads bytes that are never used)
    auto issue_gu = [&](int c) {  // by warp 0: lanes 0-3 issue one box each
        if (lane == 0) mbar_arrive_expect_tx(bar_gu, (uint32_t)(2 * a.kc * 32 * (BPB + 2)));
        __syncwarp();
        const int y = e * KBH + c * a.kc, m = lane & 1;
        if (lane < 2)
            tma_load_2d(smem_u32(gu_codes + (size_t)m * a.kc * 32 * BPB), &a.tm[m], 32 * BITS * ib, y, bar_gu, pol);
        else if (lane < 4)
            tma_load_2d(smem_u32(smem + L.gu_scales + (size_t)m * a.kc * 64), &a.tm[2 + m], 32 * ib, y, bar_gu, pol);
    };
    // down rows [c*rc, c*rc + nr) of this I-block: one code run, one scale run (warp 0, lanes 4-5)
    auto issue_d = [&](int c) {
        const int r0 = c * a.rc, nr = min(a.rc, a.H - r0);
        if (lane == 0) mbar_arrive_expect_tx(bar_d, (uint32_t)(nr * (BPB + 2)));
        __syncwarp();
        const size_t base = ((size_t)e * nIB + ib) * a.H + r0;
        if (lane == 4) bulk_g2s(smem_u32(d_codes), a.codes[2] + base * BPB, (uint32_t)(nr * BPB), bar_d, pol);
        if (lane == 5) bulk_g2s(smem_u32(smem + L.d_scales), a.scales[2] + base, (uint32_t)(nr * 2), bar_d, pol);
    };

    // buffer state (identical in every thread: all take the same path)
    int gu_chunk = 0, d_chunk = 0;       // chunk in (or on its way into) each buffer
    bool gu_ready = false, d_ready = false, x_ready = false;
    uint32_t gu_ph = 0, d_ph = 0, x_ph = 0;  // completed phases of each barrier
    if (warp == 0) {
        issue_gu(0);
        issue_d(0);
    }
    __syncwarp();

    bool failed = false;
    for (int c0 = 0; c0 < ne && !failed; c0 += a.tc) {
        const int nt = min(a.tc, ne - c0);
        if (c0 > 0 && tid < nt) {  // later passes (more than tc tokens): from the permutation arrays
            const int p = pb + c0 + tid;
            int t = __ldcg(a.perm_tok + p);
            const int j = __ldcg(a.perm_slot + p);
            float wv = 0.f;
            if (t < 0 || t >= a.T || j < 0 || j >= a.k) {  // a caller's bad permutation: no contribution
                set_status(MOEQ_STATUS_BAD_INDEX);
                t = 0;
            } else if (a.y) {
                wv = __ldcg(a.w + (size_t)t * a.k + j);
            }
            tok[tid] = t;
            wt[tid] = wv;
        }
        __syncthreads();
        // 1. the pass's quantised activations (route_mode 1: staged once for all tokens)
        if (!x_staged) {
            if (tid == 0) issue_x(false, nt);
            x_pending = true;
            if (tid < nt) xrow[tid] = tid;
        } else if (tid < nt) {
            xrow[tid] = tok[tid];
        }
        if (!x_ready) {
            const bool ok = mbar_wait(bar_x, x_ph & 1, abort_flag, wl);
            if (__syncthreads_or(!ok)) {
                failed = true;
                break;
            }
            ++x_ph;
            x_pending = false;
            x_ready = x_staged;
            MOEQ_TL(2, 3);
        } else {
            __syncthreads();
        }
        // 2. gate / up: warp (m, q) sums K-blocks q, q+4, ... of matrix m
        const int m = warp >> 2, q4 = warp & 3;
        float acc[MAXNT];
#pragma unroll
        for (int s = 0; s < MAXNT; ++s) acc[s] = 0.f;
        for (int gc = 0; gc < ngc; ++gc) {
            if (gu_chunk != gc) {  // only when the slice is streamed in pieces
                __syncthreads();
                if (warp == 0) issue_gu(gc);
                gu_chunk = gc;
                gu_ready = false;
            }
            if (!gu_ready) {
                const bool ok = mbar_wait(bar_gu, gu_ph & 1, abort_flag, wl);
                if (__syncthreads_or(!ok)) {
                    failed = true;
                    break;
                }
                ++gu_ph;
                gu_ready = true;
                MOEQ_TL(2, 4);
            }
            const int kb0 = gc * a.kc, nkb = min(a.kc, KBH - kb0);
#define MOEQ_GU(NT_)                                                                                             \
    gu_accumulate<BITS, (NT_ < MAXNT ? NT_ : MAXNT), MAXNT>(acc, gu_codes, gu_scales, xpack, xs, xsum, xrow, m, q4, a.kc, kb0, nkb, KBH, lane); \
    break
            if (MAXNT == 1) {
                gu_accumulate<BITS, 1, MAXNT>(acc, gu_codes, gu_scales, xpack, xs, xsum, xrow, m, q4, a.kc, kb0, nkb, KBH, lane);
            } else {
                switch (nt) {
                    case 1: MOEQ_GU(1);
                    case 2: MOEQ_GU(2);
                    case 3: MOEQ_GU(3);
                    case 4: MOEQ_GU(4);
                    case 5: MOEQ_GU(5);
                    case 6: MOEQ_GU(6);
                    case 7: MOEQ_GU(7);
                    default: MOEQ_GU(8);
                }
            }
#undef MOEQ_GU
        }
        if (failed) break;
#pragma unroll
        for (int s = 0; s < MAXNT; ++s) part[((m * 4 + q4) * kGvTok + s) * 32 + lane] = acc[s];
        __syncthreads();
        MOEQ_TL(2, 5);
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
            if (a.qh_out) a.qh_out[p * a.I + 32 * ib + lane] = (int8_t)q;
            if (a.sh_out && lane == 0) a.sh_out[p * nIB + ib] = sh;
        }
        __syncthreads();
        MOEQ_TL(2, 6);
        // 4. down projection of I-block ib, 4 consecutive output rows per thread
        for (int dc = 0; dc < ndc; ++dc) {
            if (d_chunk != dc) {
                __syncthreads();
                if (warp == 0) issue_d(dc);
                d_chunk = dc;
                d_ready = false;
            }
            if (!d_ready) {
                const bool ok = mbar_wait(bar_d, d_ph & 1, abort_flag, wl);
                if (__syncthreads_or(!ok)) {
                    failed = true;
                    break;
                }
                ++d_ph;
                d_ready = true;
                MOEQ_TL(2, 7);
            }
            const int r0 = dc * a.rc, nr = min(a.rc, a.H - r0);
            for (int g = tid; g < nr / 4; g += blockDim.x) {
                const int rl = 4 * g, n0 = r0 + rl;
                BlockCodes<BITS> c[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) c[r] = smem_block<BITS>(d_codes + (size_t)(rl + r) * BPB);
                const uint2 sv = *reinterpret_cast<const uint2 *>(d_scales + rl);
                const float sd[4] = {half_bits_to_float(sv.x & 0xffffu), half_bits_to_float(sv.x >> 16),
                                     half_bits_to_float(sv.y & 0xffffu), half_bits_to_float(sv.y >> 16)};
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
        }
        __syncthreads();
    }
    MOEQ_TL(2, 8);
    if (failed && tid == 0) {
        // drain the copies still in flight before the CTA's shared memory is released
        if (!gu_ready) mbar_drain(bar_gu, gu_ph & 1, abort_flag);
        if (!d_ready) mbar_drain(bar_d, d_ph & 1, abort_flag);
        if (x_pending) mbar_drain(bar_x, x_ph & 1, abort_flag);
    }
}

}  // namespace moeq
