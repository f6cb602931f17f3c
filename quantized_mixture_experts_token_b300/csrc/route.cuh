// route.cuh -- router logits, top-k + renormalised softmax, and the decode
// fast path that also builds the token-to-expert permutation.
//
// Routers run on the GPU and pick 10 of 512 experts per token ("Strata - the
// details", sections "How it works" and "Which model?").
#pragma once

#include "async.cuh"

namespace moeq {

// ---------------------------------------------------------------- top-k

// Order-preserving map of fp32 onto uint32 (larger float -> larger key); -0 is
// folded onto +0 so that equal values compare equal.
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One warp ranks one token's E logits (E <= 1024), lane l holding logits l,
// l+32, ... as order keys.  Result: the k largest in descending order, ties
// to the lower expert index, and their softmax weights.
//
// Threshold pass: tau = the k-th largest of the 32 lane maxima.  The k lanes
// with the largest maxima hold k values >= tau, so every one of the top k is
// >= tau; typically only a dozen keys pass.  The candidates are compacted into
// shared memory and each is ranked by counting the candidates ordered before
// it.  More than 64 candidates (heavy ties) fall back to k rounds of a
// warp-wide arg-max.  Must be called by whole warps of a CTA of at most 8 warps.
template <int PER>  // ceil(E / 32), <= 32
__device__ __forceinline__ void warp_topk(const float *row, int E, int k, int32_t *idx_out, float *w_out,
                                          int *sel_idx /* smem [k] or null */, float *sel_w = nullptr) {
    __shared__ uint2 s_cand[8][64];  // (key, expert) per warp
    __shared__ uint2 s_top[8][kMaxK];
    const int lane = threadIdx.x & 31, wid = (threadIdx.x >> 5) & 7;
    __syncwarp();  // a previous call of this warp is done with the tables
    uint32_t key[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < E ? order_key(ld_cg(row + e)) : 0u;  // 0: below every finite value's key
    }
    uint32_t lm = 0u;
#pragma unroll
    for (int i = 0; i < PER; ++i) lm = max(lm, key[i]);
    MOEQ_TL(9, 0);  // (tracing builds) the logits are in registers
    int gt = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) gt += __shfl_sync(0xffffffffu, lm, j) > lm;
    const uint32_t tau = __reduce_min_sync(0xffffffffu, gt < k ? lm : 0xffffffffu);
    uint32_t cm = 0u;
    int c = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i)
        if (key[i] >= tau) {
            cm |= 1u << i;
            ++c;
        }
    const int total = __reduce_add_sync(0xffffffffu, c);
    if (total <= 32) {
        // usual case: one candidate per lane, ranked by 32 register shuffles
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int pos = incl - c;
#pragma unroll
        for (int i = 0; i < PER; ++i)
            if ((cm >> i) & 1u) s_cand[wid][pos++] = make_uint2(key[i], (uint32_t)(lane + 32 * i));
        __syncwarp();
        const uint2 me = lane < total ? s_cand[wid][lane] : make_uint2(0u, 0xffffffffu);
        int r = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const uint32_t ok = __shfl_sync(0xffffffffu, me.x, j), oe = __shfl_sync(0xffffffffu, me.y, j);
            r += (j < total) && ((ok > me.x) || (ok == me.x && oe < me.y));
        }
        if (lane < total && r < k) s_top[wid][r] = me;
    } else if (total <= 64) {
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int pos = incl - c;
#pragma unroll
        for (int i = 0; i < PER; ++i)
            if ((cm >> i) & 1u) s_cand[wid][pos++] = make_uint2(key[i], (uint32_t)(lane + 32 * i));
        __syncwarp();
        for (int q = lane; q < total; q += 32) {
            const uint2 me = s_cand[wid][q];
            int r = 0;
            for (int j = 0; j < total; ++j) {
                const uint2 o = s_cand[wid][j];
                r += (o.x > me.x) || (o.x == me.x && o.y < me.y);
            }
            if (r < k) s_top[wid][r] = me;
        }
    } else {
        uint32_t taken = 0u;  // bit i: slot i already selected
        for (int j = 0; j < k; ++j) {
            uint32_t bk = 0u;
            int bi = 0;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const uint32_t ki = ((taken >> i) & 1u) ? 0u : key[i];
                if (ki > bk) {  // strict: the lowest slot wins among equal keys
                    bk = ki;
                    bi = i;
                }
            }
            const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
            const int be = __reduce_min_sync(0xffffffffu, bk == mk ? lane + 32 * bi : 0x7fffffff);
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            if (lane == j) s_top[wid][j] = make_uint2(mk, (uint32_t)be);
        }
    }
    __syncwarp();
    const float top0 = key_value(s_top[wid][0].x);
    float my_w = 0.f;
    int my_idx = 0;
    if (lane < k) {
        const uint2 t = s_top[wid][lane];
        my_w = key_value(t.x);
        my_idx = (int)t.y;
    }
    // softmax over the k selected logits, relative to the largest
    float ex = lane < k ? expf(my_w - top0) : 0.0f;
    float den = warp_sum(ex);
    if (lane < k) {
        const float wv = __fdiv_rn(ex, den);
        if (idx_out) idx_out[lane] = my_idx;
        if (w_out) w_out[lane] = wv;
        if (sel_idx) sel_idx[lane] = my_idx;
        if (sel_w) sel_w[lane] = wv;
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

// CTA = 8 warps over 4 experts.  The CTA's 4 router rows (H fp32 values each,
// 32 KB at H = 2048) are fetched into shared memory by one bulk asynchronous
// copy issued BEFORE the grid waits for the previous kernel on the stream
// (programmatic dependent launch): the router weights stream in while the
// previous layer's experts still run.  Warp w then covers the H-slice
// [w*H/8, (w+1)*H/8) for all 4 experts, so every x value loaded is used 4
// times; each lane keeps 4 x (tokens) accumulators and the H-slice partials
// are summed over the 8 warps in a fixed order (deterministic).  In the fused
// decode path the CTAs also quantise x per 32-block for the expert kernel.
constexpr int kRouteRows = 4;
constexpr int kRouteTok = 16;   // tokens per pass (register accumulators)
constexpr int kRouteHC = 2048;  // router columns held in shared memory at once
constexpr int kFusedMaxT = 64;  // largest T the fused decode tail handles (64-bit token masks)

// Fused decode work of the router kernel (mode > 0): y = residual ? x : 0, x
// quantised per 32-block for the expert kernel, and in mode 2 the routing
// itself by the last CTA to finish (top-k, grouping by expert into UnitRec
// records).
struct DecodeTail {
    int mode;  // 0: logits only; 1: + y init and x quantisation; 2: + routing tail
    int k;
    int32_t *idx;
    float *w;
    int32_t *perm_tok, *perm_slot, *inv;
    UnitRec *units;
    int *ctrl;  // [0] arrival counter, [1] number of units
    float *y;
    int residual;
    int8_t *qx;  // x quantised per 32-block [T][H], its scales [T][H/32] and code sums
    float *sx;
    int *xsum;
    int bits;  // of the expert weights: 2-bit codes are stored in the dp4a order (see qx)
};

// Dynamic shared memory of route_gemv_kernel: the router rows of one column
// chunk, later reused by the fused tail's tables.
struct RouteSmem {
    int bar, wr, sel, selw, mask, unit, pb, total;
};

__host__ __device__ inline RouteSmem route_smem(int H, int E) {
    RouteSmem L;
    L.bar = 0;
    L.wr = 16;
    const int hc = H < kRouteHC ? H : kRouteHC;
    const int wr_bytes = kRouteRows * hc * 4;
    L.sel = 16;                                // [kFusedMaxT][kMaxK] int
    L.selw = L.sel + kFusedMaxT * kMaxK * 4;   // [kFusedMaxT][kMaxK] float
    L.mask = L.selw + kFusedMaxT * kMaxK * 4;  // [E] uint64
    L.unit = L.mask + E * 8;                   // [E] int
    L.pb = L.unit + E * 4;                     // [E] int
    const int tail_end = L.pb + E * 4;
    L.total = (16 + wr_bytes > tail_end ? 16 + wr_bytes : tail_end);
    return L;
}

// Router partial dot products of this warp's columns [h_begin, h_end) of one
// shared-memory chunk for up to NT tokens (nt <= NT active).
template <int NT, int AT>
__device__ __forceinline__ void route_accumulate(float (&acc)[kRouteRows][AT], const float *wr, int hc, int nr,
                                                 const float *x, int H, int t0, int c0, int h_begin, int h_end,
                                                 int lane, int nt) {
    for (int h = h_begin + 4 * lane; h < h_end; h += 128) {
        float4 wv[kRouteRows];
#pragma unroll
        for (int r = 0; r < kRouteRows; ++r)
            wv[r] = r < nr ? *reinterpret_cast<const float4 *>(wr + r * hc + h) : make_float4(0.f, 0.f, 0.f, 0.f);
        // the tokens' x values first, all in flight at once (a load behind each
        // token's branch would wait out one L2 latency per token); a slot past the
        // call's tokens reads token t0 and is not used
        float4 xv[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t)
            xv[t] = *reinterpret_cast<const float4 *>(x + (size_t)(t0 + (t < nt ? t : 0)) * H + c0 + h);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t < nt) {
#pragma unroll
                for (int r = 0; r < kRouteRows; ++r)
                    acc[r][t] = fmaf(wv[r].x, xv[t].x,
                                     fmaf(wv[r].y, xv[t].y, fmaf(wv[r].z, xv[t].z, fmaf(wv[r].w, xv[t].w, acc[r][t]))));
            }
        }
    }
}

// Warp sums of V <= 32 values per lane at once (a reduce-scatter): each step
// sends half of the remaining values to the lane `o` away and keeps the half
// selected by that lane bit, so after log2(V) steps lane l holds a partial of
// value l >> (5 - log2 V), completed by xor-sums over the remaining lane bits.
// 31 shuffles for 32 values, where one warp sum each would take 160.
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[V], int lane) {
    static_assert(V >= 2 && V <= 32 && (V & (V - 1)) == 0, "V a power of two <= 32");
#pragma unroll
    for (int n = V, o = 16; n > 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float mine = up ? v[n / 2 + i] : v[i];
            const float other = up ? v[i] : v[n / 2 + i];
            v[i] = mine + __shfl_xor_sync(0xffffffffu, other, o);
        }
    }
    float r = v[0];
#pragma unroll
    for (int o = 16 / V; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

template <int NT, int AT>
__device__ __forceinline__ void route_reduce(const float (&acc)[kRouteRows][AT], float (*part)[kRouteRows][kRouteTok],
                                             int warp, int lane) {
    if (NT == 1) {
#pragma unroll
        for (int r = 0; r < kRouteRows; ++r) {
            const float s = warp_sum(acc[r][0]);
            if (lane == 0) part[warp][r][0] = s;
        }
        return;
    }
    // value i = r * NT + t, reduced in groups of at most 32 values
    constexpr int V = kRouteRows * NT, G = V > 32 ? 32 : V, LG = G == 32 ? 5 : G == 16 ? 4 : G == 8 ? 3 : 2;
#pragma unroll
    for (int g0 = 0; g0 < V; g0 += G) {
        float v[G];
#pragma unroll
        for (int i = 0; i < G; ++i) v[i] = acc[(g0 + i) / NT][(g0 + i) % NT];
        const float s = warp_reduce_scatter<G>(v, lane);
        if ((lane & ((32 >> LG) - 1)) == 0) {
            const int i = g0 + (lane >> (5 - LG));
            part[warp][i / NT][i % NT] = s;
        }
    }
}

// MAXT: the most tokens of a call (1 or kRouteTok).  The single-token
// instantiation keeps one accumulator per router row and none of the routing
// tail: B = 1 decode launches run it, with less code to fetch per CTA.
template <int PER, int MAXT>
__global__ void __launch_bounds__(256) route_gemv_kernel(const float *__restrict__ x, int T, int H,
                                                         const float *__restrict__ Wr,
                                                         const float *__restrict__ bias, int E,
                                                         float *logits, DecodeTail tail) {
    __shared__ float part[8][kRouteRows][kRouteTok];
    __shared__ int s_last;
    __shared__ int s_abort;
    __shared__ int s_nunits, s_npairs;
    extern __shared__ __align__(16) unsigned char rsm[];
    const RouteSmem L = route_smem(H, E);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t wl = wait_limit();
    const int e0 = blockIdx.x * kRouteRows;
    const int nr = min(kRouteRows, E - e0);
    const int hc = min(H, kRouteHC), nhc = (H + hc - 1) / hc;
    const uint32_t bar = smem_u32(rsm + L.bar);
    float *wr = reinterpret_cast<float *>(rsm + L.wr);  // [kRouteRows][hc]

    if (tid == 0) {
        mbar_init(bar, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint64_t pol = l2_evict_first();
    auto issue = [&](int c) {  // router columns [c*hc, c*hc + w) of the CTA's rows (thread 0)
        const int c0 = c * hc, w = min(hc, H - c0);
        mbar_arrive_expect_tx(bar, (uint32_t)(nr * w * 4));
        if (w == H) {
            bulk_g2s(smem_u32(wr), Wr + (size_t)e0 * H, (uint32_t)(nr * H * 4), bar, pol);
        } else {
            for (int r = 0; r < nr; ++r)
                bulk_g2s(smem_u32(wr + r * hc), Wr + (size_t)(e0 + r) * H + c0, (uint32_t)(w * 4), bar, pol);
        }
    };
    if (tid == 0) issue(0);  // router weights are read-only inputs: no need to wait for the stream
    MOEQ_TL(1, 0);
    pdl_trigger();
    pdl_wait();  // x (and the buffers written below) belong to earlier work on the stream
    MOEQ_TL(1, 1);

    int loaded = 0;
    bool ready = false, failed = false;
    uint32_t ph = 0;
    for (int t0 = 0; t0 < T && !failed; t0 += kRouteTok) {
        const int nt = min(kRouteTok, T - t0);
        float acc[kRouteRows][MAXT];
#pragma unroll
        for (int r = 0; r < kRouteRows; ++r)
#pragma unroll
            for (int t = 0; t < MAXT; ++t) acc[r][t] = 0.f;
        for (int c = 0; c < nhc; ++c) {
            if (loaded != c) {  // only when H > kRouteHC
                __syncthreads();
                if (tid == 0) issue(c);
                loaded = c;
                ready = false;
            }
            if (!ready) {
                const bool ok = mbar_wait(bar, ph & 1, &s_abort, wl);
                if (__syncthreads_or(!ok)) {
                    failed = true;
                    break;
                }
                ++ph;
                ready = true;
                MOEQ_TL(1, 2);
            }
            const int c0 = c * hc, w = min(hc, H - c0);
            const int ws = w / 8;  // multiple of 16
            const int hb = warp * ws, he = hb + ws;
            if (MAXT == 1 || nt == 1) route_accumulate<1, MAXT>(acc, wr, hc, nr, x, H, t0, c0, hb, he, lane, nt);
            else if (nt == 2) route_accumulate<2, MAXT>(acc, wr, hc, nr, x, H, t0, c0, hb, he, lane, nt);
            else if (nt <= 4) route_accumulate<4, MAXT>(acc, wr, hc, nr, x, H, t0, c0, hb, he, lane, nt);
            else if (nt <= 8) route_accumulate<8, MAXT>(acc, wr, hc, nr, x, H, t0, c0, hb, he, lane, nt);
            else route_accumulate<16, MAXT>(acc, wr, hc, nr, x, H, t0, c0, hb, he, lane, nt);
        }
        if (failed) break;
        if (MAXT == 1 || nt == 1) route_reduce<1, MAXT>(acc, part, warp, lane);
        else if (nt == 2) route_reduce<2, MAXT>(acc, part, warp, lane);
        else if (nt <= 4) route_reduce<4, MAXT>(acc, part, warp, lane);
        else if (nt <= 8) route_reduce<8, MAXT>(acc, part, warp, lane);
        else route_reduce<16, MAXT>(acc, part, warp, lane);
        __syncthreads();
        MOEQ_TL(1, 5);
        if (tid < kRouteRows * kRouteTok) {
            const int r = tid / kRouteTok, t = tid % kRouteTok;
            if (t < nt && r < nr) {
                float s = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) s += part[w8][r][t];
                s += bias ? bias[e0 + r] : 0.f;
                logits[(size_t)(t0 + t) * E + e0 + r] = s;
            }
        }
        __syncthreads();
    }
    // after the logits (the critical output): x is now in this SM's L1
    if (tail.mode > 0) {
        // y = residual ? x : 0, before any expert adds into it
        const size_t n = (size_t)T * H;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + tid; i < n; i += (size_t)gridDim.x * blockDim.x)
            tail.y[i] = tail.residual ? x[i] : 0.0f;
        // x quantised per 32-block for the expert kernel: warp j of CTA b takes
        // blocks b + j*gridDim, b + (j+8)*gridDim, ... (one block per CTA first)
        const int KBH = H / 32;
        for (int job = blockIdx.x + warp * gridDim.x; job < T * KBH; job += gridDim.x * 8) {
            const int t = job / KBH, b = job - t * KBH;
            const float v = x[(size_t)t * H + 32 * b + lane];
            const float sc = block_scale(warp_absmax(v));
            const int q = block_code(v, sc);
            tail.qx[(size_t)t * H + 32 * b + (tail.bits == 2 ? pack_pos2(lane) : lane)] = (int8_t)q;
            const int qs = warp_sum_int(q);
            if (lane == 0) {
                tail.sx[job] = sc;
                tail.xsum[job] = qs;
            }
        }
    }

    if (failed && tid == 0 && !ready) mbar_drain(bar, ph & 1, &s_abort);  // the copy in flight lands first
    MOEQ_TL(1, 3);
    if (MAXT == 1 || tail.mode < 2) return;  // the routing tail serves T >= 3 only

    // ---- the last CTA to finish ranks every token and groups the pairs by expert.
    // The barrier orders this CTA's logit and quantisation writes before thread
    // 0's device-scope fence (cumulative), which precedes its arrival.  A CTA
    // whose wait gave up still arrives (after flagging ctrl[3]), so the counter
    // is always completed and re-armed; the last CTA then publishes no work.
    __syncthreads();
    if (tid == 0) {
        if (failed) atomicExch(&tail.ctrl[3], 1);
        __threadfence();
        const int prev = atomicAdd(&tail.ctrl[0], 1);
        s_last = (prev == (int)gridDim.x - 1);
        s_nunits = 0;
        s_npairs = 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (__ldcg(&tail.ctrl[3])) {  // some CTA's logits are missing: no expert work this call
        if (tid == 0) {
            tail.ctrl[1] = 0;
            tail.ctrl[3] = 0;
            tail.ctrl[0] = 0;
        }
        return;
    }

    int(*s_sel)[kMaxK] = reinterpret_cast<int(*)[kMaxK]>(rsm + L.sel);
    float(*s_selw)[kMaxK] = reinterpret_cast<float(*)[kMaxK]>(rsm + L.selw);
    unsigned long long *s_mask = reinterpret_cast<unsigned long long *>(rsm + L.mask);  // bit t: token t picked e
    int *s_unit = reinterpret_cast<int *>(rsm + L.unit);
    int *s_pb = reinterpret_cast<int *>(rsm + L.pb);
    const int k = tail.k, P = T * k;
    for (int t = warp; t < T; t += 8)
        warp_topk<PER>(logits + (size_t)t * E, E, k, tail.idx + (size_t)t * k, tail.w + (size_t)t * k, s_sel[t],
                       s_selw[t]);
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) s_mask[s_sel[p / k][p % k]] = 0ull;
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) atomicOr(&s_mask[s_sel[p / k][p % k]], 1ull << (p / k));
    __syncthreads();
    // one unit per distinct expert, created by the pair of its first token; the
    // order of units (and of their pair ranges) is arbitrary -- every unit adds
    // into y independently
    for (int p = tid; p < P; p += blockDim.x) {
        const int t = p / k, e = s_sel[t][p - t * k];
        const unsigned long long m = s_mask[e];
        if (__ffsll((long long)m) - 1 != t) continue;
        const int n = __popcll(m);
        const int u = atomicAdd(&s_nunits, 1);
        const int pb = atomicAdd(&s_npairs, n);
        s_unit[e] = u;
        s_pb[e] = pb;
        *reinterpret_cast<int4 *>(&tail.units[u]) = make_int4(e, pb, n, 0);
    }
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int t = p / k, j = p - t * k, e = s_sel[t][j];
        const int r = __popcll(s_mask[e] & ((1ull << t) - 1ull));
        const int pos = s_pb[e] + r;
        tail.perm_tok[pos] = t;
        tail.perm_slot[pos] = j;
        tail.inv[p] = pos;
        if (r < kUnitTok) {
            tail.units[s_unit[e]].tok[r] = t;
            tail.units[s_unit[e]].w[r] = s_selw[t][j];
        }
    }
    if (tid == 0) {
        tail.ctrl[1] = s_nunits;
        tail.ctrl[0] = 0;  // re-arm the arrival counter for the next call
    }
    MOEQ_TL(1, 4);
}

}  // namespace moeq
