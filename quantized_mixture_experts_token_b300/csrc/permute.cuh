// permute.cuh -- deterministic token-to-expert grouping, and the work plan
// (active experts, 128-token tiles) the expert kernels run over.
//
// The pages' prompt path multiplies each expert once for all of a chunk's
// tokens that picked it ("Strata - the details", "Speed (measured)"), which
// needs the (token, slot) pairs grouped by expert.
#pragma once

#include "common.cuh"

namespace moeq {

// Single CTA, 1024 threads.  Pair p = (t, j) sets bit t of its expert's token
// bitmap; an expert's count is the popcount of its bitmap and the rank of
// token t inside it is the popcount of the bits below t.  Ranks therefore
// follow token order by construction (a stable counting sort) and never
// depend on the order in which atomics land.  k distinct experts per token
// make (e, t) unique.
__global__ void __launch_bounds__(1024) permute_kernel(const int32_t *__restrict__ idx, int T, int k, int E,
                                                       unsigned *masks /* [E][W] */, int *prefix /* [E][W] */,
                                                       int32_t *counts, int32_t *offsets, int32_t *perm_tok,
                                                       int32_t *perm_slot, int32_t *inv) {
    __shared__ int s_off[kMaxE];
    __shared__ int s_scan[33];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int W = (T + 31) / 32;
    const size_t nm = (size_t)E * W;
    for (size_t i = tid; i < nm; i += nt) masks[i] = 0u;
    __syncthreads();
    const int P = T * k;
    for (int p = tid; p < P; p += nt) {
        const int e = idx[p], t = p / k;
        if (e < 0 || e >= E) {
            set_status(MOEQ_STATUS_BAD_INDEX);
            inv[p] = -1;  // a rejected pair has no sorted position
            continue;
        }
        const unsigned bit = 1u << (t & 31);
        if (atomicOr(&masks[(size_t)e * W + (t >> 5)], bit) & bit)
            set_status(MOEQ_STATUS_BAD_INDEX);  // the same expert twice in one row
    }
    __syncthreads();
    for (int e = tid; e < E; e += nt) {
        int run = 0;
        for (int w = 0; w < W; ++w) {
            prefix[(size_t)e * W + w] = run;
            run += __popc(__ldcg(&masks[(size_t)e * W + w]));
        }
        counts[e] = run;
        s_off[e] = run;
    }
    __syncthreads();
    const int total = block_exclusive_scan(s_off, E, s_scan);
    for (int e = tid; e < E; e += nt) offsets[e] = s_off[e];
    if (tid == 0) offsets[E] = total;
    __syncthreads();
    for (int p = tid; p < P; p += nt) {
        const int e = idx[p], t = p / k, j = p - t * k;
        if (e < 0 || e >= E) continue;
        const size_t wi = (size_t)e * W + (t >> 5);
        const int pos = s_off[e] + __ldcg(&prefix[wi]) + __popc(__ldcg(&masks[wi]) & ((1u << (t & 31)) - 1u));
        perm_tok[pos] = t;
        perm_slot[pos] = j;
        inv[p] = pos;
    }
}

// ---------------------------------------------------------------- multi-CTA
// The same stable counting sort spread over the GPU, for large T.  Tokens are
// split into chunks of kPermChunkWords 32-token words.
//   permute_count_kernel   one CTA per chunk: the chunk's token bitmaps of
//                          every expert (shared-memory atomics), their
//                          prefix popcounts inside the chunk, and the chunk's
//                          count per expert;
//   permute_scan_kernel    one CTA: per-expert chunk bases (scan over chunks),
//                          counts, offsets (scan over experts);
//   permute_scatter_kernel one thread per pair: rank = chunk base + prefix of
//                          the words before it + popcount of the bits below.
constexpr int kPermChunkWords = 8;  // 256 tokens per chunk

__global__ void __launch_bounds__(256) permute_count_kernel(const int32_t *__restrict__ idx, int T, int k, int E,
                                                            unsigned *masks /* [E][W] */, int *wprefix /* [E][W] */,
                                                            int *chunk_count /* [NC][E] */) {
    __shared__ unsigned s_mask[kMaxE * kPermChunkWords];
    const int W = (T + 31) / 32, c = blockIdx.x;
    const int w0 = c * kPermChunkWords, nw = min(kPermChunkWords, W - w0);
    for (int i = threadIdx.x; i < E * kPermChunkWords; i += blockDim.x) s_mask[i] = 0u;
    __syncthreads();
    const int t0 = w0 * 32, t1 = min(T, (w0 + nw) * 32);
    for (int p = t0 * k + threadIdx.x; p < t1 * k; p += blockDim.x) {
        const int e = idx[p], t = p / k;
        if (e < 0 || e >= E) {
            set_status(MOEQ_STATUS_BAD_INDEX);
            continue;
        }
        const unsigned bit = 1u << (t & 31);
        if (atomicOr(&s_mask[e * kPermChunkWords + (t >> 5) - w0], bit) & bit)
            set_status(MOEQ_STATUS_BAD_INDEX);  // the same expert twice in one row
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int i = 0; i < nw; ++i) {
            const unsigned m = s_mask[e * kPermChunkWords + i];
            masks[(size_t)e * W + w0 + i] = m;
            wprefix[(size_t)e * W + w0 + i] = run;
            run += __popc(m);
        }
        chunk_count[(size_t)c * E + e] = run;
    }
}

__global__ void __launch_bounds__(1024) permute_scan_kernel(int NC, int E, const int *__restrict__ chunk_count,
                                                            int *chunk_base /* [NC][E] */, int32_t *counts,
                                                            int32_t *offsets) {
    __shared__ int s_off[kMaxE];
    __shared__ int s_scan[33];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int c = 0; c < NC; ++c) {
            chunk_base[(size_t)c * E + e] = run;
            run += chunk_count[(size_t)c * E + e];
        }
        counts[e] = run;
        s_off[e] = run;
    }
    __syncthreads();
    const int total = block_exclusive_scan(s_off, E, s_scan);
    for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = s_off[e];
    if (threadIdx.x == 0) offsets[E] = total;
}

__global__ void __launch_bounds__(256) permute_scatter_kernel(const int32_t *__restrict__ idx, int T, int k, int E,
                                                              const unsigned *__restrict__ masks,
                                                              const int *__restrict__ wprefix,
                                                              const int *__restrict__ chunk_base,
                                                              const int32_t *__restrict__ offsets, int32_t *perm_tok,
                                                              int32_t *perm_slot, int32_t *inv) {
    const int W = (T + 31) / 32, P = T * k;
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P; p += gridDim.x * blockDim.x) {
        const int e = idx[p], t = p / k, j = p - t * k;
        if (e < 0 || e >= E) {
            inv[p] = -1;  // rejected in permute_count_kernel
            continue;
        }
        const int w = t >> 5;
        const size_t wi = (size_t)e * W + w;
        const int pos = offsets[e] + chunk_base[(size_t)(w / kPermChunkWords) * E + e] + wprefix[wi] +
                        __popc(masks[wi] & ((1u << (t & 31)) - 1u));
        perm_tok[pos] = t;
        perm_slot[pos] = j;
        inv[p] = pos;
    }
}

// Work plan from offsets: the number of experts with at least one pair and
// their UnitRec records (for the decode expert kernel; units may be NULL), and
// two lists of (expert, first sorted position, rows) tiles, of up to tile_n
// and up to tile_n2 pairs (for the two tensor-core kernels; multiples of 16 in
// [kTileMin, kTileMax]), counted in ctrl[2] and ctrl[kCtrlTiles2].
constexpr int kTileMin = 64, kTileMax = 128;
constexpr int kCtrlTiles2 = 8;

struct Tile {
    int e, p0, n, pad;
};

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t *__restrict__ offsets, int E, int T, int *ctrl,
                                                    UnitRec *units, const int32_t *__restrict__ perm_tok,
                                                    const int32_t *__restrict__ perm_slot,
                                                    const float *__restrict__ w, int k, Tile *tiles, int tile_n,
                                                    Tile *tiles2, int tile_n2) {
    __shared__ int s_act[kMaxE];
    __shared__ int s_til[kMaxE];
    __shared__ int s_til2[kMaxE];
    __shared__ int s_scan[33];
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    const long long P = (long long)T * k;
    if (tid == 0) s_bad = (offsets[0] != 0 || offsets[E] < 0 || offsets[E] > P);
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        const int c = offsets[e + 1] - offsets[e];
        if (c < 0) s_bad = 1;
        s_act[e] = c > 0;
        s_til[e] = (c + tile_n - 1) / tile_n;
        s_til2[e] = (c + tile_n2 - 1) / tile_n2;
    }
    __syncthreads();
    if (s_bad) {  // offsets that are not a prefix sum over [0, T*k]: no work at all
        if (tid == 0) {
            set_status(MOEQ_STATUS_BAD_INDEX);
            ctrl[1] = 0;
            ctrl[2] = 0;
            ctrl[kCtrlTiles2] = 0;
        }
        return;
    }
    const int n_active = block_exclusive_scan(s_act, E, s_scan);
    const int n_tiles = block_exclusive_scan(s_til, E, s_scan);
    const int n_tiles2 = block_exclusive_scan(s_til2, E, s_scan);
    for (int e = tid; e < E; e += blockDim.x) {
        const int o = offsets[e], c = offsets[e + 1] - o;
        if (c > 0 && units) {
            UnitRec *r = units + s_act[e];
            *reinterpret_cast<int4 *>(r) = make_int4(e, o, c, 0);
            for (int i = 0; i < min(c, kUnitTok); ++i) {
                int t = perm_tok[o + i];
                const int j = perm_slot[o + i];
                float wv = 0.f;
                if (t < 0 || t >= T || j < 0 || j >= k) {  // no contribution from a bad pair
                    set_status(MOEQ_STATUS_BAD_INDEX);
                    t = 0;
                } else if (w) {
                    wv = w[(size_t)t * k + j];
                }
                r->tok[i] = t;
                r->w[i] = wv;
            }
        }
        for (int i = 0; i * tile_n < c; ++i) {
            Tile tl;
            tl.e = e;
            tl.p0 = o + i * tile_n;
            tl.n = min(tile_n, c - i * tile_n);
            tl.pad = 0;
            tiles[s_til[e] + i] = tl;
        }
        for (int i = 0; i * tile_n2 < c; ++i) {
            Tile tl;
            tl.e = e;
            tl.p0 = o + i * tile_n2;
            tl.n = min(tile_n2, c - i * tile_n2);
            tl.pad = 0;
            tiles2[s_til2[e] + i] = tl;
        }
    }
    if (tid == 0) {
        ctrl[1] = n_active;
        ctrl[2] = n_tiles;
        ctrl[kCtrlTiles2] = n_tiles2;
    }
}

// The trivial routing of a shared expert: every token is pair t of the single
// expert 0 with weight 1 (offsets {0, T}, perm_tok = identity, perm_slot = 0).
__global__ void shared_plan_kernel(int T, int32_t *__restrict__ offsets, int32_t *__restrict__ perm_tok,
                                   int32_t *__restrict__ perm_slot, float *__restrict__ w) {
    const int i0 = blockIdx.x * blockDim.x + threadIdx.x;
    if (i0 == 0) {
        offsets[0] = 0;
        offsets[1] = T;
    }
    for (int t = i0; t < T; t += gridDim.x * blockDim.x) {
        perm_tok[t] = t;
        perm_slot[t] = 0;
        w[t] = 1.0f;
    }
}

}  // namespace moeq
