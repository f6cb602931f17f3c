// ffn_mma8.cuh -- the experts for many tokens per expert on the warp-level
// int8 tensor path (mma.sync m16n8k32, s8 x s8 -> s32), with every 32-block
// product an exact integer dot scaled by its two block scales in fp32
// registers: the exact-block reading of the block format, on the int8 MMAs that
// the pages' fused prompt-expert kernels use ("Strata - the details", "Speed
// (measured)": 0.1.13 quantised-activation MMQ kernels, 0.1.36 fused int8
// tensor-core prompt-expert kernels).
//
// sm_103a has no int8 tcgen05 MMA, so this path runs on the legacy warp-level
// tensor instructions.  It is the measured comparison point for the tcgen05
// grouped GEMM (ffn_gemm.cuh), selected with MOEQ_MODE_GEMM_S8; the automatic
// mode never picks it.
//
// Work item = (tile of <= 64 sorted pairs of one expert, block of weight rows):
//   gate/up: 64 rows of gate and the same 64 rows of up; warp w holds rows
//            16w .. 16w + 15 of both, so SwiGLU needs no exchange, and the
//            int8 re-quantisation of h per 32 rows goes through shared memory;
//   down:    128 rows of W_down; warp w holds rows 32w .. 32w + 31.  w * D is
//            added into y with vector reductions, D stored per sorted pair.
// Operands stream through a three-stage cp.async ring of K = 128 (4 blocks):
// the tile's int8 activation rows (zero-filled past the tile's pairs), their
// block scales, and the weight codes and scales of the item's rows.
#pragma once

#include "async.cuh"
#include "permute.cuh"

namespace moeq {

constexpr int kM8Tile = 64;                  // sorted pairs per tile: 8 MMA n8 tiles
constexpr int kM8KS = 4;                     // 32-blocks per pipeline stage
constexpr int kM8Stages = 3;
constexpr int kM8Threads = 128;
constexpr int kM8XRow = kM8KS * 32 + 16;     // activation row in shared memory (16 B pad: no ldmatrix bank conflicts)

struct Mma8Args {
    int T, H, I, E, k;
    const uint8_t *codes[3];
    const uint16_t *scales[3];
    const Tile *tiles;
    const int *ntiles;  // number of tiles (written by the plan kernel)
    const int32_t *perm_tok, *perm_slot;
    const float *w;
    // int8 activation rows and their 32-block scales: x per token [T, H]
    // (gate/up) or h per sorted pair [T*k, I] (down)
    const int8_t *aq;
    const float *as;
    int8_t *qh;  // gate/up outputs [T*k, I], [T*k, I/32]
    float *sh;
    float *y, *out_sorted;  // down outputs
};

template <bool GATEUP, int BITS>
struct Mma8Cfg {
    static constexpr int NA = GATEUP ? 2 : 1;     // weight matrices per item
    static constexpr int MTW = GATEUP ? 1 : 2;    // m16 tiles per warp and matrix
    static constexpr int ROWS = 4 * 16 * MTW;     // weight rows per item
    static constexpr int BPB = 4 * BITS;          // code bytes per row and 32-block
    static constexpr int X_BYTES = kM8Tile * kM8XRow;
    static constexpr int XS_BYTES = kM8Tile * kM8KS * 4;
    static constexpr int WC_BYTES = NA * kM8KS * ROWS * BPB;
    static constexpr int WS_BYTES = NA * kM8KS * ROWS * 2;
    static constexpr int STAGE_BYTES = X_BYTES + XS_BYTES + WC_BYTES + WS_BYTES;
    static constexpr int EPI_LD = ROWS + 4;       // staging row (floats): conflict-free writes by (token, row)
    static constexpr int EPI_BYTES = kM8Tile * EPI_LD * 4;
    static constexpr int SMEM = kM8Stages * STAGE_BYTES + EPI_BYTES;
    static_assert(STAGE_BYTES % 16 == 0 && (ROWS * BPB) % 16 == 0 && (ROWS * 2) % 16 == 0, "16-byte copies");
};

// ------------------------------------------------------------ PTX helpers

// 16-byte global -> shared copy; src_bytes = 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// d = A (16 x 32 s8, row) * B (32 x 8 s8, col), s32, from a zero accumulator.
__device__ __forceinline__ void mma_s8_16832(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
}

// Four 2-bit codes (bits 2i of `x`, element i) -> four int8 levels code - 2 (byte i).
__device__ __forceinline__ uint32_t levels2(uint32_t x) {
    const uint32_t u = x | (x << 12);
    const uint32_t t = (u | (u << 6)) & 0x03030303u;  // code i in byte i
    return (t + 0x7E7E7E7Eu) ^ 0x80808080u;           // per byte: code + 126 < 256, then flip to code - 2
}

// Four 3-bit codes (bits 3i of `v`, element i) -> four int8 levels code - 4.
__device__ __forceinline__ uint32_t levels3(uint32_t v) {
    const uint32_t t = (v & 7u) | ((v << 5) & 0x700u) | ((v << 10) & 0x70000u) | ((v << 15) & 0x7000000u);
    return (t + 0x7C7C7C7Cu) ^ 0x80808080u;
}

// A fragment word: the four levels of `row` (its code bytes at `row_codes` for
// one 32-block) at K positions k0 .. k0 + 3 (k0 a multiple of 4).
template <int BITS>
__device__ __forceinline__ uint32_t a_word(const unsigned char *row_codes, int k0) {
    if (BITS == 2) return levels2(row_codes[k0 >> 2]);
    const int off = 3 * k0, wi = off >> 5, sh = off & 31;
    const uint32_t *w32 = reinterpret_cast<const uint32_t *>(row_codes);
    const uint32_t lo = w32[wi], hi = sh > 20 ? w32[wi + 1] : 0u;  // 12 bits from bit `off`
    return levels3(__funnelshift_r(lo, hi, sh) & 0xFFFu);
}

// ------------------------------------------------------------------ kernel

// Persistent: CTA c walks the items q = c, c + gridDim.x, ...; item q covers
// tile q / MT and weight rows (q % MT) * ROWS ...
template <bool GATEUP, int BITS>
__global__ void __launch_bounds__(kM8Threads) ffn_mma8_kernel(const __grid_constant__ Mma8Args a) {
    using C = Mma8Cfg<GATEUP, BITS>;
    constexpr int NA = C::NA, MTW = C::MTW, ROWS = C::ROWS, BPB = C::BPB, NF = NA * MTW;
    const int K = GATEUP ? a.H : a.I;   // reduction length
    const int NR = GATEUP ? a.I : a.H;  // rows of each weight matrix
    const int KB = K / 32, nst = K / (32 * kM8KS), MT = NR / ROWS;
    const int n_items = *a.ntiles * MT;

    extern __shared__ __align__(16) unsigned char sm8[];
    float *stage_out = reinterpret_cast<float *>(sm8 + kM8Stages * C::STAGE_BYTES);
    __shared__ int s_src[kM8Tile];  // source activation row of each tile column (-1: none)
    __shared__ int s_tok[kM8Tile];
    __shared__ float s_w[kM8Tile];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;

    for (int q = blockIdx.x; q < n_items; q += gridDim.x) {
        const Tile tl = a.tiles[q / MT];
        const int m0 = (q % MT) * ROWS, n = tl.n;
        if (tid < kM8Tile) {
            int src = -1, tok = 0;
            float wv = 0.f;
            if (tid < n) {
                const int p = tl.p0 + tid;
                const int t = a.perm_tok[p], js = a.perm_slot[p];
                if (t < 0 || t >= a.T || js < 0 || js >= a.k) {  // a caller's bad permutation: no contribution
                    set_status(MOEQ_STATUS_BAD_INDEX);
                } else {
                    src = GATEUP ? t : p;
                    tok = t;
                    if (!GATEUP && a.w) wv = a.w[(size_t)t * a.k + js];
                }
            }
            s_src[tid] = src;
            s_tok[tid] = tok;
            s_w[tid] = wv;
        }
        __syncthreads();

        auto load = [&](int st) {
            unsigned char *base = sm8 + (st % kM8Stages) * C::STAGE_BYTES;
            const int kb0 = st * kM8KS;
            for (int c = tid; c < kM8Tile * 8; c += kM8Threads) {  // activation rows: 8 x 16 B each
                const int r = c >> 3, ch = c & 7, src = s_src[r];
                cp_async16(smem_u32(base + r * kM8XRow + ch * 16), a.aq + (size_t)(src < 0 ? 0 : src) * K + kb0 * 32 + ch * 16,
                           src < 0 ? 0u : 16u);
            }
            for (int r = tid; r < kM8Tile; r += kM8Threads) {  // their scales of the stage's 4 blocks
                const int src = s_src[r];
                cp_async16(smem_u32(base + C::X_BYTES + r * 16), a.as + (size_t)(src < 0 ? 0 : src) * KB + kb0,
                           src < 0 ? 0u : 16u);
            }
            constexpr int CCH = ROWS * BPB / 16, SCH = ROWS * 2 / 16;
            for (int c = tid; c < NA * kM8KS * CCH; c += kM8Threads) {  // codes: [matrix][block][row][BPB]
                const int mb = c / CCH, ch = c % CCH, m = mb / kM8KS, b = mb % kM8KS;
                const uint8_t *src = a.codes[GATEUP ? m : 2] + (((size_t)tl.e * KB + kb0 + b) * NR + m0) * BPB;
                cp_async16(smem_u32(base + C::X_BYTES + C::XS_BYTES + mb * ROWS * BPB + ch * 16), src + ch * 16, 16u);
            }
            for (int c = tid; c < NA * kM8KS * SCH; c += kM8Threads) {  // scales: [matrix][block][row]
                const int mb = c / SCH, ch = c % SCH, m = mb / kM8KS, b = mb % kM8KS;
                const uint16_t *src = a.scales[GATEUP ? m : 2] + ((size_t)tl.e * KB + kb0 + b) * NR + m0;
                cp_async16(smem_u32(base + C::X_BYTES + C::XS_BYTES + C::WC_BYTES + mb * ROWS * 2 + ch * 16),
                           src + ch * 8, 16u);
            }
        };

        float acc[NF][8][4];
#pragma unroll
        for (int f = 0; f < NF; ++f)
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[f][j][i] = 0.f;
        const int n8 = (n + 7) >> 3;  // live n8 tiles (warp-uniform)

        load(0);
        cp_async_commit();
        if (nst > 1) load(1);
        cp_async_commit();
        for (int st = 0; st < nst; ++st) {
            cp_async_wait<1>();  // this thread's copies of stage st have landed
            __syncthreads();     // everyone's have; the slot of stage st - 1 is free
            if (st + 2 < nst) load(st + 2);
            cp_async_commit();
            const unsigned char *base = sm8 + (st % kM8Stages) * C::STAGE_BYTES;
            const float *xs = reinterpret_cast<const float *>(base + C::X_BYTES);
            const unsigned char *wc = base + C::X_BYTES + C::XS_BYTES;
            const __half *wsc = reinterpret_cast<const __half *>(wc + C::WC_BYTES);
#pragma unroll
            for (int b = 0; b < kM8KS; ++b) {
                uint32_t af[NF][4];
                float sw[NF][2];
#pragma unroll
                for (int f = 0; f < NF; ++f) {
                    const int m = f / MTW, mt = f % MTW;
                    const int r0 = 16 * (warp * MTW + mt) + gid;
                    const unsigned char *c0 = wc + (m * kM8KS + b) * ROWS * BPB + r0 * BPB;
                    const unsigned char *c1 = c0 + 8 * BPB;
                    af[f][0] = a_word<BITS>(c0, 4 * tig);
                    af[f][1] = a_word<BITS>(c1, 4 * tig);
                    af[f][2] = a_word<BITS>(c0, 16 + 4 * tig);
                    af[f][3] = a_word<BITS>(c1, 16 + 4 * tig);
                    const __half *sc = wsc + (m * kM8KS + b) * ROWS + r0;
                    sw[f][0] = __half2float(sc[0]);
                    sw[f][1] = __half2float(sc[8]);
                }
#pragma unroll
                for (int jp = 0; jp < 4; ++jp) {  // n8 tiles 2 jp, 2 jp + 1
                    if (2 * jp >= n8) break;
                    uint32_t bf[4];
                    {
                        const int mat = lane >> 3;  // ldmatrix: lanes 8i .. 8i + 7 address the rows of matrix i
                        const int tok = (2 * jp + (mat >> 1)) * 8 + (lane & 7);
                        ldmatrix_x4(smem_u32(base + tok * kM8XRow + b * 32 + (mat & 1) * 16), bf[0], bf[1], bf[2], bf[3]);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = 2 * jp + h, c0 = 8 * j + 2 * tig;
                        if (j >= n8) break;
                        const float sa0 = xs[c0 * kM8KS + b], sa1 = xs[(c0 + 1) * kM8KS + b];
#pragma unroll
                        for (int f = 0; f < NF; ++f) {
                            int d[4];
                            mma_s8_16832(d, af[f], bf[2 * h], bf[2 * h + 1]);
                            acc[f][j][0] = fmaf((float)d[0], sw[f][0] * sa0, acc[f][j][0]);
                            acc[f][j][1] = fmaf((float)d[1], sw[f][0] * sa1, acc[f][j][1]);
                            acc[f][j][2] = fmaf((float)d[2], sw[f][1] * sa0, acc[f][j][2]);
                            acc[f][j][3] = fmaf((float)d[3], sw[f][1] * sa1, acc[f][j][3]);
                        }
                    }
                }
            }
        }

        // ------------------------------------------------------ epilogue
        // accumulator (f, j, i): row 16 (warp MTW + f % MTW) + gid + 8 (i >> 1),
        // tile column 8 j + 2 tig + (i & 1)
        if (GATEUP) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j >= n8) break;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float Gv = acc[0][j][i], Uv = acc[1][j][i];
                    const float h = __fdiv_rn(Gv, 1.0f + expf(-Gv)) * Uv;
                    stage_out[(8 * j + 2 * tig + (i & 1)) * C::EPI_LD + 16 * warp + gid + 8 * (i >> 1)] = h;
                }
            }
            __syncthreads();
            // int8 re-quantisation per (pair, 32 rows): one warp per block, lane = row
            constexpr int QB = ROWS / 32;
            for (int pr = warp; pr < n * QB; pr += kM8Threads / 32) {
                const int c = pr / QB, qb = pr % QB;
                if (s_src[c] < 0) continue;
                const float h = stage_out[c * C::EPI_LD + 32 * qb + lane];
                const float s = block_scale(warp_absmax(h));
                const int code = block_code(h, s);
                const size_t p = (size_t)(tl.p0 + c);
                a.qh[p * a.I + m0 + 32 * qb + lane] = (int8_t)code;
                if (lane == 0) a.sh[p * (a.I / 32) + (m0 >> 5) + qb] = s;
            }
        } else {
#pragma unroll
            for (int f = 0; f < NF; ++f)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j >= n8) break;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        stage_out[(8 * j + 2 * tig + (i & 1)) * C::EPI_LD + 16 * (warp * MTW + f) + gid + 8 * (i >> 1)] =
                            acc[f][j][i];
                }
            __syncthreads();
            // one warp per pair: lane = 4 consecutive rows
            for (int c = warp; c < n; c += kM8Threads / 32) {
                if (s_src[c] < 0) continue;
                const float4 D = *reinterpret_cast<const float4 *>(stage_out + c * C::EPI_LD + 4 * lane);
                if (a.out_sorted)
                    *reinterpret_cast<float4 *>(a.out_sorted + (size_t)(tl.p0 + c) * a.H + m0 + 4 * lane) = D;
                if (a.y) {
                    const float wv = s_w[c];
                    red_add_v4(a.y + (size_t)s_tok[c] * a.H + m0 + 4 * lane, wv * D.x, wv * D.y, wv * D.z, wv * D.w);
                }
            }
        }
        __syncthreads();  // the tables and the staging area are reused by the next item
    }
}

}  // namespace moeq
