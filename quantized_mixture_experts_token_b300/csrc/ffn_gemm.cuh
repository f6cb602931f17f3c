// ffn_gemm.cuh -- the experts for many tokens per expert (prompt chunks): a
// grouped GEMM on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// Prior art: the pages move their prompt experts from FP16-expanded weights to
// quantised MMQ kernels (0.1.13) and then to fused int8 tensor-core kernels
// (0.1.36) ("Strata - the details", "Speed (measured)").  sm_103a has no int8
// tcgen05 MMA, so the block products are formed on the fp16 path in a way that
// keeps them as exact as the int8 reading:
//   * A (weights, M = 128 rows of one expert matrix): level * s_w with level in
//     {-2,-1,0,1} and s_w fp16 -- exact in fp16;
//   * B (activations, N = up to 128 sorted tokens): v = q * s_a * 2^-e split
//     into fp16 hi + lo (hi + lo == v to ~2^-22), two MMAs into one fp32
//     accumulator, so the per-32-block activation scale is carried without an
//     epilogue per K-block;
//   * e is a per-row power of two, undone exactly in the epilogue.
//
// Kernel shape (one CTA per (128-row M tile, <=128-token N tile), 8 warps):
//   warps 0-3  producers: cp.async the raw 2-bit codes / fp16 scales of the A
//              tile and the gathered B rows into a 3-4 stage ring, then unpack
//              the codes into the 128B-swizzled K-major fp16 A tile;
//   warp 4     allocates TMEM and issues tcgen05.mma from one thread;
//   warps 4-7  epilogue: tcgen05.ld the accumulator (lane = M row), then
//              gate/up: h = silu(G) * U and int8 re-quantisation per 32 rows
//                       (one warp = one quantisation block), stored as q_h, s_h;
//              down:    D * 2^e, weighted by the routing weight and added into
//                       y (red.add), or stored per sorted pair.
// Every mbarrier wait is bounded; a wait that gives up records
// MOEQ_STATUS_WAIT_TIMEOUT, the CTA drains its copies and MMAs, frees TMEM
// and returns.
#pragma once

#include "async.cuh"
#include "permute.cuh"

namespace moeq {

constexpr int kGmM = 128;  // MMA M: weight rows per CTA
constexpr int kGmN = 128;  // max tokens per tile (MMA N)
constexpr int kGmK = 64;   // K per pipeline stage = one 128-byte swizzle row of fp16

struct GemmArgs {
    int T, H, I, E, k;
    const uint8_t *codes[3];
    const uint16_t *scales[3];
    const Tile *tiles;
    const int *ctrl;  // ctrl[2] = number of tiles
    const int32_t *perm_tok, *perm_slot;
    const float *w;
    const __half *bhi, *blo;  // B rows: x by token (gate/up) or h by sorted position (down)
    const int *brow_exp;      // their power-of-two exponents
    int8_t *qh;               // gate/up outputs [T*k, I]
    float *sh;                // [T*k, I/32]
    float *y, *out_sorted;    // down outputs
};

template <bool GATEUP, int BITS>
struct GemmCfg {
    static constexpr int NA = GATEUP ? 2 : 1;
    static constexpr int STAGES = GATEUP ? 3 : 4;
    static constexpr int BPB = 4 * BITS;
    static constexpr int A_BYTES = kGmM * kGmK * 2;  // 16 KB
    static constexpr int B_BYTES = kGmN * kGmK * 2;  // 16 KB (hi or lo)
    static constexpr int TILE_BYTES = NA * A_BYTES + 2 * B_BYTES;
    static constexpr int RAW_CODES = NA * 2 * kGmM * BPB;  // 2 K-blocks per stage
    static constexpr int RAW_SCALES = NA * 2 * kGmM * 2;
    static constexpr int RAW_BYTES = RAW_CODES + RAW_SCALES;
    static constexpr int TMEM_COLS = 256;
    static constexpr size_t SMEM = 1024 /*align slack*/ + (size_t)STAGES * (TILE_BYTES + RAW_BYTES) + 2048;
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Shared-memory matrix descriptor (tcgen05): K-major, 128-byte swizzle, 8-row
// core groups 1024 bytes apart.  Fields: start address >> 4 (bits 0-13),
// leading byte offset >> 4 (16-29, unused for swizzled K-major: 1), stride
// byte offset >> 4 (32-45), descriptor version 1 (bits 46-47), swizzle mode
// 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B fp16 (bits 7-9, 10-12 = 0), both K-major, N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
__device__ __forceinline__ uint32_t f16_idesc(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128B-swizzled,
// K-major tile whose rows are 128 bytes long.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// fp16 pair {lut[c0], lut[c1]} for the codes in bits 0-1 / 8-9 of `two`.
__device__ __forceinline__ uint32_t lut_pair(uint32_t lut_lo, uint32_t lut_hi, uint32_t two) {
    return __byte_perm(lut_lo, lut_hi, two * 34u + 0x1010u);
}

// ------------------------------------------------------------------ kernel

template <bool GATEUP, int BITS>
__global__ void __launch_bounds__(256, 1) ffn_gemm_kernel(GemmArgs a) {
    using C = GemmCfg<GATEUP, BITS>;
    const int MT = (GATEUP ? a.I : a.H) / kGmM;
    const int tile_idx = blockIdx.x / MT, mt = blockIdx.x % MT;
    if (tile_idx >= a.ctrl[2]) return;
    const Tile tile = a.tiles[tile_idx];
    const int e = tile.e, p0 = tile.p0, nval = tile.n;
    const int nround = (nval + 15) & ~15;
    const int K = GATEUP ? a.H : a.I;
    const int KB = K / 32, nk = K / kGmK;
    const int NR = GATEUP ? a.I : a.H;  // rows of each A matrix
    const int m0 = mt * kGmM;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *tiles_base = smem;                                    // STAGES x TILE_BYTES
    unsigned char *raw_base = smem + (size_t)C::STAGES * C::TILE_BYTES;  // STAGES x RAW_BYTES
    unsigned char *misc = raw_base + (size_t)C::STAGES * C::RAW_BYTES;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(misc);
    uint64_t *empty_bar = full_bar + C::STAGES;
    uint64_t *acc_bar = empty_bar + C::STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_exp = reinterpret_cast<int *>(misc + 256);    // [kGmN] B-row exponents
    int *s_tok = s_exp + kGmN;                            // [kGmN] token of each B row
    float *s_wt = reinterpret_cast<float *>(s_tok + kGmN);  // [kGmN] routing weight of each row

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 128);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(acc_bar), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid < kGmN) {
        const int j = min(tid, nval - 1);
        const int p = p0 + j;
        const int t = a.perm_tok[p];
        s_tok[tid] = t;
        s_exp[tid] = a.brow_exp[GATEUP ? t : p];
        s_wt[tid] = (!GATEUP && a.w) ? a.w[(size_t)t * a.k + a.perm_slot[p]] : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        // ------------------------------------------------------ producers
        const int r = tid;  // A row of this thread
        const uint8_t *cptr[2];
        const uint16_t *sptr[2];
#pragma unroll
        for (int m = 0; m < C::NA; ++m) {
            const int mat = GATEUP ? m : 2;
            cptr[m] = a.codes[mat] + ((size_t)e * KB * NR + m0 + r) * C::BPB;
            sptr[m] = a.scales[mat] + (size_t)e * KB * NR + m0 + (r & ~1);
        }
        // B rows this thread copies: chunk c, rows rb + 16 i
        const int bc = tid & 7, rb = tid >> 3;
        auto issue = [&](int ks) {
            const int s = ks % C::STAGES;
            unsigned char *tb = tiles_base + (size_t)s * C::TILE_BYTES;
            unsigned char *rw = raw_base + (size_t)s * C::RAW_BYTES;
            const uint32_t bhi_s = smem_u32(tb + C::NA * C::A_BYTES);
            const uint32_t blo_s = bhi_s + C::B_BYTES;
            const int k0 = ks * kGmK;
            for (int i = 0; i < 8; ++i) {
                const int row = rb + 16 * i;
                if (row >= nround) break;
                const int src_row = GATEUP ? s_tok[row] : p0 + min(row, nval - 1);
                const size_t off = (size_t)src_row * K + k0 + 8 * bc;
                const uint32_t so = sw128_off(row, bc);
                cp_async_16(bhi_s + so, a.bhi + off);
                cp_async_16(blo_s + so, a.blo + off);
            }
#pragma unroll
            for (int m = 0; m < C::NA; ++m)
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int kb = 2 * ks + b;
                    const uint32_t cdst = smem_u32(rw + ((m * 2 + b) * kGmM + r) * C::BPB);
                    const uint8_t *csrc = cptr[m] + (size_t)kb * NR * C::BPB;
                    if (BITS == 2) {
                        cp_async_8(cdst, csrc);
                    } else {
                        cp_async_4(cdst, csrc);
                        cp_async_4(cdst + 4, csrc + 4);
                        cp_async_4(cdst + 8, csrc + 8);
                    }
                    const uint32_t sdst = smem_u32(rw + C::RAW_CODES + ((m * 2 + b) * kGmM + (r & ~1)) * 2);
                    cp_async_4(sdst, sptr[m] + (size_t)kb * NR);
                }
        };
        // prologue: steps 0 .. STAGES-2 in flight
        for (int ks = 0; ks < C::STAGES - 1; ++ks) {
            if (ks < nk) issue(ks);
            cp_async_commit();
        }
        bool ok = true;
        for (int ks = 0; ks < nk && ok; ++ks) {
            const int s = ks % C::STAGES;
            cp_async_wait<C::STAGES - 2>();  // this thread's copies of step ks have landed
            __syncwarp();                    // ... and those of the lane sharing its scale word
            unsigned char *tb = tiles_base + (size_t)s * C::TILE_BYTES;
            const unsigned char *rw = raw_base + (size_t)s * C::RAW_BYTES;
#pragma unroll
            for (int m = 0; m < C::NA; ++m) {
                const uint32_t at = smem_u32(tb + m * C::A_BYTES);
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const uint16_t sbits = *reinterpret_cast<const uint16_t *>(rw + C::RAW_CODES + ((m * 2 + b) * kGmM + r) * 2);
                    const __half sc = __ushort_as_half(sbits);
                    if (BITS == 2) {
                        const uint2 cw = *reinterpret_cast<const uint2 *>(rw + ((m * 2 + b) * kGmM + r) * C::BPB);
                        const __half m2 = __hmul(sc, __float2half(-2.0f)), m1 = __hneg(sc);
                        const uint32_t lut_lo = (uint32_t)__half_as_ushort(m2) | ((uint32_t)__half_as_ushort(m1) << 16);
                        const uint32_t lut_hi = (uint32_t)__half_as_ushort(sc) << 16;  // {0, s}
#pragma unroll
                        for (int c = 0; c < 4; ++c) {  // 16-byte chunk = 8 elements = 2 code bytes
                            const uint32_t word = c < 2 ? cw.x : cw.y;
                            const uint32_t d0 = (word >> (16 * (c & 1))) & 0xffu;
                            const uint32_t d1 = (word >> (16 * (c & 1) + 8)) & 0xffu;
                            const uint32_t q0 = lut_pair(lut_lo, lut_hi, (d0 & 3u) | ((d0 & 0xCu) << 6));
                            const uint32_t q1 = lut_pair(lut_lo, lut_hi, ((d0 >> 4) & 3u) | ((d0 & 0xC0u) << 2));
                            const uint32_t q2 = lut_pair(lut_lo, lut_hi, (d1 & 3u) | ((d1 & 0xCu) << 6));
                            const uint32_t q3 = lut_pair(lut_lo, lut_hi, ((d1 >> 4) & 3u) | ((d1 & 0xC0u) << 2));
                            st_shared_v4(at + sw128_off(r, 4 * b + c), q0, q1, q2, q3);
                        }
                    } else {
                        // 3-bit levels -4..3 times s: +-3s need not be exact in fp16 (documented;
                        // the GEMV path is exact for 3-bit)
                        const uint32_t *cw = reinterpret_cast<const uint32_t *>(rw + ((m * 2 + b) * kGmM + r) * C::BPB);
                        const uint32_t w0 = cw[0], w1 = cw[1], w2 = cw[2];
                        const float sf = __half2float(sc);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t q[4];
#pragma unroll
                            for (int h2 = 0; h2 < 4; ++h2) {
                                __half hv[2];
#pragma unroll
                                for (int u = 0; u < 2; ++u) {
                                    const int i = 8 * c + 2 * h2 + u, off = 3 * i, wi = off >> 5, sh = off & 31;
                                    const uint32_t lo = wi == 0 ? w0 : (wi == 1 ? w1 : w2);
                                    const uint32_t hi = wi == 0 ? w1 : (wi == 1 ? w2 : 0u);
                                    const int code = (int)(__funnelshift_r(lo, hi, sh) & 7u);
                                    hv[u] = __float2half_rn((float)(code - 4) * sf);
                                }
                                q[h2] = (uint32_t)__half_as_ushort(hv[0]) | ((uint32_t)__half_as_ushort(hv[1]) << 16);
                            }
                            st_shared_v4(at + sw128_off(r, 4 * b + c), q[0], q[1], q[2], q[3]);
                        }
                    }
                }
            }
            fence_proxy_async();
            mbar_arrive(smem_u32(&full_bar[s]));
            // refill the stage step ks-1 used with step ks + STAGES - 1 once its MMAs are done
            const int nx = ks + C::STAGES - 1;
            if (nx < nk) {
                if (ks >= 1) {
                    const int ps = (ks - 1) % C::STAGES;
                    ok = mbar_wait(smem_u32(&empty_bar[ps]), ((ks - 1) / C::STAGES) & 1, abort_flag);
                }
                ok = __all_sync(0xffffffffu, ok);
                __syncwarp();
                if (ok) issue(nx);
            }
            cp_async_commit();
        }
        cp_async_wait_all();
    } else if (warp == 4) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = f16_idesc(kGmM, nround);
            bool ok = true;
            for (int ks = 0; ks < nk; ++ks) {
                const int s = ks % C::STAGES;
                if (!mbar_wait(smem_u32(&full_bar[s]), (ks / C::STAGES) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tb = smem_u32(tiles_base + (size_t)s * C::TILE_BYTES);
                const uint32_t bhi_s = tb + C::NA * C::A_BYTES, blo_s = bhi_s + C::B_BYTES;
#pragma unroll
                for (int kk = 0; kk < kGmK / 16; ++kk) {
                    const uint64_t bh = sw128_desc(bhi_s + 32 * kk), bl = sw128_desc(blo_s + 32 * kk);
#pragma unroll
                    for (int m = 0; m < C::NA; ++m) {
                        const uint64_t ad = sw128_desc(tb + m * C::A_BYTES + 32 * kk);
                        const uint32_t acc_col = tmem + (uint32_t)(m * kGmN);
                        mma_f16(acc_col, ad, bh, idesc, (ks | kk) != 0);
                        mma_f16(acc_col, ad, bl, idesc, 1u);
                    }
                }
                mma_commit(smem_u32(&empty_bar[s]));
            }
            (void)ok;
            mma_commit(smem_u32(acc_bar));  // completes when every MMA issued above is done
        }
        __syncwarp();
    }

    if (warp >= 4) {
        // ------------------------------------------------------ epilogue
        // the issuer always commits acc_bar, so this wait also drains in-flight MMAs
        bool ok = mbar_wait(smem_u32(acc_bar), 0, abort_flag, false);
        ok = __all_sync(0xffffffffu, ok && !*abort_flag);
        tc_fence_after();
        if (ok) {
            const int ew = warp - 4;
            const int row = 32 * ew + lane;  // accumulator lane = A row
            const uint32_t tl = tmem + ((uint32_t)(32 * ew) << 16);
            for (int c0 = 0; c0 < nround; c0 += 16) {
                float acc0[16];
                tmem_ld16(tl + (uint32_t)c0, acc0);
                if (GATEUP) {
                    float acc1[16];
                    tmem_ld16(tl + (uint32_t)(kGmN + c0), acc1);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = c0 + jj;
                        if (j >= nval) break;
                        const float sc = exp2i(s_exp[j]);
                        const float G = acc0[jj] * sc, U = acc1[jj] * sc;
                        const float h = __fdiv_rn(G, 1.0f + expf(-G)) * U;
                        const float s = block_scale(warp_absmax(h));
                        const int q = block_code(h, s);
                        const size_t p = (size_t)(p0 + j);
                        a.qh[p * a.I + m0 + row] = (int8_t)q;
                        if (lane == 0) a.sh[p * (a.I / 32) + (m0 + row) / 32] = s;
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = c0 + jj;
                        if (j >= nval) break;
                        const float D = acc0[jj] * exp2i(s_exp[j]);
                        if (a.y) atomicAdd(a.y + (size_t)s_tok[j] * a.H + m0 + row, s_wt[j] * D);
                        if (a.out_sorted) a.out_sorted[(size_t)(p0 + j) * a.H + m0 + row] = D;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
    }
}

}  // namespace moeq
