// ffn_gemm.cuh -- the experts for many tokens per expert (prompt chunks): a
// grouped GEMM on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// Prior art: the pages move their prompt experts from FP16-expanded weights to
// quantised MMQ kernels (0.1.13) and then to fused int8 tensor-core kernels
// (0.1.36) ("Strata - the details", "Speed (measured)").  sm_103a has no int8
// tcgen05 MMA, so the block products are formed on the fp16 path in a way that
// keeps them as exact as the int8 reading:
//   * A (weights, M = 128 rows of one expert matrix): level * s_w with s_w
//     fp16.  2-bit levels {-2,-1,0,1} make it exact in fp16.  3-bit levels
//     reach +-3, whose product needs up to 13 significant bits, so the 3-bit
//     panel is split into fp16 hi + lo (lo exact: at most 2 significant bits)
//     and each product takes a third MMA, A_lo * B_hi (A_lo * B_lo, ~2^-22
//     relative, is dropped like the rest of the B split's residue);
//   * B (activations, N = up to 128 sorted tokens): v = q * s_a * 2^-e split
//     into fp16 hi + lo (hi + lo == v to ~2^-22), two MMAs into one fp32
//     accumulator, so the per-32-block activation scale is carried without an
//     epilogue per K-block;
//   * e is a per-row power of two, undone exactly in the epilogue.
//
// Work item = (tile of <= 128 sorted pairs of one expert, 128-row block of its
// weight matrix); the epilogue reads the accumulator (lane = weight row):
//   gate/up: h = silu(G) * U and int8 re-quantisation per 32 rows (one warp =
//            one quantisation block), stored as q_h, s_h;
//   down:    D * 2^e, weighted by the routing weight and added into y
//            (fp32 atomics), or stored per sorted pair.
// The kernel is persistent and warp-specialised (see ffn_gemm_kernel).
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
    // B operand image (fp16, see split_rows_kernel): [K/64][hi, lo][bimg_rows][64],
    // rows = sorted pair positions, chunks pre-swizzled per tile; x of the pair's
    // token (gate/up) or its h (down)
    const __half *bimg;
    long long bimg_rows;
    const int *brow_exp;  // power-of-two exponents of the B rows, per sorted pair
    int8_t *qh;               // gate/up outputs [T*k, I]
    float *sh;                // [T*k, I/32]
    float *y, *out_sorted;    // down outputs
};

// ------------------------------------------------------------ PTX helpers

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

// Bulk reduction of `bytes` of fp32 values from shared memory into global
// memory (dst[i] += src[i]), tracked by this thread's bulk async-group.
__device__ __forceinline__ void bulk_reduce_add_f32(float *gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 accumulator columns of this thread's TMEM lane.  The load
// and its wait are one asm statement, so no use of the destination registers
// can be scheduled before the asynchronous load has completed.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
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
struct GemmCfg {
    static constexpr int NA = GATEUP ? 2 : 1;  // weight matrices per work item (gate + up, or down)
    static constexpr int BPB = 4 * BITS;
    // operand ring, K = 64 per stage (MOEQ_GEMM_STAGES overrides the depth at build time)
#if defined(MOEQ_GEMM_STAGES_GU) && defined(MOEQ_GEMM_STAGES_DN)
    static constexpr int STAGES = GATEUP ? MOEQ_GEMM_STAGES_GU : MOEQ_GEMM_STAGES_DN;
#elif defined(MOEQ_GEMM_STAGES)
    static constexpr int STAGES = MOEQ_GEMM_STAGES;
#else
    static constexpr int STAGES = 2;
#endif
    static constexpr int RSTAGES = (GATEUP && BITS == 3) ? 4 : 6;  // raw-code ring (runs further ahead)
    static constexpr int A_BYTES = kGmM * kGmK * 2;                // fp16 weight tile
    static constexpr int NAT = BITS == 3 ? 2 : 1;                  // weight tiles per matrix: hi (, lo)
    static constexpr int B_BYTES = kGmN * kGmK * 2;                // fp16 activation tile (hi or lo)
    static constexpr int SLOT_BYTES = NAT * NA * A_BYTES + 2 * B_BYTES;  // A [part][matrix], then B hi, lo
    static constexpr int RAW_CODES = NA * 2 * kGmM * BPB;  // two K-blocks per stage
    static constexpr int RAW_SCALES = NA * 2 * kGmM * 2;
    static constexpr int RAW_BYTES = RAW_CODES + RAW_SCALES;
    static constexpr int ACC_COLS = NA * kGmN;      // one accumulator buffer (fp32 columns)
    static constexpr int TMEM_COLS = 2 * ACC_COLS;  // double buffered: 512 (gate/up) or 256 (down)
    static constexpr int NUM_BARS = 2 * RSTAGES + 3 * STAGES + 5;
    static constexpr int MISC_BYTES = 8 * NUM_BARS + 16 + 3 * 2 * kGmN * 4;
    // down: per epilogue warp two staging buffers of 16 tokens x its 32 rows of
    // w * D (fp32) that it adds into y with bulk reductions
    static constexpr int STAGE_BYTES = GATEUP ? 0 : 2 * 16 * kGmM * 4;
    static constexpr size_t SMEM =
        1024 + (size_t)STAGES * SLOT_BYTES + (size_t)RSTAGES * RAW_BYTES + MISC_BYTES + 128 + STAGE_BYTES;
    static constexpr int UNPACK = 128;                   // unpack threads (warps 2 .. 2 + UNPACK/32 - 1)
    static constexpr int THREADS = 64 + UNPACK + 128;    // producer, MMA, unpack, epilogue warps
    static constexpr int PIECES = NA * 2 * 128 / UNPACK;  // (matrix, K-block) pieces per unpack thread and stage
};

// Tracing builds: cycles each role spends in each wait, per CTA and kernel.
#ifdef MOEQ_TIMELINE
__device__ unsigned long long g_gemm_waits[2][256][16];
#define MOEQ_GW(slot, expr)                                                  \
    ([&]() {                                                                 \
        const long long c0_ = clock64();                                     \
        const bool r_ = (expr);                                              \
        gw[slot] += (unsigned long long)(clock64() - c0_);                   \
        return r_;                                                           \
    }())
#define MOEQ_GW_DECL unsigned long long gw[16] = {}; const long long gw_t0 = clock64()
#define MOEQ_GW_FLUSH(lo, hi, total_slot)                                                      \
    do {                                                                                       \
        gw[total_slot] = (unsigned long long)(clock64() - gw_t0);                              \
        for (int i_ = (lo); i_ <= (hi); ++i_)                                                  \
            atomicAdd(&g_gemm_waits[GATEUP ? 0 : 1][blockIdx.x & 255][i_], gw[i_]);            \
    } while (0)
#else
#define MOEQ_GW(slot, expr) (expr)
#define MOEQ_GW_DECL \
    do {             \
    } while (0)
#define MOEQ_GW_FLUSH(lo, hi, total_slot) \
    do {                                  \
    } while (0)
#endif

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Named barrier over n threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_sync_or(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %3, 0;\n\tbar.red.or.pred p, %1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(n), "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Persistent grouped GEMM: one CTA per SM walks the work items q = blockIdx.x,
// blockIdx.x + gridDim.x, ... where q = (tile, 128-row M block).  Each item is
// K/64 pipeline stages; stage g of this CTA uses operand slot g % STAGES and
// raw slot g % RSTAGES, so every role derives the same slot and phase from g.
//   warp 0     producer: bulk copies of the raw codes/scales (RSTAGES ahead)
//              and of the tile's B rows (hi, lo: one contiguous, pre-swizzled
//              run each per K stage) into the operand slots, on mbarriers
//   warp 1     TMEM owner; lane 0 issues the MMAs (hi and lo per K step)
//   warps 2-5  unpack: row r of the weight tile, codes -> fp16 level*scale
//   warps 6-9  epilogue on the other accumulator buffer (TMEM lane quadrant
//              = warp % 4), so item i's epilogue overlaps item i+1's MMAs
// Every wait is bounded; a wait that gives up raises the CTA's abort flag,
// every role leaves its loop, copies and MMAs are drained and TMEM is freed.
template <bool GATEUP, int BITS>
__global__ void __launch_bounds__(GemmCfg<GATEUP, BITS>::THREADS, 1) ffn_gemm_kernel(const __grid_constant__ GemmArgs a) {
    using C = GemmCfg<GATEUP, BITS>;
    constexpr int NA = C::NA, BPB = C::BPB, S = C::STAGES, R = C::RSTAGES;
    const int MT = (GATEUP ? a.I : a.H) / kGmM;
    const int K = GATEUP ? a.H : a.I;
    const int KB = K / 32, nk = K / kGmK;
    const int NR = GATEUP ? a.I : a.H;  // rows of each weight matrix
    const int n_items = a.ctrl[2] * MT;
    const int nq = n_items > (int)blockIdx.x ? (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int G = nq * nk;  // pipeline stages of this CTA

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *slots = smem;                                       // S x SLOT_BYTES
    unsigned char *raws = smem + (size_t)S * C::SLOT_BYTES;            // R x RAW_BYTES
    uint64_t *bars = reinterpret_cast<uint64_t *>(raws + (size_t)R * C::RAW_BYTES);
    uint64_t *raw_full = bars, *raw_empty = bars + R;
    uint64_t *a_full = bars + 2 * R, *b_full = a_full + S, *slot_empty = b_full + S;
    uint64_t *acc_full = slot_empty + S, *acc_empty = acc_full + 2, *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_tok = reinterpret_cast<int *>(tmem_slot + 4);  // [2][kGmN] per accumulator buffer
    int *s_exp = s_tok + 2 * kGmN;
    float *s_wt = reinterpret_cast<float *>(s_exp + 2 * kGmN);
    float *s_stage = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(s_wt + 2 * kGmN) + 127) & ~(uintptr_t)127);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t wl = wait_limit();
    [[maybe_unused]] constexpr int TLK = GATEUP ? 5 : 6;  // timeline kernel id (tracing builds)
    if (tid == 0) {
        for (int i = 0; i < R; ++i) {
            mbar_init(smem_u32(&raw_full[i]), 1);
            mbar_init(smem_u32(&raw_empty[i]), C::UNPACK);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&a_full[i]), C::UNPACK);
            mbar_init(smem_u32(&b_full[i]), 1);
            mbar_init(smem_u32(&slot_empty[i]), 1);
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
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // work item j of this CTA -> (tile, first weight row)
    auto item_tile = [&](int j) { return a.tiles[((int)blockIdx.x + j * (int)gridDim.x) / MT]; };
    auto item_m0 = [&](int j) { return (((int)blockIdx.x + j * (int)gridDim.x) % MT) * kGmM; };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        MOEQ_GW_DECL;
        const uint64_t pol = l2_evict_first();
        // raw cursor: runs up to R stages ahead of the operand cursor
        int rj = 0, rks = 0, rs = 0, graw = 0;
        uint32_t rph = 0;
        Tile rtl = nq > 0 ? item_tile(0) : Tile{};
        int rm0 = nq > 0 ? item_m0(0) : 0;
        int s = 0, gb = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int j = 0; j < nq && ok; ++j) {
            const Tile tl = item_tile(j);
            const int nround = (tl.n + 15) & ~15;
            for (int ks = 0; ks < nk; ++ks) {
                const int g = j * nk + ks;
                for (; graw < G && graw < g + R; ++graw) {
                    if (!__all_sync(0xffffffffu, MOEQ_GW(0, mbar_wait(smem_u32(&raw_empty[rs]), rph ^ 1, abort_flag, wl)))) {
                        ok = false;
                        break;
                    }
                    const uint32_t rbar = smem_u32(&raw_full[rs]);
                    if (lane == 0) mbar_arrive_expect_tx(rbar, (uint32_t)C::RAW_BYTES);
                    __syncwarp();
                    if (lane < 4 * NA) {  // lanes [0, 2NA): codes of (matrix, block); [2NA, 4NA): scales
                        const int mb = lane % (2 * NA), m = mb >> 1, kb = 2 * rks + (mb & 1);
                        const int mat = GATEUP ? m : 2;
                        const size_t blk = ((size_t)rtl.e * KB + kb) * NR + rm0;
                        unsigned char *rw = raws + (size_t)rs * C::RAW_BYTES;
                        if (lane < 2 * NA)
                            bulk_g2s(smem_u32(rw + mb * kGmM * BPB), a.codes[mat] + blk * BPB, kGmM * BPB, rbar, pol);
                        else
                            bulk_g2s(smem_u32(rw + C::RAW_CODES + mb * kGmM * 2), a.scales[mat] + blk, kGmM * 2, rbar,
                                     pol);
                    }
                    if (++rs == R) {
                        rs = 0;
                        rph ^= 1;
                    }
                    if (++rks == nk) {
                        rks = 0;
                        if (++rj < nq) {
                            rtl = item_tile(rj);
                            rm0 = item_m0(rj);
                        }
                    }
                }
                if (!ok) break;
                // B rows of this stage: hi/lo of sorted pairs p0 .. p0 + nround, K columns
                // [64 ks, 64 ks + 64), one contiguous run of 128-byte rows per half
                if (!__all_sync(0xffffffffu, MOEQ_GW(1, mbar_wait(smem_u32(&slot_empty[s]), ph ^ 1, abort_flag, wl)))) {
                    ok = false;
                    break;
                }
                const uint32_t bbar = smem_u32(&b_full[s]);
                // tiles of <= kGmN/2 rows: the lo rows follow the hi rows, so that one MMA
                // of N = 2 nround forms both products (see the MMA warp)
                const uint32_t bhi = smem_u32(slots + (size_t)s * C::SLOT_BYTES + C::NAT * NA * C::A_BYTES),
                               blo = nround <= kGmN / 2 ? bhi + (uint32_t)(nround * 128) : bhi + C::B_BYTES;
                if (lane == 0) mbar_arrive_expect_tx(bbar, (uint32_t)(2 * nround * kGmK * 2));
                __syncwarp();
                if (lane < 2)
                    bulk_g2s(lane ? blo : bhi,
                             a.bimg + ((size_t)(2 * ks + lane) * (size_t)a.bimg_rows + (size_t)tl.p0) * kGmK,
                             (uint32_t)(nround * kGmK * 2), bbar, 0);
                gb = g + 1;
                if (++s == S) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        if (lane == 0) MOEQ_GW_FLUSH(0, 2, 2);
        if (!ok && lane == 0) {  // drain the copies still in flight
            for (int g2 = max(0, graw - R); g2 < graw; ++g2)
                mbar_drain(smem_u32(&raw_full[g2 % R]), (g2 / R) & 1, abort_flag);
            for (int g2 = max(0, gb - S); g2 < gb; ++g2)
                mbar_drain(smem_u32(&b_full[g2 % S]), (g2 / S) & 1, abort_flag);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA
        if (lane == 0) {
            MOEQ_GW_DECL;
            // descriptors: slot s, matrix m, K step kk = base + ((s*SLOT + m*A) >> 4) + 2 kk
            const uint64_t d0 = sw128_desc(smem_u32(slots));
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            Tile next = nq > 0 ? item_tile(0) : Tile{};
            for (int j = 0; j < nq && ok; ++j) {
                const Tile tl = next;
                if (j + 1 < nq) next = item_tile(j + 1);  // consumed one item later
                // a tile of nround <= kGmN / 2 rows has B = [hi rows; lo rows] and takes one MMA
                // of N = 2 nround per product: hi into accumulator columns [0, nround), lo into
                // [nround, 2 nround), added in the epilogue (an MMA costs about the same down
                // to N = 64, so this halves the time of small tiles); larger tiles take two MMAs
                // (hi, lo) into the same columns
                const int nround = (tl.n + 15) & ~15;
                const bool cat = nround <= kGmN / 2;
                const uint32_t idesc = f16_idesc(kGmM, cat ? 2 * nround : nround);
                const int buf = j & 1;
                if (!MOEQ_GW(3, mbar_wait(smem_u32(&acc_empty[buf]), ((j >> 1) & 1) ^ 1, abort_flag, wl))) break;
                MOEQ_TL_TAG(TLK, 0, ((unsigned)j << 8) | blockIdx.x);
                tc_fence_after();
                const uint32_t acc0 = tmem + (uint32_t)(buf * C::ACC_COLS);
                for (int ks = 0; ks < nk; ++ks) {
                    if (!MOEQ_GW(4, mbar_wait(smem_u32(&a_full[s]), ph, abort_flag, wl)) ||
                        !MOEQ_GW(5, mbar_wait(smem_u32(&b_full[s]), ph, abort_flag, wl))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (ks == 0) MOEQ_TL_TAG(TLK, 1, ((unsigned)j << 8) | blockIdx.x);
                    const uint64_t ds = d0 + (uint64_t)((s * C::SLOT_BYTES) >> 4);
                    const uint64_t dbh = ds + (uint64_t)((C::NAT * NA * C::A_BYTES) >> 4);
                    const uint64_t dbl = dbh + (uint64_t)(C::B_BYTES >> 4);
#pragma unroll
                    for (int kk = 0; kk < kGmK / 16; ++kk) {
#pragma unroll
                        for (int m = 0; m < NA; ++m) {
                            const uint64_t ad = ds + (uint64_t)((m * C::A_BYTES) >> 4) + 2 * kk;
                            const uint32_t acc = acc0 + (uint32_t)(m * kGmN);
                            mma_f16(acc, ad, dbh + 2 * kk, idesc, (ks | kk) != 0);
                            if (!cat) mma_f16(acc, ad, dbl + 2 * kk, idesc, 1u);
                            if (C::NAT == 2)  // 3-bit: the weight panel's lo part against B hi (and lo when cat)
                                mma_f16(acc, ad + (uint64_t)((NA * C::A_BYTES) >> 4), dbh + 2 * kk, idesc, 1u);
                        }
                    }
                    mma_commit(smem_u32(&slot_empty[s]));
                    if (++s == S) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (ok) mma_commit(smem_u32(&acc_full[buf]));
                MOEQ_TL_TAG(TLK, 2, ((unsigned)j << 8) | blockIdx.x);
            }
            MOEQ_GW_FLUSH(3, 6, 6);
            // every MMA issued above is complete once this commit lands
            mma_commit(smem_u32(drain));
            mbar_drain(smem_u32(drain), 0, abort_flag);
        }
        __syncwarp();
    } else if (warp < 2 + C::UNPACK / 32) {
        // ----------------------------------------------------------- unpack
        // thread u: row r = u % 128 of the tile and PIECES of the stage's (matrix,
        // K-block) pieces, piece index = (u / 128) * PIECES + pi, matrix = index / 2
        const int u = tid - 64, r = u & 127, part = u >> 7;
        constexpr int WPT = C::PIECES;
        MOEQ_GW_DECL;
        int rs = 0, s = 0;
        uint32_t rph = 0, ph = 0;
        bool ok = true;
        for (int g = 0; g < G && ok; ++g) {
            if (!MOEQ_GW(7, mbar_wait(smem_u32(&raw_full[rs]), rph, abort_flag, wl))) break;
            if (u == 0 && g % nk == 0) MOEQ_TL_TAG(TLK, 5, ((unsigned)(g / nk) << 8) | blockIdx.x);
            const unsigned char *rw = raws + (size_t)rs * C::RAW_BYTES;
            uint32_t cw[WPT][BITS];
            uint16_t sbits[WPT];
#pragma unroll
            for (int pi = 0; pi < WPT; ++pi) {
                const int pc = part * WPT + pi, m = pc >> 1, b = pc & 1;
                const uint32_t *cp = reinterpret_cast<const uint32_t *>(rw + ((m * 2 + b) * kGmM + r) * BPB);
#pragma unroll
                for (int i = 0; i < BITS; ++i) cw[pi][i] = cp[i];
                sbits[pi] = *reinterpret_cast<const uint16_t *>(rw + C::RAW_CODES + ((m * 2 + b) * kGmM + r) * 2);
            }
            mbar_arrive(smem_u32(&raw_empty[rs]));
            if (++rs == R) {
                rs = 0;
                rph ^= 1;
            }
            if (!MOEQ_GW(8, mbar_wait(smem_u32(&slot_empty[s]), ph ^ 1, abort_flag, wl))) break;
            unsigned char *sb = slots + (size_t)s * C::SLOT_BYTES;
#pragma unroll
            for (int pi = 0; pi < WPT; ++pi) {
                const int pc = part * WPT + pi, m = pc >> 1, b = pc & 1;
                const uint32_t at = smem_u32(sb + m * C::A_BYTES);
                const __half sc = __ushort_as_half(sbits[pi]);
                if (BITS == 2) {
                    const __half m2 = __hmul(sc, __float2half(-2.0f)), m1 = __hneg(sc);
                    const uint32_t lut_lo = (uint32_t)__half_as_ushort(m2) | ((uint32_t)__half_as_ushort(m1) << 16);
                    const uint32_t lut_hi = (uint32_t)__half_as_ushort(sc) << 16;  // {0, s}
#pragma unroll
                    for (int c = 0; c < 4; ++c) {  // 16-byte chunk = 8 elements = 2 code bytes
                        const uint32_t word = cw[pi][c >> 1];
                        const uint32_t d0 = (word >> (16 * (c & 1))) & 0xffu;
                        const uint32_t d1 = (word >> (16 * (c & 1) + 8)) & 0xffu;
                        const uint32_t q0 = lut_pair(lut_lo, lut_hi, (d0 & 3u) | ((d0 & 0xCu) << 6));
                        const uint32_t q1 = lut_pair(lut_lo, lut_hi, ((d0 >> 4) & 3u) | ((d0 & 0xC0u) << 2));
                        const uint32_t q2 = lut_pair(lut_lo, lut_hi, (d1 & 3u) | ((d1 & 0xCu) << 6));
                        const uint32_t q3 = lut_pair(lut_lo, lut_hi, ((d1 >> 4) & 3u) | ((d1 & 0xC0u) << 2));
                        st_shared_v4(at + sw128_off(r, 4 * b + c), q0, q1, q2, q3);
                    }
                } else {
                    // 3-bit levels -4..3 times s: v = level * s is exact in fp32; hi = fp16(v)
                    // and lo = v - hi (exact in fp16) go to the hi and lo panels
                    const float sf = __half2float(sc);
                    const uint32_t at_lo = smem_u32(sb + (NA + m) * C::A_BYTES);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t qv[4], lv[4];
#pragma unroll
                        for (int h2 = 0; h2 < 4; ++h2) {
                            __half hv[2], lo[2];
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const int i = 8 * c + 2 * h2 + e2, off = 3 * i, wi = off >> 5, sh = off & 31;
                                const uint32_t lo_w = cw[pi][wi];
                                const uint32_t hi_w = wi + 1 < BITS ? cw[pi][wi + 1] : 0u;
                                const int code = (int)(__funnelshift_r(lo_w, hi_w, sh) & 7u);
                                const float v = (float)(code - 4) * sf;
                                hv[e2] = __float2half_rn(v);
                                lo[e2] = __float2half_rn(v - __half2float(hv[e2]));
                            }
                            qv[h2] = (uint32_t)__half_as_ushort(hv[0]) | ((uint32_t)__half_as_ushort(hv[1]) << 16);
                            lv[h2] = (uint32_t)__half_as_ushort(lo[0]) | ((uint32_t)__half_as_ushort(lo[1]) << 16);
                        }
                        st_shared_v4(at_lo + sw128_off(r, 4 * b + c), lv[0], lv[1], lv[2], lv[3]);
                        st_shared_v4(at + sw128_off(r, 4 * b + c), qv[0], qv[1], qv[2], qv[3]);
                    }
                }
            }
            fence_proxy_async();
            mbar_arrive(smem_u32(&a_full[s]));
            if (u == 0 && g % nk == nk - 1) MOEQ_TL_TAG(TLK, 6, ((unsigned)(g / nk) << 8) | blockIdx.x);
            if (++s == S) {
                s = 0;
                ph ^= 1;
            }
        }
        if (u == 0) MOEQ_GW_FLUSH(7, 9, 9);
    } else {
        // --------------------------------------------------------- epilogue
        const int et = tid - 64 - C::UNPACK;      // 0..127: table entry this thread loads
        const int row = 32 * (warp & 3) + lane;   // accumulator lane = weight row
        const uint32_t tl_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        MOEQ_GW_DECL;
        bool dead = false;  // after an abort the loop still meets every named barrier
        int nstage = 0;     // staging buffers used so far (down)
        for (int j = 0; j < nq; ++j) {
            const Tile tl = item_tile(j);
            const int m0 = item_m0(j);
            const int buf = j & 1, p0 = tl.p0, nval = tl.n, nround = (nval + 15) & ~15;
            {
                const int p = p0 + min(et, nval - 1);
                int t = a.perm_tok[p];
                const int js = a.perm_slot[p];
                float wv = 0.f;
                if (t < 0 || t >= a.T || js < 0 || js >= a.k) {  // a caller's bad permutation: no contribution
                    set_status(MOEQ_STATUS_BAD_INDEX);
                    t = 0;
                } else if (!GATEUP && a.w) {
                    wv = a.w[(size_t)t * a.k + js];
                }
                s_tok[buf * kGmN + et] = t;
                s_exp[buf * kGmN + et] = a.brow_exp[p];
                s_wt[buf * kGmN + et] = wv;
            }
            named_sync(1, 128);
            if (dead) continue;
            // one decision for all four epilogue warps (they meet at named barriers below)
            if (named_sync_or(3, 128, !MOEQ_GW(10, mbar_wait(smem_u32(&acc_full[buf]), (j >> 1) & 1, abort_flag, wl)))) {
                dead = true;
                continue;
            }
            tc_fence_after();
            if (et == 0) MOEQ_TL_TAG(TLK, 3, ((unsigned)j << 8) | blockIdx.x);
            const int *etab = s_exp + buf * kGmN;
            const uint32_t acc = tl_lane + (uint32_t)(buf * C::ACC_COLS);
            const bool cat = nround <= kGmN / 2;  // lo products in columns [nround, 2 nround) (MMA warp)
            for (int c0 = 0; c0 < nround; c0 += 16) {
                float acc0[16];
                tmem_ld16(acc + (uint32_t)c0, acc0);
                if (cat) {
                    float lo0[16];
                    tmem_ld16(acc + (uint32_t)(nround + c0), lo0);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) acc0[jj] += lo0[jj];
                }
                if (GATEUP) {
                    float acc1[16];
                    tmem_ld16(acc + (uint32_t)(kGmN + c0), acc1);
                    if (cat) {
                        float lo1[16];
                        tmem_ld16(acc + (uint32_t)(kGmN + nround + c0), lo1);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) acc1[jj] += lo1[jj];
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int jc = c0 + jj;
                        if (jc >= nval) break;
                        const float sc = exp2i(etab[jc]);
                        const float Gv = acc0[jj] * sc, Uv = acc1[jj] * sc;
                        const float h = __fdiv_rn(Gv, 1.0f + expf(-Gv)) * Uv;
                        const float s = block_scale(warp_absmax(h));
                        const int q = block_code(h, s);
                        const size_t p = (size_t)(p0 + jc);
                        a.qh[p * a.I + m0 + row] = (int8_t)q;
                        if (lane == 0) a.sh[p * (a.I / 32) + (m0 + row) / 32] = s;
                    }
                } else {
                    const int *ttab = s_tok + buf * kGmN;
                    const float *wtab = s_wt + buf * kGmN;
                    if (a.y) {
                        // w * D of these 16 pairs -> this warp's staging buffer [pair][its 32
                        // rows] -> one 128-byte bulk reduction per pair into
                        // y[token][m0 + 32 (warp % 4) ...]; warps proceed independently
                        const int q = warp & 3;
                        float *stg = s_stage + ((nstage & 1) * 4 + q) * 16 * 32;
                        bulk_wait_read<1>();  // (issuing lanes) this buffer's previous reductions have read it
                        __syncwarp();
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int jc = c0 + jj;
                            stg[jj * 32 + lane] = wtab[jc] * acc0[jj] * exp2i(etab[jc]);
                        }
                        fence_proxy_async();
                        __syncwarp();
                        if (lane < 16) {
                            if (c0 + lane < nval)
                                bulk_reduce_add_f32(a.y + (size_t)ttab[c0 + lane] * a.H + m0 + 32 * q,
                                                    smem_u32(stg + lane * 32), 32 * 4);
                            bulk_commit();
                        }
                        ++nstage;
                    }
                    if (a.out_sorted) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int jc = c0 + jj;
                            if (jc >= nval) break;
                            a.out_sorted[(size_t)(p0 + jc) * a.H + m0 + row] = acc0[jj] * exp2i(etab[jc]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&acc_empty[buf]));
            if (et == 0) MOEQ_TL_TAG(TLK, 4, ((unsigned)j << 8) | blockIdx.x);
        }
        if (!GATEUP && lane < 16) bulk_wait_all();  // reductions done before the CTA exits
        if (et == 0) MOEQ_GW_FLUSH(10, 11, 11);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
    }
}

}  // namespace moeq
