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
//     relative, is dropped like the rest of the B split's residue).  The
//     panel lives in tensor memory (the MMA's A operand from TMEM), written by
//     the unpack warps with tcgen05.st: the tcgen05 ordering rules (commit ->
//     mbarrier -> fence) then cover its reuse.  Ordinary shared-memory stores
//     into an operand slot released by a tcgen05.commit were measured to race
//     with the tensor core's reads of that slot;
//   * B (activations, N = up to TILE_N sorted tokens): v = q * s_a * 2^-e split
//     into fp16 hi + lo (hi + lo == v to ~2^-22), two MMAs into one fp32
//     accumulator, so the per-32-block activation scale is carried without an
//     epilogue per K-block;
//   * e is a per-row power of two, undone exactly in the epilogue.
//
// Work item = (tile of <= TILE_N sorted pairs of one expert, 128-row block of
// its weight matrix); the epilogue reads the accumulator (lane = weight row):
//   gate/up: h = silu(G) * U and int8 re-quantisation per 32 rows (one warp =
//            one quantisation block), stored as q_h, s_h;
//   down:    D * 2^e, weighted by the routing weight and added into y with
//            one 128-byte bulk reduction per pair and 32 rows, or stored per
//            sorted pair.
// The kernel is persistent and warp-specialised (see ffn_gemm_kernel).
#pragma once

#include "async.cuh"
#include "permute.cuh"

namespace moeq {

constexpr int kGmM = 128;  // MMA M: weight rows per CTA (= TMEM lanes)
constexpr int kGmK = 64;   // K per pipeline stage = one 128-byte swizzle row of fp16
constexpr int kTmemCols = 512;

struct GemmArgs {
    int T, H, I, E, k;
    const uint8_t *codes[3];
    const uint16_t *scales[3];
    const Tile *tiles;
    const int *ntiles;  // number of tiles (written by the plan kernel)
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

// D (TMEM) (+)= A (TMEM: lane = row, 8 columns = 16 fp16 of K) * B (shared memory).
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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
    // 2-bit: two blocks share each stage's token rows (514 -> 485 us per 4K chunk).
    // 3-bit keeps one: two would leave TMEM room for a single accumulator buffer
    // (16K-token 3-bit chunk 6.9 -> 7.9 ms)
    static constexpr int DOWN_NA = BITS == 2 ? 2 : 1;
    // weight blocks per work item: gate and up (the same 128 rows of each), or
    // DOWN_NA consecutive 128-row blocks of down
    static constexpr int NA = GATEUP ? 2 : DOWN_NA;
    static constexpr int BPB = 4 * BITS;
    static constexpr int NAT = BITS == 3 ? 2 : 1;  // weight panels per matrix: hi (, lo)
    // tokens per tile (MMA N): TMEM holds NBUF accumulator buffers of NA x TILE_N
    // columns and PSTAGES weight panels of NAT x NA x 32 columns (K = 64 fp16).
    // 3-bit gate/up needs 128 columns per panel stage, so it keeps 128-token
    // tiles (half the MMAs of 64-token ones) with one accumulator buffer: its
    // epilogue then does not overlap the next item's MMAs.  Down (8 stages per
    // item, a comparatively long epilogue) has room for three
    static constexpr int NBUF = NA == 2 ? (BITS == 3 ? 1 : 2) : 3;
    static constexpr int TILE_N = (NA == 2 && BITS == 2) ? 96 : 128;
    static constexpr int ACC_COLS = NA * TILE_N;           // one accumulator buffer (fp32 columns)
    static constexpr int A_COLS = NAT * NA * (kGmK / 2);   // one stage of weight panels
    static constexpr int A_BASE = NBUF * ACC_COLS;         // first panel column
#if defined(MOEQ_GEMM_PSTAGES)
    static constexpr int PSTAGES = MOEQ_GEMM_PSTAGES;
#else
    static constexpr int PSTAGES = (kTmemCols - A_BASE) / A_COLS > 4 ? 4 : (kTmemCols - A_BASE) / A_COLS;
#endif
    // token-row ring in shared memory, refilled by bulk copies (MOEQ_GEMM_STAGES overrides)
#if defined(MOEQ_GEMM_STAGES)
    static constexpr int STAGES = MOEQ_GEMM_STAGES;
#else
    static constexpr int STAGES = GATEUP ? (BITS == 2 ? 6 : 4) : 5;
#endif
    static constexpr int RSTAGES = 6;                    // raw-code ring (runs further ahead)
    static constexpr int B_BYTES = TILE_N * kGmK * 2;    // fp16 activation tile (hi or lo)
    static constexpr int SLOT_BYTES = 2 * B_BYTES;       // B hi, lo
    static constexpr int RAW_CODES = NA * 2 * kGmM * BPB;  // two K-blocks per stage
    static constexpr int RAW_SCALES = NA * 2 * kGmM * 2;
    static constexpr int RAW_BYTES = RAW_CODES + RAW_SCALES;
    static constexpr int NUM_BARS = 2 * RSTAGES + 2 * STAGES + 2 * PSTAGES + 2 * NBUF + 1;
    static constexpr int MISC_BYTES = 8 * NUM_BARS + 16 + 3 * NBUF * TILE_N * 4;
    // down: per epilogue warp two staging buffers of 16 tokens x its 32 rows of
    // w * D (fp32) that it adds into y with bulk reductions
    static constexpr int STAGE_BYTES = GATEUP ? 0 : 2 * 16 * kGmM * 4;
    static constexpr size_t SMEM =
        1024 + (size_t)STAGES * SLOT_BYTES + (size_t)RSTAGES * RAW_BYTES + MISC_BYTES + 128 + STAGE_BYTES;
    static constexpr int UNPACK = 128;                   // unpack threads (warps 2 .. 5)
    static constexpr int ISSUERS = NA;  // MMA-issuing threads: one per weight block of an item
    // producer, MMA, unpack, epilogue warps (+ a second MMA warp after them:
    // with two issuers, each issues the MMAs of one of the item's matrices)
    static constexpr int THREADS = 64 + UNPACK + 128 + 32 * (ISSUERS - 1);
    static constexpr int PIECES = NA * 2;                // (matrix, K-block) pieces per unpack thread and stage
    static_assert(PSTAGES >= 2 && A_BASE + PSTAGES * A_COLS <= kTmemCols, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(TILE_N % 16 == 0 && TILE_N >= kTileMin && TILE_N <= kTileMax && B_BYTES % 1024 == 0, "tile shape");
};

// The MMAs of one K = 64 stage, from one thread: for each K step kk and matrix
// m, D_m (+)= A_m,kk (TMEM) * B_kk (shared memory).  CAT: B = [hi rows; lo
// rows] in one MMA of twice the tile's N; otherwise the hi and lo products are
// two MMAs into the same accumulator.  NAT == 2 (3-bit) adds the weight
// panel's lo part against B hi.  The sequence has no branch: a conditional
// branch between tcgen05.mma instructions was measured to double their cost
// to the issuing thread (45 -> 93 cycles at N = 32 .. 96).
template <int NA, int M0, int M1, int NAT, int TN, bool CAT>
__device__ __forceinline__ void mma_stage(uint32_t acc0, uint32_t ap, uint64_t dbh, uint64_t dbl, uint32_t idesc,
                                          uint32_t accumulate) {
#pragma unroll
    for (int kk = 0; kk < kGmK / 16; ++kk) {
#pragma unroll
        for (int m = M0; m < M1; ++m) {
            const uint32_t at = ap + (uint32_t)(m * (kGmK / 2) + 8 * kk);
            const uint32_t acc = acc0 + (uint32_t)(m * TN);
            mma_f16_ta(acc, at, dbh + 2 * kk, idesc, kk ? 1u : accumulate);
            if (!CAT) mma_f16_ta(acc, at, dbl + 2 * kk, idesc, 1u);
            if (NAT == 2) mma_f16_ta(acc, at + (uint32_t)(NA * (kGmK / 2)), dbh + 2 * kk, idesc, 1u);
        }
    }
}

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
// K/64 pipeline stages; stage g of this CTA uses token slot g % STAGES, panel
// stage g % PSTAGES and raw slot g % RSTAGES, so every role derives the same
// slots and phases from g.
//   warp 0     producer: bulk copies of the raw codes/scales (RSTAGES ahead)
//              and of the tile's B rows (hi, lo: one contiguous, pre-swizzled
//              run each per K stage) into the token slots, on mbarriers
//   warp 1     TMEM owner; lane 0 issues the MMAs (A from TMEM, B from shared
//              memory; with two weight blocks per item, those of the first)
//   warps 2-5  unpack: codes -> fp16 level*scale, written into the TMEM panel
//              stage with tcgen05.st; warp w writes the 32 weight rows of its
//              TMEM lane quadrant w % 4
//   warps 6-9  epilogue on the other accumulator buffer (TMEM lane quadrant
//              = warp % 4), so item i's epilogue overlaps item i+1's MMAs
//              (with one buffer, 3-bit gate/up, the MMAs wait for it)
//   warp 10    items of two weight blocks (gate/up; 2-bit down): lane 0
//              issues the second block's MMAs while warp 1 issues the
//              first's (a second issuing thread on another SM
//              sub-partition); the stage and accumulator barriers then
//              expect a commit from each
// Every wait is bounded; a wait that gives up raises the CTA's abort flag,
// every role leaves its loop, copies and MMAs are drained and TMEM is freed.
template <bool GATEUP, int BITS>
__global__ void __launch_bounds__(GemmCfg<GATEUP, BITS>::THREADS, 1) ffn_gemm_kernel(const __grid_constant__ GemmArgs a) {
    using C = GemmCfg<GATEUP, BITS>;
    constexpr int NA = C::NA, BPB = C::BPB, S = C::STAGES, R = C::RSTAGES, PS = C::PSTAGES, TN = C::TILE_N;
    // work items per tile; with H an odd multiple of 128 the last down item has one block
    const int MT = GATEUP ? a.I / kGmM : (a.H + kGmM * NA - 1) / (kGmM * NA);
    const int K = GATEUP ? a.H : a.I;
    const int KB = K / 32, nk = K / kGmK;
    const int NR = GATEUP ? a.I : a.H;  // rows of each weight matrix
    const int n_items = *a.ntiles * MT;
    const int nq = n_items > (int)blockIdx.x ? (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int G = nq * nk;  // pipeline stages of this CTA

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *slots = smem;                                       // S x SLOT_BYTES (B hi, lo)
    unsigned char *raws = smem + (size_t)S * C::SLOT_BYTES;            // R x RAW_BYTES
    uint64_t *bars = reinterpret_cast<uint64_t *>(raws + (size_t)R * C::RAW_BYTES);
    uint64_t *raw_full = bars, *raw_empty = bars + R;
    uint64_t *b_full = bars + 2 * R, *b_empty = b_full + S;
    uint64_t *a_full = b_empty + S, *a_empty = a_full + PS;
    uint64_t *acc_full = a_empty + PS, *acc_empty = acc_full + C::NBUF, *drain = acc_empty + C::NBUF;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_tok = reinterpret_cast<int *>(tmem_slot + 4);  // [NBUF][TN] per accumulator buffer
    int *s_exp = s_tok + C::NBUF * TN;
    float *s_wt = reinterpret_cast<float *>(s_exp + C::NBUF * TN);
    float *s_stage = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(s_wt + C::NBUF * TN) + 127) & ~(uintptr_t)127);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t wl = wait_limit();
    [[maybe_unused]] constexpr int TLK = GATEUP ? 5 : 6;  // timeline kernel id (tracing builds)
    if (tid == 0) {
        for (int i = 0; i < R; ++i) {
            mbar_init(smem_u32(&raw_full[i]), 1);
            mbar_init(smem_u32(&raw_empty[i]), C::UNPACK);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&b_full[i]), 1);
            mbar_init(smem_u32(&b_empty[i]), C::ISSUERS);
        }
        for (int i = 0; i < PS; ++i) {
            mbar_init(smem_u32(&a_full[i]), C::UNPACK);
            mbar_init(smem_u32(&a_empty[i]), C::ISSUERS);
        }
        for (int i = 0; i < C::NBUF; ++i) {
            mbar_init(smem_u32(&acc_full[i]), C::ISSUERS);
            mbar_init(smem_u32(&acc_empty[i]), 128);
        }
        mbar_init(smem_u32(drain), C::ISSUERS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // work item j of this CTA -> (tile, first weight row)
    auto item_tile = [&](int j) { return a.tiles[((int)blockIdx.x + j * (int)gridDim.x) / MT]; };
    auto item_m0 = [&](int j) { return (((int)blockIdx.x + j * (int)gridDim.x) % MT) * (GATEUP ? kGmM : kGmM * NA); };

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
                    // weight blocks of this item inside the matrix (the second block of a down
                    // item past the last row is not fetched; its panel and accumulator are unused)
                    const int nbv = GATEUP ? NA : min(NA, (NR - rm0) / kGmM);
                    if (lane == 0) mbar_arrive_expect_tx(rbar, (uint32_t)(C::RAW_BYTES / NA * nbv));
                    __syncwarp();
                    if (lane < 4 * NA && ((lane % (2 * NA)) >> 1) < nbv) {  // lanes [0, 2NA): codes of (matrix, block); [2NA, 4NA): scales
                        const int mb = lane % (2 * NA), m = mb >> 1, kb = 2 * rks + (mb & 1);
                        const int mat = GATEUP ? m : 2;
                        const size_t blk = ((size_t)rtl.e * KB + kb) * NR + rm0 + (GATEUP ? 0 : m * kGmM);
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
                if (!__all_sync(0xffffffffu, MOEQ_GW(1, mbar_wait(smem_u32(&b_empty[s]), ph ^ 1, abort_flag, wl)))) {
                    ok = false;
                    break;
                }
                const uint32_t bbar = smem_u32(&b_full[s]);
                // tiles of <= TILE_N/2 rows: the lo rows follow the hi rows, so that one MMA
                // of N = 2 nround forms both products (see the MMA warp)
                const uint32_t bhi = smem_u32(slots + (size_t)s * C::SLOT_BYTES),
                               blo = nround <= TN / 2 ? bhi + (uint32_t)(nround * 128) : bhi + C::B_BYTES;
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
    } else if (warp == 1 || warp == 2 + C::UNPACK / 32 + 4) {
        // -------------------------------------------------------------- MMA
        if (lane == 0) {
            MOEQ_GW_DECL;
            // B descriptors: slot s, K step kk = base + ((s * SLOT) >> 4) + 2 kk;
            // A in TMEM: panel stage ps, matrix m, K step kk at column
            // A_BASE + ps A_COLS + m 32 + 8 kk (lo panel of 3-bit: + NA 32)
            const uint64_t d0 = sw128_desc(smem_u32(slots));
            int s = 0, ps = 0;
            uint32_t ph = 0, pph = 0;
            bool ok = true;
            Tile next = nq > 0 ? item_tile(0) : Tile{};
            for (int j = 0; j < nq && ok; ++j) {
                const Tile tl = next;
                if (j + 1 < nq) next = item_tile(j + 1);  // consumed one item later
                // a tile of nround <= TILE_N / 2 rows has B = [hi rows; lo rows] and takes one
                // MMA of N = 2 nround per product: hi into accumulator columns [0, nround), lo
                // into [nround, 2 nround), added in the epilogue; larger tiles take two MMAs
                // (hi, lo) into the same columns
                const int nround = (tl.n + 15) & ~15;
                const bool cat = nround <= TN / 2;
                const uint32_t idesc = f16_idesc(kGmM, cat ? 2 * nround : nround);
                const int buf = j % C::NBUF;
                if (!MOEQ_GW(3, mbar_wait(smem_u32(&acc_empty[buf]), ((j / C::NBUF) & 1) ^ 1, abort_flag, wl))) break;
                MOEQ_TL_TAG(TLK, 0, ((unsigned)j << 8) | blockIdx.x);
                tc_fence_after();
                const uint32_t acc0 = tmem + (uint32_t)(buf * C::ACC_COLS);
                for (int ks = 0; ks < nk; ++ks) {
                    if (!MOEQ_GW(4, mbar_wait(smem_u32(&a_full[ps]), pph, abort_flag, wl)) ||
                        !MOEQ_GW(5, mbar_wait(smem_u32(&b_full[s]), ph, abort_flag, wl))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (ks == 0) MOEQ_TL_TAG(TLK, 1, ((unsigned)j << 8) | blockIdx.x);
                    const uint64_t dbh = d0 + (uint64_t)((s * C::SLOT_BYTES) >> 4);
                    const uint64_t dbl = dbh + (uint64_t)(C::B_BYTES >> 4);
                    const uint32_t ap = tmem + (uint32_t)(C::A_BASE + ps * C::A_COLS);
                    if (C::ISSUERS == 1) {
                        if (cat) mma_stage<NA, 0, NA, C::NAT, TN, true>(acc0, ap, dbh, dbl, idesc, ks != 0);
                        else mma_stage<NA, 0, NA, C::NAT, TN, false>(acc0, ap, dbh, dbl, idesc, ks != 0);
                    } else if (warp == 1) {
                        if (cat) mma_stage<NA, 0, 1, C::NAT, TN, true>(acc0, ap, dbh, dbl, idesc, ks != 0);
                        else mma_stage<NA, 0, 1, C::NAT, TN, false>(acc0, ap, dbh, dbl, idesc, ks != 0);
                    } else {
                        if (cat) mma_stage<NA, 1, 2, C::NAT, TN, true>(acc0, ap, dbh, dbl, idesc, ks != 0);
                        else mma_stage<NA, 1, 2, C::NAT, TN, false>(acc0, ap, dbh, dbl, idesc, ks != 0);
                    }
                    mma_commit(smem_u32(&a_empty[ps]));
                    mma_commit(smem_u32(&b_empty[s]));
                    if (++s == S) {
                        s = 0;
                        ph ^= 1;
                    }
                    if (++ps == PS) {
                        ps = 0;
                        pph ^= 1;
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
        // warp w writes TMEM lanes 32 (w % 4) .. + 31: thread = weight row r of the
        // item's 128-row block, all (matrix, K-block) pieces of its row per stage
        const int q = warp & 3, r = 32 * q + lane;
        const uint32_t t_row = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)C::A_BASE;
        constexpr int WPT = C::PIECES;
        MOEQ_GW_DECL;
        int rs = 0, ps = 0;
        uint32_t rph = 0, pph = 0;
        bool ok = true;
        for (int g = 0; g < G && ok; ++g) {
            if (!__all_sync(0xffffffffu, MOEQ_GW(7, mbar_wait(smem_u32(&raw_full[rs]), rph, abort_flag, wl)))) break;
            if (r == 0 && g % nk == 0) MOEQ_TL_TAG(TLK, 5, ((unsigned)(g / nk) << 8) | blockIdx.x);
            const unsigned char *rw = raws + (size_t)rs * C::RAW_BYTES;
            uint32_t cw[WPT][BITS];
            uint16_t sbits[WPT];
#pragma unroll
            for (int pi = 0; pi < WPT; ++pi) {  // piece pi = (matrix pi / 2, K-block pi % 2)
                const uint32_t *cp = reinterpret_cast<const uint32_t *>(rw + (pi * kGmM + r) * BPB);
#pragma unroll
                for (int i = 0; i < BITS; ++i) cw[pi][i] = cp[i];
                sbits[pi] = *reinterpret_cast<const uint16_t *>(rw + C::RAW_CODES + (pi * kGmM + r) * 2);
            }
            mbar_arrive(smem_u32(&raw_empty[rs]));
            if (++rs == R) {
                rs = 0;
                rph ^= 1;
            }
            // the panel stage is free once the MMAs that read it have completed
            if (!__all_sync(0xffffffffu, MOEQ_GW(8, mbar_wait(smem_u32(&a_empty[ps]), pph ^ 1, abort_flag, wl)))) break;
            tc_fence_after();
            const uint32_t tp = t_row + (uint32_t)(ps * C::A_COLS);
#pragma unroll
            for (int m = 0; m < NA; ++m) {
                uint32_t hv[32], lv[32];  // the row's 64 K values of matrix m: K-block 0 then 1, 2 fp16 per word
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int pi = 2 * m + b;
                    const __half sc = __ushort_as_half(sbits[pi]);
                    if (BITS == 2) {
                        const __half m2 = __hmul(sc, __float2half(-2.0f)), m1 = __hneg(sc);
                        const uint32_t lut_lo = (uint32_t)__half_as_ushort(m2) | ((uint32_t)__half_as_ushort(m1) << 16);
                        const uint32_t lut_hi = (uint32_t)__half_as_ushort(sc) << 16;  // {0, s}
#pragma unroll
                        for (int c = 0; c < 4; ++c) {  // 8 elements = 2 code bytes
                            const uint32_t word = cw[pi][c >> 1];
                            const uint32_t d0 = (word >> (16 * (c & 1))) & 0xffu;
                            const uint32_t d1 = (word >> (16 * (c & 1) + 8)) & 0xffu;
                            uint32_t *o = hv + 16 * b + 4 * c;
                            o[0] = lut_pair(lut_lo, lut_hi, (d0 & 3u) | ((d0 & 0xCu) << 6));
                            o[1] = lut_pair(lut_lo, lut_hi, ((d0 >> 4) & 3u) | ((d0 & 0xC0u) << 2));
                            o[2] = lut_pair(lut_lo, lut_hi, (d1 & 3u) | ((d1 & 0xCu) << 6));
                            o[3] = lut_pair(lut_lo, lut_hi, ((d1 >> 4) & 3u) | ((d1 & 0xC0u) << 2));
                        }
                    } else {
                        // 3-bit levels -4..3 times s: v = level * s is exact in fp32; hi = fp16(v)
                        // and lo = v - hi (exact in fp16) go to the hi and lo panels
                        const float sf = __half2float(sc);
#pragma unroll
                        for (int h2 = 0; h2 < 16; ++h2) {
                            __half hh[2], ll[2];
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const int i = 2 * h2 + e2, off = 3 * i, wi = off >> 5, sh = off & 31;
                                const uint32_t lo_w = cw[pi][wi];
                                const uint32_t hi_w = wi + 1 < BITS ? cw[pi][wi + 1] : 0u;
                                const int code = (int)(__funnelshift_r(lo_w, hi_w, sh) & 7u);
                                const float v = (float)(code - 4) * sf;
                                hh[e2] = __float2half_rn(v);
                                ll[e2] = __float2half_rn(v - __half2float(hh[e2]));
                            }
                            hv[16 * b + h2] = (uint32_t)__half_as_ushort(hh[0]) | ((uint32_t)__half_as_ushort(hh[1]) << 16);
                            lv[16 * b + h2] = (uint32_t)__half_as_ushort(ll[0]) | ((uint32_t)__half_as_ushort(ll[1]) << 16);
                        }
                    }
                }
                tmem_st32(tp + (uint32_t)(m * (kGmK / 2)), hv);
                if (C::NAT == 2) tmem_st32(tp + (uint32_t)((NA + m) * (kGmK / 2)), lv);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&a_full[ps]));
            if (r == 0 && g % nk == nk - 1) MOEQ_TL_TAG(TLK, 6, ((unsigned)(g / nk) << 8) | blockIdx.x);
            if (++ps == PS) {
                ps = 0;
                pph ^= 1;
            }
        }
        if (r == 0) MOEQ_GW_FLUSH(7, 9, 9);
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
            const int buf = j % C::NBUF, p0 = tl.p0, nval = tl.n, nround = (nval + 15) & ~15;
            if (et < TN) {
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
                s_tok[buf * TN + et] = t;
                s_exp[buf * TN + et] = a.brow_exp[p];
                s_wt[buf * TN + et] = wv;
            }
            named_sync(1, 128);
            if (dead) continue;
            // one decision for all four epilogue warps (they meet at named barriers below)
            if (named_sync_or(3, 128, !MOEQ_GW(10, mbar_wait(smem_u32(&acc_full[buf]), (j / C::NBUF) & 1, abort_flag, wl)))) {
                dead = true;
                continue;
            }
            tc_fence_after();
            if (et == 0) MOEQ_TL_TAG(TLK, 3, ((unsigned)j << 8) | blockIdx.x);
            const int *etab = s_exp + buf * TN;
            const uint32_t acc = tl_lane + (uint32_t)(buf * C::ACC_COLS);
            const bool cat = nround <= TN / 2;  // lo products in columns [nround, 2 nround) (MMA warp)
            // down: one pass per 128-row block of the item (accumulator m); gate/up: one pass
            const int nbv = GATEUP ? 1 : min(NA, (a.H - m0) / kGmM);
            for (int mb = 0; mb < nbv; ++mb) {
            const uint32_t accm = acc + (uint32_t)(mb * TN);
            const int r0 = m0 + mb * kGmM;  // first weight row of this pass
            for (int c0 = 0; c0 < nround; c0 += 16) {
                float acc0[16];
                tmem_ld16(accm + (uint32_t)c0, acc0);
                if (cat) {
                    float lo0[16];
                    tmem_ld16(accm + (uint32_t)(nround + c0), lo0);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) acc0[jj] += lo0[jj];
                }
                if (GATEUP) {
                    float acc1[16];
                    tmem_ld16(acc + (uint32_t)(TN + c0), acc1);
                    if (cat) {
                        float lo1[16];
                        tmem_ld16(acc + (uint32_t)(TN + nround + c0), lo1);
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
                    const int *ttab = s_tok + buf * TN;
                    const float *wtab = s_wt + buf * TN;
                    if (a.y) {
                        // w * D of these 16 pairs -> this warp's staging buffer [pair][its 32
                        // rows] -> one 128-byte bulk reduction per pair into
                        // y[token][r0 + 32 (warp % 4) ...]; warps proceed independently
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
                                bulk_reduce_add_f32(a.y + (size_t)ttab[c0 + lane] * a.H + r0 + 32 * q,
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
                            a.out_sorted[(size_t)(p0 + jc) * a.H + r0 + row] = acc0[jj] * exp2i(etab[jc]);
                        }
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
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace moeq
