// moeq.cu -- libmoeq: host side of the C ABI declared in include/moeq.h, and
// the one translation unit that instantiates every kernel.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "combine.cuh"
#include "common.cuh"
#include "ffn_gemm.cuh"
#include "ffn_gemv.cuh"
#include "ffn_mma8.cuh"
#include "permute.cuh"
#include "quant.cuh"
#include "route.cuh"
#include "route_tc.cuh"

using namespace moeq;

namespace {

thread_local std::string g_err;

// kernel tracing (moe_trace_events)
thread_local cudaEvent_t *g_trace = nullptr;
thread_local int g_trace_n = 0, g_trace_c = 0;

// Under stream capture a plain cudaEventRecord only expresses a dependency;
// cudaEventRecordExternal makes it an event-record node that fires on replay.
void trace_record(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cs);
    if (cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, s);
}
void trace_begin(cudaStream_t s) {
    if (g_trace_n) trace_record(g_trace[g_trace_c], s);
}
void trace_end(cudaStream_t s) {
    if (g_trace_n) {
        trace_record(g_trace[g_trace_c + 1], s);
        g_trace_c = (g_trace_c + 2) % g_trace_n;
    }
}

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int ok() {
    g_err.clear();
    return MOEQ_OK;
}

int cuda_check(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return MOEQ_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Token count up to which the router logits come from the GEMV router kernel.
constexpr int kRouteGemvMaxT = 64;
// Token count up to which auto mode runs the routed experts as GEMVs: measured
// on B300 (2048/512/512, top-10, 2-bit, experts read from HBM), the GEMV path
// took 39 / 181 / 552 / 766 / 1237 us per layer at T = 8 / 64 / 256 / 512 / 1024
// against 177 / 614 / 1003 / 1029 / 1066 us for the grouped GEMM.
constexpr int kExpertGemvMaxT = 512;
// Token count up to which the decode fast path fuses routing and permutation.
constexpr int kFusedRouteMaxT = kFusedMaxT;  // (the router kernel's tail handles up to 64 tokens)
// Token count up to which every expert CTA ranks the router logits itself.
#ifdef MOEQ_INCTA_ROUTE_MAXT
constexpr int kInCtaRouteMaxT = MOEQ_INCTA_ROUTE_MAXT;
#else
constexpr int kInCtaRouteMaxT = 2;
#endif

struct Layout {
    size_t ctrl, logits, idx, w, counts, offsets, perm_tok, perm_slot, inv, masks, prefix, chunk_count, chunk_base, units,
        tiles, tiles2, qx, sx,
        ex, xsum, ximg, qh, sh, eh, himg, total;
};

Layout layout(long long T, long long H, long long I, long long E, long long k) {
    Layout L;
    size_t off = 0;
    auto take = [&](long long bytes) {
        size_t o = off;
        off += ((size_t)(bytes > 0 ? bytes : 0) + 255) & ~(size_t)255;
        return o;
    };
    const long long P = T * k, W = (T + 31) / 32;
    const long long max_tiles = (P + kTileMin - 1) / kTileMin + E;
    L.ctrl = take(256);
    L.logits = take(T * E * 4);
    L.idx = take(P * 4);
    L.w = take(P * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm_tok = take(P * 4);
    L.perm_slot = take(P * 4);
    L.inv = take(P * 4);
    L.masks = take(E * W * 4);
    L.prefix = take(E * W * 4);
    const long long NC = (W + kPermChunkWords - 1) / kPermChunkWords;
    L.chunk_count = take(NC * E * 4);
    L.chunk_base = take(NC * E * 4);
    L.units = take(E * (long long)sizeof(UnitRec));
    L.tiles = take(max_tiles * (long long)sizeof(Tile));
    L.tiles2 = take(max_tiles * (long long)sizeof(Tile));
    L.qx = take(T * H);
    L.sx = take(T * (H / 32) * 4);
    L.ex = take(P * 4);
    L.xsum = take(T * (H / 32) * 4);
    L.ximg = take(2 * (P + kTileMax) * H * 2);  // hi + lo operand image, kTileMax rows of slack
    L.qh = take(P * I);
    L.sh = take(P * (I / 32) * 4);
    L.eh = take(P * 4);
    L.himg = take(2 * (P + kTileMax) * I * 2);
    L.total = off;
    return L;
}

int check_shape(int T, int H, int I, int E, int k) {
    if (T < 0) return fail(MOEQ_ERR_ARG, "T = %d < 0", T);
    if (E < 1 || E > kMaxE) return fail(MOEQ_ERR_SHAPE, "E = %d outside [1, %d]", E, kMaxE);
    if (k < 1 || k > E || k > kMaxK) return fail(MOEQ_ERR_SHAPE, "k = %d outside [1, min(E, %d)]", k, kMaxK);
    if (H < 128 || H > 16384 || H % 128) return fail(MOEQ_ERR_SHAPE, "H = %d: need a multiple of 128 in [128, 16384]", H);
    if (I < 128 || I > 4096 || I % 128) return fail(MOEQ_ERR_SHAPE, "I = %d: need a multiple of 128 in [128, 4096]", I);
    if ((long long)T * k > (1ll << 26)) return fail(MOEQ_ERR_SHAPE, "T*k = %lld too large", (long long)T * k);
    return MOEQ_OK;
}

#define REQ_PTR(p)                                                                                  \
    do {                                                                                            \
        if (!(p)) return fail(MOEQ_ERR_ARG, "%s is NULL", #p);                                      \
        if (!aligned((p), 16)) return fail(MOEQ_ERR_ALIGN, "%s is not 16-byte aligned", #p);        \
    } while (0)
#define OPT_PTR(p)                                                                                  \
    do {                                                                                            \
        if ((p) && !aligned((p), 16)) return fail(MOEQ_ERR_ALIGN, "%s is not 16-byte aligned", #p); \
    } while (0)

int check_ws(void *ws, size_t ws_bytes, const Layout &L) {
    if (!ws) return fail(MOEQ_ERR_ARG, "ws is NULL");
    if (!aligned(ws, 256)) return fail(MOEQ_ERR_ALIGN, "ws is not 256-byte aligned");
    if (ws_bytes < L.total) return fail(MOEQ_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, L.total);
    return MOEQ_OK;
}

int check_weights(const moe_qweights *wq, int H, int I, int E) {
    if (!wq) return fail(MOEQ_ERR_ARG, "weights is NULL");
    if (wq->bits != 2 && wq->bits != 3) return fail(MOEQ_ERR_SHAPE, "bits = %d (need 2 or 3)", wq->bits);
    if (wq->H != H || wq->I != I || wq->E != E)
        return fail(MOEQ_ERR_ARG, "weights describe E=%d H=%d I=%d, call uses E=%d H=%d I=%d", wq->E, wq->H, wq->I,
                    E, H, I);
    for (int m = 0; m < 3; ++m) {
        if (!wq->codes[m] || !wq->scales[m]) return fail(MOEQ_ERR_ARG, "weight matrix %d is NULL", m);
        if (!aligned(wq->codes[m], 16) || !aligned(wq->scales[m], 16))
            return fail(MOEQ_ERR_ALIGN, "weight matrix %d is not 16-byte aligned", m);
    }
    return MOEQ_OK;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

template <int PER>
void launch_topk(const float *logits, int T, int E, int k, int32_t *idx, float *w, cudaStream_t s) {
    const int blocks = (T * 32 + 255) / 256;
    topk_kernel<PER><<<blocks, 256, 0, s>>>(logits, T, E, k, idx, w);
}

void topk_dispatch(const float *logits, int T, int E, int k, int32_t *idx, float *w, cudaStream_t s) {
    const int per = (E + 31) / 32;
    if (per <= 1) launch_topk<1>(logits, T, E, k, idx, w, s);
    else if (per <= 2) launch_topk<2>(logits, T, E, k, idx, w, s);
    else if (per <= 4) launch_topk<4>(logits, T, E, k, idx, w, s);
    else if (per <= 8) launch_topk<8>(logits, T, E, k, idx, w, s);
    else if (per <= 16) launch_topk<16>(logits, T, E, k, idx, w, s);
    else launch_topk<32>(logits, T, E, k, idx, w, s);
}

// Largest dynamic shared memory a CTA may opt into on this device.
int max_smem_optin() {
    static int v = 0;
    if (!v) {
        int dev = 0, val = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&val, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess && val > 0)
            v = val;
        else
            v = 48 * 1024;
    }
    return v;
}

// Launch with programmatic stream serialisation: the kernel may start while the
// previous kernel on the stream finishes; it calls pdl_wait() before touching
// anything that earlier work produces.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int PER, int MAXT>
int launch_route_gemv_t(const float *x, int T, int H, const float *Wr, const float *bias, int E, float *logits,
                        const DecodeTail &tail, cudaStream_t s) {
    const size_t smem = route_smem(H, E).total;
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(route_gemv_kernel<PER, MAXT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "route smem attribute: %s", cudaGetErrorString(e));
    }
    const unsigned blocks = (unsigned)((E + kRouteRows - 1) / kRouteRows);
    cudaError_t e = launch_pdl(route_gemv_kernel<PER, MAXT>, blocks, 256, smem, s, x, T, H, Wr, bias, E, logits, tail);
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "route_gemv_kernel: %s", cudaGetErrorString(e));
    return MOEQ_OK;
}

// One token (and no routing tail): the single-token router kernel.
template <int PER>
int launch_route_gemv(const float *x, int T, int H, const float *Wr, const float *bias, int E, float *logits,
                      const DecodeTail &tail, cudaStream_t s) {
    if (T == 1 && tail.mode < 2) return launch_route_gemv_t<PER, 1>(x, T, H, Wr, bias, E, logits, tail, s);
    return launch_route_gemv_t<PER, kRouteTok>(x, T, H, Wr, bias, E, logits, tail, s);
}

int route_gemv_dispatch(const float *x, int T, int H, const float *Wr, const float *bias, int E, float *logits,
                        const DecodeTail &tail, cudaStream_t s) {
    const int per = (E + 31) / 32;
    if (per <= 1) return launch_route_gemv<1>(x, T, H, Wr, bias, E, logits, tail, s);
    if (per <= 2) return launch_route_gemv<2>(x, T, H, Wr, bias, E, logits, tail, s);
    if (per <= 4) return launch_route_gemv<4>(x, T, H, Wr, bias, E, logits, tail, s);
    if (per <= 8) return launch_route_gemv<8>(x, T, H, Wr, bias, E, logits, tail, s);
    if (per <= 16) return launch_route_gemv<16>(x, T, H, Wr, bias, E, logits, tail, s);
    return launch_route_gemv<32>(x, T, H, Wr, bias, E, logits, tail, s);
}

int tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint64_t esize, uint64_t cols, uint64_t rows,
            uint32_t box_c, uint32_t box_r, CUtensorMapSwizzle swz);
int max_smem_optin();

// Router logits of a prompt chunk on the tensor cores (3xTF32).
int route_tc(const float *x, int T, int H, const float *Wr, const float *bias, int E, float *logits, cudaStream_t s) {
    RouteTcArgs g{};
    g.T = T;
    g.H = H;
    g.E = E;
    g.bias = bias;
    g.logits = logits;
    if (int rc = tmap_2d(&g.tm_x, x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)H, (uint64_t)T, kRtK, kRtM,
                         CU_TENSOR_MAP_SWIZZLE_128B))
        return rc;
    if (int rc = tmap_2d(&g.tm_w, Wr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)H, (uint64_t)E, kRtK, kRtN,
                         CU_TENSOR_MAP_SWIZZLE_128B))
        return rc;
    if ((int)kRtSmem > max_smem_optin()) return fail(MOEQ_ERR_SHAPE, "router GEMM needs %zu bytes of shared memory", kRtSmem);
    cudaError_t e = cudaFuncSetAttribute(route_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRtSmem);
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "router smem attribute: %s", cudaGetErrorString(e));
    dim3 grid((E + kRtN - 1) / kRtN, (T + kRtM - 1) / kRtM);
    trace_begin(s);
    route_tc_kernel<<<grid, 320, kRtSmem, s>>>(g);
    trace_end(s);
    return cuda_check("route_tc_kernel");
}

// Router logits + top-k (unfused).
int route_unfused(const float *x, int T, int H, const float *Wr, const float *bias, int E, int k, int32_t *idx,
                  float *w, float *logits, cudaStream_t s) {
    if (T <= kRouteGemvMaxT) {
        DecodeTail none{};
        if (int rc = route_gemv_dispatch(x, T, H, Wr, bias, E, logits, none, s)) return rc;
    } else {
        if (int rc = route_tc(x, T, H, Wr, bias, E, logits, s)) return rc;
    }
    topk_dispatch(logits, T, E, k, idx, w, s);
    return MOEQ_OK;
}

// cuTensorMapEncodeTiled from the driver (looked up once, no link-time libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D TMA map over a row-major [rows][cols] array of esize-byte elements with
// box {box_c, box_r}; zero fill outside the array.
int tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint64_t esize, uint64_t cols, uint64_t rows,
            uint32_t box_c, uint32_t box_r, CUtensorMapSwizzle swz) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
    if (!enc) return fail(MOEQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * esize};
    cuuint32_t box[2] = {box_c, box_r};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOEQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return MOEQ_OK;
}

template <int BITS, int PER, int MAXNT>
int launch_gemv(GemvArgs g, int T, int k, int E, cudaStream_t s) {
    const int cap = max_smem_optin();
    g.kc = std::min(g.H / 32, kGvMaxKB);
    g.rc = std::min(g.H, kGvMaxRows);
    g.tc = MAXNT;
    auto need = [&]() { return (int)gemv_smem(g.H, BITS, g.kc, g.rc, g.tc).total; };
    while (need() > cap && g.tc > 1) g.tc /= 2;
    while (need() > cap && g.kc > 4) g.kc = (g.kc + 1) / 2;
    while (need() > cap && g.rc > 128) g.rc /= 2;
    const int smem = need();
    if (smem > cap) return fail(MOEQ_ERR_SHAPE, "expert GEMV needs %d bytes of shared memory (%d available)", smem, cap);
    if (g.route_mode == 1 && T > g.tc) return fail(MOEQ_ERR_SHAPE, "in-CTA routing needs T <= %d here", g.tc);
    const uint64_t rows = (uint64_t)E * (uint64_t)(g.H / 32);  // (expert, K-block) rows of gate/up
    for (int m = 0; m < 2; ++m) {
        if (int rc = tmap_2d(&g.tm[m], g.codes[m], CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, (uint64_t)g.I * BITS, rows,
                             32 * BITS, (uint32_t)g.kc, CU_TENSOR_MAP_SWIZZLE_NONE))
            return rc;
        if (int rc = tmap_2d(&g.tm[2 + m], g.scales[m], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (uint64_t)g.I, rows, 32,
                             (uint32_t)g.kc, CU_TENSOR_MAP_SWIZZLE_NONE))
            return rc;
    }
    cudaError_t e = cudaFuncSetAttribute(ffn_gemv_kernel<BITS, PER, MAXNT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "gemv smem attribute: %s", cudaGetErrorString(e));
    const long long units = std::min<long long>((long long)T * k, E);
    const long long blocks = units * (g.I / 32);
    if (blocks == 0) return MOEQ_OK;
    trace_begin(s);
    e = launch_pdl(ffn_gemv_kernel<BITS, PER, MAXNT>, (unsigned)blocks, 256, (size_t)smem, s, g);
    trace_end(s);
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "ffn_gemv_kernel: %s", cudaGetErrorString(e));
    return cuda_check("ffn_gemv_kernel");
}

int gemv_dispatch(const GemvArgs &g, int bits, int T, int k, int E, cudaStream_t s) {
    const int per = (E + 31) / 32;
    // one token: the single-token kernel (every unit then holds one pair)
#define MOEQ_GEMV(P_)                                                                              \
    return T == 1 ? (bits == 2 ? launch_gemv<2, P_, 1>(g, T, k, E, s) : launch_gemv<3, P_, 1>(g, T, k, E, s)) \
                  : (bits == 2 ? launch_gemv<2, P_, kGvTok>(g, T, k, E, s) : launch_gemv<3, P_, kGvTok>(g, T, k, E, s))
    if (per <= 1) MOEQ_GEMV(1);
    if (per <= 2) MOEQ_GEMV(2);
    if (per <= 4) MOEQ_GEMV(4);
    if (per <= 8) MOEQ_GEMV(8);
    if (per <= 16) MOEQ_GEMV(16);
    MOEQ_GEMV(32);
#undef MOEQ_GEMV
}

int sm_count() {
    static int v = 0;
    if (!v) {
        int dev = 0, val = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&val, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && val > 0)
            v = val;
        else
            v = 148;
    }
    return v;
}

// The persistent grouped GEMM: one CTA per SM (at most one per work item).
template <bool GATEUP, int BITS>
int launch_gemm(const GemmArgs &g, long long max_tiles, cudaStream_t s) {
    using C = GemmCfg<GATEUP, BITS>;
    if ((int)C::SMEM > max_smem_optin()) return fail(MOEQ_ERR_SHAPE, "grouped GEMM needs %zu bytes of shared memory", C::SMEM);
    cudaError_t e = cudaFuncSetAttribute(ffn_gemm_kernel<GATEUP, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "gemm smem attribute: %s", cudaGetErrorString(e));
    const int MT = (GATEUP ? g.I : g.H) / kGmM;
    const long long items = max_tiles * MT;
    if (items == 0) return MOEQ_OK;
    const unsigned blocks = (unsigned)std::min<long long>(items, sm_count());
    trace_begin(s);
    ffn_gemm_kernel<GATEUP, BITS><<<blocks, C::THREADS, C::SMEM, s>>>(g);
    trace_end(s);
    return cuda_check("ffn_gemm_kernel");
}

// The warp-level int8 grouped GEMM (comparison path): persistent, as many
// CTAs as fit on the GPU (at most one per work item).
template <bool GATEUP, int BITS>
int launch_mma8(const Mma8Args &g, long long max_tiles, cudaStream_t s) {
    using C = Mma8Cfg<GATEUP, BITS>;
    if (C::SMEM > max_smem_optin()) return fail(MOEQ_ERR_SHAPE, "int8 GEMM needs %d bytes of shared memory", C::SMEM);
    cudaError_t e = cudaFuncSetAttribute(ffn_mma8_kernel<GATEUP, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM);
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "int8 GEMM smem attribute: %s", cudaGetErrorString(e));
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ffn_mma8_kernel<GATEUP, BITS>, kM8Threads, C::SMEM);
    if (e != cudaSuccess || per_sm < 1) return fail(MOEQ_ERR_CUDA, "int8 GEMM occupancy query failed");
    const long long items = max_tiles * ((GATEUP ? g.I : g.H) / C::ROWS);
    if (items == 0) return MOEQ_OK;
    const unsigned blocks = (unsigned)std::min<long long>(items, (long long)sm_count() * per_sm);
    trace_begin(s);
    ffn_mma8_kernel<GATEUP, BITS><<<blocks, kM8Threads, C::SMEM, s>>>(g);
    trace_end(s);
    return cuda_check("ffn_mma8_kernel");
}

// The token-to-expert permutation on the whole GPU (three small kernels).
int permute_multi(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offsets, int32_t *perm_tok,
                  int32_t *perm_slot, int32_t *inv, void *ws, const Layout &L, cudaStream_t s) {
    const int W = (T + 31) / 32, NC = (W + kPermChunkWords - 1) / kPermChunkWords;
    unsigned *masks = at<unsigned>(ws, L.masks);
    int *wprefix = at<int>(ws, L.prefix), *ccount = at<int>(ws, L.chunk_count), *cbase = at<int>(ws, L.chunk_base);
    permute_count_kernel<<<NC, 256, 0, s>>>(idx, T, k, E, masks, wprefix, ccount);
    permute_scan_kernel<<<1, 1024, 0, s>>>(NC, E, ccount, cbase, counts, offsets);
    const long long P = (long long)T * k;
    const unsigned blocks = (unsigned)std::min<long long>((P + 255) / 256, (long long)sm_count() * 8);
    permute_scatter_kernel<<<blocks, 256, 0, s>>>(idx, T, k, E, masks, wprefix, cbase, offsets, perm_tok, perm_slot,
                                                  inv);
    return cuda_check("permute kernels");
}

// Experts over an existing permutation.
int experts(const float *x, int T, const moe_qweights *wq, int k, const int32_t *offsets, const int32_t *perm_tok,
            const int32_t *perm_slot, const float *w, float *out_sorted, float *y, int residual, int mode,
            int8_t *qh_out, float *sh_out, void *ws, const Layout &L, cudaStream_t s, bool init_y = true,
            const int32_t *inv = nullptr) {
    const int H = wq->H, I = wq->I, E = wq->E, bits = wq->bits;
    const long long P = (long long)T * k;
    if (mode == MOEQ_MODE_AUTO) mode = T <= kExpertGemvMaxT ? MOEQ_MODE_GEMV : MOEQ_MODE_GEMM;
    int *ctrl = at<int>(ws, L.ctrl);
    if (y && init_y) {
        const size_t n = (size_t)T * H;
        const int blocks = (int)std::min<size_t>((n / 4 + 255) / 256, 148 * 16);
        if (blocks > 0) init_y_kernel<<<blocks, 256, 0, s>>>(x, y, n, residual);
    }
    if (T == 0) return cuda_check("init_y_kernel");
    const bool s8 = mode == MOEQ_MODE_GEMM_S8;
    plan_kernel<<<1, 1024, 0, s>>>(offsets, E, T, ctrl, mode == MOEQ_MODE_GEMV ? at<UnitRec>(ws, L.units) : nullptr,
                                   perm_tok, perm_slot, y ? w : nullptr, k, at<Tile>(ws, L.tiles),
                                   s8 ? kM8Tile : bits == 2 ? GemmCfg<true, 2>::TILE_N : GemmCfg<true, 3>::TILE_N,
                                   at<Tile>(ws, L.tiles2),
                                   s8 ? kM8Tile : bits == 2 ? GemmCfg<false, 2>::TILE_N : GemmCfg<false, 3>::TILE_N);
    if (int rc = cuda_check("plan_kernel")) return rc;
    if (s8) {
        // both GEMMs on the warp-level int8 path: x quantised per token, gate/up
        // re-quantises h in its epilogue, down reads those int8 rows directly
        int8_t *qx = at<int8_t>(ws, L.qx);
        float *sx = at<float>(ws, L.sx);
        quant_rows_kernel<<<T, 256, 0, s>>>(x, H, qx, sx, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                            0);
        if (int rc = cuda_check("quant_rows_kernel(x)")) return rc;
        const long long max_tiles = (P + kM8Tile - 1) / kM8Tile + E;
        Mma8Args g{};
        g.T = T;
        g.H = H;
        g.I = I;
        g.E = E;
        g.k = k;
        for (int m = 0; m < 3; ++m) {
            g.codes[m] = wq->codes[m];
            g.scales[m] = wq->scales[m];
        }
        g.tiles = at<Tile>(ws, L.tiles);
        g.ntiles = ctrl + 2;
        g.perm_tok = perm_tok;
        g.perm_slot = perm_slot;
        g.w = w;
        g.aq = qx;
        g.as = sx;
        g.qh = qh_out ? qh_out : at<int8_t>(ws, L.qh);
        g.sh = sh_out ? sh_out : at<float>(ws, L.sh);
        int rc = bits == 2 ? launch_mma8<true, 2>(g, max_tiles, s) : launch_mma8<true, 3>(g, max_tiles, s);
        if (rc) return rc;
        g.tiles = at<Tile>(ws, L.tiles2);
        g.ntiles = ctrl + kCtrlTiles2;
        g.aq = g.qh;
        g.as = g.sh;
        g.y = y;
        g.out_sorted = out_sorted;
        return bits == 2 ? launch_mma8<false, 2>(g, max_tiles, s) : launch_mma8<false, 3>(g, max_tiles, s);
    }
    if (mode == MOEQ_MODE_GEMV) {
        if (out_sorted) cudaMemsetAsync(out_sorted, 0, (size_t)P * H * sizeof(float), s);
        quant_rows_kernel<<<T, 256, 0, s>>>(x, H, at<int8_t>(ws, L.qx), at<float>(ws, L.sx), nullptr, nullptr,
                                            nullptr, nullptr, nullptr, nullptr, at<int>(ws, L.xsum), bits == 2);
        if (int rc = cuda_check("quant_rows_kernel(x)")) return rc;
        GemvArgs g{};
        g.x = x;
        g.qx = at<int8_t>(ws, L.qx);
        g.sx = at<float>(ws, L.sx);
        g.xsum = at<int>(ws, L.xsum);
        g.T = T;
        g.H = H;
        g.I = I;
        g.E = E;
        g.k = k;
        for (int m = 0; m < 3; ++m) {
            g.codes[m] = wq->codes[m];
            g.scales[m] = wq->scales[m];
        }
        g.perm_tok = perm_tok;
        g.perm_slot = perm_slot;
        g.w = w;
        g.units = at<UnitRec>(ws, L.units);
        g.ctrl = ctrl;
        g.route_mode = 0;
        g.y = y;
        g.out_sorted = out_sorted;
        g.qh_out = qh_out;
        g.sh_out = sh_out;
        return gemv_dispatch(g, bits, T, k, E, s);
    }
    // grouped tensor-core GEMMs
    int *ex = at<int>(ws, L.ex);
    __half *ximg = at<__half>(ws, L.ximg);
    int8_t *qh = qh_out ? qh_out : at<int8_t>(ws, L.qh);
    float *sh = sh_out ? sh_out : at<float>(ws, L.sh);
    int *eh = at<int>(ws, L.eh);
    __half *himg = at<__half>(ws, L.himg);
    const long long img_rows = P + kTileMax;  // a tile's rows may run up to kTileMax - 1 past P
    // x quantised per token and its fp16 hi/lo rows written in sorted pair
    // order (pre-swizzled per tile), in one pass, so that every GEMM tile reads
    // one contiguous run of B rows per K stage.  The pairs' sorted positions
    // come from the permutation's inverse (computed here when not given).
    if (!inv) {
        int32_t *winv = at<int32_t>(ws, L.inv);
        cudaMemsetAsync(winv, 0xFF, (size_t)P * sizeof(int32_t), s);  // -1: a pair the permutation rejected
        const unsigned pr_blocks = (unsigned)std::min<long long>((P + 255) / 256, (long long)sm_count() * 8);
        pair_rows_kernel<<<pr_blocks, 256, 0, s>>>(perm_tok, perm_slot, (int)P, T, k, winv);
        if (int rc = cuda_check("pair_rows_kernel")) return rc;
        inv = winv;
        // rows of a caller's inconsistent permutation that no pair claims: zeroed
        const unsigned or_blocks = (unsigned)std::min<long long>((P + 7) / 8, (long long)sm_count() * 16);
        orphan_rows_kernel<<<or_blocks, 256, 0, s>>>(perm_tok, perm_slot, (int)P, T, k, inv, H, ximg, img_rows, ex);
        if (int rc = cuda_check("orphan_rows_kernel")) return rc;
    }
    const unsigned qs_blocks = (unsigned)std::min<long long>(((long long)T + 7) / 8, (long long)sm_count() * 16);
    quant_split_kernel<<<qs_blocks, 256, 0, s>>>(x, T, H, k, inv, offsets, E, ximg, img_rows, ex);
    if (int rc = cuda_check("quant_split_kernel")) return rc;
    const unsigned split_blocks = (unsigned)std::min<long long>((P + 7) / 8, (long long)sm_count() * 16);
    const long long max_tiles = (P + kTileMin - 1) / kTileMin + E;
    GemmArgs g{};
    g.T = T;
    g.H = H;
    g.I = I;
    g.E = E;
    g.k = k;
    for (int m = 0; m < 3; ++m) {
        g.codes[m] = wq->codes[m];
        g.scales[m] = wq->scales[m];
    }
    g.tiles = at<Tile>(ws, L.tiles);
    g.ntiles = ctrl + 2;
    g.perm_tok = perm_tok;
    g.perm_slot = perm_slot;
    g.w = w;
    g.bimg = ximg;
    g.bimg_rows = img_rows;
    g.brow_exp = ex;
    g.qh = qh;
    g.sh = sh;
    int rc = bits == 2 ? launch_gemm<true, 2>(g, max_tiles, s) : launch_gemm<true, 3>(g, max_tiles, s);
    if (rc) return rc;
    split_rows_kernel<<<split_blocks, 256, 0, s>>>(qh, sh, I, nullptr, (int)P, (int)P, offsets, E, himg, img_rows, eh);
    if ((rc = cuda_check("split_rows_kernel(h)"))) return rc;
    g.bimg = himg;
    g.tiles = at<Tile>(ws, L.tiles2);
    g.ntiles = ctrl + kCtrlTiles2;
    g.brow_exp = eh;
    g.y = y;
    g.out_sorted = out_sorted;
    return bits == 2 ? launch_gemm<false, 2>(g, max_tiles, s) : launch_gemm<false, 3>(g, max_tiles, s);
}

// Scratch of moe_permute_noalloc: token bitmaps [E][W] then prefix counts
// [E][W], W = ceil(T/32), each at most kNoAllocWords 32-bit words.
constexpr size_t kNoAllocWords = 65536;
__device__ __align__(256) unsigned g_permute_scratch[2 * kNoAllocWords];

// Device address of g_permute_scratch, looked up once per device ordinal.
constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

int noalloc_scratch(unsigned **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(MOEQ_ERR_ARG, "device ordinal %d not supported", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_permute_scratch);
        if (e != cudaSuccess || !p)
            return fail(MOEQ_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<unsigned *>(g_scratch_addr[dev]);
    return MOEQ_OK;
}

}  // namespace

extern "C" {

const char *moe_last_error_string(void) { return g_err.c_str(); }

const char *moe_version(void) { return "moeq 0.1.0 sm_103a"; }

int moe_trace_events(void *const *events, int n) {
    if (n < 0 || (n & 1) || (n > 0 && !events)) return fail(MOEQ_ERR_ARG, "need an even number of events");
    static thread_local cudaEvent_t store[4096];
    if (n > 4096) return fail(MOEQ_ERR_ARG, "at most 4096 trace events");
    for (int i = 0; i < n; ++i) store[i] = (cudaEvent_t)events[i];
    g_trace = n ? store : nullptr;
    g_trace_n = n;
    g_trace_c = 0;
    return ok();
}

size_t moe_workspace_bytes(int T, int H, int I, int E, int k, int bits) {
    if (check_shape(T, H, I, E, k) != MOEQ_OK || (bits != 2 && bits != 3)) return 0;
    return layout(T, H, I, E, k).total;
}

int moe_route_topk(const float *x, int T, int H, const float *Wr, const float *bias, int E, int k, int32_t *idx_out,
                   float *w_out, void *ws, size_t ws_bytes, void *stream) {
    if (int rc = check_shape(T, H, 128, E, k)) return rc;
    REQ_PTR(x);
    REQ_PTR(Wr);
    OPT_PTR(bias);
    REQ_PTR(idx_out);
    REQ_PTR(w_out);
    const Layout L = layout(T, H, 128, E, k);
    if (ws_bytes < L.logits + (size_t)T * E * 4) return fail(MOEQ_ERR_WORKSPACE, "workspace too small for logits");
    if (!ws || !aligned(ws, 256)) return fail(MOEQ_ERR_ALIGN, "ws missing or not 256-byte aligned");
    if (T == 0) return ok();
    cudaStream_t s = (cudaStream_t)stream;
    if (int rc = route_unfused(x, T, H, Wr, bias, E, k, idx_out, w_out, at<float>(ws, L.logits), s)) return rc;
    if (int rc = cuda_check("moe_route_topk")) return rc;
    return ok();
}

int moe_permute(const int32_t *idx, int T, int k, int E, int32_t *counts_out, int32_t *offsets_out,
                int32_t *perm_tok_out, int32_t *perm_slot_out, int32_t *inv_out, void *ws, size_t ws_bytes,
                void *stream) {
    if (int rc = check_shape(T, 128, 128, E, k)) return rc;
    REQ_PTR(counts_out);
    REQ_PTR(offsets_out);
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {
        cudaMemsetAsync(counts_out, 0, (size_t)E * 4, s);
        cudaMemsetAsync(offsets_out, 0, (size_t)(E + 1) * 4, s);
        if (int rc = cuda_check("moe_permute")) return rc;
        return ok();
    }
    REQ_PTR(idx);
    REQ_PTR(perm_tok_out);
    REQ_PTR(perm_slot_out);
    REQ_PTR(inv_out);
    const Layout L = layout(T, 128, 128, E, k);
    if (!ws || !aligned(ws, 256)) return fail(MOEQ_ERR_ALIGN, "ws missing or not 256-byte aligned");
    if (ws_bytes < L.chunk_base + (size_t)E * (((T + 31) / 32 + kPermChunkWords - 1) / kPermChunkWords) * 4)
        return fail(MOEQ_ERR_WORKSPACE, "workspace too small");
    if (int rc = permute_multi(idx, T, k, E, counts_out, offsets_out, perm_tok_out, perm_slot_out, inv_out, ws, L, s))
        return rc;
    return ok();
}

int moe_permute_noalloc(const int32_t *idx, int T, int k, int E, int32_t *counts_out, int32_t *offsets_out,
                        int32_t *perm_tok_out, int32_t *perm_slot_out, int32_t *inv_out, void *stream) {
    if (int rc = check_shape(T, 128, 128, E, k)) return rc;
    REQ_PTR(counts_out);
    REQ_PTR(offsets_out);
    const size_t words = (size_t)E * (size_t)((T + 31) / 32);
    if (words > kNoAllocWords)
        return fail(MOEQ_ERR_SHAPE, "moe_permute_noalloc: E * ceil(T/32) = %zu exceeds its fixed scratch of %zu words",
                    words, kNoAllocWords);
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {
        cudaMemsetAsync(counts_out, 0, (size_t)E * 4, s);
        cudaMemsetAsync(offsets_out, 0, (size_t)(E + 1) * 4, s);
        if (int rc = cuda_check("moe_permute_noalloc")) return rc;
        return ok();
    }
    REQ_PTR(idx);
    REQ_PTR(perm_tok_out);
    REQ_PTR(perm_slot_out);
    REQ_PTR(inv_out);
    unsigned *scratch = nullptr;
    if (int rc = noalloc_scratch(&scratch)) return rc;
    // permute_kernel zeroes the bitmaps itself before use
    permute_kernel<<<1, 1024, 0, s>>>(idx, T, k, E, scratch, reinterpret_cast<int *>(scratch + kNoAllocWords),
                                      counts_out, offsets_out, perm_tok_out, perm_slot_out, inv_out);
    if (int rc = cuda_check("permute_kernel(noalloc)")) return rc;
    return ok();
}

int moe_quantize_act(const float *x, int T, int H, int8_t *q_out, float *s_out, void *stream) {
    if (T < 0) return fail(MOEQ_ERR_ARG, "T < 0");
    if (H < 32 || H % 32 || H > (1 << 20)) return fail(MOEQ_ERR_SHAPE, "H = %d must be a positive multiple of 32", H);
    if (T == 0) return ok();
    REQ_PTR(x);
    REQ_PTR(q_out);
    REQ_PTR(s_out);
    quant_rows_kernel<<<T, 256, 0, (cudaStream_t)stream>>>(x, H, q_out, s_out, nullptr, nullptr, nullptr, nullptr,
                                                            nullptr, nullptr, nullptr, 0);
    if (int rc = cuda_check("quant_rows_kernel")) return rc;
    return ok();
}

int moe_expert_ffn_q2(const float *x, int T, const moe_qweights *weights, int k, const int32_t *offsets,
                      const int32_t *perm_tok, const int32_t *perm_slot, const float *w, float *out_sorted, float *y,
                      int residual, int mode, int8_t *qh_out, float *sh_out, void *ws, size_t ws_bytes,
                      void *stream) {
    if (!weights) return fail(MOEQ_ERR_ARG, "weights is NULL");
    const int H = weights->H, I = weights->I, E = weights->E;
    if (int rc = check_shape(T, H, I, E, k)) return rc;
    if (int rc = check_weights(weights, H, I, E)) return rc;
    if (mode < MOEQ_MODE_AUTO || mode > MOEQ_MODE_GEMM_S8) return fail(MOEQ_ERR_ARG, "mode = %d", mode);
    if (!out_sorted && !y) return fail(MOEQ_ERR_ARG, "need out_sorted or y");
    OPT_PTR(out_sorted);
    OPT_PTR(y);
    OPT_PTR(qh_out);
    OPT_PTR(sh_out);
    if (T > 0) {
        REQ_PTR(x);
        REQ_PTR(offsets);
        REQ_PTR(perm_tok);
        REQ_PTR(perm_slot);
        if (y) REQ_PTR(w);
    }
    const Layout L = layout(T, H, I, E, k);
    if (int rc = check_ws(ws, ws_bytes, L)) return rc;
    if (int rc = experts(x, T, weights, k, offsets, perm_tok, perm_slot, w, out_sorted, y, residual, mode, qh_out,
                         sh_out, ws, L, (cudaStream_t)stream))
        return rc;
    return ok();
}

int moe_shared_expert_q2(const float *x, int T, const moe_qweights *shared, float *y, int accumulate, int mode,
                         void *ws, size_t ws_bytes, void *stream) {
    if (!shared) return fail(MOEQ_ERR_ARG, "shared is NULL");
    const int H = shared->H, I = shared->I;
    if (shared->E != 1) return fail(MOEQ_ERR_ARG, "a shared expert is one expert (E = %d)", shared->E);
    if (int rc = check_shape(T, H, I, 1, 1)) return rc;
    if (int rc = check_weights(shared, H, I, 1)) return rc;
    if (mode < MOEQ_MODE_AUTO || mode > MOEQ_MODE_GEMM_S8) return fail(MOEQ_ERR_ARG, "mode = %d", mode);
    if (T > 0) {
        REQ_PTR(x);
        REQ_PTR(y);
    }
    const Layout L = layout(T, H, I, 1, 1);
    if (int rc = check_ws(ws, ws_bytes, L)) return rc;
    if (T == 0) return ok();
    const cudaStream_t s = (cudaStream_t)stream;
    int32_t *offsets = at<int32_t>(ws, L.offsets), *perm_tok = at<int32_t>(ws, L.perm_tok);
    int32_t *perm_slot = at<int32_t>(ws, L.perm_slot);
    float *w = at<float>(ws, L.w);
    const unsigned blocks = (unsigned)std::min<long long>((T + 255) / 256, (long long)sm_count() * 4);
    shared_plan_kernel<<<blocks, 256, 0, s>>>(T, offsets, perm_tok, perm_slot, w);
    if (int rc = cuda_check("shared_plan_kernel")) return rc;
    if (int rc = experts(x, T, shared, 1, offsets, perm_tok, perm_slot, w, nullptr, y, 0, mode, nullptr, nullptr, ws,
                         L, s, /*init_y=*/accumulate == 0))
        return rc;
    return ok();
}

int moe_combine(const float *out_sorted, const int32_t *inv, const float *w, int T, int k, int H,
                const float *residual_x, float *y_out, void *stream) {
    if (T < 0 || k < 1 || k > kMaxK) return fail(MOEQ_ERR_ARG, "bad T or k");
    if (H < 4 || H % 4) return fail(MOEQ_ERR_SHAPE, "H = %d must be a positive multiple of 4", H);
    if (T == 0) return ok();
    REQ_PTR(out_sorted);
    REQ_PTR(inv);
    REQ_PTR(w);
    OPT_PTR(residual_x);
    REQ_PTR(y_out);
    combine_kernel<<<T, 256, 0, (cudaStream_t)stream>>>(out_sorted, inv, w, k, H, (long long)T * k, residual_x,
                                                            y_out);
    if (int rc = cuda_check("combine_kernel")) return rc;
    return ok();
}

int moe_layer_forward(const float *x, int T, const float *Wr, const float *bias, const moe_qweights *weights, int k,
                      int residual, float *y_out, int32_t *idx_out, float *w_out, int mode, void *ws,
                      size_t ws_bytes, void *stream) {
    if (!weights) return fail(MOEQ_ERR_ARG, "weights is NULL");
    const int H = weights->H, I = weights->I, E = weights->E;
    if (int rc = check_shape(T, H, I, E, k)) return rc;
    if (int rc = check_weights(weights, H, I, E)) return rc;
    if (mode < MOEQ_MODE_AUTO || mode > MOEQ_MODE_GEMM_S8) return fail(MOEQ_ERR_ARG, "mode = %d", mode);
    OPT_PTR(bias);
    OPT_PTR(idx_out);
    OPT_PTR(w_out);
    if (T > 0) {
        REQ_PTR(x);
        REQ_PTR(Wr);
        REQ_PTR(y_out);
    }
    const Layout L = layout(T, H, I, E, k);
    if (int rc = check_ws(ws, ws_bytes, L)) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) return ok();
    int32_t *idx = idx_out ? idx_out : at<int32_t>(ws, L.idx);
    float *w = w_out ? w_out : at<float>(ws, L.w);
    int32_t *counts = at<int32_t>(ws, L.counts), *offsets = at<int32_t>(ws, L.offsets);
    int32_t *perm_tok = at<int32_t>(ws, L.perm_tok), *perm_slot = at<int32_t>(ws, L.perm_slot);
    int32_t *inv = at<int32_t>(ws, L.inv);
    if (mode == MOEQ_MODE_AUTO) mode = T <= kExpertGemvMaxT ? MOEQ_MODE_GEMV : MOEQ_MODE_GEMM;
    if (T <= kFusedRouteMaxT && mode == MOEQ_MODE_GEMV) {
        // decode: two kernels chained by programmatic dependent launch.  The
        // router kernel also sets y = residual ? x : 0 and quantises x.  For
        // T <= kInCtaRouteMaxT every expert CTA ranks the logits itself (one
        // warp per token, no separate routing step); above that the router's
        // last CTA groups the pairs into per-expert records once.
        const bool in_cta = T <= kInCtaRouteMaxT;
        DecodeTail tail{};
        tail.mode = in_cta ? 1 : 2;
        tail.k = k;
        tail.idx = idx;
        tail.w = w;
        tail.perm_tok = perm_tok;
        tail.perm_slot = perm_slot;
        tail.inv = inv;
        tail.units = at<UnitRec>(ws, L.units);
        tail.ctrl = at<int>(ws, L.ctrl);
        tail.y = y_out;
        tail.residual = residual;
        tail.qx = at<int8_t>(ws, L.qx);
        tail.sx = at<float>(ws, L.sx);
        tail.xsum = at<int>(ws, L.xsum);
        tail.bits = weights->bits;
        float *logits = at<float>(ws, L.logits);
        if (int rc = route_gemv_dispatch(x, T, H, Wr, bias, E, logits, tail, s)) return rc;
        GemvArgs g{};
        g.x = x;
        g.qx = tail.qx;
        g.sx = tail.sx;
        g.xsum = tail.xsum;
        g.T = T;
        g.H = H;
        g.I = I;
        g.E = E;
        g.k = k;
        for (int m = 0; m < 3; ++m) {
            g.codes[m] = weights->codes[m];
            g.scales[m] = weights->scales[m];
        }
        g.perm_tok = perm_tok;
        g.perm_slot = perm_slot;
        g.w = w;
        g.units = tail.units;
        g.ctrl = tail.ctrl;
        g.route_mode = in_cta ? 1 : 0;
        g.logits = logits;
        g.idx_out = idx_out;
        g.w_out = w_out;
        g.y = y_out;
        if (int rc = gemv_dispatch(g, weights->bits, T, k, E, s)) return rc;
        return ok();
    }
    if (int rc = route_unfused(x, T, H, Wr, bias, E, k, idx, w, at<float>(ws, L.logits), s)) return rc;
    if (int rc = cuda_check("route")) return rc;
    if (int rc = permute_multi(idx, T, k, E, counts, offsets, perm_tok, perm_slot, inv, ws, L, s)) return rc;
    if (int rc = experts(x, T, weights, k, offsets, perm_tok, perm_slot, w, nullptr, y_out, residual, mode, nullptr,
                         nullptr, ws, L, s, true, inv))
        return rc;
    return ok();
}

#ifdef MOEQ_TIMELINE
// Tracing build only (not part of the C ABI): copies up to max_entries
// timeline entries (2 x uint64 each) to host memory, returns their number and
// clears the ring.
int moe_timeline_read(unsigned long long *host, int max_entries) {
    cudaDeviceSynchronize();
    unsigned n = 0;
    cudaMemcpyFromSymbol(&n, g_tl_n, sizeof n);
    const int m = (int)std::min<unsigned>(std::min<unsigned>(n, kTlEntries), (unsigned)max_entries);
    if (m > 0) cudaMemcpyFromSymbol(host, g_tl, (size_t)m * 16);
    unsigned zero = 0;
    cudaMemcpyToSymbol(g_tl_n, &zero, sizeof zero);
    return m;
}
#endif

#ifdef MOEQ_TIMELINE
// Tracing build only: copies the per-CTA wait counters of the two GEMMs
// ([2][256][16] uint64) to host memory and clears them.
int moe_gemm_waits_read(unsigned long long *host) {
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(host, g_gemm_waits, sizeof(g_gemm_waits));
    static unsigned long long zero[2][256][16];
    cudaMemcpyToSymbol(g_gemm_waits, zero, sizeof(zero));
    return 0;
}
#endif

int moe_set_wait_limit(uint64_t ns) {
    constexpr uint64_t kMaxLimitNs = 60ull * 1000000000ull;
    if (ns > kMaxLimitNs) return fail(MOEQ_ERR_ARG, "wait limit %llu ns above 60 s", (unsigned long long)ns);
    const uint64_t v = ns ? ns : kDefaultWaitLimitNs;
    cudaError_t e = cudaMemcpyToSymbol(g_wait_limit_ns, &v, sizeof v);
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "wait limit: %s", cudaGetErrorString(e));
    return ok();
}

int moe_get_device_status(void *stream, int *status_out) {
    if (!status_out) return fail(MOEQ_ERR_ARG, "status_out is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
    int st = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&st, g_status, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    if (e != cudaSuccess) return fail(MOEQ_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    *status_out = st;
    if (st) return fail(MOEQ_ERR_DEVICE, "device status 0x%x", st);
    return ok();
}

}  // extern "C"
