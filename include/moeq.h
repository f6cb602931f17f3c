/*
 * moeq.h -- C ABI of libmoeq, a routed mixture-of-experts FFN layer on 2-bit
 * (and 3-bit) block-quantised expert weights for NVIDIA B300 (sm_103a).
 *
 * The layer is the hot path of the MoE model the Strata pages describe: 512
 * experts per layer, 10 of them active per token ("Strata - the details",
 * section "Which model?"; upstream Strata README, "How does it work?"), with
 * the router and the cached experts on the GPU ("Strata - the details",
 * section "How it works") and prompt chunks multiplied on int8 tensor-core
 * kernels ("Strata - the details", section "Speed (measured)", engine 0.1.36
 * note).  Here every expert is resident in device memory and nothing runs on
 * the CPU.
 *
 * Conventions for every call
 * --------------------------
 * - Pointers named x, Wr, bias, idx, w, y, counts, offsets, perm_*, inv, q, s,
 *   out_sorted, qh, sh, ws and the weight codes/scales are DEVICE pointers in
 *   memory the caller allocated (cudaMalloc / PyTorch).  The library never
 *   allocates or frees device memory and keeps no pointer after a call returns.
 * - Row-major, densely packed arrays; fp32 = IEEE binary32, fp16 scales are
 *   passed as their 16-bit patterns.  Every device pointer must be 16-byte
 *   aligned; ws must be 256-byte aligned.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *   asynchronous: they enqueue kernels on `stream` and return without a host
 *   synchronisation (moe_get_device_status is the one exception).
 * - Return value: MOEQ_OK, or a negative MOEQ_ERR_* code, checked on the host
 *   before anything is enqueued; moe_last_error_string() (thread-local) then
 *   describes the failure.  No C++ exception crosses this interface.
 * - A workspace `ws` of at least moe_workspace_bytes(...) bytes is scratch
 *   owned by the library for the duration of the call; its content before
 *   and after a call is unspecified, except that a workspace must be zeroed
 *   once (cudaMemset) before its first use and must not be shared by calls
 *   that may run concurrently.
 * - Device-side waits (pipeline barriers inside the tensor-core kernels) are
 *   bounded; when one gives up the kernel records MOEQ_STATUS_WAIT_TIMEOUT in
 *   a per-device status word that moe_get_device_status() returns.
 *
 * Weight storage, per expert and per matrix of N output rows and K inputs:
 *   codes [E][K/32][N][4*bits bytes], scales [E][K/32][N] fp16.
 *   2-bit: element i of a 32-block is in byte i/4 at bit 2*(i%4); its value is
 *          (code - 2) * scale, i.e. levels {-2,-1,0,1} * scale.
 *   3-bit: element i occupies bits 3i..3i+2 of the block's 96-bit
 *          little-endian word; value (code - 4) * scale, levels -4..3.
 *   gate and up are [N=I, K=H]; down is [N=H, K=I].
 *   The pages name the Q2_0 format but not its bits; this layout is the
 *   library's and keeps one K-block of all rows contiguous.
 */
#ifndef MOEQ_H
#define MOEQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOEQ_OK 0
#define MOEQ_ERR_ARG -1        /* null pointer, non-positive size, k > E ... */
#define MOEQ_ERR_SHAPE -2      /* unsupported shape (see each call) */
#define MOEQ_ERR_ALIGN -3      /* pointer not 16-byte aligned (ws: 256) */
#define MOEQ_ERR_WORKSPACE -4  /* ws_bytes < moe_workspace_bytes(...) */
#define MOEQ_ERR_CUDA -5       /* a CUDA launch or query failed */
#define MOEQ_ERR_DEVICE -6     /* a kernel reported a device-side error */

#define MOEQ_STATUS_WAIT_TIMEOUT 0x1 /* a bounded device wait gave up */
#define MOEQ_STATUS_BAD_INDEX 0x2    /* an expert index outside [0, E) reached a kernel */

#define MOEQ_MODE_AUTO 0 /* GEMV for T <= 512 (faster there on B300), grouped GEMM otherwise */
#define MOEQ_MODE_GEMV 1 /* per-expert split GEMV with fused SwiGLU/down/combine */
#define MOEQ_MODE_GEMM 2 /* grouped tcgen05 tensor-core GEMMs */
/* Grouped GEMMs on the warp-level int8 tensor path (mma.sync s8), every
 * 32-block product an exact integer dot scaled in registers: the int8 MMAs of
 * the pages' fused prompt-expert kernels ("Strata - the details", "Speed
 * (measured)", 0.1.36).  A comparison path, slower than MOEQ_MODE_GEMM on
 * B300; MOEQ_MODE_AUTO never selects it. */
#define MOEQ_MODE_GEMM_S8 3

/* Supported shapes: H and I multiples of 128, 128 <= H <= 16384,
 * 128 <= I <= 4096, 1 <= E <= 1024, 1 <= k <= min(E, 32), T >= 0. */

typedef struct moe_qweights {
    int bits;                  /* 2 or 3 */
    int E, H, I;               /* experts, hidden size, expert intermediate size */
    const uint8_t *codes[3];   /* gate, up, down (device) */
    const uint16_t *scales[3]; /* gate, up, down fp16 bits (device) */
} moe_qweights;

/*
 * Router and top-k ("Strata - the details", "How it works": routers run on
 * the GPU; 10 of 512 experts per token, "Which model?").
 *   L[t,e] = sum_h x[t,h] Wr[e,h] + bias[e]      (fp32 accumulation)
 *   idx[t,0..k-1] = the k largest L[t,.] in descending order (tie: lower e)
 *   w[t,j] = exp(L_j - L_0) / sum_j' exp(L_j' - L_0)  (softmax renormalised
 *            over the selected experts)
 * x [T,H] fp32, Wr [E,H] fp32, bias [E] fp32 or NULL; idx_out [T,k] int32,
 * w_out [T,k] fp32.  T = 0 is a no-op.
 * For T <= 64 the router rows are fetched while the previous kernel on
 * `stream` is still finishing (programmatic dependent launch), so Wr must be
 * complete before the call is enqueued: do not write it from work that is
 * still pending on `stream` (weights are written once, then synchronised).
 * x and every other input are read only after earlier work has completed.
 */
int moe_route_topk(const float *x, int T, int H, const float *Wr, const float *bias, int E, int k,
                   int32_t *idx_out, float *w_out, void *ws, size_t ws_bytes, void *stream);

/*
 * Token-to-expert permutation (the grouping behind the pages' per-expert
 * prompt kernels, "Strata - the details", "Speed (measured)"): the T*k pairs
 * (t, j), in row-major order, stably sorted by expert idx[t,j].
 *   counts_out [E]      pairs per expert
 *   offsets_out [E+1]   exclusive prefix sum of counts (offsets[E] = T*k)
 *   perm_tok_out [T*k]  sorted position -> token t
 *   perm_slot_out [T*k] sorted position -> slot j
 *   inv_out [T,k]       (t, j) -> sorted position
 * Deterministic: ranks inside an expert follow token order, never arrival
 * order.  Rows of idx must hold k distinct experts in [0, E).
 */
int moe_permute(const int32_t *idx, int T, int k, int E, int32_t *counts_out, int32_t *offsets_out,
                int32_t *perm_tok_out, int32_t *perm_slot_out, int32_t *inv_out, void *ws, size_t ws_bytes,
                void *stream);

/*
 * moe_permute without a workspace.  The pages have no counterpart to this
 * entry point; it exists for callers that cannot allocate device memory --
 * for example code embedded in a host framework that owns every device
 * allocation, or a hot path that must never reach the CUDA allocator -- and so
 * cannot provide the `ws` that moe_permute needs.
 *
 * Same arguments, outputs and results as moe_permute, bit for bit.  Its
 * scratch (the per-expert token bitmaps and their prefix counts) lives in one
 * fixed 512 KiB array in device memory that the library declares statically;
 * every GPU that loads the library holds that array until the process exits.
 * Limit: E * ceil(T / 32) <= 65536 (for E = 512 that is T <= 4096); larger
 * sizes return MOEQ_ERR_SHAPE and launch nothing.  The call allocates and
 * frees nothing.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any CUDA stream capture.  All calls share the one array, so calls
 * whose kernels may overlap on the GPU (other streams, other host threads)
 * race and must be serialised by the caller.  Each call clears the part of
 * the array it needs, so no state carries over from the previous call.
 */
int moe_permute_noalloc(const int32_t *idx, int T, int k, int E, int32_t *counts_out, int32_t *offsets_out,
                        int32_t *perm_tok_out, int32_t *perm_slot_out, int32_t *inv_out, void *stream);

/*
 * Activation quantisation to int8 per 32-element block (the quantised-
 * activation prompt-expert kernels, "Strata - the details", "Speed
 * (measured)"): for each block, in fp32, s = amax/127 (IEEE division),
 * q = clamp(rint(v/s), -127, 127) with rint rounding half to even; a block of
 * zeros has s = 0, q = 0.  x [T,H] fp32 -> q_out [T,H] int8, s_out [T,H/32].
 * Bit-identical to any IEEE implementation of the same rule.
 */
int moe_quantize_act(const float *x, int T, int H, int8_t *q_out, float *s_out, void *stream);

/*
 * The experts ("Strata - the details", "How it works": the experts a token
 * selects run on the GPU; "Speed (measured)", engine 0.1.36: prompt experts on
 * fused int8 tensor-core kernels, 0.1.13: quantised-activation MMQ kernels
 * instead of FP16-expanded weights).  The FFN form (SwiGLU) and the 2-bit
 * block format are not on the pages; they are this library's readings.
 * For every sorted pair p (token t = perm_tok[p], expert e with
 * offsets[e] <= p < offsets[e+1]):
 *   G = W_gate[e] x_q, U = W_up[e] x_q        (x_q: x quantised as above)
 *   h = silu(G) * U, re-quantised per 32-block along I by the same rule
 *   D_p = W_down[e] h_q                         [H]
 * with every 32-block product an exact integer dot scaled by the two block
 * scales.  Outputs (at least one of out_sorted, y non-NULL):
 *   out_sorted [T*k, H] fp32   D_p in sorted order
 *   y [T, H] fp32              y[t] = (residual ? x[t] : 0) + sum_j w[t,j] D_(t,j)
 *   qh_out [T*k, I] int8, sh_out [T*k, I/32] fp32  (optional, may be NULL)
 *                              the quantised SwiGLU activations h_q
 * w [T,k] fp32 routing weights (needed when y != NULL).  mode: MOEQ_MODE_*.
 * The order of the k additions into y is unspecified (fp32 atomics);
 * out_sorted, qh and sh do not depend on it.
 * offsets/perm_tok/perm_slot are moe_permute's outputs (the pair's slot j
 * picks its weight w[t,j]; inv is not needed here).  offsets that are not an
 * exclusive prefix sum within [0, T*k], or a token or slot out of range, make
 * the kernels skip the affected work and raise MOEQ_STATUS_BAD_INDEX instead
 * of reading or writing out of bounds.
 */
int moe_expert_ffn_q2(const float *x, int T, const moe_qweights *weights, int k, const int32_t *offsets,
                      const int32_t *perm_tok, const int32_t *perm_slot, const float *w, float *out_sorted,
                      float *y, int residual, int mode, int8_t *qh_out, float *sh_out, void *ws,
                      size_t ws_bytes, void *stream);

/*
 * A shared expert ("Strata — the details", How it works: the shared experts
 * stay on the GPU beside the routers): one dense SwiGLU expert that every
 * token passes through, added to the layer output with weight 1 (the pages do
 * not state a gate, so none is applied).
 *   y[t] = (accumulate ? y[t] : 0) + W_down h_q(t),  h = silu(W_gate x_q) * (W_up x_q)
 * with the same block formats and rounding rules as moe_expert_ffn_q2; in fact
 * it is moe_expert_ffn_q2 with E = 1, k = 1 and every routing weight 1.
 * shared: E = 1, its own H and I (I a multiple of 128).  x [T,H], y [T,H]
 * fp32 device arrays, 16-byte aligned; y is read only when accumulate != 0
 * (call it after moe_layer_forward with accumulate = 1 to add the shared
 * expert to the routed mixture).  ws: moe_workspace_bytes(T, H, I, 1, 1, bits)
 * bytes.  mode: MOEQ_MODE_*.  The additions into y are fp32 atomics.
 * Errors: MOEQ_ERR_ARG (NULL pointer, E != 1, bad mode), MOEQ_ERR_SHAPE,
 * MOEQ_ERR_ALIGN, MOEQ_ERR_WORKSPACE, MOEQ_ERR_CUDA; nothing is launched on an
 * argument error.
 */
int moe_shared_expert_q2(const float *x, int T, const moe_qweights *shared, float *y, int accumulate, int mode,
                         void *ws, size_t ws_bytes, void *stream);

/*
 * Weighted gather-combine (each token's output mixes the k experts it picked,
 * upstream Strata README, "How does it work?": each word needs only 10 of the
 * 24,576 experts; the residual add between layers is the stack's, attention
 * being left out):
 *   y[t,:] = (residual_x ? residual_x[t,:] : 0)
 *            + sum_{j=0..k-1} w[t,j] out_sorted[inv[t,j],:]
 * summed in j order in fp32 (deterministic).  out_sorted [T*k,H], inv [T,k],
 * w [T,k], residual_x [T,H] or NULL, y_out [T,H]; H a multiple of 4.  Needs no
 * workspace.  A pair whose inv is outside [0, T*k) (moe_permute writes -1 for
 * a rejected expert index) adds nothing and raises MOEQ_STATUS_BAD_INDEX.
 */
int moe_combine(const float *out_sorted, const int32_t *inv, const float *w, int T, int k, int H,
                const float *residual_x, float *y_out, void *stream);

/*
 * The whole routed expert-FFN layer as the pages' engine runs it per layer
 * ("Strata - the details", "How it works": routers on the GPU, then each
 * token's selected experts; prompt chunks batched per expert, "Speed
 * (measured)"): route + top-k, permutation, experts and combine, all on
 * `stream` with no host synchronisation.  y_out [T,H] = (residual ? x : 0) +
 * the routed mixture.  idx_out/w_out [T,k] optional (may be NULL).
 * Decode calls (T <= 64 in GEMV mode) run as two kernels chained by
 * programmatic dependent launch; the router weights Wr are fetched before the
 * previous kernel on `stream` has finished (see moe_route_topk), so a stack
 * of layers streams layer l+1's router while layer l's experts run.
 */
int moe_layer_forward(const float *x, int T, const float *Wr, const float *bias, const moe_qweights *weights,
                      int k, int residual, float *y_out, int32_t *idx_out, float *w_out, int mode, void *ws,
                      size_t ws_bytes, void *stream);

/* Bytes of workspace every call above needs for these sizes (0 on bad shapes).
 * The pages size their prompt-chunk buffers to fit borrowed cache slots
 * ("Strata - the details", "How it works"); here the caller allocates one
 * buffer of this size per stream and passes it to every call. */
size_t moe_workspace_bytes(int T, int H, int I, int E, int k, int bits);

/* Device-side failure report (the pages' engine ends a stuck request with an
 * error instead of hanging, "Strata - the details", "Troubleshooting").
 * Synchronises `stream`, returns in *status_out the MOEQ_STATUS_* bits that
 * kernels on the current device recorded since the last call, and clears them.
 * Returns MOEQ_ERR_DEVICE when any bit was set.  After
 * MOEQ_STATUS_WAIT_TIMEOUT the outputs of the calls since the last check are
 * unspecified; the workspace stays usable (its counters are re-armed). */
int moe_get_device_status(void *stream, int *status_out);

/* The bound of every device-side pipeline wait, in nanoseconds, on the current
 * device (the counterpart of the pages' watchdog, "Strata - the details",
 * "Troubleshooting": STRATA_WATCHDOG_S ends a request that makes no progress).
 * 0 restores the default of 2 s; at most 60 s.  A wait that runs out raises
 * MOEQ_STATUS_WAIT_TIMEOUT, and its kernel drains the copies and tensor-core
 * operations it issued (bounded separately, 2 s) and returns.  Takes effect
 * for kernels launched after the call returns; call it with no library work
 * in flight on the device (it writes device memory synchronously). */
int moe_set_wait_limit(uint64_t ns);

/* Thread-local text of the last error returned on this thread ("" if none). */
const char *moe_last_error_string(void);

/*
 * Kernel tracing (the pages' engine reports per-tier counters with --stats,
 * "Strata - the details", "Speed (measured)"; this is the device-time
 * counterpart).  events: an array of n cudaEvent_t handles (n even) that the
 * caller created, or NULL to switch tracing off.  While set, every launch of
 * an expert kernel (the GEMV, and each of the two tensor-core GEMMs) and of the
 * prompt-chunk router GEMM (T > 64) on the calling thread is bracketed by
 * cudaEventRecord(events[c]) and
 * cudaEventRecord(events[c+1]) on the call's stream, c advancing by 2 modulo
 * n and starting at 0 after each moe_trace_events call.  Works inside CUDA
 * graph capture (the records become graph nodes).  Returns MOEQ_ERR_ARG for an
 * odd n or n < 0.
 */
int moe_trace_events(void *const *events, int n);

/* Library version string, e.g. "moeq 0.1.0 sm_103a". */
const char *moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOEQ_H */
