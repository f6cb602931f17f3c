/*
 * moe_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, CPU reference of the routed expert-FFN layer, written from
 * the layer's definition for checking the CUDA library against.  Only the test
 * suite, the package smoke check and the benchmark's CPU-baseline leg may load
 * it; the product never calls it.  It shares no code with the CUDA path.
 *
 * What the layer computes (the Strata pages describe the model -- 512 experts
 * per layer, 10 of them active per token, routers and cached experts on the
 * GPU -- in "Strata - the details", sections "Which model?" and "How it
 * works", and the upstream Strata README, "How does it work?"; the pages do
 * not write the arithmetic out, so the readings below are this library's and
 * are listed with it):
 *
 *   1. router logits   L[t,e] = sum_h x[t,h] Wr[e,h] + b[e]          (fp64)
 *   2. top-k           the k largest L[t,.], descending, ties -> lower e
 *      weights         w[t,j] = exp(L_j - L_0) / sum_j' exp(L_j' - L_0)
 *                      (softmax renormalised over the k selected), stored fp32
 *   3. permutation     (t, j) pairs in row-major order, stably sorted by expert
 *   4. activations     per 32-block, in fp32: s = amax / 127,
 *                      q = clamp(rint(x / s), -127, 127); s = 0 -> q = 0
 *   5. gate / up       G_i = sum_kb s_w[i,kb] s_x[kb] (sum_32 qw * qx)  (fp64,
 *                      the 32-element block dot is an exact integer)
 *   6. SwiGLU          h_i = G_i / (1 + exp(-G_i)) * U_i in fp64, rounded to
 *                      fp32, then quantised by the rule of step 4 along I
 *   7. down            D_n = sum_kb s_w[n,kb] s_h[kb] (sum_32 qw * qh)  (fp64)
 *   8. combine         y[t] = sum_j w[t,j] D_j  (+ x[t] when residual), fp64,
 *                      stored fp32
 *
 * Weight storage (one [N rows, K in] matrix per expert, block-column-major):
 *   codes [E][K/32][N][4*bits bytes], scales [E][K/32][N] fp16.
 *   2-bit element i of a block: byte i/4, bits 2*(i%4); value code - 2.
 *   3-bit element i of a block: bits 3i..3i+2 of the 96-bit LE block word;
 *   value code - 4.
 *
 * Built with -O2 -ffp-contract=off and without fast-math, so the fp32
 * quantiser of step 4 is IEEE single precision division and rintf
 * (round half to even).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- helpers */

/* IEEE binary16 bits -> double, decoded field by field. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int man = h & 1023;
    double v;
    if (expo == 0)
        v = ldexp((double)man, -24);
    else if (expo == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + man), expo - 25);
    return sign ? -v : v;
}

/* Code (unsigned field) of element kk of row n of one expert's [N, K] matrix. */
int oracle_weight_code(const uint8_t *codes, int bits, int N, int n, int kk)
{
    int bpb = 4 * bits;
    int kb = kk / 32, i = kk % 32;
    const uint8_t *blk = codes + ((size_t)kb * N + n) * bpb;
    int bit = bits * i;
    unsigned v = blk[bit / 8];
    if (bit / 8 + 1 < bpb)
        v |= (unsigned)blk[bit / 8 + 1] << 8;
    return (int)((v >> (bit % 8)) & ((1u << bits) - 1));
}

/* Signed level of that element: code - 2 (2-bit) or code - 4 (3-bit). */
int oracle_weight_level(const uint8_t *codes, int bits, int N, int n, int kk)
{
    return oracle_weight_code(codes, bits, N, n, kk) - (1 << (bits - 1));
}

double oracle_weight_scale(const uint16_t *scales, int N, int n, int kb)
{
    return oracle_half_to_double(scales[(size_t)kb * N + n]);
}

/* Dequantised weight element, for the dense brute-force cross-check. */
double oracle_weight_value(const uint8_t *codes, const uint16_t *scales, int bits, int N, int n, int kk)
{
    return (double)oracle_weight_level(codes, bits, N, n, kk) * oracle_weight_scale(scales, N, n, kk / 32);
}

/* ------------------------------------------------------ step 4: quantiser */

void oracle_quantize_block32(const float *v, int n, int8_t *q, float *s)
{
    for (int b = 0; b < n / 32; ++b) {
        const float *vb = v + 32 * b;
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(vb[i]);
            if (a > amax)
                amax = a;
        }
        float sc = amax / 127.0f;
        s[b] = sc;
        for (int i = 0; i < 32; ++i) {
            if (sc == 0.0f) {
                q[32 * b + i] = 0;
                continue;
            }
            float r = rintf(vb[i] / sc);
            if (r > 127.0f)
                r = 127.0f;
            if (r < -127.0f)
                r = -127.0f;
            q[32 * b + i] = (int8_t)r;
        }
    }
}

/* --------------------------------------------------- steps 1-2: routing */

void oracle_router_logits_token(const float *x, int H, const float *Wr, const float *bias, int E, double *L)
{
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h)
            acc += (double)x[h] * (double)Wr[(size_t)e * H + h];
        L[e] = acc + (bias ? (double)bias[e] : 0.0);
    }
}

void oracle_topk_softmax_token(const double *L, int E, int k, int32_t *idx, float *w)
{
    /* selection: k passes, each taking the largest logit not yet taken;
     * strict '>' keeps the lower expert index on an exact tie */
    char *taken = (char *)calloc((size_t)E, 1);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            if (best < 0 || L[e] > L[best])
                best = e;
        }
        taken[best] = 1;
        idx[j] = best;
    }
    free(taken);
    double m = L[idx[0]], den = 0.0;
    for (int j = 0; j < k; ++j)
        den += exp(L[idx[j]] - m);
    for (int j = 0; j < k; ++j)
        w[j] = (float)(exp(L[idx[j]] - m) / den);
}

/* ------------------------------------------------------ step 3: permutation */

void oracle_permute(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                    int32_t *perm_tok, int32_t *perm_slot, int32_t *inv)
{
    memset(counts, 0, sizeof(int32_t) * (size_t)E);
    for (int p = 0; p < T * k; ++p)
        counts[idx[p]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    memcpy(cursor, offsets, sizeof(int32_t) * (size_t)E);
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = idx[t * k + j];
            int pos = cursor[e]++;
            perm_tok[pos] = t;
            perm_slot[pos] = j;
            inv[t * k + j] = pos;
        }
    free(cursor);
}

/* ------------------------------------------------- steps 5-7: one expert */

/* Exact integer dot of one 32-block of a weight row with 32 int8 values. */
static int64_t block_dot(const uint8_t *codes, int bits, int N, int n, int kb, const int8_t *q32)
{
    int64_t d = 0;
    for (int i = 0; i < 32; ++i)
        d += (int64_t)oracle_weight_level(codes, bits, N, n, 32 * kb + i) * (int64_t)q32[i];
    return d;
}

/*
 * One token through one expert.  qx/sx: the token's quantised activations
 * (H values, H/32 scales).  Outputs (any may be NULL except D):
 *   G, U [I] fp64; h [I] fp32; qh [I], sh [I/32]; hdist [I] = distance (in
 *   units of the quantisation step) of h/s_h to the nearest rounding boundary;
 *   D [H] fp64.
 */
void oracle_expert_token(const int8_t *qx, const float *sx, int H, int I, int bits,
                         const uint8_t *cg, const uint16_t *sg, const uint8_t *cu, const uint16_t *su,
                         const uint8_t *cd, const uint16_t *sd,
                         double *G_out, double *U_out, float *h_out, int8_t *qh_out, float *sh_out,
                         double *hdist_out, double *D)
{
    float *h = (float *)malloc(sizeof(float) * (size_t)I);
    int8_t *qh = (int8_t *)malloc((size_t)I);
    float *sh = (float *)malloc(sizeof(float) * (size_t)(I / 32));
    for (int i = 0; i < I; ++i) {
        double G = 0.0, U = 0.0;
        for (int kb = 0; kb < H / 32; ++kb) {
            double sa = (double)sx[kb];
            G += oracle_weight_scale(sg, I, i, kb) * sa * (double)block_dot(cg, bits, I, i, kb, qx + 32 * kb);
            U += oracle_weight_scale(su, I, i, kb) * sa * (double)block_dot(cu, bits, I, i, kb, qx + 32 * kb);
        }
        double h64 = G / (1.0 + exp(-G)) * U;
        h[i] = (float)h64;
        if (G_out)
            G_out[i] = G;
        if (U_out)
            U_out[i] = U;
    }
    oracle_quantize_block32(h, I, qh, sh);
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int kb = 0; kb < I / 32; ++kb)
            acc += oracle_weight_scale(sd, H, n, kb) * (double)sh[kb] * (double)block_dot(cd, bits, H, n, kb, qh + 32 * kb);
        D[n] = acc;
    }
    if (h_out)
        memcpy(h_out, h, sizeof(float) * (size_t)I);
    if (qh_out)
        memcpy(qh_out, qh, (size_t)I);
    if (sh_out)
        memcpy(sh_out, sh, sizeof(float) * (size_t)(I / 32));
    if (hdist_out)
        for (int i = 0; i < I; ++i) {
            double s = (double)sh[i / 32];
            if (s == 0.0) {
                hdist_out[i] = 0.5;
                continue;
            }
            double r = fabs((double)h[i] / s);
            hdist_out[i] = fabs(r - floor(r) - 0.5);
        }
    free(h);
    free(qh);
    free(sh);
}

/* ----------------------------------------------------- the whole layer */

typedef struct {
    const float *x;
    int T, H, I, E, k, bits;
    const float *Wr, *bias;
    const uint8_t *codes[3];
    const uint16_t *scales[3];
    int residual;
    const int32_t *tokens; /* which tokens to compute */
    int n_tokens;
    int32_t *idx;  /* [n_tokens, k] */
    float *w;      /* [n_tokens, k] */
    float *y;      /* [n_tokens, H] */
    float *h;      /* [n_tokens, k, I] or NULL */
    int8_t *qh;    /* [n_tokens, k, I] or NULL */
    float *sh;     /* [n_tokens, k, I/32] or NULL */
    double *hdist; /* [n_tokens, k, I] or NULL */
    double *D;     /* [n_tokens, k, H] or NULL */
    int first, last;
} layer_job;

static void layer_token(const layer_job *J, int r)
{
    int t = J->tokens[r];
    int H = J->H, I = J->I, E = J->E, k = J->k;
    size_t Ecb_g = (size_t)(H / 32) * I * (4 * J->bits), Esc_g = (size_t)(H / 32) * I;
    size_t Ecb_d = (size_t)(I / 32) * H * (4 * J->bits), Esc_d = (size_t)(I / 32) * H;
    const float *xt = J->x + (size_t)t * H;
    double *L = (double *)malloc(sizeof(double) * (size_t)E);
    oracle_router_logits_token(xt, H, J->Wr, J->bias, E, L);
    int32_t *idx = J->idx + (size_t)r * k;
    float *w = J->w + (size_t)r * k;
    oracle_topk_softmax_token(L, E, k, idx, w);
    free(L);
    int8_t *qx = (int8_t *)malloc((size_t)H);
    float *sx = (float *)malloc(sizeof(float) * (size_t)(H / 32));
    oracle_quantize_block32(xt, H, qx, sx);
    double *D = (double *)malloc(sizeof(double) * (size_t)H);
    double *yacc = (double *)calloc((size_t)H, sizeof(double));
    for (int j = 0; j < k; ++j) {
        int e = idx[j];
        size_t rj = (size_t)r * k + j;
        oracle_expert_token(qx, sx, H, I, J->bits,
                            J->codes[0] + e * Ecb_g, J->scales[0] + e * Esc_g,
                            J->codes[1] + e * Ecb_g, J->scales[1] + e * Esc_g,
                            J->codes[2] + e * Ecb_d, J->scales[2] + e * Esc_d,
                            NULL, NULL, J->h ? J->h + rj * I : NULL,
                            J->qh ? J->qh + rj * I : NULL, J->sh ? J->sh + rj * (I / 32) : NULL,
                            J->hdist ? J->hdist + rj * I : NULL, D);
        for (int n = 0; n < H; ++n)
            yacc[n] += (double)w[j] * D[n];
        if (J->D)
            memcpy(J->D + rj * H, D, sizeof(double) * (size_t)H);
    }
    for (int n = 0; n < H; ++n)
        J->y[(size_t)r * H + n] = (float)(yacc[n] + (J->residual ? (double)xt[n] : 0.0));
    free(qx);
    free(sx);
    free(D);
    free(yacc);
}

static void *layer_worker(void *arg)
{
    const layer_job *J = (const layer_job *)arg;
    for (int r = J->first; r < J->last; ++r)
        layer_token(J, r);
    return NULL;
}

/*
 * The layer for a list of tokens of a T-token batch (every token's output
 * depends only on that token, so a list gives the exact outputs of those
 * rows).  Threads split the token list into contiguous ranges.
 */
int oracle_layer(const float *x, int T, int H, int I, int E, int k, int bits,
                 const float *Wr, const float *bias,
                 const uint8_t *cg, const uint16_t *sg, const uint8_t *cu, const uint16_t *su,
                 const uint8_t *cd, const uint16_t *sd, int residual,
                 const int32_t *tokens, int n_tokens, int nthreads,
                 int32_t *idx_out, float *w_out, float *y_out,
                 float *h_out, int8_t *qh_out, float *sh_out, double *hdist_out, double *D_out)
{
    if (H % 32 || I % 32 || k < 1 || k > E || (bits != 2 && bits != 3))
        return -1;
    for (int r = 0; r < n_tokens; ++r)
        if (tokens[r] < 0 || tokens[r] >= T)
            return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > n_tokens)
        nthreads = n_tokens > 0 ? n_tokens : 1;
    layer_job base = {x, T, H, I, E, k, bits, Wr, bias, {cg, cu, cd}, {sg, su, sd}, residual,
                      tokens, n_tokens, idx_out, w_out, y_out, h_out, qh_out, sh_out, hdist_out, D_out, 0, 0};
    layer_job *jobs = (layer_job *)malloc(sizeof(layer_job) * (size_t)nthreads);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = base;
        jobs[i].first = (int)((long long)n_tokens * i / nthreads);
        jobs[i].last = (int)((long long)n_tokens * (i + 1) / nthreads);
        pthread_create(&th[i], NULL, layer_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i)
        pthread_join(th[i], NULL);
    free(jobs);
    free(th);
    return 0;
}

/* Router logits of a whole batch (the tests use them to keep routing margins). */
typedef struct {
    const float *x;
    int H, E;
    const float *Wr, *bias;
    double *L;
    int first, last;
} logit_job;

static void *logit_worker(void *arg)
{
    const logit_job *J = (const logit_job *)arg;
    for (int t = J->first; t < J->last; ++t)
        oracle_router_logits_token(J->x + (size_t)t * J->H, J->H, J->Wr, J->bias, J->E, J->L + (size_t)t * J->E);
    return NULL;
}

int oracle_router_logits(const float *x, int T, int H, const float *Wr, const float *bias, int E,
                         double *L, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > T)
        nthreads = T > 0 ? T : 1;
    logit_job *jobs = (logit_job *)malloc(sizeof(logit_job) * (size_t)nthreads);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) {
        logit_job j = {x, H, E, Wr, bias, L, (int)((long long)T * i / nthreads), (int)((long long)T * (i + 1) / nthreads)};
        jobs[i] = j;
        pthread_create(&th[i], NULL, logit_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i)
        pthread_join(th[i], NULL);
    free(jobs);
    free(th);
    return 0;
}

int oracle_topk_softmax(const double *L, int T, int E, int k, int32_t *idx, float *w)
{
    if (k < 1 || k > E)
        return -1;
    for (int t = 0; t < T; ++t)
        oracle_topk_softmax_token(L + (size_t)t * E, E, k, idx + (size_t)t * k, w + (size_t)t * k);
    return 0;
}

/* Column kk of one expert's dequantised [N, K] matrix (N values, fp64). */
void oracle_weight_column(const uint8_t *codes, const uint16_t *scales, int bits, int N, int kk, double *out)
{
    for (int n = 0; n < N; ++n)
        out[n] = oracle_weight_value(codes, scales, bits, N, n, kk);
}
