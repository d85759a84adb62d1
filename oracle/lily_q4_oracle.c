/*
 * CPU oracle for the MLX-affine 4-bit mixture-of-experts hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg load this library.  It shares no code,
 * header, table or helper with the CUDA library; the two meet only through the
 * seeded input generator.
 *
 * What it computes (plain definitions, written out loop by loop):
 *
 *  - Weight format: MLX affine 4-bit weights in groups of 64 (Lily README,
 *    first paragraph and "Requirements"; Lily-vs-MLX report, "Hardware and
 *    software").  The pages name the format only; the reading taken here is
 *    w = s*q + b with q the 4-bit code, eight codes per uint32 along K, lowest
 *    nibble first, and one bf16 (s, b) pair per 64 consecutive K.  The code is
 *    dequantised in fp32 (s*q is exact there) and widened to fp64.
 *  - Router: fp64 dot products of the bf16 token with each bf16 router row,
 *    plus an optional fp32 per-expert offset.
 *  - Top-k: experts sorted by (logit descending, index ascending), first k
 *    taken.  The fork page's "Exactness" section notes that near-ties in the
 *    expert router flip choices; ties here go to the lower index.
 *  - Gates: softmax over the selected k logits (equal to a full softmax
 *    renormalised over the k, the full denominator cancels).
 *  - Expert: h = silu(Wg x) * (Wu x), o = Wd h, all fp64.
 *  - Shared expert (the fork page's "The model" section lists the shared
 *    expert among the dense tensors): o_s the same way, scaled by
 *    sigmoid(g_shared . x).
 *  - Output: y = sum_i p_i o_i + sigma o_s.
 *  - LM head with greedy argmax (Lily README, first paragraph: Lily decodes
 *    greedily; report "Measurement contract": greedy token selection without
 *    logprobs): fp64 logits, argmax with ties to the lower id.
 *  - Affine 8-bit matrices (the report's checkpoint keeps its router gates at
 *    8 bits, "Hardware and software"; the fork page's q4-xl conversion keeps the
 *    shared expert and the LM head at 8 bits, "The model"): the same
 *    w = s*q + b with q in 0..255, four codes per uint32 along K, lowest byte
 *    first (the 4-bit packing with 8-bit fields), one bf16 (s, b) pair per 64 K.
 *  - Full-vocabulary log-sum-exp and log-probabilities of those logits (report
 *    "Measurement contract": the MLX path computes both over the whole
 *    vocabulary): lse = log sum_n exp(l_n), logprob_n = l_n - lse,
 *    in fp64 (the sum is taken after subtracting the maximum, which changes
 *    nothing mathematically).
 *
 * Parallelism: OpenMP only splits independent output rows / tokens across
 * threads; every dot product is summed in plain k order by one thread.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_GROUP 64

static float orc_bf16(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* 4-bit code k of row n: word k/8, nibble k%8 (lowest nibble first). */
static unsigned orc_code(const uint32_t *w, int K, int n, int k) {
    uint32_t word = w[(size_t)n * (size_t)(K / 8) + (size_t)(k / 8)];
    return (word >> (4u * (unsigned)(k % 8))) & 0xFu;
}

/* Dequantised weight (n, k): fp32 s*q + b, widened to double. */
static double orc_weight(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                         int K, int n, int k) {
    size_t gi = (size_t)n * (size_t)(K / ORC_GROUP) + (size_t)(k / ORC_GROUP);
    float sf = orc_bf16(s[gi]);
    float bf = orc_bf16(b[gi]);
    float q = (float)orc_code(w, K, n, k);
    float wf = sf * q + bf;
    return (double)wf;
}

int orc_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* 8-bit code k of row n: word k/4, byte k%4 (lowest byte first). */
static unsigned orc_code8(const uint32_t *w, int K, int n, int k) {
    uint32_t word = w[(size_t)n * (size_t)(K / 4) + (size_t)(k / 4)];
    return (word >> (8u * (unsigned)(k % 4))) & 0xFFu;
}

/* Dequantised 8-bit weight (n, k): fp32 s*q + b (s*q exact: 8 x 8 significant bits),
 * widened to double. */
static double orc_weight8(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                          int K, int n, int k) {
    size_t gi = (size_t)n * (size_t)(K / ORC_GROUP) + (size_t)(k / ORC_GROUP);
    float wf = orc_bf16(s[gi]) * (float)orc_code8(w, K, n, k) + orc_bf16(b[gi]);
    return (double)wf;
}

void orc_q8_unpack(const uint32_t *w, int N, int K, uint8_t *q) {
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            q[(size_t)n * K + k] = (uint8_t)orc_code8(w, K, n, k);
}

void orc_q8_pack(const uint8_t *q, int N, int K, uint32_t *w) {
    for (int n = 0; n < N; ++n)
        for (int m = 0; m < K / 4; ++m) {
            uint32_t word = 0;
            for (int j = 0; j < 4; ++j)
                word |= ((uint32_t)q[(size_t)n * K + 4 * m + j]) << (8 * j);
            w[(size_t)n * (K / 4) + m] = word;
        }
}

void orc_q8_dequant(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                    int N, int K, double *out) {
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            out[(size_t)n * K + k] = orc_weight8(w, s, b, K, n, k);
}

/* out[n] = sum_k W^[n,k] x[k] for an 8-bit matrix, x given in fp64. */
void orc_q8_matvec(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                   int N, int K, const double *x, double *out) {
    for (int n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k)
            acc += orc_weight8(w, s, b, K, n, k) * x[k];
        out[n] = acc;
    }
}

/* 8-bit LM head: logits[n] for bf16 x (rows split over threads); returns the argmax
 * (ties to the lower id). */
int orc_q8_lm_head(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                   int N, int K, const uint16_t *x, double *logits) {
    double *xd = (double *)malloc(sizeof(double) * (size_t)K);
    for (int k = 0; k < K; ++k) xd[k] = (double)orc_bf16(x[k]);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k)
            acc += orc_weight8(w, s, b, K, n, k) * xd[k];
        logits[n] = acc;
    }
    free(xd);
    int best = 0;
    for (int n = 1; n < N; ++n)
        if (logits[n] > logits[best]) best = n;
    return best;
}

/* out[N][K] = dequantised matrix. */
void orc_q4_dequant(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                    int N, int K, double *out) {
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            out[(size_t)n * K + k] = orc_weight(w, s, b, K, n, k);
}

/* Unpack codes: q[N][K] (0..15). */
void orc_q4_unpack(const uint32_t *w, int N, int K, uint8_t *q) {
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            q[(size_t)n * K + k] = (uint8_t)orc_code(w, K, n, k);
}

/* Pack codes q[N][K] (0..15) into words. */
void orc_q4_pack(const uint8_t *q, int N, int K, uint32_t *w) {
    for (int n = 0; n < N; ++n)
        for (int m = 0; m < K / 8; ++m) {
            uint32_t word = 0;
            for (int j = 0; j < 8; ++j)
                word |= ((uint32_t)(q[(size_t)n * K + 8 * m + j] & 0xF)) << (4 * j);
            w[(size_t)n * (K / 8) + m] = word;
        }
}

/* out[n] = sum_k W^[n,k] x[k], x given in fp64. */
void orc_q4_matvec(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                   int N, int K, const double *x, double *out) {
    for (int n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k)
            acc += orc_weight(w, s, b, K, n, k) * x[k];
        out[n] = acc;
    }
}

/* LM head: logits[n] for bf16 x, rows split over threads; returns the argmax
 * (ties to the lower id). */
int orc_lm_head(const uint32_t *w, const uint16_t *s, const uint16_t *b,
                int N, int K, const uint16_t *x, double *logits) {
    double *xd = (double *)malloc(sizeof(double) * (size_t)K);
    for (int k = 0; k < K; ++k) xd[k] = (double)orc_bf16(x[k]);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k)
            acc += orc_weight(w, s, b, K, n, k) * xd[k];
        logits[n] = acc;
    }
    free(xd);
    int best = 0;
    for (int n = 1; n < N; ++n)
        if (logits[n] > logits[best]) best = n;
    return best;
}

/* lse = log(sum_n exp(l[n])) over n < N, and logprob[n] = l[n] - lse when logprob is
 * not NULL.  A NaN logit gives NaN; a +inf logit gives +inf; all -inf gives -inf. */
double orc_log_sum_exp(const double *l, int N, double *logprob) {
    double m = -INFINITY;
    int nan = 0;
    for (int n = 0; n < N; ++n) {
        if (l[n] != l[n]) nan = 1;
        else if (l[n] > m) m = l[n];
    }
    double lse;
    if (nan) lse = NAN;
    else if (isinf(m)) lse = m;
    else {
        double sum = 0.0;
        for (int n = 0; n < N; ++n) sum += exp(l[n] - m);
        lse = m + log(sum);
    }
    if (logprob)
        for (int n = 0; n < N; ++n) logprob[n] = l[n] - lse;
    return lse;
}

/* Router logits for one token. */
void orc_router(const uint16_t *Wr, const float *bias, int E, int H,
                const uint16_t *x, double *logits) {
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h)
            acc += (double)orc_bf16(Wr[(size_t)e * H + h]) * (double)orc_bf16(x[h]);
        if (bias) acc += (double)bias[e];
        logits[e] = acc;
    }
}

/* Top-k by (logit desc, index asc), then softmax over the k selected. */
void orc_topk(const double *logits, int E, int k, int32_t *idx, double *p) {
    int *order = (int *)malloc(sizeof(int) * (size_t)E);
    for (int e = 0; e < E; ++e) order[e] = e;
    /* insertion sort: a before b iff l[a] > l[b], or equal and a < b */
    for (int i = 1; i < E; ++i) {
        int cur = order[i];
        int j = i - 1;
        while (j >= 0) {
            int o = order[j];
            int before = (logits[cur] > logits[o]) || (logits[cur] == logits[o] && cur < o);
            if (!before) break;
            order[j + 1] = o;
            --j;
        }
        order[j + 1] = cur;
    }
    double lmax = logits[order[0]];
    double denom = 0.0;
    for (int i = 0; i < k; ++i) denom += exp(logits[order[i]] - lmax);
    for (int i = 0; i < k; ++i) {
        idx[i] = order[i];
        p[i] = exp(logits[order[i]] - lmax) / denom;
    }
    free(order);
}

double orc_sigmoid_gate(const uint16_t *g, int H, const uint16_t *x) {
    double acc = 0.0;
    for (int h = 0; h < H; ++h) acc += (double)orc_bf16(g[h]) * (double)orc_bf16(x[h]);
    return 1.0 / (1.0 + exp(-acc));
}

/* W^ x for 4-bit (bits = 4) or 8-bit (bits = 8) codes. */
static void orc_matvec_bits(int bits, const uint32_t *w, const uint16_t *s, const uint16_t *b,
                            int N, int K, const double *x, double *out) {
    if (bits == 8) orc_q8_matvec(w, s, b, N, K, x, out);
    else orc_q4_matvec(w, s, b, N, K, x, out);
}

/* One SwiGLU expert with codes of `bits` bits: o[H] = Wd (silu(Wg x) * (Wu x)); gate/up
 * [I x H], down [H x I]. */
static void orc_expert_bits(int bits, const uint32_t *gw, const uint16_t *gs, const uint16_t *gb,
                            const uint32_t *uw, const uint16_t *us, const uint16_t *ub,
                            const uint32_t *dw, const uint16_t *ds, const uint16_t *db,
                            int H, int I, const double *x, double *o) {
    double *g = (double *)malloc(sizeof(double) * (size_t)I);
    double *u = (double *)malloc(sizeof(double) * (size_t)I);
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    orc_matvec_bits(bits, gw, gs, gb, I, H, x, g);
    orc_matvec_bits(bits, uw, us, ub, I, H, x, u);
    for (int i = 0; i < I; ++i) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
    orc_matvec_bits(bits, dw, ds, db, H, I, h, o);
    free(g);
    free(u);
    free(h);
}

/* One SwiGLU expert with 4-bit codes. */
void orc_expert(const uint32_t *gw, const uint16_t *gs, const uint16_t *gb,
                const uint32_t *uw, const uint16_t *us, const uint16_t *ub,
                const uint32_t *dw, const uint16_t *ds, const uint16_t *db,
                int H, int I, const double *x, double *o) {
    orc_expert_bits(4, gw, gs, gb, uw, us, ub, dw, ds, db, H, I, x, o);
}

typedef struct {
    const uint32_t *w;
    const uint16_t *s;
    const uint16_t *b;
} orc_mat;

typedef struct {
    int32_t H, E, k, I;
    orc_mat gate, up, down;          /* stacked over E: [E][N][..] */
    int32_t has_shared;
    orc_mat sh_gate, sh_up, sh_down; /* single matrices */
    const uint16_t *router;          /* bf16 [E][H] (router_bits 16) */
    const float *router_bias;        /* fp32 [E] or NULL */
    const uint16_t *shared_gate;     /* bf16 [H] or NULL */
    int32_t shared_bits;             /* 4 (or 0) or 8: codes of the shared expert */
    int32_t router_bits;             /* 16 (or 0): bf16 router; 8: router8 */
    orc_mat router8;                 /* affine 8-bit router [E][H/4] codes, [E][H/64] s, b */
} orc_layer;

/* Router logits of one token from an affine 8-bit router, fp64 (+ offsets). */
static void orc_router8(const orc_mat *R, const float *bias, int E, int H, const uint16_t *x,
                        double *logits) {
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h)
            acc += orc_weight8(R->w, R->s, R->b, H, e, h) * (double)orc_bf16(x[h]);
        if (bias) acc += (double)bias[e];
        logits[e] = acc;
    }
}

static void orc_layer_router(const orc_layer *L, const uint16_t *xt, double *lg) {
    if (L->router_bits == 8) orc_router8(&L->router8, L->router_bias, L->E, L->H, xt, lg);
    else orc_router(L->router, L->router_bias, L->E, L->H, xt, lg);
}

static orc_mat orc_expert_mat(orc_mat m, int e, int N, int K) {
    orc_mat r;
    r.w = m.w + (size_t)e * N * (K / 8);
    r.s = m.s + (size_t)e * N * (K / ORC_GROUP);
    r.b = m.b + (size_t)e * N * (K / ORC_GROUP);
    return r;
}

/* Whole MoE layer for T tokens x[T][H] (bf16).  Outputs (any may be NULL except y):
 *   y[T][H] fp64, idx[T][k], p[T][k], logits[T][E], sigma[T]. */
void orc_moe(const orc_layer *L, const uint16_t *x, int T, double *y,
             int32_t *idx_out, double *p_out, double *logits_out, double *sigma_out) {
    const int H = L->H, E = L->E, k = L->k, I = L->I;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
        const uint16_t *xt = x + (size_t)t * H;
        double *xd = (double *)malloc(sizeof(double) * (size_t)H);
        double *lg = (double *)malloc(sizeof(double) * (size_t)E);
        double *o = (double *)malloc(sizeof(double) * (size_t)H);
        int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
        double *p = (double *)malloc(sizeof(double) * (size_t)k);
        for (int h = 0; h < H; ++h) xd[h] = (double)orc_bf16(xt[h]);
        orc_layer_router(L, xt, lg);
        orc_topk(lg, E, k, idx, p);
        double *yt = y + (size_t)t * H;
        for (int h = 0; h < H; ++h) yt[h] = 0.0;
        for (int i = 0; i < k; ++i) {
            int e = idx[i];
            orc_mat g = orc_expert_mat(L->gate, e, I, H);
            orc_mat u = orc_expert_mat(L->up, e, I, H);
            orc_mat d = orc_expert_mat(L->down, e, H, I);
            orc_expert(g.w, g.s, g.b, u.w, u.s, u.b, d.w, d.s, d.b, H, I, xd, o);
            for (int h = 0; h < H; ++h) yt[h] += p[i] * o[h];
        }
        double sigma = 0.0;
        if (L->has_shared) {
            sigma = orc_sigmoid_gate(L->shared_gate, H, xt);
            orc_expert_bits(L->shared_bits == 8 ? 8 : 4, L->sh_gate.w, L->sh_gate.s, L->sh_gate.b,
                            L->sh_up.w, L->sh_up.s, L->sh_up.b, L->sh_down.w, L->sh_down.s,
                            L->sh_down.b, H, I, xd, o);
            for (int h = 0; h < H; ++h) yt[h] += sigma * o[h];
        }
        if (idx_out) memcpy(idx_out + (size_t)t * k, idx, sizeof(int32_t) * (size_t)k);
        if (p_out) memcpy(p_out + (size_t)t * k, p, sizeof(double) * (size_t)k);
        if (logits_out) memcpy(logits_out + (size_t)t * E, lg, sizeof(double) * (size_t)E);
        if (sigma_out) sigma_out[t] = sigma;
        free(xd);
        free(lg);
        free(o);
        free(idx);
        free(p);
    }
}

/* Router logits only, for T tokens (used to measure top-k gaps). */
void orc_router_tokens(const orc_layer *L, const uint16_t *x, int T, double *logits) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        orc_layer_router(L, x + (size_t)t * L->H, logits + (size_t)t * L->E);
}
