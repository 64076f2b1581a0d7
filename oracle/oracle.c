/*
 * Oracle for the batch-1 fine-grained MoE verify step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark can check the CUDA library against a plain,
 * slow, obviously correct restatement of what the step computes. It shares
 * no code, header, table or constant with the CUDA library.
 *
 * Sources (web pages on the subject; section names as printed on them):
 *  - "llm-decoding" blog post, us-homepage.pages.dev:
 *      §"What batch-1 latency actually is" and §"The exact architecture":
 *        128 experts, top-8 routed plus one always-on shared expert,
 *        expert FFN width 704, hidden 2816, 30 layers, tied 262,144-word
 *        lm_head.
 *      §"Where the 7.36 GB goes": gate, up and down matrices of 2816x704
 *        per expert.
 *      §"Lever 1: fewer bytes (FP8 weights)" and §"Why halving the weight
 *        bytes bought only 17 percent": weights stored in 8 bits,
 *        dequantised and multiplied at higher precision.
 *      §"Lever 2: fewer passes (native MTP)": the target verifies the
 *        drafted tokens in one pass and keeps those it would have produced.
 *      §"What we learned": the output is identical to ordinary decoding.
 *  - "Anton, chapter 10: Making Gemma fly" (lyb.re), §"Making Gemma fly":
 *        the big model verifies the drafter's guesses in one pass.
 *  The benchmark configurations of the build fix the parts the pages leave
 *  open: softmax then top-8 renormalised routing, GELU-tanh gating, E4M3
 *  weights with one fp32 scale per output row, a unit-gain RMSNorm with
 *  eps 1e-6 before each layer and a residual add after it.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - the shared expert is a 704-wide expert stored after the routed ones and
 *    enters the sum with weight 1;
 *  - top-k and argmax ties go to the lower index;
 *  - accepted length a is the longest prefix of drafts equal to the target's
 *    argmax at the preceding position, and the next token is the target's
 *    argmax at position a.
 *
 * Arithmetic: every sum is accumulated in double precision in natural index
 * order. Activations arrive as doubles (callers pass exactly the bf16 or
 * fp32 values that define the input). E4M3 and bf16 codes are decoded by the
 * format's formula, never through a hardware conversion.
 *
 * Parallelism: OpenMP splits loops over independent output elements only;
 * no sum is split, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Number formats                                                       */
/* ------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("fn" flavour): sign, 4 exponent bits with bias 7, 3 mantissa
 * bits. Exponent field 0 holds subnormals m/8 * 2^-6. There are no
 * infinities; S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 * 2^8 = 448. */
double fgmo_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int exp_field = (code >> 3) & 0xF;
    int mant = code & 0x7;
    double mag;
    if (exp_field == 0xF && mant == 0x7)
        return NAN;
    if (exp_field == 0)
        mag = ldexp((double)mant / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, exp_field - 7);
    return sign ? -mag : mag;
}

/* Nearest E4M3 code, ties to the even code, saturating at +-448; NaN maps to
 * the positive NaN code. Done by exhaustive search over the 127 finite
 * non-negative codes, which are ordered by magnitude. */
uint8_t fgmo_e4m3_encode(double v)
{
    uint8_t best = 0;
    double best_err = INFINITY;
    double a;
    int c;
    if (isnan(v))
        return 0x7F;
    a = fabs(v);
    if (a >= 448.0) {
        best = 0x7E;
    } else {
        for (c = 0; c <= 0x7E; ++c) {
            double err = fabs(fgmo_e4m3_decode((uint8_t)c) - a);
            if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
                best_err = err;
                best = (uint8_t)c;
            }
        }
    }
    return (uint8_t)(best | (v < 0 || (v == 0 && signbit(v)) ? 0x80 : 0));
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double fgmo_bf16_decode(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits), ties to even. */
uint16_t fgmo_bf16_round(double v)
{
    double q;
    float f;
    uint32_t u;
    int e;
    if (isnan(v))
        return 0x7FC0;
    if (v == 0.0)
        return signbit(v) ? 0x8000 : 0x0000;
    frexp(v, &e);                 /* |v| in [2^(e-1), 2^e) */
    if (e < -125)
        e = -125;                 /* below the normal range the step is fixed */
    q = ldexp(nearbyint(ldexp(v, 8 - e)), e - 8);
    if (fabs(q) > 3.3895313892515355e38)   /* beyond the largest finite bf16 */
        q = copysign(INFINITY, v);
    f = (float)q;                 /* exact: q has at most 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

void fgmo_bf16_round_array(const double *v, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = fgmo_bf16_round(v[i]);
}

/* Per-row weight quantiser: scale = max|row| / 448 (fp32), code = nearest
 * E4M3 of w / scale; an all-zero row gets scale 1. */
void fgmo_quantize_rows(const float *w, int64_t rows, int64_t cols, uint8_t *q, float *scale)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        const float *row = w + r * cols;
        float amax = 0.0f, s;
        int64_t c;
        for (c = 0; c < cols; ++c)
            if (fabsf(row[c]) > amax)
                amax = fabsf(row[c]);
        s = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[r] = s;
        for (c = 0; c < cols; ++c)
            q[r * cols + c] = fgmo_e4m3_encode((double)(row[c] / s));
    }
}

/* ------------------------------------------------------------------ */
/* Model pieces                                                         */
/* ------------------------------------------------------------------ */

/* tanh-approximated GELU: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))). */
double fgmo_gelu_tanh(double x)
{
    const double k = sqrt(2.0 / M_PI);
    return 0.5 * x * (1.0 + tanh(k * (x + 0.044715 * x * x * x)));
}

/* Unit-gain RMSNorm of each of the M rows of h: x / sqrt(mean(x^2) + eps). */
void fgmo_rmsnorm(const double *h, int M, int H, double eps, double *out)
{
    int t, j;
    for (t = 0; t < M; ++t) {
        double ss = 0.0, r;
        for (j = 0; j < H; ++j)
            ss += h[(int64_t)t * H + j] * h[(int64_t)t * H + j];
        r = 1.0 / sqrt(ss / H + eps);
        for (j = 0; j < H; ++j)
            out[(int64_t)t * H + j] = h[(int64_t)t * H + j] * r;
    }
}

/* Shapes of one MoE layer. Experts 0..E-1 are routed; when n_shared is 1,
 * expert E is the always-on shared expert. */
typedef struct {
    int H;        /* hidden width */
    int F;        /* expert FFN width */
    int E;        /* routed experts */
    int k;        /* experts picked per token */
    int n_shared; /* 0 or 1 */
} fgmo_dims;

/* One MoE layer's parameters, all host pointers.
 *   router_w  bf16 bits [E][H]
 *   router_b  fp32 [E] or NULL (added to the logits)
 *   gate_q, up_q  E4M3 [E+n_shared][F][H];  gate_s, up_s  fp32 [E+n_shared][F]
 *   down_q        E4M3 [E+n_shared][H][F];  down_s        fp32 [E+n_shared][H] */
typedef struct {
    const uint16_t *router_w;
    const float *router_b;
    const uint8_t *gate_q;
    const float *gate_s;
    const uint8_t *up_q;
    const float *up_s;
    const uint8_t *down_q;
    const float *down_s;
} fgmo_layer;

/* Router for one token: logits l = W_r x + b, softmax over all E experts,
 * the k largest (ties to the lower index) renormalised to sum to 1.
 * Writes ids[k] (descending weight), w[k], logits[E] (may be NULL) and
 * returns the logit margin between the k-th and (k+1)-th choice (INFINITY
 * when k == E). */
double fgmo_router_token(const double *x, const uint16_t *router_w, const float *router_b,
                         int H, int E, int k, int32_t *ids, double *w, double *logits_out)
{
    double *l = (double *)malloc(sizeof(double) * E);
    double *p = (double *)malloc(sizeof(double) * E);
    char *taken = (char *)calloc(E, 1);
    double lmax = -INFINITY, z = 0.0, ptop = 0.0, margin = INFINITY, kth = 0.0;
    int e, j, i;
    for (e = 0; e < E; ++e) {
        double acc = 0.0;
        for (j = 0; j < H; ++j)
            acc += fgmo_bf16_decode(router_w[(int64_t)e * H + j]) * x[j];
        l[e] = acc + (router_b ? (double)router_b[e] : 0.0);
        if (l[e] > lmax)
            lmax = l[e];
    }
    for (e = 0; e < E; ++e) {
        p[e] = exp(l[e] - lmax);
        z += p[e];
    }
    for (e = 0; e < E; ++e)
        p[e] /= z;
    /* selection by repeated maximum over the untaken experts */
    for (i = 0; i < k; ++i) {
        int best = -1;
        for (e = 0; e < E; ++e)
            if (!taken[e] && (best < 0 || l[e] > l[best]))
                best = e;
        taken[best] = 1;
        ids[i] = best;
        kth = l[best];
    }
    for (e = 0; e < E; ++e)
        if (!taken[e] && kth - l[e] < margin)
            margin = kth - l[e];
    for (i = 0; i < k; ++i)
        ptop += p[ids[i]];
    for (i = 0; i < k; ++i)
        w[i] = p[ids[i]] / ptop;
    if (logits_out)
        memcpy(logits_out, l, sizeof(double) * E);
    free(l);
    free(p);
    free(taken);
    return margin;
}

/* A gated-GELU MLP of width F: gate/up rows [F][H] and down rows [H][F] as
 * E4M3 codes with one fp32 scale per row. An expert is its F = 704 case; the
 * always-on dense MLP that "llm-decoding" §"Where the 7.36 GB goes" counts at
 * 2816x2112 is its F = 2112 case. */
typedef struct {
    int F;
    const uint8_t *gate_q;   /* [F][H] */
    const float *gate_s;     /* [F] */
    const uint8_t *up_q;     /* [F][H] */
    const float *up_s;       /* [F] */
    const uint8_t *down_q;   /* [H][F] */
    const float *down_s;     /* [H] */
} fgmo_mlp;

/* The MLP on one token x[H]: g = s_g * (Q_g x), u = s_u * (Q_u x),
 * a = gelu_tanh(g) * u, out = s_d * (Q_d a). Weights are dequantised code by
 * code from E4M3 with their row scale. */
void fgmo_mlp_token(int H, const fgmo_mlp *m, const double *x, double *out)
{
    const int F = m->F;
    double *a = (double *)malloc(sizeof(double) * F);
    int i, j;
#pragma omp parallel for schedule(static)
    for (i = 0; i < F; ++i) {
        double g = 0.0, u = 0.0;
        int jj;
        for (jj = 0; jj < H; ++jj) {
            g += fgmo_e4m3_decode(m->gate_q[(int64_t)i * H + jj]) * x[jj];
            u += fgmo_e4m3_decode(m->up_q[(int64_t)i * H + jj]) * x[jj];
        }
        g *= (double)m->gate_s[i];
        u *= (double)m->up_s[i];
        a[i] = fgmo_gelu_tanh(g) * u;
    }
#pragma omp parallel for schedule(static)
    for (j = 0; j < H; ++j) {
        double acc = 0.0;
        int ii;
        for (ii = 0; ii < F; ++ii)
            acc += fgmo_e4m3_decode(m->down_q[(int64_t)j * F + ii]) * a[ii];
        out[j] = (double)m->down_s[j] * acc;
    }
    free(a);
}

/* Expert e of a layer applied to one token x[H]. */
void fgmo_expert_token(const fgmo_dims *d, const fgmo_layer *L, int expert, const double *x,
                       double *out)
{
    const int H = d->H, F = d->F;
    fgmo_mlp m;
    m.F = F;
    m.gate_q = L->gate_q + (int64_t)expert * F * H;
    m.gate_s = L->gate_s + (int64_t)expert * F;
    m.up_q = L->up_q + (int64_t)expert * F * H;
    m.up_s = L->up_s + (int64_t)expert * F;
    m.down_q = L->down_q + (int64_t)expert * H * F;
    m.down_s = L->down_s + (int64_t)expert * H;
    fgmo_mlp_token(H, &m, x, out);
}

/* One MoE layer on M tokens x[M][H]:
 *   y_t = sum_i w_{t,i} * expert_{ids_{t,i}}(x_t) + shared(x_t).
 * shared: the MLP `dense` when given (any width; the layer's own shared
 * expert is then not used), else expert E when d->n_shared, else nothing.
 * ids[M][k], w[M][k], margin[M] and logits[M][E] are outputs (logits may be
 * NULL). */
void fgmo_moe_layer_dense(const fgmo_dims *d, const fgmo_layer *L, const fgmo_mlp *dense, const double *x,
                          int M, double *y, int32_t *ids, double *w, double *margin, double *logits)
{
    const int H = d->H;
    double *tmp = (double *)malloc(sizeof(double) * H);
    int t, i, j;
    for (t = 0; t < M; ++t) {
        const double *xt = x + (int64_t)t * H;
        double *yt = y + (int64_t)t * H;
        margin[t] = fgmo_router_token(xt, L->router_w, L->router_b, H, d->E, d->k,
                                      ids + (int64_t)t * d->k, w + (int64_t)t * d->k,
                                      logits ? logits + (int64_t)t * d->E : NULL);
        for (j = 0; j < H; ++j)
            yt[j] = 0.0;
        for (i = 0; i < d->k; ++i) {
            fgmo_expert_token(d, L, ids[(int64_t)t * d->k + i], xt, tmp);
            for (j = 0; j < H; ++j)
                yt[j] += w[(int64_t)t * d->k + i] * tmp[j];
        }
        if (dense || d->n_shared) {
            if (dense)
                fgmo_mlp_token(H, dense, xt, tmp);
            else
                fgmo_expert_token(d, L, d->E, xt, tmp);
            for (j = 0; j < H; ++j)
                yt[j] += tmp[j];
        }
    }
    free(tmp);
}

void fgmo_moe_layer(const fgmo_dims *d, const fgmo_layer *L, const double *x, int M, double *y,
                    int32_t *ids, double *w, double *margin, double *logits)
{
    fgmo_moe_layer_dense(d, L, NULL, x, M, y, ids, w, margin, logits);
}

/* One layer of the stack: h <- h + layer(RMSNorm(h)), in place. */
void fgmo_stack_layer(const fgmo_dims *d, const fgmo_layer *L, double *h, int M, double eps,
                      int32_t *ids, double *w, double *margin)
{
    const int64_t n = (int64_t)M * d->H;
    double *xn = (double *)malloc(sizeof(double) * n);
    double *y = (double *)malloc(sizeof(double) * n);
    int64_t i;
    fgmo_rmsnorm(h, M, d->H, eps, xn);
    fgmo_moe_layer(d, L, xn, M, y, ids, w, margin, NULL);
    for (i = 0; i < n; ++i)
        h[i] += y[i];
    free(xn);
    free(y);
}

/* Logits of one vocabulary row v for the M hidden rows: z[t] = sum_j E[v][j] h_t[j],
 * summed in natural j order. The two storage formats of the embedding: */
typedef void (*fgmo_row_logits)(const void *rows, int64_t v, int H, const double *h, int M, double *z);

typedef struct {
    const uint8_t *q;     /* [V][H] E4M3 codes */
    const float *scale;   /* [V] fp32 row scales */
} fgmo_fp8_rows;

/* bf16 rows, decoded by the format's formula. */
static void row_logits_bf16(const void *rows, int64_t v, int H, const double *h, int M, double *z)
{
    const uint16_t *emb = (const uint16_t *)rows;
    int j, t;
    for (t = 0; t < M; ++t)
        z[t] = 0.0;
    for (j = 0; j < H; ++j) {
        double e = fgmo_bf16_decode(emb[v * H + j]);
        for (t = 0; t < M; ++t)
            z[t] += e * h[(int64_t)t * H + j];
    }
}

/* E4M3 rows with one fp32 scale per row, the expert weights' format applied to
 * the embedding: z = s_v * (Q_v h), the same form as the gate/up products. */
static void row_logits_fp8(const void *rows, int64_t v, int H, const double *h, int M, double *z)
{
    const fgmo_fp8_rows *r = (const fgmo_fp8_rows *)rows;
    int j, t;
    for (t = 0; t < M; ++t)
        z[t] = 0.0;
    for (j = 0; j < H; ++j) {
        double e = fgmo_e4m3_decode(r->q[v * H + j]);
        for (t = 0; t < M; ++t)
            z[t] += e * h[(int64_t)t * H + j];
    }
    for (t = 0; t < M; ++t)
        z[t] *= (double)r->scale[v];
}

/* Argmax over the V rows of the logits of each token: argmax[t] (ties to the
 * lower index), maxlogit[t] and the gap to the runner-up margin[t]. Rows are
 * independent; each row is visited once for all M tokens. NaN logits never
 * win; if every logit of a token is NaN its argmax is -1. */
static void lm_head_argmax(fgmo_row_logits row_logits, const void *rows, int64_t V, int H, const double *h,
                           int M, int32_t *argmax, double *maxlogit, double *margin)
{
    int t;
    double best[16], second[16];
    int64_t bidx[16];
    if (M < 1 || M > 16)
        return;
    for (t = 0; t < M; ++t) {
        best[t] = -INFINITY;
        second[t] = -INFINITY;
        bidx[t] = -1;
    }
#pragma omp parallel
    {
        double lb[16], ls[16], z[16];
        int64_t li[16];
        int64_t v;
        int tt;
        for (tt = 0; tt < M; ++tt) {
            lb[tt] = -INFINITY;
            ls[tt] = -INFINITY;
            li[tt] = -1;
        }
#pragma omp for schedule(static)
        for (v = 0; v < V; ++v) {
            row_logits(rows, v, H, h, M, z);
            for (tt = 0; tt < M; ++tt) {
                if (z[tt] > lb[tt]) {
                    ls[tt] = lb[tt];
                    lb[tt] = z[tt];
                    li[tt] = v;
                } else if (z[tt] > ls[tt]) {
                    ls[tt] = z[tt];
                }
            }
        }
#pragma omp critical
        for (tt = 0; tt < M; ++tt) {
            /* merge (value desc, index asc) */
            if (li[tt] >= 0 && (lb[tt] > best[tt] || (lb[tt] == best[tt] && li[tt] < bidx[tt]))) {
                double old = best[tt];
                second[tt] = fmax(old, fmax(second[tt], ls[tt]));
                best[tt] = lb[tt];
                bidx[tt] = li[tt];
            } else {
                second[tt] = fmax(second[tt], lb[tt]);
            }
        }
    }
    for (t = 0; t < M; ++t) {
        argmax[t] = (int32_t)bidx[t];
        if (maxlogit)
            maxlogit[t] = best[t];
        if (margin)
            margin[t] = best[t] - second[t];
    }
}

/* Tied lm_head with argmax over the bf16 embedding rows. */
void fgmo_lm_head(const uint16_t *emb, int64_t V, int H, const double *h, int M, int32_t *argmax,
                  double *maxlogit, double *margin)
{
    lm_head_argmax(row_logits_bf16, emb, V, H, h, M, argmax, maxlogit, margin);
}

/* FP8 lm_head with argmax ("llm-decoding", §"Lever 1: fewer bytes (FP8
 * weights)": every weight, the tied 262,144-word output projection included,
 * stored in 8 bits and dequantised for the product; §"First principles:
 * compute-bound or memory-bound?" counts that projection at a fifth of a
 * token's bytes in BF16). The embedding is stored as E4M3 codes q[V][H] with
 * one fp32 scale per row, z_{t,v} = scale[v] * sum_j e4m3(q[v][j]) h_t[j];
 * outputs and tie rule as fgmo_lm_head. */
void fgmo_lm_head_fp8(const uint8_t *q, const float *scale, int64_t V, int H, const double *h, int M,
                      int32_t *argmax, double *maxlogit, double *margin)
{
    fgmo_fp8_rows rows;
    rows.q = q;
    rows.scale = scale;
    lm_head_argmax(row_logits_fp8, &rows, V, H, h, M, argmax, maxlogit, margin);
}

/* Greedy verify: target[0..M-1] are the target's argmax tokens at the M
 * positions, draft[0..M-2] the drafter's tokens d_1..d_gamma. Accepted
 * length a = largest j <= gamma with d_1..d_j equal to target_0..target_{j-1};
 * out[0] = a, out[1] = target_a (the token emitted after the accepted
 * drafts). */
void fgmo_spec_verify(const int32_t *target, const int32_t *draft, int M, int32_t *out)
{
    int a = 0;
    while (a < M - 1 && draft[a] == target[a])
        ++a;
    out[0] = a;
    out[1] = target[a];
}

/* Logits of the tied bf16 lm_head for all V rows: z[t][v] = sum_j E[v][j] h_t[j]
 * (the quantity fgmo_lm_head takes the argmax of). z is [M][V]. */
void fgmo_lm_head_logits(const uint16_t *emb, int64_t V, int H, const double *h, int M, double *z)
{
    int64_t v;
#pragma omp parallel for schedule(static)
    for (v = 0; v < V; ++v) {
        double zz[16];
        int t;
        row_logits_bf16(emb, v, H, h, M, zz);
        for (t = 0; t < M; ++t)
            z[(int64_t)t * V + v] = zz[t];
    }
}

/* Inverse CDF of the unnormalised weights w[0..V-1] at u in [0, 1): the
 * smallest v with w_0 + ... + w_v > u * (w_0 + ... + w_{V-1}), summed in
 * vocabulary order; *gap = distance from u * total to the nearest partial sum
 * (how far u is from choosing a neighbour). */
static int64_t inverse_cdf(const double *w, int64_t V, double u, double *gap)
{
    double total = 0.0, target, acc = 0.0, prev = 0.0;
    int64_t v, last = -1;
    for (v = 0; v < V; ++v)
        total += w[v];
    target = u * total;
    for (v = 0; v < V; ++v) {
        if (w[v] <= 0.0)
            continue;
        last = v;
        prev = acc;
        acc += w[v];
        if (acc > target) {
            if (gap)
                *gap = fmin(target - prev, acc - target);
            return v;
        }
    }
    if (gap)
        *gap = 0.0;   /* u * total reached the end only through rounding */
    return last;
}

/* Speculative sampling verify at temperature T > 0 ("llm-decoding",
 * §"What we learned": a proposed token is kept only if it passes the
 * distribution the full model samples from, and a rejected one falls back to
 * a real model step, so the output distribution equals ordinary decoding).
 * The drafter here proposes tokens only: its distribution at position i is
 * one-hot at d_i. Then, with p_i = softmax(z_i / T) over the V logits of
 * position i:
 *   for i = 0 .. M-2: accept d_i if u_acc[i] < p_i(d_i); otherwise emit a
 *     sample of p_i with d_i removed (renormalised), by inverse CDF at
 *     u_next[i], and stop: out = {i, sample};
 *   if all M-1 drafts pass: emit a sample of p_{M-1} at u_next[M-1]:
 *     out = {M-1, sample}.
 * z is [M][V]; u_acc [M-1] and u_next [M] are uniforms in [0, 1) supplied by
 * the caller. margin[0] = the smallest |u_acc[i] - p_i(d_i)| over the tested
 * drafts, margin[1] = the inverse-CDF gap of the emitted sample, relative to
 * the distribution's total (decisions closer than these may round either
 * way in another summation order). */
void fgmo_spec_sample(const double *z, int64_t V, int M, double T, const int32_t *draft, const double *u_acc,
                      const double *u_next, int32_t *out, double *margin)
{
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    double acc_margin = INFINITY, gap = 0.0;
    int i;
    for (i = 0; i < M; ++i) {
        const double *zi = z + (int64_t)i * V;
        double zmax = -INFINITY, total = 0.0;
        int64_t v, pick;
        for (v = 0; v < V; ++v)
            if (zi[v] > zmax)
                zmax = zi[v];
        for (v = 0; v < V; ++v) {
            w[v] = exp((zi[v] - zmax) / T);
            total += w[v];
        }
        if (i < M - 1) {
            const double pd = w[draft[i]] / total;
            acc_margin = fmin(acc_margin, fabs(u_acc[i] - pd));
            if (u_acc[i] < pd)
                continue;
            w[draft[i]] = 0.0;
        }
        pick = inverse_cdf(w, V, u_next[i], &gap);
        {
            double tot = 0.0;
            for (v = 0; v < V; ++v)
                tot += w[v];
            gap = tot > 0.0 ? gap / tot : 0.0;
        }
        out[0] = i;
        out[1] = (int32_t)pick;
        break;
    }
    if (margin) {
        margin[0] = acc_margin;
        margin[1] = gap;
    }
    free(w);
}

int fgmo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void fgmo_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Array forms used by the Python wrapper. */
void fgmo_e4m3_decode_array(const uint8_t *codes, int64_t n, double *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = fgmo_e4m3_decode(codes[i]);
}

void fgmo_e4m3_encode_array(const double *v, int64_t n, uint8_t *out)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i)
        out[i] = fgmo_e4m3_encode(v[i]);
}

void fgmo_gelu_tanh_array(const double *x, int64_t n, double *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = fgmo_gelu_tanh(x[i]);
}
