/*
 * CPU ORACLE for the streamed-expert MoE layer -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library. The product path (the CUDA library and its Python
 * binding) never calls it, and the two share no code: only the seeded input
 * generators (workload/) feed both.
 *
 * Plain, single-threaded, slow and obviously correct. Compiled twice:
 *   liboracle32.so with REAL = float  (gcc -O2 -ffp-contract=off, no fast-math, SSE2)
 *   liboracle64.so with REAL = double (bounds the fp32 oracle's own rounding error)
 *
 * What it computes, per token and per layer (sources are the pages' titles and
 * sections; the shapes and formats come from the synthetic model configuration
 * of a Gemma-4-26B-A4B-style layer):
 *
 *  - RMSNorm of the layer input ("Como executar um modelo de 26 bilhoes de
 *    parametros em dois gigabytes de memoria em um Mac comum", section "Sem
 *    dependencias do llama.cpp e MLX": hand-written RMSNorm, GEMV, MoE and
 *    quantisation kernels). Reading: eps = 1e-6, unit gain.
 *  - Router GEMV, top-8 selection and the routing weights (same page, section
 *    "Qual e o principal truque da arquitetura": the router of each layer picks
 *    the 8 experts the token needs). Reading: top-8 on the logits, ties to the
 *    lower expert index, softmax over the 8 selected logits (weights sum to 1).
 *  - 4-bit expert FFN: affine int4 codes q in 0..15 with an fp16 scale s and
 *    bias b per group of 64 along K, W = s*q + b; g = Wg n, u = Wu n,
 *    h = gelu_tanh(g) * u, y = Wd h (page "Show HN: mecanismo de codigo aberto
 *    executando Gemma 4 26B em 2 GB de RAM ...", section "Abordagem tecnica (MoE +
 *    streaming por SSD)": MoE sparsity, a 3.36 MB expert at 4 bits).
 *  - Dense shared expert on the same normalised input, bf16 weights (devtrends
 *    page, "Qual e o principal truque da arquitetura": the GPU computes the
 *    shared-expert branch while missing experts are read).
 *  - Combine: delta = shared + sum_i w_i * y_i in top-k order; out = bf16(x + delta).
 *  - 16-slot LFU expert cache per layer (devtrends page, "Qual e o principal
 *    truque da arquitetura": 16 slots, LFU). Reading: textbook LFU, see or_lfu_step.
 *  - The attention half of a decoder layer for one token with RoPE and an FP16
 *    KV cache (devtrends page, "Qual e o principal truque da arquitetura": the
 *    shared core and the FP16 KV cache stay resident; "Sem dependencias do
 *    llama.cpp e MLX": hand-written attention and RoPE kernels). The pages give
 *    no attention shapes or conventions; the reading is a plain pre-norm
 *    grouped-query attention, see or_attn_decode.
 *
 * Threads. The plain build is single-threaded. The same file is also built with
 * -fopenmp (liboracle32mt.so), which only spreads the independent output rows
 * of the router, the dequantisation and the matrix-vector products over the
 * host's cores; each row is still summed by one thread in the order below, so
 * that build's results are bit-identical to the single-threaded ones. It
 * exists to time the oracle on all cores.
 *
 * Canonical reduction order (used for sum x^2 and for the router dot products,
 * so that the top-8 selection is reproducible bit for bit): 32 partial sums,
 * partial l accumulating the terms k = l, l+32, l+64, ... in increasing k; then
 * five butterfly rounds p_l <- p_l + p_(l xor d) for d = 16, 8, 4, 2, 1; the
 * result is p_0. All other sums run sequentially in increasing index.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef REAL
#define REAL float
#endif

#if REAL_IS_DOUBLE
#define R_SQRT sqrt
#define R_EXP exp
#define R_TANH tanh
#else
#define R_SQRT sqrtf
#define R_EXP expf
#define R_TANH tanhf
#endif

#define OR_GROUP 64

/* ---------------------------------------------------------------- encodings */

/* IEEE binary16 -> fp32 (exact). */
float or_half_to_float(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t ex = (uint32_t)(h >> 10) & 0x1Fu;
    uint32_t man = (uint32_t)h & 0x3FFu;
    float v;
    if (ex == 0) {
        v = ldexpf((float)man, -24);                 /* zero or subnormal: man * 2^-24 */
    } else if (ex == 31) {
        v = man ? NAN : INFINITY;
    } else {
        v = ldexpf((float)(man + 1024u), (int)ex - 25); /* (1024 + man) * 2^(ex - 15 - 10) */
    }
    return sign ? -v : v;
}

/* bf16 -> fp32 (exact: bf16 is the top half of an fp32). */
float or_bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even. */
uint16_t or_float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* fp32 -> IEEE binary16, round to nearest, ties to even (overflow -> inf, NaN kept). */
uint16_t or_float_to_half(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t sign = (u >> 16) & 0x8000u;
    if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
    float a = fabsf(f);
    if (a == 0.0f) return (uint16_t)sign;
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7C00u);     /* rounds past the largest finite value */
    /* a = m * 2^e with the spacing of binary16 at a: 2^(e - 10) for normal values (e >= -14), 2^-24 below */
    int e;
    frexpf(a, &e);                                            /* a in [2^(e-1), 2^e) */
    int q = e - 1 - 10;
    if (q < -24) q = -24;
    float steps = ldexpf(a, -q);                              /* exact: a / 2^q */
    float fl = floorf(steps);
    float rem = steps - fl;
    uint32_t n = (uint32_t)fl;
    if (rem > 0.5f || (rem == 0.5f && (n & 1u))) n += 1u;    /* n * 2^q is the rounded magnitude */
    /* encode n * 2^q: subnormal when q = -24 and n < 1024 */
    uint32_t bits;
    if (q == -24 && n < 1024u) {
        bits = n;
    } else {
        int ex = q + 25;                                       /* biased exponent of n * 2^q with n in [1024, 2048] */
        if (n == 2048u) { n = 1024u; ex += 1; }
        if (ex >= 31) return (uint16_t)(sign | 0x7C00u);
        bits = ((uint32_t)ex << 10) | (n - 1024u);
    }
    return (uint16_t)(sign | bits);
}

static REAL to_bf16_real(REAL v) { return (REAL)or_bf16_to_float(or_float_to_bf16((float)v)); }
static REAL to_f16_real(REAL v) { return (REAL)or_half_to_float(or_float_to_half((float)v)); }

/* Operand formats of the tensor-core reading: values are rounded from fp32 to this format before
 * their products (OR_FMT_NONE: kept as they are, the fp32 reading). */
enum { OR_FMT_NONE = 0, OR_FMT_BF16 = 1, OR_FMT_F16 = 2 };
static REAL to_fmt(REAL v, int fmt) {
    if (fmt == OR_FMT_BF16) return to_bf16_real(v);
    if (fmt == OR_FMT_F16) return to_f16_real(v);
    return v;
}

/* ------------------------------------------------------- canonical reduction */

/* Sum of t[0..n) in the canonical order described in the header. */
static REAL canonical_sum(const REAL* t, int n) {
    REAL p[32], q[32];
    for (int l = 0; l < 32; ++l) p[l] = (REAL)0;
    for (int l = 0; l < 32; ++l)
        for (int k = l; k < n; k += 32) p[l] = p[l] + t[k];
    for (int d = 16; d >= 1; d >>= 1) {
        for (int l = 0; l < 32; ++l) q[l] = p[l] + p[l ^ d];
        memcpy(p, q, sizeof(p));
    }
    return p[0];
}

/* ------------------------------------------------------------------ RMSNorm */

/* r = 1 / sqrt(mean(x^2) + eps); the normalised input is n_k = r * x_k. */
REAL or_rms_scale(const uint16_t* x, int H, double eps) {
    REAL* t = (REAL*)malloc(sizeof(REAL) * (size_t)H);
    for (int k = 0; k < H; ++k) {
        REAL xk = (REAL)or_bf16_to_float(x[k]);
        t[k] = xk * xk;                       /* exact: bf16 * bf16 fits fp32 */
    }
    REAL ss = canonical_sum(t, H);
    free(t);
    REAL ms = ss / (REAL)H;
    return (REAL)1 / R_SQRT(ms + (REAL)eps);
}

void or_normalise(const uint16_t* x, int H, REAL r, REAL* n) {
    for (int k = 0; k < H; ++k) n[k] = r * (REAL)or_bf16_to_float(x[k]);
}

/* ------------------------------------------------------------------- router */

/* z_e = (r * d_e) + bias_e with d_e = sum_k Wr[e,k] x_k in canonical order. */
void or_router_logits(const uint16_t* x, int H, const uint16_t* Wr, int E, const float* bias,
                      REAL r, REAL* z) {
#pragma omp parallel for schedule(static)
    for (int e = 0; e < E; ++e) {
        REAL* t = (REAL*)malloc(sizeof(REAL) * (size_t)H);
        for (int k = 0; k < H; ++k)
            t[k] = (REAL)or_bf16_to_float(Wr[(size_t)e * H + k]) * (REAL)or_bf16_to_float(x[k]);
        REAL d = canonical_sum(t, H);
        REAL v = r * d;
        if (bias) v = v + (REAL)bias[e];
        z[e] = v;
        free(t);
    }
}

/* a ranks before b: larger value first, equal values -> lower index; NaN below everything. */
static int ranks_before(REAL za, int a, REAL zb, int b) {
    int na = isnan(za), nb = isnan(zb);
    if (na || nb) return (na == nb) ? (a < b) : nb;
    if (za > zb) return 1;
    if (za < zb) return 0;
    return a < b;
}

/* Indices of the k best logits, best first (selection by repeated scan). */
void or_topk(const REAL* z, int E, int k, int32_t* idx) {
    char* taken = (char*)calloc((size_t)E, 1);
    for (int i = 0; i < k; ++i) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            if (best < 0 || ranks_before(z[e], e, z[best], best)) best = e;
        }
        idx[i] = best;
        taken[best] = 1;
    }
    free(taken);
}

/* w_i = exp(z_i - z_max) / sum_j exp(z_j - z_max) over the k selected logits. */
void or_softmax_selected(const REAL* z, const int32_t* idx, int k, REAL* w) {
    REAL zmax = z[idx[0]];
    for (int i = 1; i < k; ++i)
        if (z[idx[i]] > zmax) zmax = z[idx[i]];
    REAL sum = (REAL)0;
    for (int i = 0; i < k; ++i) {
        w[i] = R_EXP(z[idx[i]] - zmax);
        sum = sum + w[i];
    }
    for (int i = 0; i < k; ++i) w[i] = w[i] / sum;
}

/* -------------------------------------------------------------- dequantise */

/* W = s * q + b. s * q is exact (11-bit * 4-bit), so this is one rounding. */
REAL or_dequant(uint8_t q, uint16_t s, uint16_t b) {
    REAL sv = (REAL)or_half_to_float(s);
    REAL bv = (REAL)or_half_to_float(b);
    REAL p = sv * (REAL)q;
    return p + bv;
}

/* Dense [R, K] matrix from codes q[R][K] and s, b [R][K/64]; fmt rounds each weight (OR_FMT_*). */
void or_dequant_matrix(const uint8_t* q, const uint16_t* s, const uint16_t* b, int R, int K,
                       int fmt, REAL* W) {
    int G = K / OR_GROUP;
#pragma omp parallel for schedule(static)
    for (int j = 0; j < R; ++j)
        for (int k = 0; k < K; ++k) {
            size_t gi = (size_t)j * G + (size_t)(k / OR_GROUP);
            REAL w = or_dequant(q[(size_t)j * K + k], s[gi], b[gi]);
            W[(size_t)j * K + k] = to_fmt(w, fmt);
        }
}

/* -------------------------------------------------------------------- FFN */

/* gelu(v) = 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))) (Hendrycks & Gimpel 2016, tanh form). */
REAL or_gelu(REAL v) {
    const REAL c = (REAL)0.7978845608028654;
    const REAL a = (REAL)0.044715;
    REAL v3 = v * v * v;
    REAL inner = c * (v + a * v3);
    REAL t = R_TANH(inner);
    return (REAL)0.5 * v * ((REAL)1 + t);
}

/* y[R] = W[R,K] v[K], sequential in k. */
static void matvec(const REAL* W, int R, int K, const REAL* v, REAL* y) {
#pragma omp parallel for schedule(static)
    for (int j = 0; j < R; ++j) {
        REAL acc = (REAL)0;
        for (int k = 0; k < K; ++k) acc = acc + W[(size_t)j * K + k] * v[k];
        y[j] = acc;
    }
}

typedef struct {
    const uint8_t* q[3];   /* gate [I][H], up [I][H], down [H][I] */
    const uint16_t* s[3];  /* fp16 scales  [I][H/64], [I][H/64], [H][I/64] */
    const uint16_t* b[3];  /* fp16 biases, same shapes */
} or_expert;

/*
 * One routed expert on the input v[H]:
 *   g = c (Wg v), u = c (Wu v), h = gelu(g) * u, y = Wd h,   c = in_scale.
 * The fp32 reading (formats OR_FMT_NONE) takes v = n (the normalised input) and
 * c = 1. A tensor-core reading rounds the operands of each product before it
 * (accumulation stays in REAL): Wg, Wu and v to fmt_gu, Wd and h to fmt_d (bf16
 * or fp16); there the layer passes the raw layer input (see or_layer_combine)
 * and applies the RMS scale to the two dot products after them, as the router
 * applies it. Equal to the first form in real arithmetic.
 */
void or_expert_ffn(const REAL* v, int H, int I, const or_expert* ex, int fmt_gu, int fmt_d, REAL in_scale,
                   REAL* y) {
    REAL* Wg = (REAL*)malloc(sizeof(REAL) * (size_t)I * H);
    REAL* Wu = (REAL*)malloc(sizeof(REAL) * (size_t)I * H);
    REAL* Wd = (REAL*)malloc(sizeof(REAL) * (size_t)H * I);
    REAL* nn = (REAL*)malloc(sizeof(REAL) * (size_t)H);
    REAL* g = (REAL*)malloc(sizeof(REAL) * (size_t)I);
    REAL* u = (REAL*)malloc(sizeof(REAL) * (size_t)I);
    REAL* h = (REAL*)malloc(sizeof(REAL) * (size_t)I);
    or_dequant_matrix(ex->q[0], ex->s[0], ex->b[0], I, H, fmt_gu, Wg);
    or_dequant_matrix(ex->q[1], ex->s[1], ex->b[1], I, H, fmt_gu, Wu);
    or_dequant_matrix(ex->q[2], ex->s[2], ex->b[2], H, I, fmt_d, Wd);
    for (int k = 0; k < H; ++k) nn[k] = to_fmt(v[k], fmt_gu);
    matvec(Wg, I, H, nn, g);
    matvec(Wu, I, H, nn, u);
    for (int j = 0; j < I; ++j) {
        g[j] = in_scale * g[j];
        u[j] = in_scale * u[j];
        REAL hj = or_gelu(g[j]) * u[j];
        h[j] = to_fmt(hj, fmt_d);
    }
    matvec(Wd, H, I, h, y);
    free(Wg); free(Wu); free(Wd); free(nn); free(g); free(u); free(h);
}

/* Dense shared expert with bf16 weights: gate [S,H], up [S,H], down [H,S]; the
 * input v, fmt (for v and h; the weights are bf16 already) and in_scale as for
 * or_expert_ffn. */
void or_shared_ffn(const REAL* v, int H, int S, const uint16_t* Wg16, const uint16_t* Wu16,
                   const uint16_t* Wd16, int fmt, REAL in_scale, REAL* y) {
    REAL* Wg = (REAL*)malloc(sizeof(REAL) * (size_t)S * H);
    REAL* Wu = (REAL*)malloc(sizeof(REAL) * (size_t)S * H);
    REAL* Wd = (REAL*)malloc(sizeof(REAL) * (size_t)H * S);
    REAL* nn = (REAL*)malloc(sizeof(REAL) * (size_t)H);
    REAL* g = (REAL*)malloc(sizeof(REAL) * (size_t)S);
    REAL* u = (REAL*)malloc(sizeof(REAL) * (size_t)S);
    REAL* h = (REAL*)malloc(sizeof(REAL) * (size_t)S);
    for (size_t i = 0; i < (size_t)S * H; ++i) {
        Wg[i] = (REAL)or_bf16_to_float(Wg16[i]);
        Wu[i] = (REAL)or_bf16_to_float(Wu16[i]);
        Wd[i] = (REAL)or_bf16_to_float(Wd16[i]);
    }
    for (int k = 0; k < H; ++k) nn[k] = to_fmt(v[k], fmt);
    matvec(Wg, S, H, nn, g);
    matvec(Wu, S, H, nn, u);
    for (int j = 0; j < S; ++j) {
        g[j] = in_scale * g[j];
        u[j] = in_scale * u[j];
        REAL hj = or_gelu(g[j]) * u[j];
        h[j] = to_fmt(hj, fmt);
    }
    matvec(Wd, H, S, h, y);
    free(Wg); free(Wu); free(Wd); free(nn); free(g); free(u); free(h);
}

/*
 * Routing of one token: r, the logits z[E], the top-k ids (best first) and
 * the routing weights w[k].
 */
void or_route(const uint16_t* x, int H, const uint16_t* Wr, int E, const float* bias, int k,
              double eps, REAL* r_out, REAL* z, int32_t* idx, REAL* w) {
    REAL r = or_rms_scale(x, H, eps);
    or_router_logits(x, H, Wr, E, bias, r, z);
    or_topk(z, E, k, idx);
    or_softmax_selected(z, idx, k, w);
    *r_out = r;
}

/*
 * Combine for one token, given its routing (idx only selects which experts
 * the caller passed in ex[0..k)):
 *   delta_j = shared_j + sum_{i in top-k order} w_i * y_ij ;  out_j = bf16(x_j + delta_j).
 * Wsg may be NULL (no shared expert). The fp32 reading (tc = 0) feeds the FFNs
 * n = r x. The tensor-core reading (tc = 1) feeds them the raw input and applies
 * the scale after the gate and up dot products (see or_expert_ffn): the shared
 * expert takes bf16 operands (its bf16 weights, x, h) with scale r; the routed
 * experts take fp16 operands for gate/up (the dequantised weights and x p, where
 * p = 2^e is the power of two with r = m 2^e, m in [1, 2): an exact scaling that
 * keeps the fp16 operand near unit size whatever the size of x) with scale
 * m = r / p, and bf16 operands for down (the dequantised weights and h, whose
 * range fp16 does not always hold).
 */
void or_layer_combine(const uint16_t* x, int H, int I, REAL r, int k, const or_expert* ex,
                      const REAL* w, int S, const uint16_t* Wsg, const uint16_t* Wsu,
                      const uint16_t* Wsd, int tc, uint16_t* out, REAL* delta) {
    REAL* n = (REAL*)malloc(sizeof(REAL) * (size_t)H);
    REAL* v = (REAL*)malloc(sizeof(REAL) * (size_t)H);
    REAL* y = (REAL*)malloc(sizeof(REAL) * (size_t)H);
    REAL in_scale = (REAL)1, routed_scale = (REAL)1;
    if (tc) {
        int e;
        frexp((double)r, &e);                               /* r = m 2^(e-1), m in [1, 2) */
        const REAL p = (REAL)ldexp(1.0, e - 1);
        for (int j = 0; j < H; ++j) {
            n[j] = (REAL)or_bf16_to_float(x[j]);
            v[j] = n[j] * p;                                /* exact: a power of two */
        }
        in_scale = r;
        routed_scale = r / p;                               /* exact: m */
    } else {
        or_normalise(x, H, r, n);
        for (int j = 0; j < H; ++j) v[j] = n[j];
    }
    for (int j = 0; j < H; ++j) delta[j] = (REAL)0;
    if (Wsg) {
        or_shared_ffn(n, H, S, Wsg, Wsu, Wsd, tc ? OR_FMT_BF16 : OR_FMT_NONE, in_scale, y);
        for (int j = 0; j < H; ++j) delta[j] = y[j];
    }
    for (int i = 0; i < k; ++i) {
        or_expert_ffn(v, H, I, &ex[i], tc ? OR_FMT_F16 : OR_FMT_NONE, tc ? OR_FMT_BF16 : OR_FMT_NONE, routed_scale,
                      y);
        for (int j = 0; j < H; ++j) delta[j] = delta[j] + w[i] * y[j];
    }
    for (int j = 0; j < H; ++j) {
        REAL o = (REAL)or_bf16_to_float(x[j]) + delta[j];
        out[j] = or_float_to_bf16((float)o);
    }
    free(n); free(v); free(y);
}

/* ------------------------------------------------------------ LFU simulator */

typedef struct {
    int32_t step, layer, expert, hit, slot, evicted;
} or_cache_event;

typedef struct {
    int n_layers, n_slots;
    int32_t* expert;     /* [L][S], -1 = empty */
    int64_t* count;      /* use count since admission */
    int64_t* last_use;   /* step of the last use */
} or_lfu;

or_lfu* or_lfu_new(int n_layers, int n_slots) {
    or_lfu* c = (or_lfu*)calloc(1, sizeof(or_lfu));
    size_t n = (size_t)n_layers * n_slots;
    c->n_layers = n_layers;
    c->n_slots = n_slots;
    c->expert = (int32_t*)malloc(sizeof(int32_t) * n);
    c->count = (int64_t*)calloc(n, sizeof(int64_t));
    c->last_use = (int64_t*)calloc(n, sizeof(int64_t));
    for (size_t i = 0; i < n; ++i) c->expert[i] = -1;
    return c;
}

void or_lfu_free(or_lfu* c) {
    if (!c) return;
    free(c->expert); free(c->count); free(c->last_use); free(c);
}

/*
 * One (step, layer) of the per-layer LFU cache, ids[0..n) in top-k order.
 *  pass 1: each resident id is a hit: count += 1, last_use = step;
 *  pass 2: each missing id, in order, takes the lowest empty slot, else the
 *          slot not holding any of this step's ids with the smallest count,
 *          then the oldest last_use, then the lowest index; it starts with
 *          count = 1, last_use = step.
 * Events come out in ids order. Returns the number of misses, or -1 if no
 * slot can be evicted (more ids than slots).
 */
int or_lfu_step(or_lfu* c, int step, int layer, const int32_t* ids, int n, or_cache_event* ev) {
    int S = c->n_slots;
    int32_t* ex = c->expert + (size_t)layer * S;
    int64_t* cnt = c->count + (size_t)layer * S;
    int64_t* lu = c->last_use + (size_t)layer * S;
    int misses = 0;
    for (int i = 0; i < n; ++i) {
        ev[i].step = step; ev[i].layer = layer; ev[i].expert = ids[i];
        ev[i].hit = 0; ev[i].slot = -1; ev[i].evicted = -1;
        for (int s = 0; s < S; ++s)
            if (ex[s] == ids[i]) {
                ev[i].hit = 1; ev[i].slot = s;
                cnt[s] += 1; lu[s] = step;
                break;
            }
    }
    for (int i = 0; i < n; ++i) {
        if (ev[i].hit) continue;
        misses++;
        int victim = -1;
        for (int s = 0; s < S; ++s)
            if (ex[s] < 0) { victim = s; break; }
        if (victim < 0) {
            for (int s = 0; s < S; ++s) {
                int current = 0;
                for (int j = 0; j < n; ++j) if (ex[s] == ids[j]) current = 1;
                if (current) continue;
                if (victim < 0 || cnt[s] < cnt[victim] ||
                    (cnt[s] == cnt[victim] && lu[s] < lu[victim]))
                    victim = s;
            }
        }
        if (victim < 0) return -1;
        ev[i].slot = victim;
        ev[i].evicted = ex[victim];
        ex[victim] = ids[i];
        cnt[victim] = 1;
        lu[victim] = step;
    }
    return misses;
}

void or_lfu_state(const or_lfu* c, int layer, int32_t* expert, int64_t* count, int64_t* last_use) {
    size_t o = (size_t)layer * c->n_slots;
    memcpy(expert, c->expert + o, sizeof(int32_t) * (size_t)c->n_slots);
    memcpy(count, c->count + o, sizeof(int64_t) * (size_t)c->n_slots);
    memcpy(last_use, c->last_use + o, sizeof(int64_t) * (size_t)c->n_slots);
}

/* --------------------------------------------------------------- attention */

/*
 * Attention half of a decoder layer for one token at position pos (0-based),
 * grouped-query, with RoPE and an FP16 KV cache (reading of the pages, which
 * name the kernels and the FP16 cache but give no shapes):
 *   r = 1/sqrt(sum x^2 / H + eps) (as or_rms_scale), n = r x;
 *   q = Wq n [nq*d], k = Wk n [nkv*d], v = Wv n [nkv*d]  (bf16 weights, row-major [out][H]);
 *   RoPE on every head of q and k: for j < d/2 the pair (j, j + d/2) turns by
 *     the angle pos * theta^(-2j/d):  a' = a cos - b sin,  b' = b cos + a sin
 *     (the angle, its cosine and sine in double precision);
 *   K[pos] = fp16(k'), V[pos] = fp16(v)   (caches fp16 [max_seq][nkv][d]);
 *   for each q head h, with kv head g = h / (nq / nkv):
 *     s_t = (q'_h . K[t]_g) / sqrt(d), t = 0..pos;  p = softmax(s);
 *     a_h = sum_t p_t V[t]_g;
 *   out = bf16(x + Wo a)   (Wo bf16 [H][nq*d]).
 * Sums run sequentially in increasing index. scores (nullable) receives s for
 * q head 0 (pos + 1 values); attn (nullable) receives a [nq*d].
 */
void or_attn_decode(const uint16_t* x, int H, int nq, int nkv, int d, double eps, double theta, int pos,
                    const uint16_t* Wq, const uint16_t* Wk, const uint16_t* Wv, const uint16_t* Wo,
                    uint16_t* Kc, uint16_t* Vc, uint16_t* out, REAL* scores, REAL* attn) {
    const int QD = nq * d, KD = nkv * d, half = d / 2;
    REAL r = or_rms_scale(x, H, eps);
    REAL* n = (REAL*)malloc(sizeof(REAL) * (size_t)H);
    or_normalise(x, H, r, n);
    REAL* q = (REAL*)malloc(sizeof(REAL) * (size_t)QD);
    REAL* k = (REAL*)malloc(sizeof(REAL) * (size_t)KD);
    REAL* v = (REAL*)malloc(sizeof(REAL) * (size_t)KD);
    const uint16_t* Ws[3] = {Wq, Wk, Wv};
    REAL* ys[3] = {q, k, v};
    const int rows[3] = {QD, KD, KD};
    for (int m = 0; m < 3; ++m)
        for (int j = 0; j < rows[m]; ++j) {
            REAL acc = (REAL)0;
            for (int c = 0; c < H; ++c) acc = acc + (REAL)or_bf16_to_float(Ws[m][(size_t)j * H + c]) * n[c];
            ys[m][j] = acc;
        }
    /* RoPE */
    for (int m = 0; m < 2; ++m) {
        REAL* y = ys[m];
        const int heads = m == 0 ? nq : nkv;
        for (int h = 0; h < heads; ++h)
            for (int j = 0; j < half; ++j) {
                double ang = (double)pos * pow(theta, -2.0 * (double)j / (double)d);
                REAL cs = (REAL)cos(ang), sn = (REAL)sin(ang);
                REAL a = y[h * d + j], b = y[h * d + j + half];
                y[h * d + j] = a * cs - b * sn;
                y[h * d + j + half] = b * cs + a * sn;
            }
    }
    /* the cache rows of this position */
    for (int i = 0; i < KD; ++i) {
        Kc[(size_t)pos * KD + i] = or_float_to_half((float)k[i]);
        Vc[(size_t)pos * KD + i] = or_float_to_half((float)v[i]);
    }
    /* attention over positions 0..pos */
    REAL* a = (REAL*)calloc((size_t)QD, sizeof(REAL));
    REAL* s = (REAL*)malloc(sizeof(REAL) * (size_t)(pos + 1));
    const REAL inv_sqrt_d = (REAL)1 / R_SQRT((REAL)d);
    for (int h = 0; h < nq; ++h) {
        const int g = h / (nq / nkv);
        REAL mx = -INFINITY;
        for (int t = 0; t <= pos; ++t) {
            REAL acc = (REAL)0;
            for (int j = 0; j < d; ++j)
                acc = acc + q[h * d + j] * (REAL)or_half_to_float(Kc[((size_t)t * nkv + g) * d + j]);
            s[t] = acc * inv_sqrt_d;
            if (s[t] > mx) mx = s[t];
        }
        if (h == 0 && scores)
            for (int t = 0; t <= pos; ++t) scores[t] = s[t];
        REAL l = (REAL)0;
        for (int t = 0; t <= pos; ++t) {
            s[t] = R_EXP(s[t] - mx);
            l = l + s[t];
        }
        for (int j = 0; j < d; ++j) {
            REAL acc = (REAL)0;
            for (int t = 0; t <= pos; ++t) acc = acc + s[t] * (REAL)or_half_to_float(Vc[((size_t)t * nkv + g) * d + j]);
            a[h * d + j] = acc / l;
        }
    }
    if (attn) memcpy(attn, a, sizeof(REAL) * (size_t)QD);
    /* output projection and residual */
    for (int i = 0; i < H; ++i) {
        REAL acc = (REAL)0;
        for (int c = 0; c < QD; ++c) acc = acc + (REAL)or_bf16_to_float(Wo[(size_t)i * QD + c]) * a[c];
        out[i] = or_float_to_bf16((float)((REAL)or_bf16_to_float(x[i]) + acc));
    }
    free(n);
    free(q);
    free(k);
    free(v);
    free(a);
    free(s);
}

int or_real_bytes(void) { return (int)sizeof(REAL); }

/* Threads the row loops may use: 1 in the plain build. */
#ifdef _OPENMP
#include <omp.h>
int or_threads(void) { return omp_get_max_threads(); }
#else
int or_threads(void) { return 1; }
#endif
