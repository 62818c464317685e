/*
 * CPU oracle of the greedy speculative-decoding verify pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark call this code.  It shares no code with the
 * CUDA path; the two meet only in the seeded inputs of the `synth` module.
 *
 * What it computes (plain definitions, fp32 arithmetic, every sum taken
 * sequentially in index order, no blocking or fusion):
 *
 *  - The pre-norm residual decoder of the LayerSkip summary ("Notation and
 *    Baseline Architecture": x_{l+1} = x_l + f_l(x_l), logits e = g(x_L),
 *    g = final norm + LM head), with the Llama-family blocks that page names
 *    (RMSNorm, rotary position embedding, grouped-query attention, SwiGLU FFN).
 *  - The verify pass of self-speculative decoding (LayerSkip summary, 4.3.2;
 *    DFlash README, "Architecture": the target runs [last token] + drafts in
 *    one pass against its KV cache and returns one logit row per position).
 *  - The mixture-of-experts FFN of the MoE speculative-decoding page: a
 *    softmax router, top-k experts per token plus shared experts.  Per-slot and
 *    deduplicated expert reads compute the same function, so there is one path.
 *  - A layer plan: the list of layer indices a pass runs (the layer-skip draft
 *    of the MLX self-speculation post, "Code -> the implementation", keeps a
 *    subset of the same layers with shared weights).
 *
 * Rounding points (bf16 round-to-nearest-even, everything else fp32): the
 * normalised GEMM inputs, q after RoPE, the cached k and v, the attention
 * output and the SwiGLU product.  Logits are fp32.
 *
 * Accumulators.  Every long sum (GEMM dot products, the RMSNorm sum of
 * squares, attention scores, softmax denominators and the weighted value sum)
 * runs in acc_t: fp32 by default, the precision the pass is specified in.
 * Built with -DORC_ACC64 the same sums run in fp64 and are rounded to fp32
 * where the default build holds its fp32 result; every rounding point above is
 * unchanged.  The two builds compute the same definition; how far they drift
 * apart measures how reproducible fp32 accumulation is at a given depth and
 * width, which is what the full-size tests bound an implementation by.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifdef ORC_ACC64
typedef double acc_t;
#else
typedef float acc_t;
#endif

typedef struct {
    int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    float rope_theta, norm_eps;
    int n_experts, top_k, expert_ffn, n_shared, first_moe_layer;
    int max_ctx;
} orc_cfg;

enum {
    T_EMBED = 0, T_LMHEAD, T_FINALNORM, T_ATTN_NORM, T_FFN_NORM, T_WQ, T_WK, T_WV, T_WO,
    T_GATE, T_UP, T_DOWN, T_ROUTER, T_EGATE, T_EUP, T_EDOWN, T_SGATE, T_SUP, T_SDOWN
};

typedef struct {
    orc_cfg c;
    const uint16_t *embed, *lm_head, *final_norm;
    const uint16_t **attn_norm, **ffn_norm, **wq, **wk, **wv, **wo, **gate, **up, **down, **router;
    const uint16_t **egate, **eup, **edown; /* [layer * n_experts + e] */
    const uint16_t **sgate, **sup, **sdown; /* [layer * n_shared + s] */
    float *rope_cos, *rope_sin;             /* [max_ctx][head_dim / 2] */
} orc_model;

typedef struct {
    int n_slots, max_ctx, width, len;
    float *k, *v; /* [slot][max_ctx][n_kv_heads * head_dim], bf16-rounded values */
} orc_cache;

/* ---------------------------------------------------------------- bf16 --- */
static inline float bf_widen(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a float to the nearest bf16 value (ties to even), returned as float. */
static inline float bf_round(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    u &= 0xFFFF0000u;
    float r;
    memcpy(&r, &u, 4);
    return r;
}

float orc_bf16_round(float f) { return bf_round(f); }

/* ---------------------------------------------------------- model setup --- */
orc_model* orc_create(const orc_cfg* cfg) {
    orc_model* m = (orc_model*)calloc(1, sizeof(orc_model));
    m->c = *cfg;
    int L = cfg->n_layers;
    const uint16_t*** per_layer[] = {&m->attn_norm, &m->ffn_norm, &m->wq, &m->wk, &m->wv, &m->wo,
                                     &m->gate, &m->up, &m->down, &m->router};
    for (unsigned i = 0; i < sizeof(per_layer) / sizeof(per_layer[0]); ++i)
        *per_layer[i] = (const uint16_t**)calloc((size_t)L, sizeof(void*));
    int E = cfg->n_experts > 0 ? cfg->n_experts : 1;
    int S = cfg->n_shared > 0 ? cfg->n_shared : 1;
    m->egate = (const uint16_t**)calloc((size_t)L * E, sizeof(void*));
    m->eup = (const uint16_t**)calloc((size_t)L * E, sizeof(void*));
    m->edown = (const uint16_t**)calloc((size_t)L * E, sizeof(void*));
    m->sgate = (const uint16_t**)calloc((size_t)L * S, sizeof(void*));
    m->sup = (const uint16_t**)calloc((size_t)L * S, sizeof(void*));
    m->sdown = (const uint16_t**)calloc((size_t)L * S, sizeof(void*));

    /* Rotary table: inv_freq_i = theta^(-2i/hd), angle = pos * inv_freq_i,
     * evaluated in double and stored as float. */
    int half = cfg->head_dim / 2;
    m->rope_cos = (float*)malloc(sizeof(float) * (size_t)cfg->max_ctx * half);
    m->rope_sin = (float*)malloc(sizeof(float) * (size_t)cfg->max_ctx * half);
    for (int p = 0; p < cfg->max_ctx; ++p)
        for (int i = 0; i < half; ++i) {
            double inv = pow((double)cfg->rope_theta, -2.0 * (double)i / (double)cfg->head_dim);
            double a = (double)p * inv;
            m->rope_cos[(size_t)p * half + i] = (float)cos(a);
            m->rope_sin[(size_t)p * half + i] = (float)sin(a);
        }
    return m;
}

void orc_destroy(orc_model* m) {
    if (!m) return;
    free(m->attn_norm); free(m->ffn_norm); free(m->wq); free(m->wk); free(m->wv); free(m->wo);
    free(m->gate); free(m->up); free(m->down); free(m->router);
    free(m->egate); free(m->eup); free(m->edown); free(m->sgate); free(m->sup); free(m->sdown);
    free(m->rope_cos); free(m->rope_sin);
    free(m);
}

/* Register one host tensor (bf16 bits, row-major [out][in]). */
int orc_set(orc_model* m, int kind, int layer, int expert, const uint16_t* p) {
    int L = m->c.n_layers;
    if (layer < -1 || layer >= L) return 1;
    int E = m->c.n_experts > 0 ? m->c.n_experts : 1;
    int S = m->c.n_shared > 0 ? m->c.n_shared : 1;
    switch (kind) {
        case T_EMBED: m->embed = p; return 0;
        case T_LMHEAD: m->lm_head = p; return 0;
        case T_FINALNORM: m->final_norm = p; return 0;
        case T_ATTN_NORM: m->attn_norm[layer] = p; return 0;
        case T_FFN_NORM: m->ffn_norm[layer] = p; return 0;
        case T_WQ: m->wq[layer] = p; return 0;
        case T_WK: m->wk[layer] = p; return 0;
        case T_WV: m->wv[layer] = p; return 0;
        case T_WO: m->wo[layer] = p; return 0;
        case T_GATE: m->gate[layer] = p; return 0;
        case T_UP: m->up[layer] = p; return 0;
        case T_DOWN: m->down[layer] = p; return 0;
        case T_ROUTER: m->router[layer] = p; return 0;
        case T_EGATE: if (expert < 0 || expert >= E) return 1; m->egate[(size_t)layer * E + expert] = p; return 0;
        case T_EUP: if (expert < 0 || expert >= E) return 1; m->eup[(size_t)layer * E + expert] = p; return 0;
        case T_EDOWN: if (expert < 0 || expert >= E) return 1; m->edown[(size_t)layer * E + expert] = p; return 0;
        case T_SGATE: if (expert < 0 || expert >= S) return 1; m->sgate[(size_t)layer * S + expert] = p; return 0;
        case T_SUP: if (expert < 0 || expert >= S) return 1; m->sup[(size_t)layer * S + expert] = p; return 0;
        case T_SDOWN: if (expert < 0 || expert >= S) return 1; m->sdown[(size_t)layer * S + expert] = p; return 0;
        default: return 1;
    }
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* --------------------------------------------------------------- caches --- */
orc_cache* orc_cache_create(const orc_model* m, int n_slots) {
    orc_cache* c = (orc_cache*)calloc(1, sizeof(orc_cache));
    c->n_slots = n_slots;
    c->max_ctx = m->c.max_ctx;
    c->width = m->c.n_kv_heads * m->c.head_dim;
    size_t sz = (size_t)n_slots * c->max_ctx * c->width;
    c->k = (float*)calloc(sz, sizeof(float));
    c->v = (float*)calloc(sz, sizeof(float));
    c->len = 0;
    return c;
}

void orc_cache_destroy(orc_cache* c) {
    if (!c) return;
    free(c->k); free(c->v); free(c);
}

int orc_cache_len(const orc_cache* c) { return c->len; }

/* Rollback: keep positions [0, new_len).  Growing is not allowed. */
int orc_cache_truncate(orc_cache* c, int new_len) {
    if (new_len < 0 || new_len > c->len) return 1;
    c->len = new_len;
    return 0;
}

/* Write given K/V rows (bf16 bits, [ctx][n_kv_heads*head_dim]) into one slot
 * at positions [0, ctx): synthetic-context support. */
int orc_cache_load(orc_cache* c, int slot, int ctx, const uint16_t* k, const uint16_t* v) {
    if (slot < 0 || slot >= c->n_slots || ctx < 0 || ctx > c->max_ctx) return 1;
    size_t base = (size_t)slot * c->max_ctx * c->width;
    for (size_t i = 0; i < (size_t)ctx * c->width; ++i) {
        c->k[base + i] = bf_widen(k[i]);
        c->v[base + i] = bf_widen(v[i]);
    }
    return 0;
}

int orc_cache_set_len(orc_cache* c, int len) {
    if (len < 0 || len > c->max_ctx) return 1;
    c->len = len;
    return 0;
}

/* Read back one slot's K or V rows [0, ctx) as float. */
int orc_cache_read(const orc_cache* c, int slot, int which, int ctx, float* out) {
    if (slot < 0 || slot >= c->n_slots || ctx < 0 || ctx > c->max_ctx) return 1;
    const float* src = (which ? c->v : c->k) + (size_t)slot * c->max_ctx * c->width;
    memcpy(out, src, sizeof(float) * (size_t)ctx * c->width);
    return 0;
}

/* ----------------------------------------------------------- primitives --- */
/* Y[i][r] = sum_k W[r][k] * X[i][k] for i < n, r < N; sums in k order. */
static void gemm_rows(const uint16_t* W, int N, int K, const float* X, int n, float* Y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < N; ++r) {
        const uint16_t* w = W + (size_t)r * K;
        for (int i = 0; i < n; ++i) {
            const float* x = X + (size_t)i * K;
            acc_t acc = 0;
            for (int k = 0; k < K; ++k) acc += (acc_t)bf_widen(w[k]) * x[k];
            Y[(size_t)i * N + r] = (float)acc;
        }
    }
}

/* h = bf16(x * rsqrt(mean(x^2) + eps) * g) */
static void rmsnorm_bf16(const float* x, const uint16_t* g, int d, float eps, float* h) {
    acc_t ss = 0;
    for (int k = 0; k < d; ++k) ss += (acc_t)x[k] * x[k];
    float rstd = 1.0f / sqrtf((float)(ss / (acc_t)d) + eps);
    for (int k = 0; k < d; ++k) h[k] = bf_round(x[k] * rstd * bf_widen(g[k]));
}

/* Rotate-half RoPE of one head vector at position pos. */
static void rope_apply(const orc_model* m, float* v, int pos) {
    int half = m->c.head_dim / 2;
    const float* cs = m->rope_cos + (size_t)pos * half;
    const float* sn = m->rope_sin + (size_t)pos * half;
    for (int i = 0; i < half; ++i) {
        float a = v[i], b = v[i + half];
        v[i] = a * cs[i] - b * sn[i];
        v[i + half] = b * cs[i] + a * sn[i];
    }
}

static inline float silu(float g) { return g / (1.0f + expf(-g)); }

/* Softmax attention of one query over nk keys (rows of K and V start at k0 /
 * v0 and are `stride` floats apart): out = bf16(sum_t p_t v_t / sum_t p_t),
 * p_t = exp(s_t - max s), s_t = (q . k_t) / sqrt(hd). */
static void attend_one(const float* qv, const float* k0, const float* v0, int stride, int nk, int hd, float* out) {
    const float scale = 1.0f / sqrtf((float)hd);
    float* sc = (float*)malloc(sizeof(float) * (size_t)(nk > 0 ? nk : 1));
    float mx = -INFINITY;
    for (int t = 0; t < nk; ++t) {
        const float* kv = k0 + (size_t)t * stride;
        acc_t dot = 0;
        for (int e = 0; e < hd; ++e) dot += (acc_t)qv[e] * kv[e];
        sc[t] = (float)dot * scale;
        if (sc[t] > mx) mx = sc[t];
    }
    acc_t den = 0;
    for (int t = 0; t < nk; ++t) {
        sc[t] = expf(sc[t] - mx);
        den += sc[t];
    }
    for (int e = 0; e < hd; ++e) {
        acc_t acc = 0;
        for (int t = 0; t < nk; ++t) acc += (acc_t)sc[t] * v0[(size_t)t * stride + e];
        out[e] = bf_round((float)(acc / den));
    }
    free(sc);
}

/* Router of one token: pr = softmax(logits) over E experts (in place), then
 * K ids by repeated largest-probability pick, the lowest id winning ties
 * (forced ids, when given, replace the pick).  gate = pr[id], not
 * renormalised. */
static void route_one(float* pr, int E, int K, const int* forced, int* ids, float* gates) {
    float mx = -INFINITY;
    acc_t den = 0;
    for (int e = 0; e < E; ++e) if (pr[e] > mx) mx = pr[e];
    for (int e = 0; e < E; ++e) { pr[e] = expf(pr[e] - mx); den += pr[e]; }
    for (int e = 0; e < E; ++e) pr[e] = (float)(pr[e] / den);
    char taken[1024];
    memset(taken, 0, sizeof(taken));
    for (int r = 0; r < K; ++r) {
        int best = -1;
        if (forced) {
            best = forced[r];
        } else {
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || pr[e] > pr[best])) best = e;
        }
        taken[best] = 1;
        ids[r] = best;
        gates[r] = pr[best];
    }
}

/* SwiGLU FFN of n rows: out = bf16(silu(h Wg^T) * (h Wu^T)) Wd^T. */
static void ffn_swiglu(const uint16_t* wg, const uint16_t* wu, const uint16_t* wd, int d, int f,
                       const float* h, int n, float* out) {
    float* g = (float*)malloc(sizeof(float) * (size_t)n * f);
    float* u = (float*)malloc(sizeof(float) * (size_t)n * f);
    gemm_rows(wg, f, d, h, n, g);
    gemm_rows(wu, f, d, h, n, u);
    for (size_t i = 0; i < (size_t)n * f; ++i) g[i] = bf_round(silu(g[i]) * u[i]);
    gemm_rows(wd, d, f, g, n, out);
    free(g);
    free(u);
}

/* ---------------------------------------------------------------- forward --- */
/*
 * Run tokens[0..n) at positions pos0..pos0+n-1 through the layers listed in
 * plan[0..plan_len) (cache slot s holds plan[s]'s keys and values), append
 * their k and v, and write fp32 logits of rows i >= logits_from to
 * logits[(i - logits_from) * vocab ...] when logits is not NULL.
 *
 * MoE layers write the chosen expert ids and gates to ids_out / gates_out
 * ([plan_len][n][top_k], may be NULL).  When forced_ids ([plan_len][n][top_k])
 * is given, those ids replace the top-k choice and their gates are the router
 * probabilities at those ids.  probs_out ([plan_len][n][n_experts], may be
 * NULL) receives every router probability of every MoE layer, so that a
 * caller can check a forced choice against the top-k it replaced.
 *
 * hidden_out ([plan_len][n][d_model], may be NULL) receives the residual
 * stream after each executed layer: the target hidden states from which the
 * mlx-dflash README ("Architecture") takes the draft's context features.
 *
 * Returns 0, or 1 on a bad argument (pos0 beyond the cache length, overflow).
 */
int orc_forward(const orc_model* m, orc_cache* cache, const int* plan, int plan_len, const int* tokens,
                int n, int pos0, float* logits, int logits_from, int* ids_out, float* gates_out,
                const int* forced_ids, float* probs_out, float* hidden_out) {
    const orc_cfg* c = &m->c;
    const int d = c->d_model, hd = c->head_dim, Hq = c->n_heads, Hkv = c->n_kv_heads;
    const int qw = Hq * hd, kw = Hkv * hd, group = Hq / Hkv;
    if (n <= 0 || pos0 < 0 || pos0 > cache->len || pos0 + n > cache->max_ctx) return 1;
    if (plan_len > cache->n_slots) return 1;
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= c->vocab) return 1;

    float* x = (float*)malloc(sizeof(float) * (size_t)n * d);
    float* h = (float*)malloc(sizeof(float) * (size_t)n * d);
    float* q = (float*)malloc(sizeof(float) * (size_t)n * qw);
    float* kk = (float*)malloc(sizeof(float) * (size_t)n * kw);
    float* vv = (float*)malloc(sizeof(float) * (size_t)n * kw);
    float* att = (float*)malloc(sizeof(float) * (size_t)n * qw);
    float* y = (float*)malloc(sizeof(float) * (size_t)n * d);

    for (int i = 0; i < n; ++i)
        for (int k = 0; k < d; ++k) x[(size_t)i * d + k] = bf_widen(m->embed[(size_t)tokens[i] * d + k]);

    for (int s = 0; s < plan_len; ++s) {
        const int l = plan[s];
        /* --- attention block --- */
        for (int i = 0; i < n; ++i) rmsnorm_bf16(x + (size_t)i * d, m->attn_norm[l], d, c->norm_eps, h + (size_t)i * d);
        gemm_rows(m->wq[l], qw, d, h, n, q);
        gemm_rows(m->wk[l], kw, d, h, n, kk);
        gemm_rows(m->wv[l], kw, d, h, n, vv);
        float* ck = cache->k + (size_t)s * cache->max_ctx * kw;
        float* cv = cache->v + (size_t)s * cache->max_ctx * kw;
        for (int i = 0; i < n; ++i) {
            const int pos = pos0 + i;
            for (int hh = 0; hh < Hq; ++hh) rope_apply(m, q + (size_t)i * qw + hh * hd, pos);
            for (int hh = 0; hh < Hkv; ++hh) rope_apply(m, kk + (size_t)i * kw + hh * hd, pos);
            for (int e = 0; e < qw; ++e) q[(size_t)i * qw + e] = bf_round(q[(size_t)i * qw + e]);
            for (int e = 0; e < kw; ++e) {
                ck[(size_t)pos * kw + e] = bf_round(kk[(size_t)i * kw + e]);
                cv[(size_t)pos * kw + e] = bf_round(vv[(size_t)i * kw + e]);
            }
        }
        /* token i attends to keys 0..pos0+i (causal inside the block) */
#pragma omp parallel for collapse(2) schedule(static)
        for (int i = 0; i < n; ++i)
            for (int hh = 0; hh < Hq; ++hh)
                attend_one(q + (size_t)i * qw + hh * hd, ck + (hh / group) * hd, cv + (hh / group) * hd, kw,
                           pos0 + i + 1, hd, att + (size_t)i * qw + hh * hd);
        gemm_rows(m->wo[l], d, qw, att, n, y);
        for (size_t e = 0; e < (size_t)n * d; ++e) x[e] += y[e];

        /* --- FFN block --- */
        for (int i = 0; i < n; ++i) rmsnorm_bf16(x + (size_t)i * d, m->ffn_norm[l], d, c->norm_eps, h + (size_t)i * d);
        if (c->n_experts > 0 && l >= c->first_moe_layer) {
            const int E = c->n_experts, K = c->top_k, fe = c->expert_ffn, S = c->n_shared;
            float* rl = (float*)malloc(sizeof(float) * (size_t)n * E);
            gemm_rows(m->router[l], E, d, h, n, rl);
            float* eo = (float*)malloc(sizeof(float) * (size_t)d);
            for (int i = 0; i < n; ++i) {
                float* pr = rl + (size_t)i * E;
                int chosen[64];
                float gsel[64];
                route_one(pr, E, K, forced_ids ? forced_ids + ((size_t)s * n + i) * K : NULL, chosen, gsel);
                if (probs_out) memcpy(probs_out + ((size_t)s * n + i) * E, pr, sizeof(float) * (size_t)E);
                for (int r = 0; r < K; ++r) {
                    if (ids_out) ids_out[((size_t)s * n + i) * K + r] = chosen[r];
                    if (gates_out) gates_out[((size_t)s * n + i) * K + r] = gsel[r];
                }
                float* yi = y + (size_t)i * d;
                for (int k = 0; k < d; ++k) yi[k] = 0.0f;
                const float* hi = h + (size_t)i * d;
                for (int r = 0; r < K; ++r) {
                    const int e = chosen[r];
                    const size_t ix = (size_t)l * E + e;
                    ffn_swiglu(m->egate[ix], m->eup[ix], m->edown[ix], d, fe, hi, 1, eo);
                    for (int k = 0; k < d; ++k) yi[k] += gsel[r] * eo[k];
                }
                for (int sh = 0; sh < S; ++sh) {
                    const size_t ix = (size_t)l * S + sh;
                    ffn_swiglu(m->sgate[ix], m->sup[ix], m->sdown[ix], d, fe, hi, 1, eo);
                    for (int k = 0; k < d; ++k) yi[k] += eo[k];
                }
            }
            free(eo);
            free(rl);
        } else {
            ffn_swiglu(m->gate[l], m->up[l], m->down[l], d, c->ffn_dim, h, n, y);
        }
        for (size_t e = 0; e < (size_t)n * d; ++e) x[e] += y[e];
        if (hidden_out) memcpy(hidden_out + (size_t)s * n * d, x, sizeof(float) * (size_t)n * d);
    }
    cache->len = pos0 + n;

    if (logits) {
        const uint16_t* wl = m->lm_head ? m->lm_head : m->embed;
        const int rows = n - logits_from;
        if (rows > 0) {
            for (int i = logits_from; i < n; ++i)
                rmsnorm_bf16(x + (size_t)i * d, m->final_norm, d, c->norm_eps, h + (size_t)(i - logits_from) * d);
            gemm_rows(wl, c->vocab, d, h, rows, logits);
        }
    }
    free(x); free(h); free(q); free(kk); free(vv); free(att); free(y);
    return 0;
}

/* ------------------------------------------------ DFlash context append --- */
/*
 * The conditioning path of the block draft in the mlx-dflash README
 * ("Architecture"): the target hidden states tapped at n_in layers are
 * projected by fc into one context feature per position, and the draft
 * attends over those context positions.  Reading: each layer of this model
 * computes the keys and values of a context position from its feature the
 * way it computes them from a token's residual stream (that layer's input
 * norm, its k and v projections, RoPE on k at the position), and appends them
 * to its cache; nothing else of the layer runs.
 *
 * taps: fp32 [n_in][16][d_model], rows r < m used (the tap buffer layout).
 * fc:   bf16 [d_model][n_in * d_model], input index t * d_model + i.
 * The concatenated taps are rounded to bf16 (a GEMM operand); the feature is
 * the fp32 product.  Positions len .. len + m - 1 of every slot (slot s =
 * layer s; the cache must cover every layer) are written, then len += m.
 * feat_out (may be NULL) receives the features, fp32 [m][d_model].
 * Returns 0, or 1 on a bad argument.
 */
int orc_context_append(const orc_model* m, orc_cache* cache, const uint16_t* fc, int n_in, const float* taps,
                       int rows, float* feat_out) {
    const orc_cfg* c = &m->c;
    const int d = c->d_model, hd = c->head_dim, Hkv = c->n_kv_heads, kw = Hkv * hd;
    if (n_in < 1 || rows < 1 || rows > 16 || cache->n_slots != c->n_layers) return 1;
    if (cache->len + rows > cache->max_ctx) return 1;
    const int K = n_in * d;
    float* xin = (float*)malloc(sizeof(float) * (size_t)rows * K);
    float* feat = (float*)malloc(sizeof(float) * (size_t)rows * d);
    float* h = (float*)malloc(sizeof(float) * (size_t)rows * d);
    float* kk = (float*)malloc(sizeof(float) * (size_t)rows * kw);
    float* vv = (float*)malloc(sizeof(float) * (size_t)rows * kw);
    for (int r = 0; r < rows; ++r)
        for (int t = 0; t < n_in; ++t)
            for (int i = 0; i < d; ++i)
                xin[(size_t)r * K + (size_t)t * d + i] = bf_round(taps[((size_t)t * 16 + r) * d + i]);
    gemm_rows(fc, d, K, xin, rows, feat);
    if (feat_out) memcpy(feat_out, feat, sizeof(float) * (size_t)rows * d);
    for (int l = 0; l < c->n_layers; ++l) {
        for (int r = 0; r < rows; ++r) rmsnorm_bf16(feat + (size_t)r * d, m->attn_norm[l], d, c->norm_eps, h + (size_t)r * d);
        gemm_rows(m->wk[l], kw, d, h, rows, kk);
        gemm_rows(m->wv[l], kw, d, h, rows, vv);
        float* ck = cache->k + (size_t)l * cache->max_ctx * kw;
        float* cv = cache->v + (size_t)l * cache->max_ctx * kw;
        for (int r = 0; r < rows; ++r) {
            const int pos = cache->len + r;
            for (int hh = 0; hh < Hkv; ++hh) rope_apply(m, kk + (size_t)r * kw + hh * hd, pos);
            for (int e = 0; e < kw; ++e) {
                ck[(size_t)pos * kw + e] = bf_round(kk[(size_t)r * kw + e]);
                cv[(size_t)pos * kw + e] = bf_round(vv[(size_t)r * kw + e]);
            }
        }
    }
    cache->len += rows;
    free(xin); free(feat); free(h); free(kk); free(vv);
    return 0;
}

/* Index of the largest value; the lowest index wins ties. */
int orc_argmax(const float* v, int count) {
    int best = 0;
    for (int i = 1; i < count; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

/* ------------------------------------------------ primitives for the pins --- */
void orc_gemm(const uint16_t* W, int N, int K, const float* X, int n, float* Y) { gemm_rows(W, N, K, X, n, Y); }

void orc_rmsnorm(const float* x, const uint16_t* g, int d, float eps, float* h) { rmsnorm_bf16(x, g, d, eps, h); }

void orc_rope(const orc_model* m, float* v, int pos) { rope_apply(m, v, pos); }

/* Grouped-query attention of one token: q [Hq][hd], K/V rows [nk][Hkv*hd];
 * query head h reads kv head h / (Hq / Hkv). */
void orc_attend(const float* q, const float* K, const float* V, int nk, int Hq, int Hkv, int hd, float* out) {
    int group = Hq / Hkv;
    for (int h = 0; h < Hq; ++h)
        attend_one(q + (size_t)h * hd, K + (h / group) * hd, V + (h / group) * hd, Hkv * hd, nk, hd, out + (size_t)h * hd);
}

void orc_route(float* logits, int E, int K, const int* forced, int* ids, float* gates) {
    route_one(logits, E, K, forced, ids, gates);
}
