/*
 * CPU oracle of one batch-1 Llama decode step: TEST INFRASTRUCTURE ONLY.
 * See oracle.h for what it computes, the layouts and who may use it.
 *
 * Each function follows the definition of its step, written out plainly:
 * no blocking, fusion or reordering beyond the definition.  The only
 * parallelism is over independent output rows (linear maps) and independent
 * heads (attention); every output is computed by one thread in a fixed
 * order, so results do not depend on the thread count.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

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

/* ---------------------------------------------------------------- numbers */

/* bf16 is the upper half of an IEEE binary32 */
double orc_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, binary32 exponent
 * range), ties to even, directly from the double (no intermediate float). */
uint16_t orc_bf16_from_double(double v) {
    if (isnan(v)) return 0x7FC0;
    double r;
    double a = fabs(v);
    if (a == 0.0 || isinf(v)) {
        r = v;
    } else if (a < ldexp(1.0, -126)) {
        /* subnormal range: fixed quantum 2^-133 */
        r = nearbyint(ldexp(v, 133));
        r = ldexp(r, -133);
    } else {
        int e;
        double m = frexp(v, &e);          /* v = m * 2^e, 0.5 <= |m| < 1 */
        r = nearbyint(ldexp(m, 8));       /* 8 significant bits, ties to even */
        r = ldexp(r, e - 8);
    }
    /* r is exactly representable in binary32 (or overflows to inf there) */
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits */
double orc_fp16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25);
    }
    return sign ? -v : v;
}

/* ---------------------------------------------------------------- weights */

void orc_dequant_row(const orc_linear* lin, int64_t out_features, int64_t in_features,
                     int64_t row, double* out) {
    (void)out_features;
    const int64_t k_in = in_features;
    if (lin->format == ORC_BF16) {
        const uint16_t* w = (const uint16_t*)lin->w + row * k_in;
        for (int64_t k = 0; k < k_in; ++k) out[k] = orc_bf16_to_double(w[k]);
    } else if (lin->format == ORC_INT8) {
        /* symmetric per-row: w = q * s_row */
        const int8_t* w = (const int8_t*)lin->w + row * k_in;
        double s = orc_fp16_to_double(lin->scales[row]);
        for (int64_t k = 0; k < k_in; ++k) out[k] = (double)w[k] * s;
    } else {
        /* asymmetric group-128: w = (q - z_g) * s_g */
        const int64_t ng = k_in / 128;
        const int64_t zb = (ng + 1) / 2;
        const uint8_t* w = (const uint8_t*)lin->w + row * (k_in / 2);
        const uint16_t* sc = lin->scales + row * ng;
        const uint8_t* zr = lin->zeros + row * zb;
        for (int64_t k = 0; k < k_in; ++k) {
            uint8_t byte = w[k / 2];
            int q = (k & 1) ? (byte >> 4) : (byte & 15);
            int64_t g = k / 128;
            uint8_t zbyte = zr[g / 2];
            int z = (g & 1) ? (zbyte >> 4) : (zbyte & 15);
            out[k] = (double)(q - z) * orc_fp16_to_double(sc[g]);
        }
    }
}

void orc_linear_apply(const orc_linear* lin, int64_t out_features, int64_t in_features,
                      const double* x, double* y) {
#pragma omp parallel
    {
        double* row = (double*)malloc(sizeof(double) * (size_t)in_features);
#pragma omp for schedule(static)
        for (int64_t o = 0; o < out_features; ++o) {
            orc_dequant_row(lin, out_features, in_features, o, row);
            double acc = 0.0;
            for (int64_t k = 0; k < in_features; ++k) acc += row[k] * x[k];
            y[o] = acc;
        }
        free(row);
    }
}

/* ------------------------------------------------------------ elementwise */

void orc_rmsnorm(const double* x, const uint16_t* w, int64_t n, double eps, double* out) {
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; ++i) {
        double wi = w ? orc_bf16_to_double(w[i]) : 1.0;
        out[i] = x[i] * r * wi;
    }
}

/* HF rotate-half: dims i and i + head_dim/2 form one rotation pair, turned
 * by angle pos * theta^(-2i/head_dim). */
void orc_rope(double* v, int32_t n_heads, int32_t head_dim, int64_t pos, double theta) {
    const int32_t half = head_dim / 2;
    for (int32_t hh = 0; hh < n_heads; ++hh) {
        double* x = v + (int64_t)hh * head_dim;
        for (int32_t i = 0; i < half; ++i) {
            double inv_freq = pow(theta, -2.0 * (double)i / (double)head_dim);
            double ang = (double)pos * inv_freq;
            double c = cos(ang), s = sin(ang);
            double a = x[i], b = x[i + half];
            x[i] = a * c - b * s;
            x[i + half] = b * c + a * s;
        }
    }
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

void orc_attention(const double* q, const uint16_t* k, const uint16_t* v,
                   int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                   int64_t max_seq, int64_t ctx, double* out) {
    const int32_t group = n_heads / n_kv_heads;
    const double scale = 1.0 / sqrt((double)head_dim);
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
#pragma omp for schedule(static)
        for (int32_t i = 0; i < n_heads; ++i) {
            const int32_t g = i / group;
            const double* qi = q + (int64_t)i * head_dim;
            const uint16_t* kg = k + (int64_t)g * max_seq * head_dim;
            const uint16_t* vg = v + (int64_t)g * max_seq * head_dim;
            double m = -INFINITY;
            for (int64_t t = 0; t < ctx; ++t) {
                double dot = 0.0;
                for (int32_t d = 0; d < head_dim; ++d)
                    dot += qi[d] * orc_bf16_to_double(kg[t * head_dim + d]);
                s[t] = dot * scale;
                if (s[t] > m) m = s[t];
            }
            double denom = 0.0;
            for (int64_t t = 0; t < ctx; ++t) {
                s[t] = exp(s[t] - m);
                denom += s[t];
            }
            double* oi = out + (int64_t)i * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) oi[d] = 0.0;
            for (int64_t t = 0; t < ctx; ++t) {
                double p = s[t] / denom;
                for (int32_t d = 0; d < head_dim; ++d)
                    oi[d] += p * orc_bf16_to_double(vg[t * head_dim + d]);
            }
        }
        free(s);
    }
}

/* --------------------------------------------------------------- decoder */

static int check_config(const orc_config* c) {
    if (!c || c->n_layers <= 0 || c->hidden <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 ||
        c->head_dim <= 0 || c->ffn <= 0 || c->vocab <= 0 || c->max_seq <= 0)
        return -1;
    if (c->n_heads % c->n_kv_heads) return -1;
    if (c->head_dim % 2) return -1;
    return 0;
}

int orc_decode_layers(const orc_config* c, const orc_weights* w, uint16_t* kv, double* x,
                      int64_t pos, int32_t l0, int32_t l1) {
    if (check_config(c) || !w || !kv || !x) return -1;
    if (pos < 0 || pos >= c->max_seq || l0 < 0 || l1 > c->n_layers || l0 > l1) return -1;

    const int64_t H = c->hidden, F = c->ffn, hd = c->head_dim;
    const int64_t qd = (int64_t)c->n_heads * hd, kvd = (int64_t)c->n_kv_heads * hd;
    const int64_t layer_stride = 2 * kvd * c->max_seq;     /* bf16 elements per layer */
    const int64_t kv_half = kvd * c->max_seq;              /* K block, then V block */

    double* hn = (double*)malloc(sizeof(double) * H);
    double* q = (double*)malloc(sizeof(double) * qd);
    double* kk = (double*)malloc(sizeof(double) * kvd);
    double* vv = (double*)malloc(sizeof(double) * kvd);
    double* o = (double*)malloc(sizeof(double) * qd);
    double* y = (double*)malloc(sizeof(double) * H);
    double* g = (double*)malloc(sizeof(double) * F);
    double* u = (double*)malloc(sizeof(double) * F);

    for (int32_t l = l0; l < l1; ++l) {
        const orc_layer* L = &w->layers[l];
        uint16_t* kc = kv + l * layer_stride;
        uint16_t* vc = kc + kv_half;

        /* attention block */
        orc_rmsnorm(x, L->attn_norm, H, c->rms_eps, hn);
        orc_linear_apply(&L->wq, qd, H, hn, q);
        orc_linear_apply(&L->wk, kvd, H, hn, kk);
        orc_linear_apply(&L->wv, kvd, H, hn, vv);
        orc_rope(q, c->n_heads, (int32_t)hd, pos, c->rope_theta);
        orc_rope(kk, c->n_kv_heads, (int32_t)hd, pos, c->rope_theta);
        for (int32_t gh = 0; gh < c->n_kv_heads; ++gh)
            for (int64_t d = 0; d < hd; ++d) {
                kc[((int64_t)gh * c->max_seq + pos) * hd + d] = orc_bf16_from_double(kk[gh * hd + d]);
                vc[((int64_t)gh * c->max_seq + pos) * hd + d] = orc_bf16_from_double(vv[gh * hd + d]);
            }
        orc_attention(q, kc, vc, c->n_heads, c->n_kv_heads, (int32_t)hd, c->max_seq, pos + 1, o);
        orc_linear_apply(&L->wo, H, qd, o, y);
        for (int64_t i = 0; i < H; ++i) x[i] += y[i];

        /* SwiGLU feed-forward block */
        orc_rmsnorm(x, L->ffn_norm, H, c->rms_eps, hn);
        orc_linear_apply(&L->wg, F, H, hn, g);
        orc_linear_apply(&L->wu, F, H, hn, u);
        for (int64_t j = 0; j < F; ++j) g[j] = orc_silu(g[j]) * u[j];
        orc_linear_apply(&L->wd, H, F, g, y);
        for (int64_t i = 0; i < H; ++i) x[i] += y[i];
    }
    free(hn); free(q); free(kk); free(vv); free(o); free(y); free(g); free(u);
    return 0;
}

int orc_logits_rows(const orc_config* c, const orc_weights* w, const double* x, double* logits,
                    int64_t r0, int64_t r1) {
    if (check_config(c) || !w || !x || !logits || r0 < 0 || r1 > c->vocab || r0 > r1) return -1;
    const int64_t H = c->hidden;
    double* hn = (double*)malloc(sizeof(double) * H);
    orc_rmsnorm(x, w->final_norm, H, c->rms_eps, hn);
    /* rows r0.. of the LM head are the linear map whose row 0 is row r0 */
    orc_linear lm = w->lm_head;
    if (lm.format == ORC_BF16) {
        lm.w = (const uint16_t*)lm.w + r0 * H;
    } else if (lm.format == ORC_INT8) {
        lm.w = (const int8_t*)lm.w + r0 * H;
        lm.scales += r0;
    } else {
        lm.w = (const uint8_t*)lm.w + r0 * (H / 2);
        lm.scales += r0 * (H / 128);
        lm.zeros += r0 * ((H / 128 + 1) / 2);
    }
    orc_linear_apply(&lm, r1 - r0, H, hn, logits + r0);
    free(hn);
    return 0;
}

int orc_decode_step(const orc_config* c, const orc_weights* w, uint16_t* kv,
                    int32_t token, int64_t pos, double* logits) {
    if (check_config(c) || !w || !kv) return -1;
    if (token < 0 || token >= c->vocab || pos < 0 || pos >= c->max_seq) return -1;
    const int64_t H = c->hidden;
    double* x = (double*)malloc(sizeof(double) * H);
    /* x = embedding row of the token */
    for (int64_t i = 0; i < H; ++i) x[i] = orc_bf16_to_double(w->embed[(int64_t)token * H + i]);
    int rc = orc_decode_layers(c, w, kv, x, pos, 0, c->n_layers);
    if (rc == 0 && logits) rc = orc_logits_rows(c, w, x, logits, 0, c->vocab);
    free(x);
    return rc;
}

int orc_prefill(const orc_config* c, const orc_weights* w, uint16_t* kv,
                const int32_t* tokens, int64_t n, int64_t start_pos) {
    for (int64_t i = 0; i < n; ++i) {
        int rc = orc_decode_step(c, w, kv, tokens[i], start_pos + i, NULL);
        if (rc) return rc;
    }
    return 0;
}

/* The prefill as the pages' batched form of the same decoder: every layer
 * processes all n prompt tokens before the next layer starts (a separate
 * loop nest from orc_prefill's token-by-token steps).  Per layer: RMSNorm
 * and the Q, K, V maps of every token; RoPE of each token at its position;
 * the K, V rows of all n positions written to the cache; causal attention
 * of token t over positions [0, start_pos + t]; the O map and residual; the
 * SwiGLU block and residual.  Each element is computed by the same
 * operations in the same order as in a decode step, so the cache it leaves
 * equals orc_prefill's bit for bit. */
int orc_prefill_batched(const orc_config* c, const orc_weights* w, uint16_t* kv,
                        const int32_t* tokens, int64_t n, int64_t start_pos) {
    if (check_config(c) || !w || !kv || (n > 0 && !tokens) || n < 0) return -1;
    if (start_pos < 0 || start_pos + n > c->max_seq) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (tokens[t] < 0 || tokens[t] >= c->vocab) return -1;
    if (n == 0) return 0;
    const int64_t H = c->hidden, F = c->ffn, hd = c->head_dim;
    const int64_t qd = (int64_t)c->n_heads * hd, kvd = (int64_t)c->n_kv_heads * hd;
    const int64_t layer_stride = 2 * kvd * c->max_seq;
    const int64_t kv_half = kvd * c->max_seq;

    double* X = (double*)malloc(sizeof(double) * (size_t)(n * H));    /* residual rows */
    double* Hn = (double*)malloc(sizeof(double) * (size_t)(n * H));   /* normed rows */
    double* Q = (double*)malloc(sizeof(double) * (size_t)(n * qd));
    double* K = (double*)malloc(sizeof(double) * (size_t)(n * kvd));
    double* V = (double*)malloc(sizeof(double) * (size_t)(n * kvd));
    double* O = (double*)malloc(sizeof(double) * (size_t)(n * qd));
    double* Y = (double*)malloc(sizeof(double) * (size_t)H);
    double* G = (double*)malloc(sizeof(double) * (size_t)F);
    double* U = (double*)malloc(sizeof(double) * (size_t)F);

    for (int64_t t = 0; t < n; ++t)
        for (int64_t i = 0; i < H; ++i)
            X[t * H + i] = orc_bf16_to_double(w->embed[(int64_t)tokens[t] * H + i]);

    for (int32_t l = 0; l < c->n_layers; ++l) {
        const orc_layer* L = &w->layers[l];
        uint16_t* kc = kv + l * layer_stride;
        uint16_t* vc = kc + kv_half;
        /* projections of every token, then RoPE at each token's position */
        for (int64_t t = 0; t < n; ++t) {
            orc_rmsnorm(X + t * H, L->attn_norm, H, c->rms_eps, Hn + t * H);
            orc_linear_apply(&L->wq, qd, H, Hn + t * H, Q + t * qd);
            orc_linear_apply(&L->wk, kvd, H, Hn + t * H, K + t * kvd);
            orc_linear_apply(&L->wv, kvd, H, Hn + t * H, V + t * kvd);
            orc_rope(Q + t * qd, c->n_heads, (int32_t)hd, start_pos + t, c->rope_theta);
            orc_rope(K + t * kvd, c->n_kv_heads, (int32_t)hd, start_pos + t, c->rope_theta);
        }
        /* the K, V rows of all prompt positions */
        for (int64_t t = 0; t < n; ++t)
            for (int32_t gh = 0; gh < c->n_kv_heads; ++gh)
                for (int64_t d = 0; d < hd; ++d) {
                    const int64_t at = ((int64_t)gh * c->max_seq + start_pos + t) * hd + d;
                    kc[at] = orc_bf16_from_double(K[t * kvd + gh * hd + d]);
                    vc[at] = orc_bf16_from_double(V[t * kvd + gh * hd + d]);
                }
        /* causal attention: token t sees positions 0 .. start_pos + t */
        for (int64_t t = 0; t < n; ++t)
            orc_attention(Q + t * qd, kc, vc, c->n_heads, c->n_kv_heads, (int32_t)hd, c->max_seq,
                          start_pos + t + 1, O + t * qd);
        /* O map + residual, then the SwiGLU block + residual, per token */
        for (int64_t t = 0; t < n; ++t) {
            double* x = X + t * H;
            orc_linear_apply(&L->wo, H, qd, O + t * qd, Y);
            for (int64_t i = 0; i < H; ++i) x[i] += Y[i];
            orc_rmsnorm(x, L->ffn_norm, H, c->rms_eps, Hn + t * H);
            orc_linear_apply(&L->wg, F, H, Hn + t * H, G);
            orc_linear_apply(&L->wu, F, H, Hn + t * H, U);
            for (int64_t j = 0; j < F; ++j) G[j] = orc_silu(G[j]) * U[j];
            orc_linear_apply(&L->wd, H, F, G, Y);
            for (int64_t i = 0; i < H; ++i) x[i] += Y[i];
        }
    }
    free(X); free(Hn); free(Q); free(K); free(V); free(O); free(Y); free(G); free(U);
    return 0;
}
