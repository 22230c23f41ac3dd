/*
 * CPU oracle of one batch-1 decode step of a Llama-family decoder.
 *
 * TEST INFRASTRUCTURE ONLY.  This library exists to check the CUDA decode
 * path: only the tests, the smoke check and the benchmark's CPU-baseline /
 * reference legs may load it.  It shares no code, header, table or helper
 * with the CUDA path (decode_megakernel_gb300/csrc); the two meet only in
 * the seeded inputs they are both given.
 *
 * What it computes is the plain definition of the decode step the
 * AutoMegaKernel pages target: a HuggingFace Llama-family decoder (AMK
 * summaries, "Methodology": "compiles HuggingFace Llama-family models"),
 * with RMSNorm, the QKV / O / gate-up / down / LM-head linear maps, RoPE,
 * GQA attention over a KV cache and SwiGLU (AMK "Layer 1: instructions":
 * GEMV, attention, RMSNorm; Argus "Workload and baselines": the megakernel
 * also holds KV-cache updates and the logits).  Arithmetic is IEEE double;
 * weights are the given bf16 values, or the given int8 / int4 codes
 * dequantised exactly; the KV cache is stored in bf16 (round to nearest
 * even), everything else stays in double.
 *
 * Parity pins (tests/test_oracle_pins.py): every function below is checked
 * against closed forms, invariants, library routines or brute force.
 *
 * Layouts (all row-major, host memory):
 *   bf16 linear   w  uint16 [out][in]
 *   int8 linear   w  int8   [out][in],  scales fp16 [out]
 *   int4 linear   w  uint8  [out][in/2] (low nibble = even k),
 *                 scales fp16 [out][in/128], zeros uint8 [out][ceil(in/256)]
 *                 (low nibble = even group); w = (q - z) * s
 *   KV cache      bf16 [n_layers][2 (K,V)][n_kv_heads][max_seq][head_dim]
 */
#ifndef AMK_ORACLE_H
#define AMK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BF16 = 0, ORC_INT8 = 1, ORC_INT4 = 2 };

typedef struct {
    int32_t format;          /* ORC_BF16 / ORC_INT8 / ORC_INT4 */
    const void* w;           /* codes, see layouts above */
    const uint16_t* scales;  /* fp16 bits; NULL for bf16 */
    const uint8_t* zeros;    /* int4 only */
} orc_linear;

typedef struct {
    const uint16_t* attn_norm;   /* bf16 [hidden] */
    const uint16_t* ffn_norm;    /* bf16 [hidden] */
    orc_linear wq, wk, wv, wo, wg, wu, wd;
} orc_layer;

typedef struct {
    const uint16_t* embed;       /* bf16 [vocab][hidden] */
    const uint16_t* final_norm;  /* bf16 [hidden] */
    orc_linear lm_head;          /* tied models pass embed here as bf16 */
    const orc_layer* layers;     /* [n_layers] */
} orc_weights;

typedef struct {
    int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
    int64_t max_seq;
    double rms_eps, rope_theta;
} orc_config;

/* threads used by the parallel loops (OpenMP when built with it) */
void orc_set_threads(int n);
int orc_get_threads(void);

/* number conversions */
double orc_bf16_to_double(uint16_t b);
uint16_t orc_bf16_from_double(double v);     /* round to nearest, ties to even */
double orc_fp16_to_double(uint16_t h);

/* weight element access: out[k] = W[row][k] as an exact double */
void orc_dequant_row(const orc_linear* lin, int64_t out_features, int64_t in_features,
                     int64_t row, double* out);

/* y[out] = W[out][in] x[in] */
void orc_linear_apply(const orc_linear* lin, int64_t out_features, int64_t in_features,
                      const double* x, double* y);

/* out = x / sqrt(mean(x^2) + eps) * w   (w NULL means all ones) */
void orc_rmsnorm(const double* x, const uint16_t* w, int64_t n, double eps, double* out);

/* in place rotate-half RoPE of n_heads vectors of head_dim at position pos */
void orc_rope(double* v, int32_t n_heads, int32_t head_dim, int64_t pos, double theta);

double orc_silu(double z);

/* causal GQA attention of one query position over ctx cached positions.
 * q [n_heads][head_dim]; k, v bf16 [n_kv_heads][max_seq][head_dim];
 * out [n_heads][head_dim]; q head i reads kv head i / (n_heads / n_kv_heads). */
void orc_attention(const double* q, const uint16_t* k, const uint16_t* v,
                   int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                   int64_t max_seq, int64_t ctx, double* out);

/* One decode step at position pos: writes K,V of pos into kv and, when
 * logits is not NULL, the vocab logits.  Returns 0, or -1 on bad arguments. */
int orc_decode_step(const orc_config* cfg, const orc_weights* w, uint16_t* kv,
                    int32_t token, int64_t pos, double* logits);

/* The two halves of a decode step, for bounded timing samples:
 * layers [l0, l1) applied in place to the residual x [hidden] at position
 * pos (writing their K,V of pos), and the final norm + LM-head rows
 * [r0, r1) of the vocabulary from the residual.  orc_decode_step is
 * embedding -> orc_decode_layers(0, n_layers) -> orc_logits_rows(0, vocab). */
int orc_decode_layers(const orc_config* cfg, const orc_weights* w, uint16_t* kv, double* x,
                      int64_t pos, int32_t l0, int32_t l1);
int orc_logits_rows(const orc_config* cfg, const orc_weights* w, const double* x,
                    double* logits, int64_t r0, int64_t r1);

/* n decode steps at positions start_pos.. without logits (fills the cache) */
int orc_prefill(const orc_config* cfg, const orc_weights* w, uint16_t* kv,
                const int32_t* tokens, int64_t n, int64_t start_pos);

/* The same prefill as one batched, causal loop nest: layer by layer over
 * all n tokens (projections, RoPE, the K,V rows of every position, causal
 * attention, O map, SwiGLU block).  Leaves the cache orc_prefill leaves. */
int orc_prefill_batched(const orc_config* cfg, const orc_weights* w, uint16_t* kv,
                        const int32_t* tokens, int64_t n, int64_t start_pos);

#ifdef __cplusplus
}
#endif
#endif
