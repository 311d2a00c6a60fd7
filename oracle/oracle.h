/*
 * CPU ORACLE for the GGUF-quantized Llama-style decoder forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously-correct fp64
 * restatement of what the cited pages define, used by the tests, by the
 * smoke check and by the timed CPU baseline.  No product code path may link,
 * load or call it, and it shares no code with the CUDA library.
 *
 * Sources (page title, section):
 *  - Airframe "GPU_PIPELINE.md" (Shimmy docs): per-layer operation diagram
 *    (RMS norm, Q/K/V projections, RoPE with the YaRN theta, KV write at t,
 *    QK^T/sqrt(head_dim), softmax, weighted V sum, O projection + residual,
 *    RMS norm, gate/up, SwiGLU gate*sigmoid(gate)*up, down + residual);
 *    "KV cache" buffer layout and byte formula; "Prefill" chunking;
 *    "Decode" step; "Output head" (LM head on the last position); "Sampler"
 *    (greedy = temperature 0).
 *  - "Shimmy v2.0 Architecture": "Quantization" table (Q4_0, Q8_0 32-element
 *    blocks; Q4_K, Q5_K and Q6_K super-blocks, whose byte layout the pages leave to
 *    another document: the published GGUF layout is taken), "Extended Context
 *    (YaRN)" (scale applied to all positions).
 *  - "GPU Inference — dotLLM": "Forward Pass" steps (final RmsNorm on the last
 *    token, LM head), "Attention on GPU" (causal mask, GQA group = H / KVH).
 *
 * Parity pins: every function here is pinned by CPU tests against values the
 * pages or the mathematics fix (hand-built blocks, closed forms, invariants,
 * brute force).  The whole-model composition is pinned only through those
 * parts plus chunk-invariance and decode-vs-prefill invariants: its end-to-end
 * logits are "parity unpinned" beyond that, because the pages print none.
 */
#ifndef AF_ORACLE_H
#define AF_ORACLE_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_Q4_0 = 2, ORC_Q8_0 = 8, ORC_Q4_K = 12, ORC_Q5_K = 13, ORC_Q6_K = 14 };

typedef struct orc_config {
    int32_t n_layers, n_embd, n_heads, n_kv_heads, head_dim, n_ff, n_vocab;
    int32_t wtype;      /* ORC_Q8_0 | ORC_Q4_0 | ORC_Q4_K | ORC_Q5_K | ORC_Q6_K: layer matrices and token_embd */
    int32_t kv_f16;     /* 0: f32 cache, 1: f16 cache, 2: Q8_0, 3: Q4_0 (quantized, with an fp16 window) */
    int32_t max_ctx, native_ctx;
    double rms_eps, rope_base;
    int32_t out_wtype;  /* block type of the LM head (0 = wtype) */
    int32_t kv_window;  /* quantized caches: slots within this many positions of a step's last one stay fp16 */
} orc_config;

typedef struct orc_model orc_model;

/* IEEE binary16 bits -> exact double. */
double orc_f16_to_double(uint16_t h);
/* double -> nearest binary16 value (RNE, overflow to inf), returned as double. */
double orc_round_f16(double x);
/* double -> nearest binary32 value, returned as double. */
double orc_round_f32(double x);

/* Decode k elements (a whole number of blocks: 32 elements, 256 for Q4_K / Q6_K) of GGUF blocks into exact
 * doubles. */
int orc_dequant_row(int32_t wtype, const uint8_t* blocks, int64_t k, double* out);

/* A quantized cache's replacement of one K or V row (D % 32 == 0, fp16 values) by its Q8_0 (kv_dtype 2) or Q4_0
 * (3) quantization, in place (see the quantized KV reading in oracle.cpp). */
int orc_quant_kv_row(int32_t kv_dtype, double* v, int64_t D);

/* y[i] = sum_j W[i][j] x[j] for the n rows of W (k columns, GGUF blocks). */
int orc_qgemv(int32_t wtype, const uint8_t* W, int64_t n, int64_t k, const double* x, double* y, int n_threads);
/* The same for selected rows only: y[r] for r in rows[0..n_rows). */
int orc_qgemv_rows(int32_t wtype, const uint8_t* W, int64_t k, const int64_t* rows, int64_t n_rows, const double* x,
                   double* y, int n_threads);
/* Y[m][i] = sum_j X[m][j] W[i][j]  (X: [M, k] row-major, Y: [M, n]). */
int orc_qgemm(int32_t wtype, const uint8_t* W, int64_t n, int64_t k, const double* X, int64_t M, double* Y,
              int n_threads);

/* y = w * x / sqrt(mean(x^2) + eps). */
void orc_rmsnorm(const double* x, const float* w, int64_t n, double eps, double* y);
/* yarn_scale = max_ctx / native_ctx when max_ctx > native_ctx, else 1. */
double orc_yarn_scale(int32_t max_ctx, int32_t native_ctx);
/* theta(t, i) = (t / yarn_scale) / base^(2i / head_dim). */
double orc_rope_theta(int64_t t, int32_t i, int32_t head_dim, double base, double yarn_scale);
/* Rotate pairs (2i, 2i+1) of each head of v[n_heads*head_dim] by theta(t, i). */
void orc_rope(double* v, int32_t n_heads, int32_t head_dim, int64_t t, double base, double yarn_scale);
double orc_silu(double g);
/* In-place softmax with max subtraction. */
void orc_softmax(double* s, int64_t n);
/* One query row, all heads: out[h] = softmax_j(q_h . K_j / sqrt(D)) V_j over j < n_keys.
 * K/V of kv head g at kc/vc + g * head_stride, key j at + j * head_dim. */
void orc_attention(const double* q, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, const double* kc,
                   const double* vc, int64_t head_stride, int64_t n_keys, double* out);

/* Per-layer blob section offsets, off[9] = total bytes. */
int orc_layer_offsets(const orc_config* c, uint64_t off[10]);
/* KV cache bytes: n_layers * n_kv_heads * max_ctx * head_dim * elem * 2. */
uint64_t orc_kv_bytes(const orc_config* c);

/* The model holds pointers to the caller's host blobs (not copied) and an fp64
 * KV cache with kv_slots positions (<= max_ctx; 0 means max_ctx). */
orc_model* orc_model_create(const orc_config* c, const uint8_t* const* layer_blobs, const uint8_t* token_embd,
                            const float* output_norm, const uint8_t* output, int64_t kv_slots);
/* Forward n tokens at absolute positions start_pos..start_pos+n-1 (a quantized cache: n <= kv_window, else -3).
 * logits: [n_vocab] for the last row (nullable).  capture: [n_layers+1][n][n_embd]
 * residual stream after the embedding and after each layer (nullable). */
int orc_forward(orc_model* m, const int32_t* tokens, int64_t n, int64_t start_pos, double* logits, double* capture,
                int n_threads);
/* Read cache slot (layer, kv head, pos): head_dim values of K and of V. */
int orc_kv_read(const orc_model* m, int32_t layer, int32_t kvh, int64_t pos, double* k, double* v);
/* Set cache slots pos0..pos0+n-1 of (layer, kv head): k, v [n][head_dim], stored as given (the caller passes
 * values of the cache's element type).  A plain setter: it lets a test start from a cache prefix that both sides
 * hold. */
int orc_kv_write(orc_model* m, int32_t layer, int32_t kvh, int64_t pos0, int64_t n, const double* k,
                 const double* v);
void orc_model_destroy(orc_model* m);
/* Greedy token: argmax, lowest index on ties. */
int64_t orc_argmax(const double* v, int64_t n);
// Sampler chain: repetition penalty -> temperature -> softmax -> top-p -> sample with uniform u.
// Returns the token; lo / hi (nullable) get its cumulative-mass interval within the nucleus.
int64_t orc_sample(const double* logits, int64_t V, const int32_t* recent, int64_t n_recent, double repeat_penalty,
                   double temperature, double top_p, double u, double* lo, double* hi);
// For a given token (temperature > 0): its cumulative-mass interval [lo, hi] in the sampling order as a
// fraction of the nucleus mass, its probability and the nucleus' smallest probability.  Returns 1 if the
// token is in the nucleus, 0 if not, -1 on bad arguments.
int orc_sample_interval(const double* logits, int64_t V, const int32_t* recent, int64_t n_recent,
                        double repeat_penalty, double temperature, double top_p, int64_t token, double* lo,
                        double* hi, double* p_token, double* p_boundary);

#ifdef __cplusplus
}
#endif
#endif
