/*
 * af.h — C ABI of the GB300 (sm_103a) forward pass of a GGUF-quantized
 * Llama-style decoder.
 *
 * What it computes (page title, section):
 *  - Airframe "GPU_PIPELINE.md" (Shimmy docs), per-layer operation diagram:
 *    RMS norm -> Q/K/V projections with inline dequantization -> RoPE with
 *    theta(t, i) = (t / yarn_scale) / base^(2i / head_dim) and
 *    yarn_scale = max_ctx / native_ctx when max_ctx > native_ctx -> K, V written
 *    to the KV cache at position t -> softmax(Q K^T / sqrt(head_dim)) V ->
 *    O projection + residual -> RMS norm -> gate, up -> gate*sigmoid(gate)*up
 *    -> down + residual.  "Prefill": prompts run in chunks of up to 512 tokens
 *    that fill KV slots start_pos..start_pos+n-1; only the last chunk's logits
 *    are used.  "Decode": one token at position t attends to slots 0..t.
 *    "Output head": LM head on the last position.  "KV cache": layout
 *    [n_layers][n_kv_heads][max_ctx][head_dim], K and V separate.
 *  - "Shimmy v2.0 Architecture", "Quantization": GGUF Q4_0 and Q8_0
 *    32-element blocks; "Extended Context (YaRN)": the theta scale applies to
 *    all positions.
 *  - "GPU Inference — dotLLM", "Forward Pass" (final RmsNorm on the last token,
 *    LM head, one host sync per step) and "Attention on GPU" (causal, GQA with
 *    group = n_heads / n_kv_heads).
 *
 * Conventions.
 *  - Every call returns an af_status.  Arguments are validated on the host
 *    before anything is launched; a call that fails validation changes nothing.
 *    af_last_error() returns a thread-local message for the last failure.
 *  - "_dev" pointers are device pointers on the current CUDA device; "_host"
 *    pointers are ordinary host memory.  `stream` is a cudaStream_t (NULL =
 *    legacy default stream).  Unless stated otherwise a call only enqueues
 *    work on the model's (or the given) stream and returns.
 *  - The caller owns every pointer it passes.  af_model_create and
 *    af_qweight_create copy (repack) the weights into memory they own, so the
 *    caller may free its blobs once the call has returned and the stream has
 *    been synchronised.
 *  - Weights: GGUF blocks, little-endian.
 *      Q8_0 (34 B): fp16 d, int8 q[32];             w_j = d * q_j
 *      Q4_0 (18 B): fp16 d, uint8 qs[16];            w_j = d * (n_j - 8),
 *                   n_j = qs[j] & 15 (j < 16), qs[j - 16] >> 4 (j >= 16)
 *      Q4_K (144 B per 256 weights): fp16 d, fp16 dmin, uint8 scales[12],
 *                   uint8 qs[128]; 6-bit scale s_j and min m_j of sub-block
 *                   j = e / 32 (j < 4: scales[j] & 63, scales[j + 4] & 63;
 *                   j >= 4: (scales[j + 4] & 15) | (scales[j - 4] >> 6) << 4,
 *                   (scales[j + 4] >> 4) | (scales[j] >> 6) << 4); code n_e in
 *                   the low (e % 64 < 32) or high nibble of qs[32 (e / 64) + e % 32];
 *                   w_e = d s_j n_e - dmin m_j
 *      Q5_K (176 B per 256 weights): fp16 d, fp16 dmin, uint8 scales[12] (as
 *                   Q4_K), uint8 qh[32], uint8 qs[128] (nibbles placed as Q4_K's);
 *                   the 5-bit code q_e = nibble + 16 * (bit 2 (e / 64) + (e % 64 >= 32)
 *                   of qh[e % 32]); w_e = d s_j q_e - dmin m_j
 *      Q6_K (210 B per 256 weights): uint8 ql[128], uint8 qh[64], int8
 *                   scales[16], fp16 d; with h = e / 128, k = (e % 128) / 32,
 *                   l = e % 32 the code q_e has its low 4 bits in the low (k < 2)
 *                   or high nibble of ql[64 h + 32 (k & 1) + l] and its high 2 bits
 *                   at bits 2k of qh[32 h + l]; w_e = d scales[e / 16] (q_e - 32)
 *    (Shimmy v2.0 Architecture, "Quantization": the K-quant super-blocks; their
 *    byte layout is GGUF's.)  A matrix [N, K] is N rows of K / 32 blocks each
 *    (K / 256 super-blocks for Q4_K, Q5_K and Q6_K; K must be a whole number of blocks).
 */
#ifndef AF_H
#define AF_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum af_status {
    AF_OK = 0,
    AF_EINVAL = 1,   /* bad argument: null pointer, unsupported shape or type */
    AF_ERANGE = 2,   /* position / token id / size out of range */
    AF_ENOMEM = 3,   /* device or host allocation failed (nothing leaked) */
    AF_ECUDA = 4,    /* a CUDA runtime call failed; see af_last_error() */
    AF_ETIMEOUT = 5, /* a bounded device-side wait gave up */
    AF_ENOTIMPL = 6  /* valid request this build does not implement */
} af_status;

typedef enum af_wtype { AF_Q4_0 = 2, AF_Q8_0 = 8, AF_Q4_K = 12, AF_Q5_K = 13, AF_Q6_K = 14 } af_wtype; /* GGUF's type numbers */
/* KV cache element types.  AF_KV_Q8_0 / AF_KV_Q4_0: a quantized cache with an fp16 window (dotLLM, "CUDA
 * components": "Q8_0/Q4_0 + FP16 window"): a slot is written in fp16; once it lies more than kv_window
 * positions behind a step's last position it is replaced by the Q8_0 / Q4_0 quantization of its fp16 values,
 * per 32 values along head_dim (Q8_0: d = fp16(max|v| / 127), q = clamp(round-half-away(v / d), -127, 127);
 * Q4_0: d = fp16(m / -8) with m the value of largest magnitude, n = clamp(floor(v / d + 8.5), 0, 15),
 * q = n - 8; decisions in fp32 on the fp16 values), and reads of the slot see d * q.  Decode attention reads
 * retired slots from the quantized store; prefill attention reads the fp16 copy, where a retired slot holds
 * fp16(d * q). */
typedef enum af_dtype { AF_F32 = 0, AF_F16 = 1, AF_KV_Q8_0 = 2, AF_KV_Q4_0 = 3 } af_dtype;

typedef struct af_config {
    int32_t n_layers, n_embd, n_heads, n_kv_heads, head_dim, n_ff, n_vocab;
    int32_t wtype;      /* af_wtype of every matrix and of token_embd */
    int32_t kv_dtype;   /* af_dtype of the KV cache */
    int32_t max_ctx;    /* KV slots */
    int32_t native_ctx; /* yarn_scale = max_ctx / native_ctx if max_ctx > native_ctx, else 1 */
    int32_t max_chunk;  /* largest n accepted by af_prefill (0 = 512) */
    float rms_eps;      /* RMSNorm epsilon */
    float rope_base;    /* RoPE base */
    int32_t out_wtype;  /* af_wtype of the LM head (output.weight); 0 = wtype (a Q4_K_M model: Q4_K layers and
                           embedding with a Q6_K head) */
    int32_t kv_window;  /* quantized caches: slots kept in fp16 behind a step's last position; at least max_chunk, so
                           a step is never longer than the window (ignored for AF_F32 / AF_F16) */
} af_config;

/*
 * Layer blob (Airframe "GPU_PIPELINE.md", bindless layer buffer): one device
 * buffer per layer holding, in this order, each section at a 256-byte aligned
 * offset (see af_layer_offsets):
 *   attn_norm f32[E] | attn_q [H*D, E] | attn_k [KVH*D, E] | attn_v [KVH*D, E] |
 *   attn_o [E, H*D] | ffn_norm f32[E] | ffn_gate [F, E] | ffn_up [F, E] | ffn_down [E, F]
 * Matrices are [out, in] in GGUF blocks along `in`.
 */
typedef struct af_weights {
    const void* const* layer_blob; /* host array of n_layers device pointers */
    const void* token_embd;        /* device, [n_vocab, n_embd] blocks */
    const float* output_norm;      /* device, f32 [n_embd] */
    const void* output;            /* device, [n_vocab, n_embd] blocks of out_wtype (LM head, not tied) */
} af_weights;

typedef struct af_model af_model;
typedef struct af_qweight af_qweight;

/* Section offsets of a layer blob: off[0..8] in the order above, off[9] = blob bytes. */
int af_layer_offsets(const af_config* cfg, uint64_t off[10]);

/* KV cache bytes, n_layers * n_kv_heads * max_ctx * head_dim * elem * 2
 * (Airframe "GPU_PIPELINE.md", "KV cache" size formula).  A quantized cache holds every slot twice, in fp16
 * and in the quantized store: n_layers * n_kv_heads * 2 * max_ctx * (head_dim * 2 + head_dim / 32 * B),
 * B = 34 (Q8_0) or 18 (Q4_0) bytes per 32 values.  0 on a bad config. */
uint64_t af_kv_bytes(const af_config* cfg);

/*
 * Create a model on the current device.  Repacks every matrix into the
 * model's own layout, allocates the KV cache (zeroed) and the step scratch,
 * and builds the RoPE table.  Synchronises `stream` before returning.  With
 * stream == NULL the model creates (and later destroys) a blocking stream of
 * its own, which is ordered with the legacy default stream.
 * Supported: head_dim in {64, 128}, n_heads % n_kv_heads == 0 with
 * n_heads / n_kv_heads in {1, 2, 4, 8}, n_embd, n_ff, n_heads*head_dim
 * multiples of 64, even n_vocab; quantized caches: kv_window >= max_chunk and
 * max_ctx a multiple of 4.  Errors: AF_EINVAL, AF_ENOMEM, AF_ECUDA,
 * AF_ENOTIMPL (valid but unsupported shape).  *out is NULL on failure.
 */
int af_model_create(const af_config* cfg, const af_weights* w, void* stream, af_model** out);

/*
 * Prefill n tokens (1 <= n <= max_chunk) at absolute positions
 * start_pos..start_pos+n-1 (start_pos + n <= max_ctx).  Writes those KV slots;
 * row r attends to slots 0..start_pos+r.  The caller runs longer prompts as
 * consecutive chunks with increasing start_pos.  If logits_dev is not NULL it
 * receives the n_vocab fp32 logits of the last row.  tokens_host is copied
 * into the model's page-locked staging buffer before the call returns, so the
 * caller may reuse it at once (pageable or page-locked alike); the call first
 * waits for the previous af_prefill's copy out of that buffer.  Not for stream
 * capture (use af_prefill_dev there).  Errors: AF_EINVAL, AF_ERANGE (token id
 * outside [0, n_vocab) or positions past max_ctx), AF_ECUDA.
 */
int af_prefill(af_model* m, const int32_t* tokens_host, int32_t n, int32_t start_pos, float* logits_dev);

/* As af_prefill with the token ids already in device memory.  They are not
 * validated on the host; an id outside [0, n_vocab) reads embedding row 0. */
int af_prefill_dev(af_model* m, const int32_t* tokens_dev, int32_t n, int32_t start_pos, float* logits_dev);

/*
 * One decode step: the token at position pos (0 <= pos < max_ctx) attends to
 * slots 0..pos.  token = -1 feeds the previous step's greedy token (from the
 * device, no host round trip).  logits_dev (nullable) receives the fp32
 * logits.  If next_token_host is not NULL the call synchronises the model's
 * stream once and stores the greedy token there (argmax, lowest index on
 * ties); otherwise it only enqueues.
 */
int af_decode_step(af_model* m, int32_t token, int32_t pos, float* logits_dev, int32_t* next_token_host);

/* Synchronise the model's stream.  Returns AF_ETIMEOUT if a bounded device-side
 * wait of an earlier call gave up, else AF_OK; if next_token_host is not NULL it
 * receives the greedy token of the last call that produced logits.  A reported
 * timeout is cleared (af_decode_step with next_token_host reports and clears the
 * same way), so a later call reports only what happened after it.  The outputs
 * of the calls that timed out are not valid. */
int af_model_sync(af_model* m, int32_t* next_token_host);

/* Greedy token of the last af_decode_step / af_prefill with logits (device int32, valid after the stream). */
const int32_t* af_model_next_token_dev(const af_model* m);

/* Device pointers of the model's KV cache: K and V each [n_layers][n_kv_heads][max_ctx][head_dim]
 * in kv_dtype, fp16 for a quantized cache (Airframe "GPU_PIPELINE.md", "KV cache" layout).  Owned by the
 * model. */
int af_model_kv_cache(const af_model* m, void** k_dev, void** v_dev);

/* The quantized store of a quantized cache (AF_EINVAL otherwise): per slot of [n_layers][n_kv_heads][max_ctx],
 * the codes (Q8_0: head_dim int8 values q in element order; Q4_0: head_dim / 2 bytes, byte j holding
 * n = q + 8 of element 2j in its low and of element 2j + 1 in its high nibble) in *codes, and head_dim / 32 fp16
 * scales d in *scales; k_ for K, v_ for V.  Valid for slots that have retired.  Owned by the model. */
int af_model_kv_store(const af_model* m, void** k_codes, void** k_scales, void** v_codes, void** v_scales);

/* Zero the KV cache (the service is stateless between requests) and the error word.  Steps after it start
 * again at position 0; with a quantized cache, each step must start where the previous one ended (the
 * slots that leave the window are retired by the step that passes them). */
int af_reset(af_model* m);

/* Model's stream (as given to af_model_create). */
void* af_model_stream(const af_model* m);

/* Capture the residual stream after the embedding and after every layer of the
 * next af_prefill / af_decode_step into hidden_dev [n_layers+1][n][n_embd] fp32
 * (n = that call's token count).  One-shot; test instrumentation. */
int af_debug_capture(af_model* m, float* hidden_dev);

/*
 * How af_decode_step runs (both are this library's CUDA kernels):
 *   AF_DECODE_KERNELS (default): one launch per matrix / attention, chained
 *     with programmatic dependent launch and replayed as a CUDA graph (see
 *     af_set_decode_graph).
 *   AF_DECODE_PERSISTENT: one cooperative launch per token, one CTA per SM,
 *     phases (each matrix, attention) separated by bounded grid barriers; each
 *     warp's shared-memory slot streams its next stage of weights or cache
 *     tiles whatever phase it belongs to, so copies run ahead through the
 *     barriers (Q4_0 or Q8_0 for every matrix including the LM head, an fp32 or
 *     fp16 cache, head_dim 64 or 128, group 2, 4 or 8; AF_ENOTIMPL otherwise or
 *     where it cannot be resident).  Measured slower than the default.
 */
enum { AF_DECODE_PERSISTENT = 0, AF_DECODE_KERNELS = 1 };
int af_set_decode_mode(af_model* m, int mode);
int af_get_decode_mode(const af_model* m);

/* In AF_DECODE_KERNELS mode, use (1) or stop using (0) a CUDA graph (default 1). */
int af_set_decode_graph(af_model* m, int enable);

/* Trace the next persistent af_decode_step: trace_dev (device, uint64 [5 n_layers + 3])
 * receives the GPU global timer (ns) at kernel start, after the embedding, after each
 * of the 5 phases of every layer, and at the end.  One-shot; profiling aid. */
int af_debug_trace(af_model* m, uint64_t* trace_dev);

void af_model_destroy(af_model* m);

/* Test instrumentation of the error path: with polls != 0 the first wait of every decode GEMV launched
 * afterwards polls an mbarrier that nothing arrives on `polls` times, then takes its timeout path (error
 * word set, its bulk copies drained, early return) as a real timeout would; 0 turns it off.  Synchronises
 * the model's stream.  Lets a test see AF_ETIMEOUT without a fault or a hang. */
int af_debug_stall(af_model* m, uint32_t polls);

/*
 * Standalone quantized matmuls.
 * af_qweight_create repacks a [N, K] block matrix (N even, K a whole number
 * of blocks: K % 32 == 0, K % 256 == 0 for Q4_K / Q5_K / Q6_K; K <= 32768, or
 * <= 16384 for Q8_0, else AF_ENOTIMPL) into its own device memory (and
 * scratch for the GEMV); synchronises `stream`.
 *   af_qgemv: y[i]    = sum_j W[i][j] x[j]        x_dev fp32 [K], y_dev fp32 [N]
 *   af_qgemm: Y[m][i] = sum_j X[m][j] W[i][j]     X_dev fp32 [M, K] row-major,
 *                                                 Y_dev fp32 [M, N], M >= 1
 * Calls that share one af_qweight must be ordered on one stream (they share
 * its scratch).  af_qgemv accumulates exact integer products of the weight
 * codes with x held in 16-bit fixed point per 32-element block (K-quant
 * sub-block scales and mins applied per 32 or 16 elements in fp32); af_qgemm
 * runs on the tensor cores with X and W each split into fp16 hi + lo parts
 * (three fp16 products accumulated in fp32, relative error ~1e-6 per product;
 * K-quant weights are formed in fp32 before their split).
 * af_qgemm keeps the split X in buffers of the af_qweight: the first call
 * with a larger M than before synchronises `stream` and grows them.
 */
int af_qweight_create(int32_t wtype, const void* blocks_dev, int32_t N, int32_t K, void* stream, af_qweight** out);
int af_qgemv(const af_qweight* w, const float* x_dev, float* y_dev, void* stream);
int af_qgemm(const af_qweight* w, const float* X_dev, int32_t M, float* Y_dev, void* stream);
void af_qweight_destroy(af_qweight* w);

/* Synchronise `stream` and report w's error word: AF_ETIMEOUT if a bounded device-side wait of an af_qgemv /
 * af_qgemm on w gave up since the last report (the word is then cleared; those outputs are not valid), else
 * AF_OK. */
int af_qweight_status(const af_qweight* w, void* stream);

/* Test instrumentation: as af_debug_stall, for the af_qgemv calls on w (synchronises `stream`). */
int af_qweight_debug_stall(af_qweight* w, uint32_t polls, void* stream);

/*
 * Standalone causal GQA attention for one query row at position pos over a
 * caller's cache (Airframe per-layer ops: softmax(q K^T / sqrt(D)) V over
 * slots 0..pos; dotLLM "Attention on GPU": GQA group = H / KVH).
 *   q_dev   fp32 [H*D] (already rotated)
 *   k_dev, v_dev  [KVH][ctx][D] in kv_dtype
 *   out_dev fp32 [H*D]
 * Scratch (split partials) is allocated per call and freed after the stream
 * completes (the call synchronises `stream`).  AF_ETIMEOUT if a bounded
 * device-side wait gave up.
 */
int af_attention_decode(const float* q_dev, const void* k_dev, const void* v_dev, int32_t kv_dtype, int32_t n_heads,
                        int32_t n_kv_heads, int32_t head_dim, int32_t ctx, int32_t pos, float* out_dev, void* stream);

/*
 * af_attention_decode without any device allocation (no counterpart on the
 * pages: an interface for callers that cannot allocate mid-step, e.g. a
 * serving loop that cannot take the device-wide synchronisation of cudaFree,
 * or one whose memory is all handed to its own pool).  Same arguments, same
 * kernel and same result as af_attention_decode, but stream-ordered: it does
 * not synchronise `stream`.
 * Scratch: one file-scope device array of this library (4 MiB of split
 * partials + 1024 arrival counters + an error word), used only when ctx >
 * 2048 (shorter caches take the cluster path, which merges in distributed
 * shared memory, where the device can schedule 8-CTA clusters).
 * On that path, calls with n_kv_heads > 1024 or whose partials need more than
 * 2^20 floats (n_heads * splits * (head_dim + 4), splits = max(1, 2 * SMs /
 * n_kv_heads)) return AF_ERANGE before launching.
 * Errors on the device: the call does not wait for the kernel, so it cannot
 * report AF_ETIMEOUT; if a bounded device-side wait gives up, every output
 * value of the affected kv heads is NaN instead.
 * The counters must start at zero: they are zero when the library is loaded
 * and every launch leaves them zero, a timed-out one included (each CTA
 * still arrives, and the last one resets the counter).  All calls on a device
 * share the one array, so calls that may overlap in time (different streams
 * without ordering between them) race and give wrong results: order them on
 * one stream.  The first call on each device looks up the array's address
 * (cudaGetSymbolAddress, with that device current) and loads the kernels; make
 * that first call before any stream capture.
 */
int af_attention_decode_static(const float* q_dev, const void* k_dev, const void* v_dev, int32_t kv_dtype,
                               int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t ctx, int32_t pos,
                               float* out_dev, void* stream);

/*
 * Standalone causal prefill attention (the tensor-core kernel af_prefill runs;
 * Airframe per-layer ops: softmax(q K^T / sqrt(D)) V, causal; dotLLM
 * "Attention on GPU": GQA group = H / KVH) for n query rows at positions
 * start_pos..start_pos+n-1 over a caller's cache.  Test entry point.
 *   q_dev   fp32 [n][H*D] (already rotated), row r at position start_pos + r
 *   k_dev, v_dev  [KVH][ctx][D] in kv_dtype (16-byte aligned); row r attends
 *           to slots 0..start_pos+r
 *   out_dev fp32 [n][H*D]: the fp16 hi + lo output planes of the kernel, summed
 * 1 <= n <= 512, start_pos + n <= ctx (AF_ERANGE).  The output planes are
 * allocated per call; the call synchronises `stream`.  AF_ETIMEOUT if a
 * bounded device-side wait gave up.
 */
int af_attention_prefill(const float* q_dev, const void* k_dev, const void* v_dev, int32_t kv_dtype, int32_t n_heads,
                         int32_t n_kv_heads, int32_t head_dim, int32_t ctx, int32_t start_pos, int32_t n,
                         float* out_dev, void* stream);

/*
 * Sampler chain on the device (Airframe GPU pipeline, sampler: "repetition
 * penalty -> temperature -> softmax -> top-p -> sample"): one kernel launch
 * of one 8-CTA thread-block cluster that keeps the logits in shared memory; no
 * device scratch and no allocation, so calls on different streams are
 * independent.  Asynchronous on `stream`:
 *   logits_dev  fp32 [n_vocab] (not modified), n_vocab <= 262144
 *   recent_dev  int32 [n_recent] recent token ids (device; NULL when n_recent = 0);
 *               each distinct id in [0, n_vocab) has its logit divided by
 *               repeat_penalty once (only when repeat_penalty > 1)
 *   temperature 0 -> greedy (argmax, lowest index on ties); > 0 divides the logits
 *   top_p       nucleus: the shortest prefix of the tokens sorted by
 *               (probability descending, index ascending) whose mass reaches
 *               top_p, plus every token tied with its last one; >= 1 keeps all
 *   u           the caller's uniform draw in [0, 1): the token returned is the
 *               first of that order whose cumulative mass reaches u times the
 *               nucleus mass
 *   token_dev   int32 [1] result
 * AF_EINVAL / AF_ERANGE for bad arguments (checked on the host).
 */
int af_sample(const float* logits_dev, int32_t n_vocab, const int32_t* recent_dev, int32_t n_recent,
              float repeat_penalty, float temperature, float top_p, float u, int32_t* token_dev, void* stream);

/*
 * The sampler chain (as af_sample) over a model's logits, on the model's stream:
 * the token drawn replaces the model's next-token word (af_model_next_token_dev),
 * so a following af_decode_step(m, -1, ...) feeds it.  A decode loop that
 * alternates af_decode_step(m, -1, pos, NULL, NULL) and af_model_sample(...)
 * samples on the device with no logits read back.
 *   logits_dev  the logits to sample (n_vocab fp32); NULL = the model's own
 *               buffer, which steps called with logits_dev = NULL write
 *   recent_dev, n_recent, repeat_penalty, temperature, top_p, u: as af_sample
 *   token_host  if not NULL: synchronises the model's stream once and stores
 *               the token drawn; otherwise the call only enqueues
 * AF_EINVAL / AF_ERANGE for bad arguments (checked on the host).
 */
int af_model_sample(af_model* m, const float* logits_dev, const int32_t* recent_dev, int32_t n_recent,
                    float repeat_penalty, float temperature, float top_p, float u, int32_t* token_host);

/* Thread-local message for the last failed call on this thread ("" if none). */
const char* af_last_error(void);

#ifdef __cplusplus
}
#endif
#endif
