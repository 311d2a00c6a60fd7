/*
 * Seeded synthetic inputs for the GGUF-quantized Llama-style decoder.
 *
 * This module produces INPUT DATA only: random-init weights already encoded
 * as GGUF Q8_0 / Q4_0 blocks, fp32 norm weights, token ids and activation
 * vectors.  It contains none of the forward-pass arithmetic (no decode of a
 * quantized block, no matmul, norm, RoPE or attention); both the CUDA library
 * and the CPU oracle read the bytes it writes and decode them independently.
 *
 * Random numbers: counter-based, so each element is a pure function of
 * (seed, tensor id, element index) and the output does not depend on the
 * number of threads used.
 *   key(seed, tid, i) = splitmix64( splitmix64(seed) ^ (tid << 40) ^ i )
 *   uniform(key)      = ((key >> 11) + 0.5) * 2^-53          in (0, 1)
 *   normal(seed,tid,i)= sqrt(-2 ln u1) * cos(2 pi u2),
 *                       u1 = uniform(key(seed,tid,2i)), u2 = uniform(key(seed,tid,2i+1))
 * splitmix64 is Steele/Lea/Flood's SplittableRandom finaliser as published by
 * Vigna; Box-Muller is the textbook transform.
 *
 * Block encodings (the GGUF formats named on the Shimmy v2.0 Architecture page,
 * "Quantization" table: "Q4_0 32-element block, 4-bit signed", "Q8_0 32-element
 * block, 8-bit signed"), byte layout little-endian:
 *   Q8_0 block (34 B): fp16 d | int8 q[32];            value_j = d * q_j
 *   Q4_0 block (18 B): fp16 d | uint8 qs[16];           value_j = d * (n_j - 8)
 *        n_j = qs[j] & 15 for j < 16, qs[j-16] >> 4 for j >= 16.
 * Encoder choices (test data only; any choice decodes unambiguously):
 *   Q8_0: d = max|w| / 127 (fp32), stored fp16 RNE;
 *         q = clamp(round-half-away(w / d), -127, 127); all-zero block -> d = 0, q = 0.
 *   Q4_0: m = the element of largest |w| (first on ties), d = m / -8 (fp32),
 *         stored fp16 RNE; n = clamp(floor(w / d + 8.5), 0, 15); m = 0 -> d = 0, n = 8.
 *
 * Layer blob: the Airframe GPU-pipeline page ("bindless" layer buffer layout)
 * packs one buffer per layer in the order
 *   attn_norm | attn_q | attn_k | attn_v | attn_o | ffn_norm | ffn_gate | ffn_up | ffn_down
 * Here every section starts at a 256-byte aligned offset, norms are fp32 and
 * matrices [out, in] row-major with GGUF blocks along `in`.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYN_Q8_0 8
#define SYN_Q4_0 2

static uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ULL;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ULL;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBULL;
    return x ^ (x >> 31);
}

static uint64_t syn_key(uint64_t seed, uint64_t tid, uint64_t i) {
    return splitmix64(splitmix64(seed) ^ (tid << 40) ^ i);
}

static double syn_uniform(uint64_t k) { return ((double)(k >> 11) + 0.5) * (1.0 / 9007199254740992.0); }

static double syn_normal(uint64_t seed, uint64_t tid, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = syn_uniform(syn_key(seed, tid, 2 * i));
    double u2 = syn_uniform(syn_key(seed, tid, 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

/* fp32 -> IEEE binary16 bits, round to nearest even (handles subnormals, inf). */
static uint16_t f32_to_f16_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax >= 0x7F800000u) return (uint16_t)(sign | (ax > 0x7F800000u ? 0x7E00u : 0x7C00u));
    if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* rounds to >= 65520 -> inf */
    if (ax < 0x38800000u) {                                   /* below fp16 min normal */
        if (ax < 0x33000000u) return (uint16_t)sign;          /* < half of min subnormal */
        uint32_t mant = (ax & 0x7FFFFFu) | 0x800000u;
        int e = (int)(ax >> 23);                              /* value = mant * 2^(e-150) */
        int shift = 126 - e;                                  /* to units of 2^-24 */
        uint32_t q = mant >> shift, rem = mant & ((1u << shift) - 1u), half = 1u << (shift - 1);
        if (rem > half || (rem == half && (q & 1u))) q++;
        return (uint16_t)(sign | q);
    }
    uint32_t e = (ax >> 23) - 112u; /* rebias 127 -> 15 */
    uint32_t m = ax & 0x7FFFFFu;
    uint32_t q = (e << 10) | (m >> 13), rem = m & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q++;
    return (uint16_t)(sign | q);
}

static size_t align256(size_t x) { return (x + 255u) & ~(size_t)255u; }

size_t syn_block_bytes(int wtype) { return wtype == SYN_Q8_0 ? 34u : (wtype == SYN_Q4_0 ? 18u : 0u); }

size_t syn_matrix_bytes(int wtype, int64_t n, int64_t k) { return (size_t)n * (size_t)(k / 32) * syn_block_bytes(wtype); }

/* off[0..8] = section offsets, off[9] = total bytes (multiple of 256). */
int syn_layer_offsets(int n_embd, int n_heads, int n_kv_heads, int head_dim, int n_ff, int wtype, uint64_t off[10]) {
    if (syn_block_bytes(wtype) == 0 || n_embd % 32 || n_ff % 32 || (n_heads * head_dim) % 32) return -1;
    size_t E = n_embd, QD = (size_t)n_heads * head_dim, KVD = (size_t)n_kv_heads * head_dim, F = n_ff;
    size_t sz[9] = {E * 4, syn_matrix_bytes(wtype, QD, E), syn_matrix_bytes(wtype, KVD, E),
                    syn_matrix_bytes(wtype, KVD, E), syn_matrix_bytes(wtype, E, QD), E * 4,
                    syn_matrix_bytes(wtype, F, E), syn_matrix_bytes(wtype, F, E), syn_matrix_bytes(wtype, E, F)};
    size_t o = 0;
    for (int i = 0; i < 9; i++) {
        off[i] = o;
        o = align256(o + sz[i]);
    }
    off[9] = o;
    return 0;
}

/* Encode one 32-element block. */
static void encode_block(int wtype, const float* w, uint8_t* out) {
    if (wtype == SYN_Q8_0) {
        float amax = 0.f;
        for (int j = 0; j < 32; j++) amax = fmaxf(amax, fabsf(w[j]));
        float d = amax / 127.f;
        uint16_t h = f32_to_f16_bits(d);
        memcpy(out, &h, 2);
        for (int j = 0; j < 32; j++) {
            int q = 0;
            if (d != 0.f) {
                float r = w[j] / d;
                q = (int)(r >= 0.f ? floorf(r + 0.5f) : -floorf(-r + 0.5f));
                q = q < -127 ? -127 : (q > 127 ? 127 : q);
            }
            out[2 + j] = (uint8_t)(int8_t)q;
        }
    } else {
        float m = 0.f, amax = 0.f;
        for (int j = 0; j < 32; j++)
            if (fabsf(w[j]) > amax) {
                amax = fabsf(w[j]);
                m = w[j];
            }
        float d = m / -8.f;
        uint16_t h = f32_to_f16_bits(d);
        memcpy(out, &h, 2);
        uint8_t n[32];
        for (int j = 0; j < 32; j++) {
            int v = 8;
            if (d != 0.f) {
                v = (int)floorf(w[j] / d + 8.5f);
                v = v < 0 ? 0 : (v > 15 ? 15 : v);
            }
            n[j] = (uint8_t)v;
        }
        for (int j = 0; j < 16; j++) out[2 + j] = (uint8_t)(n[j] | (n[j + 16] << 4));
    }
}

typedef struct {
    int wtype;
    uint64_t seed, tid;
    int64_t n, k, r0, r1;
    float mean, sigma;
    uint8_t* out;
} mat_job;

static void* mat_worker(void* arg) {
    mat_job* j = (mat_job*)arg;
    size_t bb = syn_block_bytes(j->wtype);
    float w[32];
    for (int64_t r = j->r0; r < j->r1; r++)
        for (int64_t b = 0; b < j->k / 32; b++) {
            for (int e = 0; e < 32; e++)
                w[e] = (float)(j->mean + j->sigma * syn_normal(j->seed, j->tid, (uint64_t)(r * j->k + b * 32 + e)));
            encode_block(j->wtype, w, j->out + ((size_t)r * (size_t)(j->k / 32) + (size_t)b) * bb);
        }
    return NULL;
}

/* Random matrix [n, k] with elements mean + sigma*N(0,1), encoded as GGUF blocks (AoS). */
int syn_gen_matrix(int wtype, uint64_t seed, uint64_t tid, int64_t n, int64_t k, float mean, float sigma,
                   uint8_t* out, int n_threads) {
    if (syn_block_bytes(wtype) == 0 || k % 32 || n < 0) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if (n_threads > n) n_threads = (int)(n > 0 ? n : 1);
    pthread_t th[256];
    mat_job jobs[256];
    for (int t = 0; t < n_threads; t++) {
        jobs[t] = (mat_job){wtype, seed, tid, n, k, n * t / n_threads, n * (t + 1) / n_threads, mean, sigma, out};
        if (t > 0) pthread_create(&th[t], NULL, mat_worker, &jobs[t]);
    }
    mat_worker(&jobs[0]);
    for (int t = 1; t < n_threads; t++) pthread_join(th[t], NULL);
    return 0;
}

/* n fp32 values mean + sigma*N(0,1). */
void syn_gen_f32(uint64_t seed, uint64_t tid, int64_t n, float mean, float sigma, float* out) {
    for (int64_t i = 0; i < n; i++) out[i] = (float)(mean + sigma * syn_normal(seed, tid, (uint64_t)i));
}

/* n token ids uniform over [0, vocab). */
void syn_gen_tokens(uint64_t seed, uint64_t tid, int64_t n, int vocab, int32_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = (int32_t)(syn_key(seed, tid, (uint64_t)i) % (uint64_t)vocab);
}

/* One layer blob.  Tensor ids: 1 + 16*layer + section. */
int syn_gen_layer(int n_embd, int n_heads, int n_kv_heads, int head_dim, int n_ff, int wtype, uint64_t seed, int layer,
                  float w_sigma, float norm_sigma, uint8_t* blob, int n_threads) {
    uint64_t off[10];
    if (syn_layer_offsets(n_embd, n_heads, n_kv_heads, head_dim, n_ff, wtype, off)) return -1;
    memset(blob, 0, off[9]);
    int64_t E = n_embd, QD = (int64_t)n_heads * head_dim, KVD = (int64_t)n_kv_heads * head_dim, F = n_ff;
    uint64_t t0 = 1 + 16 * (uint64_t)layer;
    syn_gen_f32(seed, t0 + 0, E, 1.f, norm_sigma, (float*)(blob + off[0]));
    syn_gen_matrix(wtype, seed, t0 + 1, QD, E, 0.f, w_sigma, blob + off[1], n_threads);
    syn_gen_matrix(wtype, seed, t0 + 2, KVD, E, 0.f, w_sigma, blob + off[2], n_threads);
    syn_gen_matrix(wtype, seed, t0 + 3, KVD, E, 0.f, w_sigma, blob + off[3], n_threads);
    syn_gen_matrix(wtype, seed, t0 + 4, E, QD, 0.f, w_sigma, blob + off[4], n_threads);
    syn_gen_f32(seed, t0 + 5, E, 1.f, norm_sigma, (float*)(blob + off[5]));
    syn_gen_matrix(wtype, seed, t0 + 6, F, E, 0.f, w_sigma, blob + off[6], n_threads);
    syn_gen_matrix(wtype, seed, t0 + 7, F, E, 0.f, w_sigma, blob + off[7], n_threads);
    syn_gen_matrix(wtype, seed, t0 + 8, E, F, 0.f, w_sigma, blob + off[8], n_threads);
    return 0;
}

/* Exposed for tests of the encoder's fp16 rounding. */
uint16_t syn_f32_to_f16_bits(float f) { return f32_to_f16_bits(f); }
