// CPU ORACLE — test infrastructure only (see oracle.h).  Plain fp64 code that
// follows the pages step by step; no blocking, fusion or reordering beyond a
// split of independent output rows across threads, which leaves every output's
// summation order unchanged (so results do not depend on the thread count).
#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---- number formats ------------------------------------------------------

double f16_to_double(uint16_t h) {
    int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = std::ldexp((double)m, -24);  // subnormal: m * 2^-24
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = std::ldexp((double)(1024 + m), e - 25);  // (1 + m/1024) * 2^(e-15)
    return s ? -v : v;
}

// Nearest binary16 value of x (ties to even), as a double.
double round_f16(double x) {
    if (std::isnan(x) || x == 0.0) return x;
    double a = std::fabs(x);
    if (a >= 65520.0) return std::copysign(INFINITY, x);
    int e;
    std::frexp(a, &e);                        // a = f * 2^e, f in [0.5, 1)
    int q = e - 11;                           // spacing 2^(e-11) for normals (11 significant bits)
    if (q < -24) q = -24;                     // subnormal spacing
    double scaled = std::ldexp(a, -q);        // exact
    double r = std::nearbyint(scaled);        // default rounding mode: ties to even
    return std::copysign(std::ldexp(r, q), x);
}

double round_f32(double x) { return (double)(float)x; }

// ---- GGUF blocks (Shimmy v2.0 Architecture, "Quantization") --------------

size_t block_bytes(int32_t wtype) {
    switch (wtype) {
        case ORC_Q8_0: return 34;
        case ORC_Q4_0: return 18;
        case ORC_Q4_K: return 144;
        case ORC_Q5_K: return 176;
        case ORC_Q6_K: return 210;
        default: return 0;
    }
}

// elements per block: 32, or 256 for the K-quant super-blocks
int64_t block_elems(int32_t wtype) { return (wtype == ORC_Q4_K || wtype == ORC_Q5_K || wtype == ORC_Q6_K) ? 256 : 32; }

// bytes of one row of k elements
size_t row_bytes_of(int32_t wtype, int64_t k) { return (size_t)(k / block_elems(wtype)) * block_bytes(wtype); }

// K-quant super-blocks (Shimmy v2.0 Architecture, "Quantization": "Q4_K_M super-block with row scales",
// "Q6_K super-block, 6-bit"; GPU Inference - dotLLM, "Weight Strategy": Q4_K at about 4.5 bits per weight).
// The pages leave the byte layout to another document, so the published GGUF layout is taken.
//
// Q4_K (144 B per 256 elements): fp16 d, fp16 dmin, 12 bytes holding eight 6-bit scales s_j and eight 6-bit
// mins m_j of the 32-element sub-blocks, then 128 bytes of 4-bit codes.  Element e: sub-block j = e / 32,
// value = d s_j n_e - dmin m_j.
void q4_k_scale_min(const uint8_t* sc, int j, int* s, int* m) {
    if (j < 4) {  // low six bits of bytes j and j + 4
        *s = sc[j] & 63;
        *m = sc[j + 4] & 63;
    } else {  // low four bits from byte j + 4 (s: low nibble, m: high nibble), top two bits from bytes j - 4 / j
        *s = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4);
        *m = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
    }
}

void dequant_q4_k(const uint8_t* b, double* out) {
    const double d = f16_to_double((uint16_t)(b[0] | (b[1] << 8)));
    const double dmin = f16_to_double((uint16_t)(b[2] | (b[3] << 8)));
    const uint8_t* sc = b + 4;
    const uint8_t* qs = b + 16;
    for (int e = 0; e < 256; e++) {
        int s = 0, m = 0;
        q4_k_scale_min(sc, e / 32, &s, &m);
        // 64-element group c shares 32 bytes: the low nibbles are its first 32 elements, the high its last 32
        const int c = e / 64, r = e % 64;
        const uint8_t byte = qs[32 * c + r % 32];
        const int n = r < 32 ? (byte & 15) : (byte >> 4);
        out[e] = d * (double)s * (double)n - dmin * (double)m;
    }
}

// Q5_K (176 B per 256 elements; Shimmy v2.0 Architecture: "Q5_K_M super-block, 5-bit with high-bit plane"):
// fp16 d, fp16 dmin, the 12 bytes of 6-bit scales and mins as in Q4_K, 32 bytes of high bits, 128 bytes of
// low nibbles (placed as Q4_K's).  The high bit of element e (c = e / 64, r = e % 64) is bit 2c + (r >= 32) of
// byte r % 32 of the high-bit plane; the 5-bit code is nibble + 16 * high bit; value = d s_j q_e - dmin m_j.
void dequant_q5_k(const uint8_t* b, double* out) {
    const double d = f16_to_double((uint16_t)(b[0] | (b[1] << 8)));
    const double dmin = f16_to_double((uint16_t)(b[2] | (b[3] << 8)));
    const uint8_t* sc = b + 4;
    const uint8_t* qh = b + 16;
    const uint8_t* qs = b + 48;
    for (int e = 0; e < 256; e++) {
        int s = 0, m = 0;
        q4_k_scale_min(sc, e / 32, &s, &m);
        const int c = e / 64, r = e % 64;
        const uint8_t byte = qs[32 * c + r % 32];
        const int nib = r < 32 ? (byte & 15) : (byte >> 4);
        const int hb = (qh[r % 32] >> (2 * c + (r >= 32 ? 1 : 0))) & 1;
        out[e] = d * (double)s * (double)(nib + 16 * hb) - dmin * (double)m;
    }
}

// Q6_K (210 B per 256 elements): 128 bytes of low 4-bit parts, 64 bytes of high 2-bit parts, sixteen int8
// scales of the 16-element sub-blocks, fp16 d.  Element e: value = d * scale[e / 16] * (q_e - 32).
void dequant_q6_k(const uint8_t* b, double* out) {
    const uint8_t* ql = b;
    const uint8_t* qh = b + 128;
    const int8_t* scale = reinterpret_cast<const int8_t*>(b + 192);
    const double d = f16_to_double((uint16_t)(b[208] | (b[209] << 8)));
    for (int e = 0; e < 256; e++) {
        // half h of 128 elements uses ql[64h ..] and qh[32h ..]; its quarter k (32 elements) takes the low
        // (k < 2) or high (k >= 2) nibbles of ql[64h + 32 (k & 1) ..] and bits 2k, 2k+1 of qh[32h ..]
        const int h = e / 128, k = (e % 128) / 32, l = e % 32;
        const uint8_t lo = ql[64 * h + 32 * (k & 1) + l];
        const int q = (k < 2 ? (lo & 15) : (lo >> 4)) | (((qh[32 * h + l] >> (2 * k)) & 3) << 4);
        out[e] = d * (double)scale[e / 16] * (double)(q - 32);
    }
}

// Q8_0: fp16 scale d, then 32 signed bytes q; element j = d * q_j.
// Q4_0: fp16 scale d, then 16 bytes; element j uses the low nibble of byte j
// (j < 16) or the high nibble of byte j-16 (j >= 16); value = d * (nibble - 8).
void dequant_block(int32_t wtype, const uint8_t* b, double* out) {
    uint16_t dbits = (uint16_t)(b[0] | (b[1] << 8));
    double d = f16_to_double(dbits);
    if (wtype == ORC_Q8_0) {
        for (int j = 0; j < 32; j++) out[j] = d * (double)(int8_t)b[2 + j];
    } else {
        for (int j = 0; j < 16; j++) {
            out[j] = d * (double)((b[2 + j] & 0x0F) - 8);
            out[j + 16] = d * (double)((b[2 + j] >> 4) - 8);
        }
    }
}

void dequant_row(int32_t wtype, const uint8_t* blocks, int64_t k, double* out) {
    const size_t bb = block_bytes(wtype);
    const int64_t be = block_elems(wtype);
    for (int64_t b = 0; b < k / be; b++) {
        if (wtype == ORC_Q4_K)
            dequant_q4_k(blocks + b * bb, out + b * be);
        else if (wtype == ORC_Q5_K)
            dequant_q5_k(blocks + b * bb, out + b * be);
        else if (wtype == ORC_Q6_K)
            dequant_q6_k(blocks + b * bb, out + b * be);
        else
            dequant_block(wtype, blocks + b * bb, out + b * be);
    }
}

// Run f(i) for i in [0, n) over n_threads threads (contiguous ranges).
template <class F>
void parallel_for(int64_t n, int n_threads, F f) {
    if (n_threads <= 1 || n < 2) {
        for (int64_t i = 0; i < n; i++) f(i);
        return;
    }
    if (n_threads > n) n_threads = (int)n;
    std::vector<std::thread> th;
    for (int t = 0; t < n_threads; t++)
        th.emplace_back([&, t] {
            for (int64_t i = n * t / n_threads; i < n * (t + 1) / n_threads; i++) f(i);
        });
    for (auto& x : th) x.join();
}

double dot(const double* a, const double* b, int64_t n) {
    double s = 0.0;
    for (int64_t j = 0; j < n; j++) s += a[j] * b[j];
    return s;
}

// Y[m][i] = W_i . X_m : dequantize weight row i once, then dot it with every input row.
void qgemm(int32_t wtype, const uint8_t* W, int64_t n, int64_t k, const double* X, int64_t M, double* Y,
           int n_threads) {
    const size_t row_bytes = row_bytes_of(wtype, k);
    parallel_for(n, n_threads, [&](int64_t i) {
        std::vector<double> w(k);
        dequant_row(wtype, W + (size_t)i * row_bytes, k, w.data());
        for (int64_t m = 0; m < M; m++) Y[m * n + i] = dot(w.data(), X + m * k, k);
    });
}

void rmsnorm(const double* x, const float* w, int64_t n, double eps, double* y) {
    double ss = 0.0;
    for (int64_t j = 0; j < n; j++) ss += x[j] * x[j];
    double inv = 1.0 / std::sqrt(ss / (double)n + eps);
    for (int64_t j = 0; j < n; j++) y[j] = (double)w[j] * (x[j] * inv);
}

double yarn_scale(int32_t max_ctx, int32_t native_ctx) {
    return (native_ctx > 0 && max_ctx > native_ctx) ? (double)max_ctx / (double)native_ctx : 1.0;
}

// Airframe GPU_PIPELINE.md, RoPE step: theta(t, i) = (t / yarn_scale) / base^(2i / head_dim).
double rope_theta(int64_t t, int32_t i, int32_t head_dim, double base, double ys) {
    return ((double)t / ys) / std::pow(base, (2.0 * i) / (double)head_dim);
}

// Pair (2i, 2i+1) of every head rotated by theta(t, i): [c -s; s c].
void rope(double* v, int32_t n_heads, int32_t head_dim, int64_t t, double base, double ys) {
    for (int32_t h = 0; h < n_heads; h++)
        for (int32_t i = 0; i < head_dim / 2; i++) {
            double th = rope_theta(t, i, head_dim, base, ys);
            double c = std::cos(th), s = std::sin(th);
            double* p = v + (size_t)h * head_dim + 2 * i;
            double a = p[0], b = p[1];
            p[0] = a * c - b * s;
            p[1] = a * s + b * c;
        }
}

// SwiGLU activation on the gate: gate * sigmoid(gate).
double silu(double g) { return g / (1.0 + std::exp(-g)); }

void softmax(double* s, int64_t n) {
    double mx = s[0];
    for (int64_t j = 1; j < n; j++) mx = s[j] > mx ? s[j] : mx;
    double sum = 0.0;
    for (int64_t j = 0; j < n; j++) {
        s[j] = std::exp(s[j] - mx);
        sum += s[j];
    }
    for (int64_t j = 0; j < n; j++) s[j] /= sum;
}

// scores = q_h . K_j / sqrt(head_dim), softmax over j, out_h = sum_j a_j V_j.
// GQA: query head h reads kv head h / (n_heads / n_kv_heads).
void attention(const double* q, int32_t H, int32_t KVH, int32_t D, const double* kc, const double* vc,
               int64_t head_stride, int64_t n_keys, double* out) {
    int32_t group = H / KVH;
    std::vector<double> s(n_keys);
    double scale = 1.0 / std::sqrt((double)D);
    for (int32_t h = 0; h < H; h++) {
        int32_t g = h / group;
        const double* K = kc + (size_t)g * head_stride;
        const double* V = vc + (size_t)g * head_stride;
        for (int64_t j = 0; j < n_keys; j++) s[j] = dot(q + (size_t)h * D, K + (size_t)j * D, D) * scale;
        softmax(s.data(), n_keys);
        for (int32_t d = 0; d < D; d++) {
            double acc = 0.0;
            for (int64_t j = 0; j < n_keys; j++) acc += s[j] * V[(size_t)j * D + d];
            out[(size_t)h * D + d] = acc;
        }
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// ---- quantized KV cache ---------------------------------------------------
// dotLLM, "CUDA components": a quantized KV cache, "Q8_0/Q4_0 + FP16 window".  The pages name the parts only.
// Reading: a slot is written in fp16; once it lies outside the step's window (slot <= b - W, b = the step's
// last position, W = kv_window) it is replaced by the Q8_0 / Q4_0 quantization of its fp16 values, per
// 32-element block along head_dim.  A step (a prefill chunk or a decode step) is never longer than the window
// (n <= W), so a slot retires in a later step than the one that writes it, and every row of a step sees the
// slots of that step in fp16.  The quantizer takes its decisions in fp32 on those fp16 values:
//   Q8_0: d = fp16(max|v| / 127), q = clamp(round-half-away(v / d), -127, 127)  (floor(r + 0.5) in fp32), v' = d q
//   Q4_0: m = the element of largest |v| (first on ties), d = fp16(m / -8),
//         n = clamp(floor(v / d + 8.5), 0, 15), v' = d (n - 8)
// (a zero scale gives zero values).  Every query of the step sees the same representation of a slot.
enum { KV_F32 = 0, KV_F16 = 1, KV_Q8_0 = 2, KV_Q4_0 = 3 };

void quant_kv_row(int32_t kvt, double* v, int64_t D) {
    for (int64_t b0 = 0; b0 < D; b0 += 32) {
        float x[32];
        for (int j = 0; j < 32; j++) x[j] = (float)v[b0 + j];  // fp16 values: exact in fp32
        if (kvt == KV_Q8_0) {
            float amax = 0.f;
            for (int j = 0; j < 32; j++) amax = std::fmax(amax, std::fabs(x[j]));
            const double d = round_f16((double)(amax / 127.f));
            const float df = (float)d;
            for (int j = 0; j < 32; j++) {
                int q = 0;
                if (df != 0.f) {
                    const float r = x[j] / df;
                    q = (int)(r >= 0.f ? std::floor(r + 0.5f) : -std::floor(-r + 0.5f));
                    q = q < -127 ? -127 : (q > 127 ? 127 : q);
                }
                v[b0 + j] = d * (double)q;
            }
        } else {
            float mx = 0.f, amax = 0.f;
            for (int j = 0; j < 32; j++)
                if (std::fabs(x[j]) > amax) {
                    amax = std::fabs(x[j]);
                    mx = x[j];
                }
            const double d = round_f16((double)(mx / -8.f));
            const float df = (float)d;
            for (int j = 0; j < 32; j++) {
                int q = 8;
                if (df != 0.f) {
                    q = (int)std::floor(x[j] / df + 8.5f);
                    q = q < 0 ? 0 : (q > 15 ? 15 : q);
                }
                v[b0 + j] = d * (double)(q - 8);
            }
        }
    }
}

struct orc_model {
    orc_config c;
    std::vector<const uint8_t*> layers;
    const uint8_t* token_embd;
    const float* output_norm;
    const uint8_t* output;
    uint64_t off[10];
    int64_t slots;
    std::vector<double> kcache, vcache;  // [L][KVH][slots][D], values rounded to the cache dtype
    int64_t kv_quantized = 0;            // quantized KV: slots [0, kv_quantized) hold their quantized values
    double ys;
};

extern "C" {

double orc_f16_to_double(uint16_t h) { return f16_to_double(h); }
double orc_round_f16(double x) { return round_f16(x); }
double orc_round_f32(double x) { return round_f32(x); }

int orc_quant_kv_row(int32_t kv_dtype, double* v, int64_t D) {
    if ((kv_dtype != KV_Q8_0 && kv_dtype != KV_Q4_0) || D % 32) return -1;
    quant_kv_row(kv_dtype, v, D);
    return 0;
}

int orc_dequant_row(int32_t wtype, const uint8_t* blocks, int64_t k, double* out) {
    if (!block_bytes(wtype) || k % block_elems(wtype)) return -1;
    dequant_row(wtype, blocks, k, out);
    return 0;
}

int orc_qgemv(int32_t wtype, const uint8_t* W, int64_t n, int64_t k, const double* x, double* y, int n_threads) {
    return orc_qgemm(wtype, W, n, k, x, 1, y, n_threads);
}

int orc_qgemv_rows(int32_t wtype, const uint8_t* W, int64_t k, const int64_t* rows, int64_t n_rows, const double* x,
                   double* y, int n_threads) {
    if (!block_bytes(wtype) || k % block_elems(wtype)) return -1;
    const size_t row_bytes = row_bytes_of(wtype, k);
    parallel_for(n_rows, n_threads, [&](int64_t r) {
        std::vector<double> w(k);
        dequant_row(wtype, W + (size_t)rows[r] * row_bytes, k, w.data());
        y[r] = dot(w.data(), x, k);
    });
    return 0;
}

int orc_qgemm(int32_t wtype, const uint8_t* W, int64_t n, int64_t k, const double* X, int64_t M, double* Y,
              int n_threads) {
    if (!block_bytes(wtype) || k % block_elems(wtype)) return -1;
    qgemm(wtype, W, n, k, X, M, Y, n_threads);
    return 0;
}

void orc_rmsnorm(const double* x, const float* w, int64_t n, double eps, double* y) { rmsnorm(x, w, n, eps, y); }
double orc_yarn_scale(int32_t max_ctx, int32_t native_ctx) { return yarn_scale(max_ctx, native_ctx); }
double orc_rope_theta(int64_t t, int32_t i, int32_t head_dim, double base, double ys) {
    return rope_theta(t, i, head_dim, base, ys);
}
void orc_rope(double* v, int32_t n_heads, int32_t head_dim, int64_t t, double base, double ys) {
    rope(v, n_heads, head_dim, t, base, ys);
}
double orc_silu(double g) { return silu(g); }
void orc_softmax(double* s, int64_t n) { softmax(s, n); }
void orc_attention(const double* q, int32_t H, int32_t KVH, int32_t D, const double* kc, const double* vc,
                   int64_t head_stride, int64_t n_keys, double* out) {
    attention(q, H, KVH, D, kc, vc, head_stride, n_keys, out);
}

int orc_layer_offsets(const orc_config* c, uint64_t off[10]) {
    const int32_t w = c->wtype;
    const int64_t be = block_elems(w);
    if (!block_bytes(w) || c->n_embd % be || c->n_ff % be || (c->n_heads * c->head_dim) % be) return -1;
    if (c->out_wtype && (!block_bytes(c->out_wtype) || c->n_embd % block_elems(c->out_wtype))) return -1;
    size_t E = c->n_embd, QD = (size_t)c->n_heads * c->head_dim, KVD = (size_t)c->n_kv_heads * c->head_dim;
    size_t F = c->n_ff;
    // attn_norm, attn_q, attn_k, attn_v, attn_o, ffn_norm, ffn_gate, ffn_up, ffn_down
    size_t sz[9] = {E * 4, QD * row_bytes_of(w, E), KVD * row_bytes_of(w, E), KVD * row_bytes_of(w, E),
                    E * row_bytes_of(w, QD), E * 4, F * row_bytes_of(w, E), F * row_bytes_of(w, E),
                    E * row_bytes_of(w, F)};
    size_t o = 0;
    for (int i = 0; i < 9; i++) {
        off[i] = o;
        o = align256(o + sz[i]);
    }
    off[9] = o;
    return 0;
}

// Airframe GPU_PIPELINE.md, "KV cache": L * KVH * max_ctx * head_dim * elem, times 2 (K and V).  A quantized
// cache holds every slot twice: in fp16 (as written; a retired slot holds its quantized values there) and in
// the quantized store of 34 (Q8_0) or 18 (Q4_0) bytes per 32 values ("Shimmy v2.0 Architecture",
// Quantization).  The fp16 copy is what prefill attention reads; decode reads the quantized store for retired
// slots, which is where the bandwidth goes.
uint64_t orc_kv_bytes(const orc_config* c) {
    const uint64_t rows = (uint64_t)c->n_layers * c->n_kv_heads * 2;  // K and V
    if (c->kv_f16 == KV_Q8_0 || c->kv_f16 == KV_Q4_0)
        return rows * c->max_ctx *
               ((uint64_t)c->head_dim * 2 + (uint64_t)(c->head_dim / 32) * (c->kv_f16 == KV_Q8_0 ? 34 : 18));
    return rows * c->max_ctx * c->head_dim * (c->kv_f16 ? 2 : 4);
}

orc_model* orc_model_create(const orc_config* c, const uint8_t* const* layer_blobs, const uint8_t* token_embd,
                            const float* output_norm, const uint8_t* output, int64_t kv_slots) {
    if (c->n_heads % c->n_kv_heads || c->head_dim % 2) return nullptr;
    orc_model* m = new orc_model();
    m->c = *c;
    if (orc_layer_offsets(c, m->off)) {
        delete m;
        return nullptr;
    }
    m->layers.assign(layer_blobs, layer_blobs + c->n_layers);
    m->token_embd = token_embd;
    m->output_norm = output_norm;
    m->output = output;
    m->slots = (kv_slots > 0 && kv_slots < c->max_ctx) ? kv_slots : c->max_ctx;
    size_t n = (size_t)c->n_layers * c->n_kv_heads * m->slots * c->head_dim;
    m->kcache.assign(n, 0.0);
    m->vcache.assign(n, 0.0);
    m->ys = yarn_scale(c->max_ctx, c->native_ctx);
    return m;
}

void orc_model_destroy(orc_model* m) { delete m; }

int orc_kv_read(const orc_model* m, int32_t layer, int32_t kvh, int64_t pos, double* k, double* v) {
    const orc_config& c = m->c;
    if (layer < 0 || layer >= c.n_layers || kvh < 0 || kvh >= c.n_kv_heads || pos < 0 || pos >= m->slots) return -1;
    size_t base = (((size_t)layer * c.n_kv_heads + kvh) * m->slots + pos) * c.head_dim;
    std::memcpy(k, &m->kcache[base], sizeof(double) * c.head_dim);
    std::memcpy(v, &m->vcache[base], sizeof(double) * c.head_dim);
    return 0;
}

int orc_kv_write(orc_model* m, int32_t layer, int32_t kvh, int64_t pos0, int64_t n, const double* k,
                 const double* v) {
    const orc_config& c = m->c;
    if (layer < 0 || layer >= c.n_layers || kvh < 0 || kvh >= c.n_kv_heads || pos0 < 0 || n < 0 ||
        pos0 + n > m->slots)
        return -1;
    const size_t base = (((size_t)layer * c.n_kv_heads + kvh) * m->slots + pos0) * c.head_dim;
    std::memcpy(&m->kcache[base], k, sizeof(double) * c.head_dim * n);
    std::memcpy(&m->vcache[base], v, sizeof(double) * c.head_dim * n);
    return 0;
}

int64_t orc_argmax(const double* v, int64_t n) {
    int64_t best = 0;
    for (int64_t i = 1; i < n; i++)
        if (v[i] > v[best]) best = i;
    return best;
}

// Sampler chain (Airframe GPU pipeline, "sampling applies these transformations
// in order"): repetition penalty, temperature, softmax, top-p, sample.  Readings:
// the penalty divides each distinct recent token's logit once; temperature 0 is
// greedy (argmax, lowest index on ties); the nucleus is the shortest prefix of
// the tokens sorted by (probability descending, index ascending) whose sum
// reaches top_p, extended by every token tied with its last one (top_p >= 1
// keeps everything); the sample is the first token of that order whose
// cumulative mass reaches u times the nucleus mass (u in [0, 1) is the caller's
// uniform draw).  *lo / *hi receive the token's cumulative mass interval
// (before, after) as a fraction of the nucleus mass.
namespace {

// The sampler's distribution: penalized, temperature-scaled softmax probabilities p, the order
// (probability descending, index ascending) and the nucleus length.  temperature > 0.
struct SampleDist {
    std::vector<double> p;
    std::vector<int64_t> order;
    int64_t kept = 0;
    double zk = 0.0;
};

std::vector<double> penalized(const double* logits, int64_t V, const int32_t* recent, int64_t n_recent,
                              double repeat_penalty) {
    std::vector<double> l(logits, logits + V);
    if (repeat_penalty > 1.0) {
        for (int64_t i = 0; i < n_recent; i++) {
            const int32_t t = recent[i];
            if (t < 0 || t >= V) continue;
            bool seen = false;
            for (int64_t j = 0; j < i; j++) seen = seen || recent[j] == t;
            if (!seen) l[t] /= repeat_penalty;
        }
    }
    return l;
}

SampleDist sample_dist(std::vector<double> l, double temperature, double top_p) {
    const int64_t V = (int64_t)l.size();
    SampleDist d;
    double mx = -INFINITY;
    for (int64_t i = 0; i < V; i++) {
        l[i] /= temperature;
        mx = std::fmax(mx, l[i]);
    }
    d.p.resize(V);
    double z = 0.0;
    for (int64_t i = 0; i < V; i++) {
        d.p[i] = std::exp(l[i] - mx);
        z += d.p[i];
    }
    for (int64_t i = 0; i < V; i++) d.p[i] /= z;
    d.order.resize(V);
    for (int64_t i = 0; i < V; i++) d.order[i] = i;
    const std::vector<double>& p = d.p;
    std::sort(d.order.begin(), d.order.end(),
              [&](int64_t a, int64_t b) { return p[a] > p[b] || (p[a] == p[b] && a < b); });
    d.kept = V;
    if (top_p < 1.0) {
        double c = 0.0;
        for (int64_t k = 0; k < V; k++) {
            c += p[d.order[k]];
            if (c >= top_p) {
                d.kept = k + 1;
                break;
            }
        }
        while (d.kept < V && p[d.order[d.kept]] == p[d.order[d.kept - 1]]) d.kept++;
    }
    for (int64_t k = 0; k < d.kept; k++) d.zk += p[d.order[k]];
    return d;
}

}  // namespace

int64_t orc_sample(const double* logits, int64_t V, const int32_t* recent, int64_t n_recent, double repeat_penalty,
                   double temperature, double top_p, double u, double* lo, double* hi) {
    std::vector<double> l = penalized(logits, V, recent, n_recent, repeat_penalty);
    if (temperature <= 0.0) {
        if (lo) *lo = 0.0;
        if (hi) *hi = 1.0;
        return orc_argmax(l.data(), V);
    }
    const SampleDist d = sample_dist(std::move(l), temperature, top_p);
    const double target = u * d.zk;
    double c = 0.0;
    for (int64_t k = 0; k < d.kept; k++) {
        const double before = c;
        c += d.p[d.order[k]];
        if (c >= target || k == d.kept - 1) {
            if (lo) *lo = before / d.zk;
            if (hi) *hi = c / d.zk;
            return d.order[k];
        }
    }
    return d.order[0];
}

int orc_sample_interval(const double* logits, int64_t V, const int32_t* recent, int64_t n_recent,
                        double repeat_penalty, double temperature, double top_p, int64_t token, double* lo,
                        double* hi, double* p_token, double* p_boundary) {
    if (token < 0 || token >= V || temperature <= 0.0) return -1;
    const SampleDist d = sample_dist(penalized(logits, V, recent, n_recent, repeat_penalty), temperature, top_p);
    double c = 0.0;
    int in_nucleus = 0;
    for (int64_t k = 0; k < V; k++) {
        const double before = c;
        c += d.p[d.order[k]];
        if (d.order[k] == token) {
            *lo = before / d.zk;
            *hi = c / d.zk;
            in_nucleus = k < d.kept;
            break;
        }
    }
    *p_token = d.p[token];
    *p_boundary = d.p[d.order[d.kept - 1]];
    return in_nucleus;
}

// Forward pass over n tokens at positions start_pos.. (Airframe per-layer op
// order; a decode step is the case n = 1).  All rows write their K/V before any
// row attends; row r attends to cache slots 0..start_pos+r (causal).
int orc_forward(orc_model* m, const int32_t* tokens, int64_t n, int64_t start_pos, double* logits, double* capture,
                int n_threads) {
    const orc_config& c = m->c;
    if (n <= 0 || start_pos < 0 || start_pos + n > m->slots) return -1;
    for (int64_t r = 0; r < n; r++)
        if (tokens[r] < 0 || tokens[r] >= c.n_vocab) return -2;
    const int64_t E = c.n_embd, H = c.n_heads, KVH = c.n_kv_heads, D = c.head_dim, F = c.n_ff;
    const int64_t QD = H * D, KVD = KVH * D;
    const int32_t head_wtype = c.out_wtype ? c.out_wtype : c.wtype;
    const bool quantized_kv = c.kv_f16 == KV_Q8_0 || c.kv_f16 == KV_Q4_0;
    if (quantized_kv && n > c.kv_window) return -3;  // a step longer than the window (see the reading above)
    const int64_t retire_to = start_pos + n - 1 - c.kv_window;  // last slot outside this step's window

    std::vector<double> X(n * E), Y(n * E), Q(n * QD), K(n * KVD), V(n * KVD), A(n * QD), O(n * E);
    std::vector<double> G(n * F), U(n * F), Hh(n * F);

    // embedding lookup: dequantized row of token_embd
    for (int64_t r = 0; r < n; r++)
        dequant_row(c.wtype, m->token_embd + (size_t)tokens[r] * row_bytes_of(c.wtype, E), E, &X[r * E]);
    if (capture) std::memcpy(capture, X.data(), sizeof(double) * n * E);

    for (int32_t l = 0; l < c.n_layers; l++) {
        const uint8_t* blob = m->layers[l];
        const float* attn_norm = (const float*)(blob + m->off[0]);
        const uint8_t* Wq = blob + m->off[1];
        const uint8_t* Wk = blob + m->off[2];
        const uint8_t* Wv = blob + m->off[3];
        const uint8_t* Wo = blob + m->off[4];
        const float* ffn_norm = (const float*)(blob + m->off[5]);
        const uint8_t* Wg = blob + m->off[6];
        const uint8_t* Wu = blob + m->off[7];
        const uint8_t* Wd = blob + m->off[8];

        for (int64_t r = 0; r < n; r++) rmsnorm(&X[r * E], attn_norm, E, c.rms_eps, &Y[r * E]);
        qgemm(c.wtype, Wq, QD, E, Y.data(), n, Q.data(), n_threads);
        qgemm(c.wtype, Wk, KVD, E, Y.data(), n, K.data(), n_threads);
        qgemm(c.wtype, Wv, KVD, E, Y.data(), n, V.data(), n_threads);
        for (int64_t r = 0; r < n; r++) {
            rope(&Q[r * QD], (int32_t)H, (int32_t)D, start_pos + r, c.rope_base, m->ys);
            rope(&K[r * KVD], (int32_t)KVH, (int32_t)D, start_pos + r, c.rope_base, m->ys);
        }
        // KV write at position t, rounded to the cache's element type
        for (int64_t r = 0; r < n; r++)
            for (int64_t g = 0; g < KVH; g++)
                for (int64_t d = 0; d < D; d++) {
                    size_t idx = (((size_t)l * KVH + g) * m->slots + start_pos + r) * D + d;
                    double kv = K[r * KVD + g * D + d], vv = V[r * KVD + g * D + d];
                    m->kcache[idx] = c.kv_f16 ? round_f16(kv) : round_f32(kv);  // quantized caches: fp16 first
                    m->vcache[idx] = c.kv_f16 ? round_f16(vv) : round_f32(vv);
                }
        if (quantized_kv)  // slots that left this step's window take their quantized values
            for (int64_t sl = m->kv_quantized; sl <= retire_to; sl++)
                for (int64_t g = 0; g < KVH; g++) {
                    const size_t row = (((size_t)l * KVH + g) * m->slots + sl) * D;
                    quant_kv_row(c.kv_f16, &m->kcache[row], D);
                    quant_kv_row(c.kv_f16, &m->vcache[row], D);
                }
        const double* kc = &m->kcache[(size_t)l * KVH * m->slots * D];
        const double* vc = &m->vcache[(size_t)l * KVH * m->slots * D];
        parallel_for(n, n_threads, [&](int64_t r) {
            attention(&Q[r * QD], (int32_t)H, (int32_t)KVH, (int32_t)D, kc, vc, m->slots * D, start_pos + r + 1,
                      &A[r * QD]);
        });
        qgemm(c.wtype, Wo, E, QD, A.data(), n, O.data(), n_threads);
        for (int64_t i = 0; i < n * E; i++) X[i] += O[i];

        for (int64_t r = 0; r < n; r++) rmsnorm(&X[r * E], ffn_norm, E, c.rms_eps, &Y[r * E]);
        qgemm(c.wtype, Wg, F, E, Y.data(), n, G.data(), n_threads);
        qgemm(c.wtype, Wu, F, E, Y.data(), n, U.data(), n_threads);
        for (int64_t i = 0; i < n * F; i++) Hh[i] = silu(G[i]) * U[i];
        qgemm(c.wtype, Wd, E, F, Hh.data(), n, O.data(), n_threads);
        for (int64_t i = 0; i < n * E; i++) X[i] += O[i];
        if (capture) std::memcpy(capture + (size_t)(l + 1) * n * E, X.data(), sizeof(double) * n * E);
    }
    if (logits) {
        // final RMS norm on the last position only, then the LM head
        std::vector<double> last(E);
        rmsnorm(&X[(n - 1) * E], m->output_norm, E, c.rms_eps, last.data());
        qgemm(head_wtype, m->output, c.n_vocab, E, last.data(), 1, logits, n_threads);
    }
    if (quantized_kv && retire_to + 1 > m->kv_quantized) m->kv_quantized = retire_to + 1;
    return 0;
}

}  // extern "C"
