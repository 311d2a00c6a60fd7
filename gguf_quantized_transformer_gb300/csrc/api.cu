// C ABI (include/af.h): validation, weight repacking, buffers and the launch
// sequences of prefill and decode.
//
// Launch sequence per layer (Airframe "GPU_PIPELINE.md" per-layer ops; dotLLM
// "GPU Inference", "Forward Pass" and "Synchronization Model": one stream, no
// host sync inside the pass):
//   decode : GEMV[RMSNorm | QKV -> RoPE -> q, KV write]  -> attention(split-KV)
//            -> GEMV[O -> x +=] -> GEMV[RMSNorm | gate,up -> SwiGLU]
//            -> GEMV[down -> x +=];  head: GEMV[RMSNorm | LM head -> logits, argmax]
//   prefill: RMSNorm rows -> GEMM[QKV -> RoPE, KV write] -> causal attention
//            -> GEMM[O -> x +=] -> RMSNorm rows -> GEMM[gate,up -> SwiGLU]
//            -> GEMM[down -> x +=]; LM head on the last row only.
// The decode step after its first kernel is captured once into a CUDA graph
// (position and token are read from device memory, so the graph is reused).
#include <algorithm>
#include <cstdarg>
#include <new>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"

using namespace af;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

#define CK(call)                                                                                 \
    do {                                                                                         \
        cudaError_t e_ = (call);                                                                 \
        if (e_ != cudaSuccess) return fail(AF_ECUDA, "%s: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                                           __FILE__, __LINE__);                                  \
    } while (0)

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t block_bytes(int wtype) {
    switch (wtype) {
        case AF_Q8_0: return 34;
        case AF_Q4_0: return 18;
        case AF_Q4_K: return 144;
        case AF_Q5_K: return 176;
        case AF_Q6_K: return 210;
        default: return 0;
    }
}

// bytes of one GGUF row of k weights
size_t row_bytes(int wtype, size_t k) { return k / (size_t)block_elems(wtype) * block_bytes(wtype); }

int head_wtype(const af_config* c) { return c->out_wtype ? c->out_wtype : c->wtype; }

bool kv_quantized(const af_config* c) { return c->kv_dtype == AF_KV_Q8_0 || c->kv_dtype == AF_KV_Q4_0; }

// bytes of one element of the (fp32 / fp16) cache; a quantized cache keeps an fp16 copy of every slot
size_t kv_elem(const af_config* c) { return c->kv_dtype == AF_F32 ? 4 : 2; }

// Tracks device allocations of one object so a failed create frees everything.
struct Allocs {
    std::vector<void*> p;
    void* get(size_t bytes) {
        void* q = nullptr;
        if (cudaMalloc(&q, bytes ? bytes : 1) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        p.push_back(q);
        return q;
    }
    void release(void* q) {
        for (auto& e : p)
            if (e == q) {
                cudaFree(e);
                e = nullptr;
            }
    }
    void free_all() {
        for (void* q : p) cudaFree(q);
        p.clear();
    }
};

Planes make_planes(Allocs& A, int wtype, int N, int K) {
    Planes P;
    size_t sc_off = 0;
    size_t total = planes_bytes(wtype, N, K, &sc_off);
    uint8_t* buf = (uint8_t*)A.get(total);
    if (!buf) return P;
    P.qs = buf;
    P.sc = (const __half*)(buf + sc_off);
    P.N = N;
    P.K = K;
    P.Kp = padded_k(wtype, K);
    P.wtype = wtype;
    return P;
}

cudaError_t repack_into(const Planes& P, const void* src, int N, int row0, int step, cudaStream_t s) {
    return launch_repack((const uint8_t*)src, P, N, row0, step, s);
}

struct LayerW {
    Planes qkv, o, gu, down;
    const float* attn_norm = nullptr;
    const float* ffn_norm = nullptr;
};

Epi epi_simple(int kind, float* out, int ld) {
    Epi e;
    e.kind = kind;
    e.out = out;
    e.ld = ld;
    return e;
}

int check_config(const af_config* c) {
    if (!c) return fail(AF_EINVAL, "null config");
    if (!block_bytes(c->wtype)) return fail(AF_EINVAL, "wtype must be AF_Q4_0, AF_Q8_0, AF_Q4_K, AF_Q5_K or AF_Q6_K");
    if (!block_bytes(head_wtype(c))) return fail(AF_EINVAL, "bad out_wtype");
    if (c->kv_dtype != AF_F32 && c->kv_dtype != AF_F16 && !kv_quantized(c))
        return fail(AF_EINVAL, "kv_dtype must be AF_F32, AF_F16, AF_KV_Q8_0 or AF_KV_Q4_0");
    if (c->n_layers <= 0 || c->n_embd <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
        c->n_ff <= 0 || c->n_vocab <= 0 || c->max_ctx <= 0)
        return fail(AF_EINVAL, "all sizes must be positive");
    if (c->max_chunk < 0 || c->native_ctx < 0) return fail(AF_EINVAL, "negative max_chunk / native_ctx");
    {
        const int be = std::max(block_elems(c->wtype), block_elems(head_wtype(c)));
        if (c->n_embd % be || c->n_ff % block_elems(c->wtype) || (c->n_heads * c->head_dim) % block_elems(c->wtype))
            return fail(AF_EINVAL, "n_embd, n_ff and n_heads*head_dim must be whole GGUF blocks (%d weights)", be);
    }
    if (c->n_heads % c->n_kv_heads) return fail(AF_EINVAL, "n_heads must be a multiple of n_kv_heads");
    if (!(c->rms_eps >= 0.f) || !(c->rope_base > 0.f)) return fail(AF_EINVAL, "bad rms_eps / rope_base");
    if (!attn_supported(c->n_heads, c->n_kv_heads, c->head_dim))
        return fail(AF_ENOTIMPL, "attention supports head_dim 64/128 and group size 1/2/4/8");
    if (kv_quantized(c)) {
        const int chunk = c->max_chunk ? c->max_chunk : 512;
        if (c->kv_window < chunk)
            return fail(AF_EINVAL, "kv_window (%d) must be at least max_chunk (%d): a step may not outrun the window",
                        c->kv_window, chunk);
        if (c->max_ctx % 4) return fail(AF_ENOTIMPL, "a quantized cache needs max_ctx a multiple of 4");
    }
    if (c->n_embd % 64 || c->n_ff % 64 || (c->n_heads * c->head_dim) % 64 || c->n_vocab % 2)
        return fail(AF_ENOTIMPL, "n_embd, n_ff, n_heads*head_dim must be multiples of 64 and n_vocab even");
    {
        const int kmax = std::max(std::max(c->n_embd, c->n_ff), c->n_heads * c->head_dim);
        if (padded_k(c->wtype, kmax) / chunk_weights(c->wtype) > qgemv_max_chunks())
            return fail(AF_ENOTIMPL, "matrix rows longer than %d weights", qgemv_max_chunks() * chunk_weights(c->wtype));
        if (padded_k(head_wtype(c), c->n_embd) / chunk_weights(head_wtype(c)) > qgemv_max_chunks())
            return fail(AF_ENOTIMPL, "LM head rows longer than %d weights",
                        qgemv_max_chunks() * chunk_weights(head_wtype(c)));
    }
    return AF_OK;
}

}  // namespace

struct af_model {
    af_config c{};
    cudaStream_t s = nullptr;
    bool own_stream = false;
    Allocs A;
    std::vector<LayerW> L;
    Planes emb, out;
    const float* out_norm = nullptr;
    void* kc = nullptr;
    void* vc = nullptr;
    size_t kv_layer_elems = 0;
    float2* rope = nullptr;
    int chunk = 512;
    float* x = nullptr;      // [chunk][E] residual stream
    float* q = nullptr;      // [chunk][H*D] rotated q
    float* attn = nullptr;   // [H*D] decode attention output
    float* h = nullptr;      // [F] decode SwiGLU output
    __half* y16[2] = {};     // [chunk][E] normalized activations, fp16 hi / lo (GEMM operand)
    __half* a16[2] = {};     // [chunk][H*D] attention output, fp16 hi / lo
    __half* h16[2] = {};     // [chunk][F] SwiGLU output, fp16 hi / lo
    int* tok = nullptr;      // [chunk]
    int* tok_host = nullptr;  // [chunk] page-locked staging of af_prefill's token ids
    cudaEvent_t tok_ev = nullptr;  // the copy out of tok_host has completed
    float* logits = nullptr; // [V] default logits
    GemvScratch gs;
    AttnScratch as;
    GemmSplit gsplit;  // split-K scratch of the prefill GEMMs
    StepState* st = nullptr;
    float* capture = nullptr;
    unsigned long long* trace = nullptr;
    bool use_graph = true;
    int decode_mode = AF_DECODE_KERNELS;
    DecodePlan dplan;
    LayerPlan* d_layers = nullptr;
    bool persistent_ok = false;
    cudaGraphExec_t gexec = nullptr;
    float* graph_logits = nullptr;
    unsigned err_host = 0;

    int E() const { return c.n_embd; }
    int QD() const { return c.n_heads * c.head_dim; }
    int KVD() const { return c.n_kv_heads * c.head_dim; }
    KvStore kvq;  // quantized store (kvq.qtype == 0: the cache is not quantized)

    void* kl(int l) const { return (char*)kc + (size_t)l * kv_layer_elems * kv_elem(&c); }
    void* vl(int l) const { return (char*)vc + (size_t)l * kv_layer_elems * kv_elem(&c); }
    KvLayerStore kvq_layer(int l) const {
        KvLayerStore q;
        if (!kvq.qtype) return q;
        const size_t rows = (size_t)l * kv_layer_elems / c.head_dim;  // slot rows before layer l
        const int cb = kv_code_bytes(kvq.qtype, c.head_dim);
        q.kq = kvq.kq + rows * cb;
        q.vq = kvq.vq + rows * cb;
        q.ks = kvq.ks + rows * (c.head_dim / 32);
        q.vs = kvq.vs + rows * (c.head_dim / 32);
        q.qtype = kvq.qtype;
        q.window = kvq.window;
        return q;
    }
};

namespace {
Epi epi_qkv_plan(af_model* m, int l) {
    Epi e;
    e.kind = EPI_QKV;
    e.out = m->q;
    e.ld = m->QD();
    e.qd = m->QD();
    e.kvd = m->KVD();
    e.head_dim = m->c.head_dim;
    e.max_ctx = m->c.max_ctx;
    e.kv_f16 = m->c.kv_dtype != AF_F32;
    e.kcache = m->kl(l);
    e.vcache = m->vl(l);
    e.rope = m->rope;
    return e;
}
}  // namespace

namespace {
// Synchronise the model's stream and report its error word; a reported error is cleared, so only calls that
// ran after the report can raise it again.
int read_err(af_model* m) {
    CK(cudaMemcpyAsync(&m->err_host, m->gs.err, 4, cudaMemcpyDeviceToHost, m->s));
    CK(cudaStreamSynchronize(m->s));
    if (m->err_host) {
        const unsigned code = m->err_host;
        CK(cudaMemsetAsync(m->gs.err, 0, 4, m->s));
        CK(cudaStreamSynchronize(m->s));
        return fail(AF_ETIMEOUT, "a bounded device-side wait gave up (code %u)", code);
    }
    return AF_OK;
}
}  // namespace

struct af_qweight {
    Planes p;
    Allocs A;
    GemvScratch gs;
    GemmSplit gsplit;  // split-K scratch of af_qgemm (sized for 512 rows; calls on one weight are serialized)
    __half* x16[2] = {};  // af_qgemm operand: X as fp16 hi / lo, grown on demand
    int x16_rows = 0;
};

extern "C" {

const char* af_last_error(void) { return g_err.c_str(); }

int af_layer_offsets(const af_config* c, uint64_t off[10]) {
    if (!c || !off) return fail(AF_EINVAL, "null argument");
    const int wt = c->wtype;
    if (!block_bytes(wt)) return fail(AF_EINVAL, "bad wtype");
    const int be = block_elems(wt);
    if (c->n_embd <= 0 || c->n_ff <= 0 || c->n_heads <= 0 || c->head_dim <= 0 || c->n_kv_heads <= 0 ||
        c->n_embd % be || c->n_ff % be || (c->n_heads * c->head_dim) % be)
        return fail(AF_EINVAL, "bad shape");
    const size_t E = c->n_embd, QD = (size_t)c->n_heads * c->head_dim, KVD = (size_t)c->n_kv_heads * c->head_dim;
    const size_t F = c->n_ff;
    const size_t sz[9] = {E * 4, QD * row_bytes(wt, E), KVD * row_bytes(wt, E), KVD * row_bytes(wt, E),
                          E * row_bytes(wt, QD), E * 4, F * row_bytes(wt, E), F * row_bytes(wt, E),
                          E * row_bytes(wt, F)};
    size_t o = 0;
    for (int i = 0; i < 9; i++) {
        off[i] = o;
        o = al256(o + sz[i]);
    }
    off[9] = o;
    return AF_OK;
}

uint64_t af_kv_bytes(const af_config* c) {
    if (!c || c->n_layers <= 0 || c->n_kv_heads <= 0 || c->max_ctx <= 0 || c->head_dim <= 0) return 0;
    const uint64_t rows = (uint64_t)c->n_layers * c->n_kv_heads * 2;
    if (kv_quantized(c)) {
        if (c->head_dim % 32) return 0;
        return rows * c->max_ctx *
               ((uint64_t)c->head_dim * 2 + (uint64_t)(c->head_dim / 32) * (c->kv_dtype == AF_KV_Q8_0 ? 34 : 18));
    }
    if (c->kv_dtype != AF_F32 && c->kv_dtype != AF_F16) return 0;
    return rows * c->max_ctx * c->head_dim * (c->kv_dtype == AF_F16 ? 2 : 4);
}

void af_model_destroy(af_model* m) {
    if (!m) return;
    if (m->gexec) cudaGraphExecDestroy(m->gexec);
    if (m->s) cudaStreamSynchronize(m->s);
    if (m->tok_ev) cudaEventDestroy(m->tok_ev);
    if (m->tok_host) cudaFreeHost(m->tok_host);
    m->A.free_all();
    if (m->own_stream) cudaStreamDestroy(m->s);
    delete m;
}

int af_model_create(const af_config* cfg, const af_weights* w, void* stream, af_model** out) {
    if (!out) return fail(AF_EINVAL, "null out");
    *out = nullptr;
    int rc = check_config(cfg);
    if (rc) return rc;
    if (!w || !w->layer_blob || !w->token_embd || !w->output_norm || !w->output)
        return fail(AF_EINVAL, "null weight pointer");
    for (int l = 0; l < cfg->n_layers; l++)
        if (!w->layer_blob[l]) return fail(AF_EINVAL, "null layer blob %d", l);
    uint64_t off[10];
    af_layer_offsets(cfg, off);

    af_model* m = new (std::nothrow) af_model();
    if (!m) return fail(AF_ENOMEM, "host allocation failed");
    m->c = *cfg;
    if (m->c.max_chunk == 0) m->c.max_chunk = 512;
    m->chunk = m->c.max_chunk;
    m->s = (cudaStream_t)stream;
    if (!m->s) {  // a blocking stream of our own: ordered with the legacy default stream, and capturable
        if (cudaStreamCreate(&m->s) != cudaSuccess) {
            cudaGetLastError();
            delete m;
            return fail(AF_ECUDA, "cudaStreamCreate failed");
        }
        m->own_stream = true;
    }
    const af_config& c = m->c;
    const int E = c.n_embd, QD = m->QD(), KVD = m->KVD(), F = c.n_ff, V = c.n_vocab, D = c.head_dim;
    const int wt = c.wtype;
    cudaStream_t s = m->s;
    Allocs& A = m->A;
    auto oom = [&](const char* what) {
        m->A.free_all();
        if (m->own_stream) cudaStreamDestroy(m->s);
        delete m;
        return fail(AF_ENOMEM, "device allocation failed: %s", what);
    };
    auto cuda_fail = [&](cudaError_t e, const char* what) {
        cudaStreamSynchronize(m->s);
        m->A.free_all();
        if (m->own_stream) cudaStreamDestroy(m->s);
        delete m;
        return fail(AF_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    };

    // weights
    m->L.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; l++) {
        LayerW& lw = m->L[l];
        const uint8_t* blob = (const uint8_t*)w->layer_blob[l];
        lw.qkv = make_planes(A, wt, QD + 2 * KVD, E);
        lw.o = make_planes(A, wt, E, QD);
        lw.gu = make_planes(A, wt, 2 * F, E);
        lw.down = make_planes(A, wt, E, F);
        float* norms = (float*)A.get(2 * al256((size_t)E * 4));
        if (!lw.qkv.qs || !lw.o.qs || !lw.gu.qs || !lw.down.qs || !norms) return oom("layer weights");
        lw.attn_norm = norms;
        lw.ffn_norm = (const float*)((char*)norms + al256((size_t)E * 4));
        cudaError_t e = cudaSuccess;
        if (!e) e = cudaMemcpyAsync(norms, blob + off[0], (size_t)E * 4, cudaMemcpyDeviceToDevice, s);
        if (!e) e = cudaMemcpyAsync((void*)lw.ffn_norm, blob + off[5], (size_t)E * 4, cudaMemcpyDeviceToDevice, s);
        if (!e) e = repack_into(lw.qkv, blob + off[1], QD, 0, 1, s);
        if (!e) e = repack_into(lw.qkv, blob + off[2], KVD, QD, 1, s);
        if (!e) e = repack_into(lw.qkv, blob + off[3], KVD, QD + KVD, 1, s);
        if (!e) e = repack_into(lw.o, blob + off[4], E, 0, 1, s);
        if (!e) e = repack_into(lw.gu, blob + off[6], F, 0, 2, s);  // gate rows -> even
        if (!e) e = repack_into(lw.gu, blob + off[7], F, 1, 2, s);  // up rows   -> odd
        if (!e) e = repack_into(lw.down, blob + off[8], E, 0, 1, s);
        if (e) return cuda_fail(e, "weight repack");
    }
    m->emb = make_planes(A, wt, V, E);
    m->out = make_planes(A, head_wtype(&c), V, E);
    float* onorm = (float*)A.get((size_t)E * 4);
    if (!m->emb.qs || !m->out.qs || !onorm) return oom("embedding / output");
    m->out_norm = onorm;
    {
        cudaError_t e = repack_into(m->emb, w->token_embd, V, 0, 1, s);
        if (!e) e = repack_into(m->out, w->output, V, 0, 1, s);
        if (!e) e = cudaMemcpyAsync(onorm, w->output_norm, (size_t)E * 4, cudaMemcpyDeviceToDevice, s);
        if (e) return cuda_fail(e, "output repack");
    }

    // KV cache, RoPE table
    m->kv_layer_elems = (size_t)c.n_kv_heads * c.max_ctx * D;
    const size_t kvb = (size_t)c.n_layers * m->kv_layer_elems * kv_elem(&c);  // K (or V) cache, fp16 when quantized
    m->kc = A.get(kvb);
    m->vc = A.get(kvb);
    m->rope = (float2*)A.get((size_t)c.max_ctx * (D / 2) * sizeof(float2));
    if (!m->kc || !m->vc || !m->rope) return oom("KV cache");
    if (kv_quantized(&c)) {  // the quantized store: codes and scales of every slot row
        const size_t rows = (size_t)c.n_layers * c.n_kv_heads * c.max_ctx;
        const int cb = kv_code_bytes(c.kv_dtype, D);
        m->kvq.qtype = c.kv_dtype;
        m->kvq.window = c.kv_window;
        m->kvq.kq = (uint8_t*)A.get(rows * cb);
        m->kvq.vq = (uint8_t*)A.get(rows * cb);
        m->kvq.ks = (__half*)A.get(rows * (D / 32) * 2);
        m->kvq.vs = (__half*)A.get(rows * (D / 32) * 2);
        if (!m->kvq.kq || !m->kvq.vq || !m->kvq.ks || !m->kvq.vs) return oom("quantized KV store");
    }
    const double ys = (c.native_ctx > 0 && c.max_ctx > c.native_ctx) ? (double)c.max_ctx / c.native_ctx : 1.0;
    {
        cudaError_t e = cudaMemsetAsync(m->kc, 0, kvb, s);
        if (!e) e = cudaMemsetAsync(m->vc, 0, kvb, s);
        if (!e) e = launch_rope_table(m->rope, c.max_ctx, D, (double)c.rope_base, ys, s);
        if (e) return cuda_fail(e, "KV init");
    }

    // activations and scratch
    const int S = m->chunk;
    m->x = (float*)A.get((size_t)S * E * 4);
    m->q = (float*)A.get((size_t)S * QD * 4);
    m->attn = (float*)A.get((size_t)QD * 4);
    m->h = (float*)A.get((size_t)F * 4);
    for (int i = 0; i < 2; i++) {
        m->y16[i] = (__half*)A.get((size_t)S * E * 2);
        m->a16[i] = (__half*)A.get((size_t)S * QD * 2);
        m->h16[i] = (__half*)A.get((size_t)S * F * 2);
    }
    m->tok = (int*)A.get((size_t)S * 4);
    m->logits = (float*)A.get((size_t)V * 4);
    m->st = (StepState*)A.get(sizeof(StepState));
    m->gs.err = (unsigned*)A.get(kErrWords * sizeof(unsigned));
    m->as.ns = std::max(attn_decode_splits(c.n_heads, c.n_kv_heads, c.max_ctx), decode_attn_splits(c.n_kv_heads));
    m->as.part = (float*)A.get(attn_decode_part_elems(c.n_heads, D, m->as.ns) * 4);
    m->as.cnt = (unsigned*)A.get((size_t)c.n_kv_heads * 4);
    m->as.err = m->gs.err;
    {  // split-K scratch: the largest any layer GEMM wants at a full chunk
        const int NK[4][2] = {{QD + 2 * m->KVD(), E}, {E, QD}, {2 * F, E}, {E, F}};
        size_t ws = 0;
        int tiles = 0;
        for (const auto& nk : NK) {
            ws = std::max(ws, qgemm_ws_bytes(nk[0], nk[1], S));
            tiles = std::max(tiles, qgemm_tiles(nk[0], S));
        }
        if (ws) {
            m->gsplit.ws = (float*)A.get(ws);
            m->gsplit.ws_bytes = m->gsplit.ws ? ws : 0;
            m->gsplit.cnt = (unsigned*)A.get((size_t)tiles * 4);
            m->gsplit.cnt_n = m->gsplit.cnt ? tiles : 0;
        }
    }
    if (!m->x || !m->q || !m->attn || !m->h || !m->y16[0] || !m->y16[1] || !m->a16[0] || !m->a16[1] || !m->h16[0] || !m->h16[1] || !m->tok || !m->logits || !m->st ||
        !m->gs.err || !m->as.part || !m->as.cnt)
        return oom("activations");
    // persistent decode plan: per-layer GEMV tasks on the device, barrier words
    unsigned* words = (unsigned*)A.get(4 * sizeof(unsigned));
    m->d_layers = (LayerPlan*)A.get(sizeof(LayerPlan) * c.n_layers);
    if (!words || !m->d_layers) return oom("decode plan");
    {
        DecodePlan& P = m->dplan;
        P.wtype = wt;
        P.n_layers = c.n_layers;
        P.H = c.n_heads;
        P.KVH = c.n_kv_heads;
        P.D = D;
        P.max_ctx = c.max_ctx;
        P.kv_f16 = c.kv_dtype == AF_F16;
        P.attn_splits = std::min(decode_attn_splits(c.n_kv_heads), m->as.ns);  // within the partials buffer
        P.eps = c.rms_eps;
        P.layers = m->d_layers;
        P.emb = m->emb;
        P.x = m->x;
        P.q = m->q;
        P.attn = m->attn;
        P.attn_part = m->as.part;
        P.attn_cnt = m->as.cnt;
        P.st = m->st;
        P.bar_count = words;
        P.bar_gen = words + 1;
        P.abort = words + 2;
        P.err = m->gs.err;
        std::vector<LayerPlan> lp(c.n_layers);
        // the persistent kernel decodes every matrix as one type and reads an fp32 / fp16 cache
        bool ok = head_wtype(&c) == wt && !kv_quantized(&c);
        for (int l = 0; l < c.n_layers; l++) {
            const LayerW& lw = m->L[l];
            LayerPlan& L = lp[l];
            ok = ok && decode_gemv_task(lw.qkv, L.qkv) && decode_gemv_task(lw.o, L.o) &&
                 decode_gemv_task(lw.gu, L.gu) && decode_gemv_task(lw.down, L.down);
            L.kc = m->kl(l);
            L.vc = m->vl(l);
            L.qkv.x = m->x;
            L.qkv.nw = lw.attn_norm;
            L.qkv.epi = epi_qkv_plan(m, l);
            L.o.x = m->attn;
            L.o.epi = epi_simple(EPI_RESID, m->x, E);
            L.gu.x = m->x;
            L.gu.nw = lw.ffn_norm;
            L.gu.epi = epi_simple(EPI_SWIGLU, m->h, F);
            L.down.x = m->h;
            L.down.epi = epi_simple(EPI_RESID, m->x, E);
        }
        ok = ok && decode_gemv_task(m->out, P.head);
        P.head.x = m->x;
        P.head.nw = m->out_norm;
        P.head.epi = epi_simple(EPI_LOGITS, m->logits, 0);
        P.head.epi.argmax = &m->st->argmax;
        m->persistent_ok = ok && E / num_sms() + 2 <= decode_max_cta_rows() && decode_configure(P, lp[0]);
        cudaError_t e = cudaMemcpyAsync(m->d_layers, lp.data(), sizeof(LayerPlan) * c.n_layers, cudaMemcpyHostToDevice, s);
        if (!e) e = cudaMemsetAsync(words, 0, 4 * sizeof(unsigned), s);
        if (!e) e = cudaStreamSynchronize(s);  // lp is a host temporary
        if (e) return cuda_fail(e, "decode plan");
        if (m->persistent_ok && decode_prepare(P) != cudaSuccess) {
            cudaGetLastError();
            m->persistent_ok = false;  // cannot be resident on this device
        }
    }
    {
        cudaError_t e = qgemv_prepare();
        if (!e) e = qgemm_prepare();
        if (!e) e = cudaMemsetAsync(m->gs.err, 0, kErrWords * sizeof(unsigned), s);
        if (!e) e = cudaMemsetAsync(m->as.cnt, 0, (size_t)c.n_kv_heads * 4, s);
        if (!e && m->gsplit.cnt) e = cudaMemsetAsync(m->gsplit.cnt, 0, (size_t)m->gsplit.cnt_n * 4, s);
        if (!e) e = cudaMemsetAsync(m->st, 0, sizeof(StepState), s);
        if (!e) e = cudaStreamSynchronize(s);
        if (e) return cuda_fail(e, "model init");
        if (cudaMallocHost(&m->tok_host, (size_t)S * 4) != cudaSuccess ||
            cudaEventCreateWithFlags(&m->tok_ev, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            if (m->tok_ev) cudaEventDestroy(m->tok_ev);
            if (m->tok_host) cudaFreeHost(m->tok_host);
            m->tok_ev = nullptr;
            m->tok_host = nullptr;
            return oom("token staging");
        }
    }
    *out = m;
    return AF_OK;
}

void* af_model_stream(const af_model* m) { return m ? (void*)m->s : nullptr; }

const int32_t* af_model_next_token_dev(const af_model* m) { return m ? &m->st->next_token : nullptr; }

int af_model_sync(af_model* m, int32_t* next_token_host) {
    if (!m) return fail(AF_EINVAL, "null model");
    if (next_token_host) CK(cudaMemcpyAsync(next_token_host, &m->st->next_token, 4, cudaMemcpyDeviceToHost, m->s));
    return read_err(m);
}

int af_model_kv_cache(const af_model* m, void** k_dev, void** v_dev) {
    if (!m || !k_dev || !v_dev) return fail(AF_EINVAL, "null argument");
    *k_dev = m->kc;
    *v_dev = m->vc;
    return AF_OK;
}

int af_model_kv_store(const af_model* m, void** k_codes, void** k_scales, void** v_codes, void** v_scales) {
    if (!m || !k_codes || !k_scales || !v_codes || !v_scales) return fail(AF_EINVAL, "null argument");
    if (!m->kvq.qtype) return fail(AF_EINVAL, "the model's KV cache is not quantized");
    *k_codes = m->kvq.kq;
    *k_scales = m->kvq.ks;
    *v_codes = m->kvq.vq;
    *v_scales = m->kvq.vs;
    return AF_OK;
}

int af_reset(af_model* m) {
    if (!m) return fail(AF_EINVAL, "null model");
    const size_t kvb = (size_t)m->c.n_layers * m->kv_layer_elems * kv_elem(&m->c);
    CK(cudaMemsetAsync(m->kc, 0, kvb, m->s));
    CK(cudaMemsetAsync(m->vc, 0, kvb, m->s));
    CK(cudaMemsetAsync(m->gs.err, 0, 4, m->s));
    return AF_OK;
}

int af_debug_stall(af_model* m, uint32_t polls) {
    if (!m) return fail(AF_EINVAL, "null model");
    CK(cudaStreamSynchronize(m->s));
    CK(cudaMemcpy(m->gs.err + 1, &polls, 4, cudaMemcpyHostToDevice));
    return AF_OK;
}

int af_debug_capture(af_model* m, float* hidden_dev) {
    if (!m || !hidden_dev) return fail(AF_EINVAL, "null argument");
    m->capture = hidden_dev;
    return AF_OK;
}

int af_debug_trace(af_model* m, uint64_t* trace_dev) {
    if (!m || !trace_dev) return fail(AF_EINVAL, "null argument");
    m->trace = reinterpret_cast<unsigned long long*>(trace_dev);
    return AF_OK;
}

int af_set_decode_mode(af_model* m, int mode) {
    if (!m) return fail(AF_EINVAL, "null model");
    if (mode != AF_DECODE_PERSISTENT && mode != AF_DECODE_KERNELS) return fail(AF_EINVAL, "bad decode mode");
    if (mode == AF_DECODE_PERSISTENT && !m->persistent_ok)
        return fail(AF_ENOTIMPL, "persistent decode kernel not available for this device/shape");
    m->decode_mode = mode;
    return AF_OK;
}

int af_get_decode_mode(const af_model* m) { return m ? m->decode_mode : -1; }

int af_set_decode_graph(af_model* m, int enable) {
    if (!m) return fail(AF_EINVAL, "null model");
    m->use_graph = enable != 0;
    return AF_OK;
}

}  // extern "C"

namespace {

int capture_copy(af_model* m, int slot, int n) {
    if (!m->capture) return AF_OK;
    const size_t bytes = (size_t)n * m->E() * 4;
    CK(cudaMemcpyAsync(m->capture + (size_t)slot * n * m->E(), m->x, bytes, cudaMemcpyDeviceToDevice, m->s));
    return AF_OK;
}

Epi epi_qkv(af_model* m, int l, float* qout, const int* pos_dev, int pos0) {
    Epi e;
    e.kind = EPI_QKV;
    e.out = qout;
    e.ld = m->QD();
    e.qd = m->QD();
    e.kvd = m->KVD();
    e.head_dim = m->c.head_dim;
    e.max_ctx = m->c.max_ctx;
    e.kv_f16 = m->c.kv_dtype != AF_F32;
    e.kcache = m->kl(l);
    e.vcache = m->vl(l);
    e.rope = m->rope;
    e.pos_dev = pos_dev;
    e.pos0 = pos0;
    return e;
}

// Decode body after step_begin: reads token/pos from m->st.
int decode_body(af_model* m, float* logits) {
    const af_config& c = m->c;
    cudaStream_t s = m->s;
    const int* pos_dev = &m->st->pos;
    CK(launch_embed(m->emb, &m->st->token, 1, m->x, m->E(), s));
    int rc = capture_copy(m, 0, 1);
    if (rc) return rc;
    // a quantized cache: the slot that leaves the window in this step (pos - window) retires, in every layer
    if (m->kvq.qtype)
        CK(launch_kv_retire(m->kvq, (__half*)m->kc, (__half*)m->vc, c.n_layers, c.n_kv_heads, c.max_ctx, c.head_dim,
                            pos_dev, 0, 1, s));
    for (int l = 0; l < c.n_layers; l++) {
        const LayerW& lw = m->L[l];
        const KvLayerStore qs = m->kvq_layer(l);
        CK(launch_qgemv(lw.qkv, m->x, lw.attn_norm, c.rms_eps, epi_qkv(m, l, m->q, pos_dev, 0), m->gs, s));
        CK(launch_attn_decode(m->q, m->kl(l), m->vl(l), c.kv_dtype != AF_F32, c.n_heads, c.n_kv_heads, c.head_dim,
                              c.max_ctx, pos_dev, 0, m->as, m->attn, s, qs.qtype ? &qs : nullptr));
        CK(launch_qgemv(lw.o, m->attn, nullptr, 0.f, epi_simple(EPI_RESID, m->x, m->E()), m->gs, s));
        CK(launch_qgemv(lw.gu, m->x, lw.ffn_norm, c.rms_eps, epi_simple(EPI_SWIGLU, m->h, c.n_ff), m->gs, s));
        CK(launch_qgemv(lw.down, m->h, nullptr, 0.f, epi_simple(EPI_RESID, m->x, m->E()), m->gs, s));
        rc = capture_copy(m, l + 1, 1);
        if (rc) return rc;
    }
    Epi el = epi_simple(EPI_LOGITS, logits, 0);
    el.argmax = &m->st->argmax;
    CK(launch_qgemv(m->out, m->x, m->out_norm, c.rms_eps, el, m->gs, s));
    CK(launch_step_end(m->st, s));
    return AF_OK;
}

int prefill_impl(af_model* m, const int* tok_dev, int n, int start_pos, float* logits) {
    const af_config& c = m->c;
    cudaStream_t s = m->s;
    const int E = m->E(), QD = m->QD(), F = c.n_ff;
    CK(launch_embed(m->emb, tok_dev, n, m->x, E, s));
    int rc = capture_copy(m, 0, n);
    if (rc) return rc;
    // a quantized cache: the n slots that leave the window in this step retire before any attention reads them
    if (m->kvq.qtype)
        CK(launch_kv_retire(m->kvq, (__half*)m->kc, (__half*)m->vc, c.n_layers, c.n_kv_heads, c.max_ctx, c.head_dim,
                            nullptr, start_pos - m->kvq.window, n, s));
    for (int l = 0; l < c.n_layers; l++) {
        const LayerW& lw = m->L[l];
        CK(launch_rmsnorm_rows(m->x, n, E, lw.attn_norm, c.rms_eps, m->y16[0], m->y16[1], s));
        CK(launch_qgemm(lw.qkv, m->y16[0], m->y16[1], E, n, epi_qkv(m, l, m->q, nullptr, start_pos),
                        m->gs.err, s, &m->gsplit));
        CK(launch_attn_prefill(m->q, QD, m->kl(l), m->vl(l), c.kv_dtype != AF_F32, c.n_heads, c.n_kv_heads,
                               c.head_dim, c.max_ctx, start_pos, n, m->a16[0], m->a16[1], QD, m->gs.err, s));
        CK(launch_qgemm(lw.o, m->a16[0], m->a16[1], QD, n, epi_simple(EPI_RESID, m->x, E), m->gs.err, s,
                        &m->gsplit));
        CK(launch_rmsnorm_rows(m->x, n, E, lw.ffn_norm, c.rms_eps, m->y16[0], m->y16[1], s));
        Epi eg = epi_simple(EPI_SWIGLU, nullptr, F);
        eg.out16 = m->h16[0];
        eg.out16_lo = m->h16[1];
        CK(launch_qgemm(lw.gu, m->y16[0], m->y16[1], E, n, eg, m->gs.err, s, &m->gsplit));
        CK(launch_qgemm(lw.down, m->h16[0], m->h16[1], F, n, epi_simple(EPI_RESID, m->x, E), m->gs.err, s,
                        &m->gsplit));
        rc = capture_copy(m, l + 1, n);
        if (rc) return rc;
    }
    if (logits) {
        CK(launch_step_begin(m->st, 0, start_pos + n - 1, s));  // resets the argmax word
        Epi el = epi_simple(EPI_LOGITS, logits, 0);
        el.argmax = &m->st->argmax;
        CK(launch_qgemv(m->out, m->x + (size_t)(n - 1) * E, m->out_norm, c.rms_eps, el, m->gs, s));
        CK(launch_step_end(m->st, s));
    }
    m->capture = nullptr;
    return AF_OK;
}

}  // namespace

extern "C" {

int af_prefill_dev(af_model* m, const int32_t* tokens_dev, int32_t n, int32_t start_pos, float* logits_dev) {
    if (!m || !tokens_dev) return fail(AF_EINVAL, "null argument");
    if (n < 1 || n > m->chunk) return fail(AF_ERANGE, "n=%d outside [1, max_chunk=%d]", n, m->chunk);
    if (start_pos < 0 || (int64_t)start_pos + n > m->c.max_ctx)
        return fail(AF_ERANGE, "positions %d..%d outside the cache (max_ctx %d)", start_pos, start_pos + n - 1,
                    m->c.max_ctx);
    return prefill_impl(m, tokens_dev, n, start_pos, logits_dev);
}

int af_prefill(af_model* m, const int32_t* tokens_host, int32_t n, int32_t start_pos, float* logits_dev) {
    if (!m || !tokens_host) return fail(AF_EINVAL, "null argument");
    if (n < 1 || n > m->chunk) return fail(AF_ERANGE, "n=%d outside [1, max_chunk=%d]", n, m->chunk);
    if (start_pos < 0 || (int64_t)start_pos + n > m->c.max_ctx)
        return fail(AF_ERANGE, "positions %d..%d outside the cache (max_ctx %d)", start_pos, start_pos + n - 1,
                    m->c.max_ctx);
    for (int i = 0; i < n; i++)
        if (tokens_host[i] < 0 || tokens_host[i] >= m->c.n_vocab)
            return fail(AF_ERANGE, "token %d at index %d outside [0, %d)", tokens_host[i], i, m->c.n_vocab);
    // through the model's page-locked staging buffer: the caller's buffer is free once this returns, and the
    // staging buffer is rewritten only after the previous call's copy out of it has completed
    CK(cudaEventSynchronize(m->tok_ev));
    std::memcpy(m->tok_host, tokens_host, (size_t)n * 4);
    CK(cudaMemcpyAsync(m->tok, m->tok_host, (size_t)n * 4, cudaMemcpyHostToDevice, m->s));
    CK(cudaEventRecord(m->tok_ev, m->s));
    return prefill_impl(m, m->tok, n, start_pos, logits_dev);
}

int af_decode_step(af_model* m, int32_t token, int32_t pos, float* logits_dev, int32_t* next_token_host) {
    if (!m) return fail(AF_EINVAL, "null model");
    if (pos < 0 || pos >= m->c.max_ctx) return fail(AF_ERANGE, "pos %d outside [0, %d)", pos, m->c.max_ctx);
    if (token < -1 || token >= m->c.n_vocab) return fail(AF_ERANGE, "token %d outside [-1, %d)", token, m->c.n_vocab);
    float* logits = logits_dev ? logits_dev : m->logits;
    CK(launch_step_begin(m->st, token, pos, m->s, m->dplan.bar_count));
    if (m->decode_mode == AF_DECODE_PERSISTENT) {
        DecodePlan P = m->dplan;
        P.head.epi.out = logits;
        P.capture = m->capture;
        P.trace = m->trace;
        m->capture = nullptr;
        m->trace = nullptr;
        CK(launch_decode(P, m->s));
        CK(launch_step_end(m->st, m->s));
    } else if (m->use_graph && !m->capture) {
        if (!m->gexec || m->graph_logits != logits) {
            if (m->gexec) {
                cudaGraphExecDestroy(m->gexec);
                m->gexec = nullptr;
            }
            cudaGraph_t g = nullptr;
            CK(cudaStreamBeginCapture(m->s, cudaStreamCaptureModeThreadLocal));
            int rc = decode_body(m, logits);
            cudaError_t e = cudaStreamEndCapture(m->s, &g);
            if (rc) {
                if (g) cudaGraphDestroy(g);
                return rc;
            }
            if (e != cudaSuccess) return fail(AF_ECUDA, "graph capture: %s", cudaGetErrorString(e));
            e = cudaGraphInstantiate(&m->gexec, g, 0);
            cudaGraphDestroy(g);
            if (e != cudaSuccess) {
                m->gexec = nullptr;
                return fail(AF_ECUDA, "graph instantiate: %s", cudaGetErrorString(e));
            }
            m->graph_logits = logits;
        }
        CK(cudaGraphLaunch(m->gexec, m->s));
    } else {
        int rc = decode_body(m, logits);
        m->capture = nullptr;
        if (rc) return rc;
    }
    if (next_token_host) {
        CK(cudaMemcpyAsync(next_token_host, &m->st->next_token, 4, cudaMemcpyDeviceToHost, m->s));
        return read_err(m);
    }
    return AF_OK;
}

// ---------------------------------------------------------------- standalone matmuls

void af_qweight_destroy(af_qweight* w) {
    if (!w) return;
    w->A.free_all();
    delete w;
}

int af_qweight_create(int32_t wtype, const void* blocks_dev, int32_t N, int32_t K, void* stream, af_qweight** out) {
    if (!out) return fail(AF_EINVAL, "null out");
    *out = nullptr;
    if (!block_bytes(wtype)) return fail(AF_EINVAL, "bad wtype");
    if (!blocks_dev) return fail(AF_EINVAL, "null blocks");
    if (N <= 0 || K <= 0 || K % block_elems(wtype))
        return fail(AF_EINVAL, "need N > 0 and K a positive multiple of %d", block_elems(wtype));
    if (N % 2) return fail(AF_ENOTIMPL, "N must be even");
    if (padded_k(wtype, K) / chunk_weights(wtype) > qgemv_max_chunks())
        return fail(AF_ENOTIMPL, "K above %d", qgemv_max_chunks() * chunk_weights(wtype));
    af_qweight* w = new (std::nothrow) af_qweight();
    if (!w) return fail(AF_ENOMEM, "host allocation failed");
    cudaStream_t s = (cudaStream_t)stream;
    w->p = make_planes(w->A, wtype, N, K);
    w->gs.err = (unsigned*)w->A.get(kErrWords * sizeof(unsigned));
    if (const size_t ws = qgemm_ws_bytes(N, K, 512)) {
        w->gsplit.ws = (float*)w->A.get(ws);
        w->gsplit.ws_bytes = w->gsplit.ws ? ws : 0;
        w->gsplit.cnt = (unsigned*)w->A.get((size_t)qgemm_tiles(N, 512) * 4);
        w->gsplit.cnt_n = w->gsplit.cnt ? qgemm_tiles(N, 512) : 0;
    }
    if (!w->p.qs || !w->gs.err) {
        af_qweight_destroy(w);
        return fail(AF_ENOMEM, "device allocation failed");
    }
    cudaError_t e = qgemv_prepare();
    if (!e) e = qgemm_prepare();
    if (!e) e = repack_into(w->p, blocks_dev, N, 0, 1, s);
    if (!e) e = cudaMemsetAsync(w->gs.err, 0, kErrWords * sizeof(unsigned), s);
    if (!e && w->gsplit.cnt) e = cudaMemsetAsync(w->gsplit.cnt, 0, (size_t)w->gsplit.cnt_n * 4, s);
    if (!e) e = cudaStreamSynchronize(s);
    if (e) {
        af_qweight_destroy(w);
        return fail(AF_ECUDA, "qweight repack: %s", cudaGetErrorString(e));
    }
    *out = w;
    return AF_OK;
}

int af_qgemv(const af_qweight* w, const float* x_dev, float* y_dev, void* stream) {
    if (!w || !x_dev || !y_dev) return fail(AF_EINVAL, "null argument");
    CK(launch_qgemv(w->p, x_dev, nullptr, 0.f, epi_simple(EPI_STORE, y_dev, w->p.N), w->gs, (cudaStream_t)stream));
    return AF_OK;
}

int af_qgemm(const af_qweight* wc, const float* X_dev, int32_t M, float* Y_dev, void* stream) {
    if (!wc || !X_dev || !Y_dev) return fail(AF_EINVAL, "null argument");
    if (M < 1) return fail(AF_ERANGE, "M must be >= 1");
    af_qweight* w = const_cast<af_qweight*>(wc);
    cudaStream_t s = (cudaStream_t)stream;
    if (w->x16_rows < M) {  // (re)allocate the operand planes; the old ones may still be in use
        CK(cudaStreamSynchronize(s));
        for (int i = 0; i < 2; i++) {
            w->A.release(w->x16[i]);
            w->x16[i] = (__half*)w->A.get((size_t)M * w->p.K * 2);
        }
        w->x16_rows = (w->x16[0] && w->x16[1]) ? M : 0;
        if (!w->x16_rows) return fail(AF_ENOMEM, "operand buffer");
    }
    CK(launch_split_f16(X_dev, w->x16[0], w->x16[1], (int64_t)M * w->p.K, s));
    CK(launch_qgemm(w->p, w->x16[0], w->x16[1], w->p.K, M, epi_simple(EPI_STORE, Y_dev, w->p.N), w->gs.err, s,
                    &w->gsplit));
    return AF_OK;
}

int af_qweight_status(const af_qweight* w, void* stream) {
    if (!w) return fail(AF_EINVAL, "null argument");
    cudaStream_t s = (cudaStream_t)stream;
    unsigned code = 0;
    CK(cudaMemcpyAsync(&code, w->gs.err, 4, cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    if (code) {
        CK(cudaMemsetAsync(w->gs.err, 0, 4, s));
        CK(cudaStreamSynchronize(s));
        return fail(AF_ETIMEOUT, "a bounded device-side wait gave up (code %u)", code);
    }
    return AF_OK;
}

int af_qweight_debug_stall(af_qweight* w, uint32_t polls, void* stream) {
    if (!w) return fail(AF_EINVAL, "null argument");
    CK(cudaStreamSynchronize((cudaStream_t)stream));
    CK(cudaMemcpy(w->gs.err + 1, &polls, 4, cudaMemcpyHostToDevice));
    return AF_OK;
}

// ---------------------------------------------------------------- standalone attention

int af_attention_decode(const float* q_dev, const void* k_dev, const void* v_dev, int32_t kv_dtype, int32_t H,
                        int32_t KVH, int32_t D, int32_t ctx, int32_t pos, float* out_dev, void* stream) {
    if (!q_dev || !k_dev || !v_dev || !out_dev) return fail(AF_EINVAL, "null argument");
    if (kv_dtype != AF_F32 && kv_dtype != AF_F16) return fail(AF_EINVAL, "bad kv_dtype");
    if (H <= 0 || KVH <= 0 || D <= 0 || ctx <= 0) return fail(AF_EINVAL, "sizes must be positive");
    if (!attn_supported(H, KVH, D)) return fail(AF_ENOTIMPL, "unsupported head_dim / group size");
    if (pos < 0 || pos >= ctx) return fail(AF_ERANGE, "pos %d outside [0, %d)", pos, ctx);
    cudaStream_t s = (cudaStream_t)stream;
    AttnScratch as;
    as.ns = attn_decode_splits(H, KVH, ctx);
    const size_t pe = attn_decode_part_elems(H, D, as.ns);
    if (cudaMalloc(&as.part, pe * 4) != cudaSuccess) {
        cudaGetLastError();
        return fail(AF_ENOMEM, "scratch");
    }
    if (cudaMalloc(&as.cnt, (size_t)(KVH + 1) * 4) != cudaSuccess) {  // counters, then the error word
        cudaGetLastError();
        cudaFree(as.part);
        return fail(AF_ENOMEM, "scratch");
    }
    as.err = as.cnt + KVH;
    unsigned err_host = 0;
    cudaError_t e = cudaMemsetAsync(as.cnt, 0, (size_t)(KVH + 1) * 4, s);
    if (!e) e = launch_attn_decode(q_dev, k_dev, v_dev, kv_dtype == AF_F16, H, KVH, D, ctx, nullptr, pos, as, out_dev, s);
    if (!e) e = cudaMemcpyAsync(&err_host, as.err, 4, cudaMemcpyDeviceToHost, s);
    cudaError_t e2 = cudaStreamSynchronize(s);
    cudaFree(as.part);
    cudaFree(as.cnt);
    if (e) return fail(AF_ECUDA, "attention: %s", cudaGetErrorString(e));
    if (e2) return fail(AF_ECUDA, "attention sync: %s", cudaGetErrorString(e2));
    if (err_host) return fail(AF_ETIMEOUT, "a bounded device-side wait gave up (code %u)", err_host);
    return AF_OK;
}

int af_attention_prefill(const float* q_dev, const void* k_dev, const void* v_dev, int32_t kv_dtype, int32_t H,
                         int32_t KVH, int32_t D, int32_t ctx, int32_t start_pos, int32_t n, float* out_dev,
                         void* stream) {
    if (!q_dev || !k_dev || !v_dev || !out_dev) return fail(AF_EINVAL, "null argument");
    if (kv_dtype != AF_F32 && kv_dtype != AF_F16) return fail(AF_EINVAL, "bad kv_dtype");
    if (H <= 0 || KVH <= 0 || D <= 0 || ctx <= 0) return fail(AF_EINVAL, "sizes must be positive");
    if (!attn_supported(H, KVH, D)) return fail(AF_ENOTIMPL, "unsupported head_dim / group size");
    if (n < 1 || n > 512) return fail(AF_ERANGE, "n=%d outside [1, 512]", n);
    if (start_pos < 0 || (int64_t)start_pos + n > ctx)
        return fail(AF_ERANGE, "positions %d..%d outside the cache (%d slots)", start_pos, start_pos + n - 1, ctx);
    if (((uintptr_t)q_dev | (uintptr_t)k_dev | (uintptr_t)v_dev) & 15) return fail(AF_EINVAL, "unaligned pointer");
    cudaStream_t s = (cudaStream_t)stream;
    const size_t ne = (size_t)n * H * D;
    void* buf = nullptr;  // out_hi, out_lo planes, then the error words
    if (cudaMalloc(&buf, ne * 4 + 256) != cudaSuccess) {
        cudaGetLastError();
        return fail(AF_ENOMEM, "scratch");
    }
    __half* hi = (__half*)buf;
    __half* lo = hi + ne;
    unsigned* err = (unsigned*)((char*)buf + ne * 4);
    unsigned err_host = 0;
    cudaError_t e = cudaMemsetAsync(err, 0, 4, s);
    if (!e) e = launch_attn_prefill(q_dev, (int64_t)H * D, k_dev, v_dev, kv_dtype == AF_F16, H, KVH, D, ctx, start_pos, n,
                                    hi, lo, (int64_t)H * D, err, s);
    if (!e) e = launch_join_f16(hi, lo, out_dev, (int64_t)ne, s);
    if (!e) e = cudaMemcpyAsync(&err_host, err, 4, cudaMemcpyDeviceToHost, s);
    cudaError_t e2 = cudaStreamSynchronize(s);
    cudaFree(buf);
    if (e) return fail(AF_ECUDA, "prefill attention: %s", cudaGetErrorString(e));
    if (e2) return fail(AF_ECUDA, "prefill attention sync: %s", cudaGetErrorString(e2));
    if (err_host) return fail(AF_ETIMEOUT, "a bounded device-side wait gave up (code %u)", err_host);
    return AF_OK;
}

// Same computation without allocating: the split scratch is a file-scope device
// array (attn_static.cu).  For callers that cannot allocate mid-step: a serving
// loop with work queued on other streams cannot take the device-wide
// synchronisation that cudaFree implies, and a caller that has handed the
// device's free memory to its own pool has none left to cudaMalloc.
int af_attention_decode_static(const float* q_dev, const void* k_dev, const void* v_dev, int32_t kv_dtype, int32_t H,
                               int32_t KVH, int32_t D, int32_t ctx, int32_t pos, float* out_dev, void* stream) {
    if (!q_dev || !k_dev || !v_dev || !out_dev) return fail(AF_EINVAL, "null argument");
    if (kv_dtype != AF_F32 && kv_dtype != AF_F16) return fail(AF_EINVAL, "bad kv_dtype");
    if (H <= 0 || KVH <= 0 || D <= 0 || ctx <= 0) return fail(AF_EINVAL, "sizes must be positive");
    if (!attn_supported(H, KVH, D)) return fail(AF_ENOTIMPL, "unsupported head_dim / group size");
    if (pos < 0 || pos >= ctx) return fail(AF_ERANGE, "pos %d outside [0, %d)", pos, ctx);
    AttnScratch as;
    as.ns = attn_decode_splits(H, KVH, ctx);
    // the cluster path keeps its partials in shared memory: only the split path needs the counters and partials
    if (!attn_decode_uses_cluster(ctx)) {
        if (KVH > kStaticAttnMaxKVH)
            return fail(AF_ERANGE, "n_kv_heads %d above the fixed scratch (%d)", KVH, kStaticAttnMaxKVH);
        if (attn_decode_part_elems(H, D, as.ns) > kStaticAttnPartFloats)
            return fail(AF_ERANGE, "split partials (%zu floats) above the fixed scratch (%zu)",
                        attn_decode_part_elems(H, D, as.ns), kStaticAttnPartFloats);
    }
    CK(attn_static_scratch(&as.part, &as.cnt, &as.err));
    CK(launch_attn_decode(q_dev, k_dev, v_dev, kv_dtype == AF_F16, H, KVH, D, ctx, nullptr, pos, as, out_dev,
                          (cudaStream_t)stream));
    return AF_OK;
}

// ---------------------------------------------------------------- sampler chain

}  // extern "C"

namespace {
int check_sample_args(int32_t n_vocab, const int32_t* recent_dev, int32_t n_recent, float repeat_penalty,
                      float temperature, float top_p, float u) {
    if (n_recent < 0 || (n_recent > 0 && !recent_dev)) return fail(AF_EINVAL, "bad recent-token list");
    if (n_vocab < 1 || n_vocab > sampler_max_vocab())
        return fail(AF_ERANGE, "n_vocab %d outside [1, %d]", n_vocab, sampler_max_vocab());
    if (!(repeat_penalty > 0.f) || !(temperature >= 0.f) || !(top_p == top_p))
        return fail(AF_EINVAL, "repeat_penalty must be > 0, temperature >= 0, top_p a number");
    if (!(u >= 0.f && u < 1.f)) return fail(AF_ERANGE, "u must be in [0, 1)");
    return AF_OK;
}
}  // namespace

extern "C" {

int af_sample(const float* logits_dev, int32_t n_vocab, const int32_t* recent_dev, int32_t n_recent,
              float repeat_penalty, float temperature, float top_p, float u, int32_t* token_dev, void* stream) {
    if (!logits_dev || !token_dev) return fail(AF_EINVAL, "null argument");
    if (int rc = check_sample_args(n_vocab, recent_dev, n_recent, repeat_penalty, temperature, top_p, u)) return rc;
    CK(launch_sample(logits_dev, n_vocab, recent_dev, n_recent, repeat_penalty, temperature, top_p, u, token_dev,
                     (cudaStream_t)stream));
    return AF_OK;
}

int af_model_sample(af_model* m, const float* logits_dev, const int32_t* recent_dev, int32_t n_recent,
                    float repeat_penalty, float temperature, float top_p, float u, int32_t* token_host) {
    if (!m) return fail(AF_EINVAL, "null model");
    if (int rc = check_sample_args(m->c.n_vocab, recent_dev, n_recent, repeat_penalty, temperature, top_p, u))
        return rc;
    const float* logits = logits_dev ? logits_dev : m->logits;
    CK(launch_sample(logits, m->c.n_vocab, recent_dev, n_recent, repeat_penalty, temperature, top_p, u,
                     &m->st->next_token, m->s));
    if (token_host) {
        CK(cudaMemcpyAsync(token_host, &m->st->next_token, 4, cudaMemcpyDeviceToHost, m->s));
        CK(cudaStreamSynchronize(m->s));
    }
    return AF_OK;
}

}  // extern "C"
