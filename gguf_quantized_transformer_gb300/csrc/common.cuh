// Shared device/host definitions of the CUDA library (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "af.h"  // include/ (passed with -I by the build)

namespace af {

// ---------------------------------------------------------------------------
// Repacked weight layout ("planes").
//
// A GGUF [N, K] block matrix is stored as one record per row, pitch() bytes
// apart (a multiple of 16), so R consecutive rows, scales included, are one
// contiguous range (one bulk copy per GEMV stage).  K is padded to Kp, a whole
// GEMV chunk (1024 weights; 512 for Q8_0); padding holds zero codes and zero
// scales, so it contributes 0.  The unit of the kernels is 32 weights whose
// 4-bit codes sit in 16 bytes in GGUF's Q4_0 nibble order (byte j: element j
// low, element j + 16 high); Q8_0 units are 16 weights in 16 bytes.
//   Q4_0 / Q8_0: [(Kp/32) x QB code bytes][(Kp/32) fp16 scales]  (QB = 16 / 32)
//   Q4_K: [(Kp/32) x 16 code bytes][(Kp/256) super-block records of 20 B:
//          fp16 d, fp16 dmin, then (s_j, m_j) byte pairs of its 8 sub-blocks,
//          the 6-bit scales and mins already unpacked]
//   Q5_K: as Q4_K, with a plane of the codes' high bits after the units: one word
//          per unit, element 4t + i of half h (16 elements) at bit 8i + 4h + t
//   Q6_K: [(Kp/32) x 16 bytes: low 4 bits of the codes][(Kp/32) x 8 bytes: the
//          high 2 bits, two words per unit, element 4t + i of a 16-element half
//          at bits 8i + 2t][(Kp/256) records of 18 B: fp16 d, 16 int8 scales]
//          (+ padding of the row to 16 bytes)
// qs points at row 0; sc at row 0's fp16 scales (Q4_0 / Q8_0; sc_pitch()
// halves per row).  sc_off() is the byte offset of the scales or records in a
// row, hb_off() that of the Q5_K / Q6_K high-bit plane.
// ---------------------------------------------------------------------------
constexpr int kQ4KRec = 20;  // also Q5_K's record
constexpr int kQ6KRec = 18;

__host__ __device__ inline bool is_kquant(int wtype) {
    return wtype == AF_Q4_K || wtype == AF_Q5_K || wtype == AF_Q6_K;
}

struct Planes {
    const uint8_t* qs = nullptr;
    const __half* sc = nullptr;
    int N = 0, K = 0, Kp = 0, wtype = 0;
    __host__ __device__ int qb() const { return wtype == AF_Q8_0 ? 32 : 16; }  // code bytes per 32 weights
    __host__ __device__ int sc_off() const {
        return wtype == AF_Q6_K ? (Kp / 32) * 24 : wtype == AF_Q5_K ? (Kp / 32) * 20 : (Kp / 32) * qb();
    }
    __host__ __device__ int hb_off() const { return (Kp / 32) * 16; }
    __host__ __device__ int64_t qs_pitch() const {  // bytes per row
        int64_t b;
        if (wtype == AF_Q4_K)
            b = (int64_t)(Kp / 32) * 16 + (int64_t)(Kp / 256) * kQ4KRec;
        else if (wtype == AF_Q5_K)
            b = (int64_t)(Kp / 32) * 20 + (int64_t)(Kp / 256) * kQ4KRec;
        else if (wtype == AF_Q6_K)
            b = (int64_t)(Kp / 32) * 24 + (int64_t)(Kp / 256) * kQ6KRec;
        else
            b = (int64_t)(Kp / 32) * (qb() + 2);
        return (b + 15) & ~(int64_t)15;
    }
    __host__ __device__ int sc_pitch() const { return (int)(qs_pitch() / 2); }  // halves per row
};

inline int chunk_weights(int wtype) { return wtype == AF_Q8_0 ? 512 : 1024; }
inline int padded_k(int wtype, int K) { int c = chunk_weights(wtype); return (K + c - 1) / c * c; }
inline int block_elems(int wtype) { return is_kquant(wtype) ? 256 : 32; }
inline size_t planes_bytes(int wtype, int N, int K, size_t* sc_off) {
    Planes p;
    p.wtype = wtype;
    p.Kp = padded_k(wtype, K);
    if (sc_off) *sc_off = (size_t)p.sc_off();
    return ((size_t)N * (size_t)p.qs_pitch() + 255) & ~(size_t)255;
}

// ---------------------------------------------------------------------------
// Fused epilogues, shared by the decode GEMV and the prefill GEMM.  Each is
// applied to an adjacent column pair (n, n+1) of one output row m.
// ---------------------------------------------------------------------------
enum EpiKind { EPI_STORE = 0, EPI_RESID = 1, EPI_QKV = 2, EPI_SWIGLU = 3, EPI_LOGITS = 4 };

struct Epi {
    int kind = EPI_STORE;
    float* out = nullptr;  // STORE: Y [M][ld]; RESID: x [M][ld]; QKV: q [M][ld]; SWIGLU: h [M][ld]; LOGITS: [N]
    int ld = 0;
    __half* out16 = nullptr;     // optional fp16 hi part of the SWIGLU output (GEMM operand), same ld
    __half* out16_lo = nullptr;  // its fp16 lo part: value - hi
    // EPI_QKV: columns [0, qd) are q, [qd, qd+kvd) k, [qd+kvd, qd+2kvd) v
    int qd = 0, kvd = 0, head_dim = 0, max_ctx = 0, kv_f16 = 0;
    void* kcache = nullptr;  // this layer's [KVH][max_ctx][D]
    void* vcache = nullptr;
    const float2* rope = nullptr;  // [max_ctx][D/2] (cos, sin) of theta(t, i)
    const int* pos_dev = nullptr;  // if set: position of row m is *pos_dev + m
    int pos0 = 0;                  // else: pos0 + m
    unsigned long long* argmax = nullptr;  // EPI_LOGITS: packed (value, ~index) maximum
};

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    unsigned u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // order-preserving map of floats to unsigned
    return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)idx);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

// Reads across kernels.  A kernel launched with programmatic dependent launch starts before its predecessor
// has finished, and the SM's L1 is not invalidated for it: a line that an earlier kernel cached on the same SM
// can be stale (measured: row RMSNorm reading x through L1 after griddepcontrol.wait returned old values).  So
// data written by an earlier kernel of a chain (activations, the residual, q, the position word) is read with
// ld.global.cg, which goes to L2, after griddepcontrol.wait; only data no kernel writes (weights, norm weights,
// the RoPE table) is read through L1.
__device__ __forceinline__ void epi_pair(const Epi& e, int m, int n, float v0, float v1) {
    switch (e.kind) {
        case EPI_STORE: {
            e.out[(int64_t)m * e.ld + n] = v0;
            e.out[(int64_t)m * e.ld + n + 1] = v1;
        } break;
        case EPI_RESID: {  // the residual was written by an earlier kernel: read through L2 (note above)
            float* p = e.out + (int64_t)m * e.ld + n;
            const float2 o = __ldcg(reinterpret_cast<const float2*>(p));
            *reinterpret_cast<float2*>(p) = make_float2(o.x + v0, o.y + v1);
        } break;
        case EPI_SWIGLU: {  // columns (2r, 2r+1) hold (gate_r, up_r)
            float h = silu_f(v0) * v1;
            if (e.out) e.out[(int64_t)m * e.ld + (n >> 1)] = h;
            if (e.out16) {
                const __half hh = __float2half_rn(h);
                e.out16[(int64_t)m * e.ld + (n >> 1)] = hh;
                e.out16_lo[(int64_t)m * e.ld + (n >> 1)] = __float2half_rn(h - __half2float(hh));
            }
        } break;
        case EPI_LOGITS: {
            e.out[n] = v0;
            e.out[n + 1] = v1;
            unsigned long long k = argmax_key(v0, n), k1 = argmax_key(v1, n + 1);
            atomicMax(e.argmax, k > k1 ? k : k1);
        } break;
        case EPI_QKV: {
            const int pos = (e.pos_dev ? __ldcg(e.pos_dev) : e.pos0) + m;
            const int D = e.head_dim;
            if (n < e.qd + e.kvd) {  // q or k: rotate the pair (2i, 2i+1) by theta(pos, i)
                const int d = (n < e.qd ? n : n - e.qd) % D;
                const float2 cs = e.rope[(int64_t)pos * (D / 2) + (d >> 1)];
                const float r0 = v0 * cs.x - v1 * cs.y, r1 = v0 * cs.y + v1 * cs.x;
                v0 = r0;
                v1 = r1;
            }
            if (n < e.qd) {
                if (e.out) {
                    e.out[(int64_t)m * e.ld + n] = v0;
                    e.out[(int64_t)m * e.ld + n + 1] = v1;
                }
            } else {
                const bool isk = n < e.qd + e.kvd;
                const int c = isk ? n - e.qd : n - e.qd - e.kvd;
                const int g = c / D, d = c % D;
                const int64_t idx = ((int64_t)g * e.max_ctx + pos) * D + d;
                void* base = isk ? e.kcache : e.vcache;
                if (e.kv_f16) {
                    *reinterpret_cast<__half2*>((__half*)base + idx) = __floats2half2_rn(v0, v1);
                } else {
                    *reinterpret_cast<float2*>((float*)base + idx) = make_float2(v0, v1);
                }
            }
        } break;
    }
}

// ---------------------------------------------------------------------------
// Host-side launchers (defined in the .cu files).
// ---------------------------------------------------------------------------
// Device error words of a model or a standalone weight: err[0] is the DEV_* code a kernel records when one of
// its bounded waits gives up (zero when healthy); err[1] is test instrumentation read by the decode GEMV: when
// nonzero, the GEMV's first wait polls an mbarrier nothing arrives on that many times and then takes its timeout
// path, so the error reporting can be exercised without a fault or a hang.
constexpr int kErrWords = 2;
struct GemvScratch {
    unsigned* err = nullptr;  // device, kErrWords words (above)
};

int num_sms();
constexpr int kMaxDevices = 64;  // per-device state (kernel attributes, static scratch addresses)

cudaError_t launch_repack(const uint8_t* src, const Planes& P, int N, int row0, int step, cudaStream_t s);
cudaError_t launch_rope_table(float2* tab, int max_ctx, int head_dim, double base, double yarn_scale,
                              cudaStream_t s);
cudaError_t launch_embed(const Planes& emb, const int* tok_dev, int n, float* x, int64_t ldx, cudaStream_t s);
// y = RMSNorm(x) per row, written as fp16 hi + lo planes (the tensor-core GEMM operand).
cudaError_t launch_rmsnorm_rows(const float* x, int n, int E, const float* w, float eps, __half* y_hi, __half* y_lo,
                                cudaStream_t s);
// x (fp32) -> fp16 hi + lo planes.
cudaError_t launch_split_f16(const float* x, __half* hi, __half* lo, int64_t n, cudaStream_t s);
// fp16 hi + lo planes -> out = hi + lo (fp32).
cudaError_t launch_join_f16(const __half* hi, const __half* lo, float* out, int64_t n, cudaStream_t s);

// y-part of the decode path: one matrix-vector product with optional RMSNorm
// prologue (norm_w != nullptr) and a fused epilogue.
cudaError_t launch_qgemv(const Planes& W, const float* x, const float* norm_w, float eps, const Epi& epi,
                         const GemvScratch& scr, cudaStream_t s);
// Opt the GEMV kernels in to their shared-memory ring (call once, before any stream capture).
cudaError_t qgemv_prepare();
// Largest number of K chunks (Kp / chunk_weights) a GEMV supports.
int qgemv_max_chunks();

// A 2-D TMA tensor map over an fp16 [rows][ld] array: box box_cols (innermost, 64 for SWIZZLE_128B) x box_rows,
// SWIZZLE_128B, zero fill outside the array.  false if the driver refuses it.
bool make_tmap_f16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_cols,
                   uint32_t box_rows);

// Split-K scratch of the prefill GEMM: fp32 partial tiles and one arrival counter per output tile (zero between
// launches; the last CTA of a tile resets its counter).  Launches on one stream may share it.
struct GemmSplit {
    float* ws = nullptr;
    size_t ws_bytes = 0;
    unsigned* cnt = nullptr;
    int cnt_n = 0;
};
// Workspace bytes the GEMM's split K wants for an N x K weight at M rows (0: no split), and the counters it needs.
size_t qgemm_ws_bytes(int N, int K, int M);
int qgemm_tiles(int N, int M);
// Prefill GEMM on the tensor cores: Y = X W^T for M rows with a fused epilogue.  X is given as fp16
// hi + lo planes [M][ldx] (ldx % 8 == 0, 16-byte aligned).  err: device error word.  split (nullable): scratch
// for splitting K where it pays; the split is limited to what the scratch holds.
cudaError_t launch_qgemm(const Planes& W, const __half* X_hi, const __half* X_lo, int64_t ldx, int M, const Epi& epi,
                         unsigned* err, cudaStream_t s, const GemmSplit* split = nullptr);
cudaError_t qgemm_prepare();

// Quantized KV cache (AF_KV_Q8_0 / AF_KV_Q4_0): every slot lives in the fp16 cache; slots that left the window
// also live in the quantized store, as codes (Q8_0: D int8 values in element order; Q4_0: D / 2 bytes, byte j
// = n(2j) | n(2j + 1) << 4 with n = q + 8) and D / 32 fp16 scales per slot, in the cache's
// [layer][kv head][slot] order.
struct KvStore {
    uint8_t* kq = nullptr;
    uint8_t* vq = nullptr;
    __half* ks = nullptr;
    __half* vs = nullptr;
    int qtype = 0;   // AF_KV_Q8_0 / AF_KV_Q4_0, 0 = the cache is not quantized
    int window = 0;  // slots kept fp16 behind a step's last position
};
__host__ __device__ inline int kv_code_bytes(int qtype, int D) { return qtype == AF_KV_Q8_0 ? D : D / 2; }

// One layer's view of the quantized store, for decode attention.
struct KvLayerStore {
    const uint8_t* kq = nullptr;
    const uint8_t* vq = nullptr;
    const __half* ks = nullptr;
    const __half* vs = nullptr;
    int qtype = 0;
    int window = 0;
};

// Retire slots first..first+count-1 (with pos_dev: the one slot *pos_dev - window) of every layer and kv head:
// quantize the slot's fp16 K and V rows into the store and write fp16(d q) back into the fp16 cache.  Slots
// below 0 are skipped.
cudaError_t launch_kv_retire(const KvStore& st, __half* kc, __half* vc, int L, int KVH, int max_ctx, int D,
                             const int* pos_dev, int first, int count, cudaStream_t s);

// Attention
struct AttnScratch {
    float* part = nullptr;    // [KVH][NS][G][D+2]
    unsigned* cnt = nullptr;  // [KVH], zero between launches
    unsigned* err = nullptr;  // device error word (a bounded wait gave up)
    int ns = 0;               // splits the partials have room for
};
// Whether decode attention over a cache of max_ctx slots takes the cluster path (partials merged through
// distributed shared memory: no global scratch) rather than the split path (partials and arrival counters in
// the scratch).  The path depends on the cache size only.
bool attn_decode_uses_cluster(int max_ctx);
// Splits the decode attention launches (grid.x) for this shape.
int attn_decode_splits(int n_heads, int n_kv_heads, int max_ctx);
size_t attn_decode_part_elems(int n_heads, int head_dim, int ns);
// qs (nullable): the layer's quantized store; kc, vc are then the fp16 cache and retired slots (below
// pos + 1 - window) are read from the store.
cudaError_t launch_attn_decode(const float* q, const void* kc, const void* vc, int kv_f16, int H, int KVH, int D,
                               int max_ctx, const int* pos_dev, int pos, const AttnScratch& scr, float* out,
                               cudaStream_t s, const KvLayerStore* qs = nullptr);
// Causal prefill attention on the tensor cores: S query rows at positions pos0.. (q fp32 [S][ldq], rotated),
// output as fp16 hi + lo planes [S][ldo].  err: device error word.
cudaError_t launch_attn_prefill(const float* q, int64_t ldq, const void* kc, const void* vc, int kv_f16, int H,
                                int KVH, int D, int max_ctx, int pos0, int S, __half* out_hi, __half* out_lo,
                                int64_t ldo, unsigned* err, cudaStream_t s);
bool attn_supported(int H, int KVH, int D);

// Sampler chain over the logits (one CTA): penalty, temperature, softmax, top-p, draw with uniform u.
int sampler_max_vocab();
cudaError_t launch_sample(const float* logits, int V, const int* recent, int n_recent, float penalty,
                          float temperature, float top_p, float u, int* token_out, cudaStream_t s);

// Capacity of the fixed decode-attention scratch (a file-scope device array, no allocation).
constexpr int kStaticAttnMaxKVH = 1024;                  // arrival counters (plus one error word)
constexpr size_t kStaticAttnPartFloats = (size_t)1 << 20;  // split partials (4 MiB)
// Device address of that scratch on the current device (looked up once per device).
cudaError_t attn_static_scratch(float** part, unsigned** cnt, unsigned** err);

// One GEMV of the persistent decode kernel: matrix, input, optional RMSNorm
// weight, rows per stage R and epilogue.
struct GemvTask {
    Planes W;
    const float* x = nullptr;
    const float* nw = nullptr;
    int R = 0;
    Epi epi;
};

struct LayerPlan {
    GemvTask qkv, o, gu, down;
    void* kc = nullptr;  // this layer's K cache [KVH][max_ctx][D]
    void* vc = nullptr;
};

struct StepState;

constexpr int kMaxSlotsP = 16;  // stage slots of the persistent decode kernel (one owner warp each)

struct DecodePlan {
    int wtype = 0, n_layers = 0, H = 0, KVH = 0, D = 0, max_ctx = 0, kv_f16 = 0, attn_splits = 0;
    int nslot = 0, slot_bytes = 0, att_T = 0;  // stage slots; cache slots per attention stage
    int ximg_bytes = 0, tab_bytes = 0;         // bytes of the x image / attention scratch region, of the schedule
    float eps = 0.f;
    const LayerPlan* layers = nullptr;  // device array [n_layers]
    Planes emb;
    GemvTask head;
    float* x = nullptr;
    float* q = nullptr;
    float* attn = nullptr;
    float* attn_part = nullptr;  // [KVH][splits][G][D+4]
    unsigned* attn_cnt = nullptr;  // [KVH], zero between steps
    StepState* st = nullptr;
    unsigned* bar_count = nullptr;  // grid barrier (zero-initialised)
    unsigned* bar_gen = nullptr;
    unsigned* abort = nullptr;      // raised by a CTA that timed out
    unsigned* err = nullptr;        // DEV_* code
    float* capture = nullptr;       // optional [n_layers+1][E] residual stream after embed / each layer
    unsigned long long* trace = nullptr;  // optional [2 + 5 n_layers + 1] %globaltimer at phase boundaries (CTA 0)
};

bool decode_gemv_task(const Planes& W, GemvTask& t);
int decode_attn_splits(int n_kv_heads);
int decode_max_cta_rows();
// Slot size and count, attention stage length and scratch of a plan whose head task, splits and shapes are
// set, given the host copy of a layer's tasks (every layer has the same shapes); false if the kernel cannot
// run it.
bool decode_configure(DecodePlan& p, const LayerPlan& l0);
cudaError_t decode_prepare(const DecodePlan& p);
cudaError_t launch_decode(const DecodePlan& p, cudaStream_t s);

// Decode-step bookkeeping
struct StepState {
    int token;  // token of this step
    int pos;    // position of this step
    unsigned long long argmax;
    int next_token;
    int pad;
};
cudaError_t launch_step_begin(StepState* st, int token, int pos, cudaStream_t s, unsigned* bar_count = nullptr);
cudaError_t launch_step_end(StepState* st, cudaStream_t s);

}  // namespace af
