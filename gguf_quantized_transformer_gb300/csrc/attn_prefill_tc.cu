// Causal GQA prefill attention on the 5th-generation tensor cores
// (Airframe "GPU_PIPELINE.md" per-layer ops: scores Q K^T / sqrt(head_dim),
// causal softmax over slots 0..t, weighted sum of V; dotLLM "GPU Inference",
// "Attention on GPU": GQA group = n_heads / n_kv_heads).
//
// CTA (query tile, kv head g): 128 query vectors = QT = 128/G rows x the G
// heads of the group (vector v = h * QT + row), so every K/V tile is used by
// all heads of the group.  One pass over the keys in tiles of BKV slots (64 for
// an fp16 cache, 32 for fp32), with warps specialised and the tiles pipelined:
//   warp 9      : bulk copies of each tile's raw K and V rows into a staging
//                 buffer (the next tile streams in while this one is converted);
//   warps 4..7  : convert the staged rows into the MMA operands of one of two
//                 buffers: K rows as they are (split hi + lo for fp32) and V
//                 transposed, so that keys run along K of the P V product;
//   warp 8      : one lane issues S = Q K^T for tile t, then O += P V for tile
//                 t - 1, each followed by a commit;
//   warps 0..3  : own the 128 TMEM lanes (one query vector each): the online
//                 softmax of S with the causal mask, P (fp16) into one of two
//                 buffers, and the epilogue.
// The running maximum is rescaled lazily: P uses a reference maximum that only
// moves (rescaling O in TMEM and the row sum) when a tile's maximum exceeds it
// by more than kLazy, so p <= e^kLazy and fp16 P stays in range.  O / l does not
// depend on the reference, so the result is the same as with the exact maximum.
// The output is O / l, written as the fp16 hi + lo planes the O-projection GEMM
// reads.
//
// Precision.  Q (scaled) is split into fp16 hi + lo, so the scores are
// near-fp32: S = Q_hi K + Q_lo K (+ Q_hi K_lo for an fp32 cache, which is split
// too; an fp16 cache is exact in fp16).  P is rounded to fp16 (a relative
// error <= 2^-12 per weight, so O / l moves by at most about 2^-12 of the V
// values' range; the row sum l keeps the unrounded p): O += P V_hi (+ P V_lo
// for an fp32 cache), fp32 accumulate.
//
// Operands live in shared memory in the SWIZZLE_128B K-major layout.  Every
// tcgen05.ld / st is executed by whole warps under warp-uniform conditions,
// and every mbarrier wait is bounded: a CTA that gives up records DEV_TIMEOUT,
// lets what it issued finish and frees its TMEM.
#include <math_constants.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace af {

namespace {

// Byte offset of 16-byte chunk c (8 fp16 along K) of row r in an operand of R rows stored as
// SWIZZLE_128B atoms of 64 K-elements: atom c/8 is a [R][128 B] block.
__device__ __forceinline__ uint32_t op_off(int R, int r, int c) {
    return (uint32_t)((c >> 3) * R * 128) + sw128(r, c & 7);
}

// Descriptor of the 16-wide K step kk of an operand with R rows at shared address base.
__device__ __forceinline__ uint64_t op_desc(uint32_t base, int R, int kk) {
    return umma_desc_sw128(base + (uint32_t)((kk >> 2) * R * 128 + (kk & 3) * 32));
}

__device__ __forceinline__ void ld8(const __half* p, float (&w)[8]) {
    const uint4 raw = *reinterpret_cast<const uint4*>(p);
    const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const float2 f = __half22float2(h[e]);
        w[2 * e] = f.x;
        w[2 * e + 1] = f.y;
    }
}
__device__ __forceinline__ void ld8(const float* p, float (&w)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}
// 8 floats written by an earlier kernel, read through L2
__device__ __forceinline__ void ld8_cg(const float* p, float (&w)[8]) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(p)), b = __ldcg(reinterpret_cast<const float4*>(p + 4));
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}
__device__ __forceinline__ void ld2(const float* p, float& a, float& b) {
    const float2 f = *reinterpret_cast<const float2*>(p);
    a = f.x;
    b = f.y;
}

// 2^x by the hardware's approximate base-2 exponential (relative error about 2^-22; results below 2^-126 flush
// to zero, which a probability of that size is)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 pack8_f16(const float (&w)[8]) {  // round to nearest fp16
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const __half2 hh = __floats2half2_rn(w[2 * i], w[2 * i + 1]);
        h[i] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}


constexpr int kPWarps = 10;
constexpr int kPThreads = kPWarps * 32;
constexpr int BQ = 128;          // query vectors per CTA = TMEM lanes
constexpr int kTmemCols = 256;   // S buffers at columns 0 and BKV, O at column 128 (D columns)
constexpr int kOCol = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.f * kLog2e;  // (log2 units) the reference maximum moves when a tile exceeds it by more:
                                       // p = 2^(s - m) stays below e^8

template <int D, typename KT>
struct PCfg {
    static constexpr bool SPLIT_KV = sizeof(KT) == 4;  // fp32 cache: K and V need hi + lo
    static constexpr int BKV = 64;                     // keys per tile (a whole 128-byte row of a P / V^T atom)
    static constexpr int NBUF = SPLIT_KV ? 1 : 2;      // operand buffers (an fp32 cache's hi + lo fill one's room)
    static constexpr int Q_BYTES = BQ * D * 2;         // one fp16 plane
    static constexpr int K_BYTES = BKV * D * 2;
    static constexpr int V_BYTES = D * BKV * 2;
    static constexpr int P_BYTES = BQ * BKV * 2;
    // one operand buffer: K hi (+ lo), V hi (+ lo), P
    static constexpr int B_KH = 0;
    static constexpr int B_KL = B_KH + K_BYTES;
    static constexpr int B_VH = B_KL + (SPLIT_KV ? K_BYTES : 0);
    static constexpr int B_VL = B_VH + V_BYTES;
    static constexpr int B_PH = B_VL + (SPLIT_KV ? V_BYTES : 0);
    static constexpr int BUF = (B_PH + P_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_QH = 0;
    static constexpr int OFF_QL = Q_BYTES;
    static constexpr int OFF_BUF = 2 * Q_BYTES;        // the operand buffers
    static constexpr int RAW_BYTES = BKV * D * (int)sizeof(KT);
    static constexpr int OFF_RK = OFF_BUF + NBUF * BUF;  // staging: raw K rows, then raw V rows
    static constexpr int OFF_RV = OFF_RK + RAW_BYTES;
    static constexpr int SMEM = OFF_RV + RAW_BYTES + 1024;  // + 1024-byte alignment slack
};

struct PSmem {
    uint64_t raw_full;     // staging filled (transaction bytes)
    uint64_t raw_empty;    // staging converted (4 converter warps)
    uint64_t op_full[2];   // K / V operands of buffer t % NBUF written (4 converter warps)
    uint64_t op_free[2];   // P V of buffer t % NBUF done: its operands and P are free (commit)
    uint64_t s_full[2];    // S of tile t in TMEM columns (t & 1) * BKV computed (commit)
    uint64_t p_full[2];    // P of tile t written, O rescaled if needed (4 softmax warps), indexed t & 1
    uint64_t done;         // every MMA finished (commit)
    uint32_t tmem_base;
    int fills;             // staging fills issued (for the drain on abort)
    volatile int abort;
};

// Bounded wait of a whole warp; false (warp-uniformly) after a timeout or when the CTA aborts.
__device__ __forceinline__ bool pwait(uint64_t* bar, unsigned parity, PSmem& sm, unsigned* err) {
    bool ok = false;
    for (unsigned i = 0; i < kWaitLimit && !ok; i++) {
        ok = mbar_try_wait(bar, parity);
        if (!ok && sm.abort) break;
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0 && !sm.abort) {
        sm.abort = 1;
        atomicExch(err, (unsigned)DEV_TIMEOUT);
    }
    return ok;
}
// the same for one thread (the MMA issuer and the copy producer)
__device__ __forceinline__ bool pwait1(uint64_t* bar, unsigned parity, PSmem& sm, unsigned* err) {
    for (unsigned i = 0; i < kWaitLimit; i++) {
        if (mbar_try_wait(bar, parity)) return true;
        if (sm.abort) return false;
    }
    sm.abort = 1;
    atomicExch(err, (unsigned)DEV_TIMEOUT);
    return false;
}

template <int D, int G, typename KT>
__global__ void __launch_bounds__(kPThreads, 1)
    attn_prefill_tc_kernel(const float* __restrict__ q, int64_t ldq, const KT* __restrict__ kc,
                           const KT* __restrict__ vc, int max_ctx, int pos0, int S, __half* __restrict__ out_hi,
                           __half* __restrict__ out_lo, int64_t ldo, unsigned* err) {
    using C = PCfg<D, KT>;
    constexpr int QT = BQ / G;     // query rows per CTA
    constexpr int BKV = C::BKV;
    constexpr uint32_t kIdS = idesc_f16(BQ, BKV);  // S = Q K^T: M = 128 vectors, N = BKV keys, K = D
    constexpr uint32_t kIdO = idesc_f16(BQ, D);    // O += P V: M = 128 vectors, N = D, K = BKV keys
    extern __shared__ uint8_t smem_raw[];
    __shared__ PSmem sm;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.y, r0 = blockIdx.x * QT;
    const int nrows = min(QT, S - r0);               // query rows of this tile
    const int nkeys = pos0 + r0 + nrows;             // slots 0..(last query position)
    const int ntiles = (nkeys + BKV - 1) / BKV;
    const KT* K = kc + (int64_t)g * max_ctx * D;
    const KT* V = vc + (int64_t)g * max_ctx * D;

    pdl_launch_dependents();
    if (tid == 0) {
        mbar_init(&sm.raw_full, 1);
        mbar_init(&sm.raw_empty, 4);
        for (int b = 0; b < 2; b++) {
            mbar_init(&sm.op_full[b], 4);
            mbar_init(&sm.s_full[b], 1);
            mbar_init(&sm.p_full[b], 4);
            mbar_init(&sm.op_free[b], 1);
        }
        mbar_init(&sm.done, 1);
        sm.fills = 0;
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    pdl_wait();  // q and the cache rows of this chunk are written by the previous kernel
    constexpr int NB = C::NBUF;
    auto buf = [&](int b) { return smem + C::OFF_BUF + b * C::BUF; };

    // ---- Q tile (all threads): vector v = h * QT + row, scaled by log2(e) / sqrt(D) (scores in base-2 units:
    // p = 2^(s - m) = e^(q.k/sqrt(D) - m')), split hi + lo
    {
        const float scale = rsqrtf((float)D) * kLog2e;
        for (int i = tid; i < BQ * (D / 8); i += kPThreads) {
            const int v = i / (D / 8), c = i % (D / 8);
            const int h = v / QT, rr = v % QT;
            float w[8];
            if (rr < nrows) {
                ld8_cg(q + (int64_t)(r0 + rr) * ldq + (int64_t)(g * G + h) * D + 8 * c, w);
#pragma unroll
                for (int e = 0; e < 8; e++) w[e] *= scale;
            } else {
#pragma unroll
                for (int e = 0; e < 8; e++) w[e] = 0.f;
            }
            uint4 hi, lo;
            split8(w, hi, lo);
            *reinterpret_cast<uint4*>(smem + C::OFF_QH + op_off(BQ, v, c)) = hi;
            *reinterpret_cast<uint4*>(smem + C::OFF_QL + op_off(BQ, v, c)) = lo;
        }
    }
    fence_proxy_async_shared();  // Q (generic-proxy writes) -> visible to the tensor core
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 9) {
        // ---------------- staging producer: raw K and V rows of tile t (one bulk copy each)
        if (lane == 0) {
            for (int t = 0; t < ntiles; t++) {
                if (t > 0 && !pwait1(&sm.raw_empty, (t - 1) & 1, sm, err)) break;
                const int keys = min(BKV, nkeys - t * BKV);
                const unsigned bytes = (unsigned)(keys * D * (int)sizeof(KT));
                mbar_arrive_expect_tx(&sm.raw_full, 2 * bytes);
                bulk_g2s(smem + C::OFF_RK, K + (int64_t)t * BKV * D, bytes, &sm.raw_full);
                bulk_g2s(smem + C::OFF_RV, V + (int64_t)t * BKV * D, bytes, &sm.raw_full);
                sm.fills = t + 1;
            }
            // every fill is consumed before the converters finish, so nothing is in flight past the final barrier
            // unless the CTA aborted (then the drain below waits for the last fill)
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- converters: staging -> K / V operands of buffer t % NBUF
        const int ct = tid - 128;  // 0..127
        const KT* stK = reinterpret_cast<const KT*>(smem + C::OFF_RK);
        const KT* stV = reinterpret_cast<const KT*>(smem + C::OFF_RV);
        for (int t = 0; t < ntiles; t++) {
            const int b = t % NB;
            if (!pwait(&sm.raw_full, t & 1, sm, err)) break;
            // the buffer's previous tile (t - NBUF) is multiplied: P V done
            if (t >= NB && !pwait(&sm.op_free[b], ((t - NB) / NB) & 1, sm, err)) break;
            uint8_t* ob = buf(b);
            // K tile: rows = keys, K axis = D
            for (int i = ct; i < BKV * (D / 8); i += 128) {
                const int j = i / (D / 8), c = i % (D / 8);
                const bool in = t * BKV + j < nkeys;
                if (C::SPLIT_KV) {
                    float w[8];
                    if (in) {
                        ld8(stK + (int64_t)j * D + 8 * c, w);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; e++) w[e] = 0.f;
                    }
                    uint4 hi, lo;
                    split8(w, hi, lo);
                    *reinterpret_cast<uint4*>(ob + C::B_KH + op_off(BKV, j, c)) = hi;
                    *reinterpret_cast<uint4*>(ob + C::B_KL + op_off(BKV, j, c)) = lo;
                } else {  // fp16 rows: the chunk is already the operand's
                    *reinterpret_cast<uint4*>(ob + C::B_KH + op_off(BKV, j, c)) =
                        in ? *reinterpret_cast<const uint4*>(stK + (int64_t)j * D + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // V tile transposed: rows = d, K axis = keys (thread: dims 2dp, 2dp + 1 of 8 keys)
            for (int i = ct; i < (D / 2) * (BKV / 8); i += 128) {
                const int dp = i % (D / 2), kg = i / (D / 2);
                if constexpr (!C::SPLIT_KV) {  // fp16: word e holds (dim 2dp, dim 2dp + 1) of key 8kg + e
                    uint32_t wv[8];
#pragma unroll
                    for (int e = 0; e < 8; e++)
                        wv[e] = t * BKV + 8 * kg + e < nkeys
                                    ? *reinterpret_cast<const uint32_t*>(stV + (int64_t)(8 * kg + e) * D + 2 * dp)
                                    : 0u;
                    uint4 a4, b4;
                    a4.x = __byte_perm(wv[0], wv[1], 0x5410); b4.x = __byte_perm(wv[0], wv[1], 0x7632);
                    a4.y = __byte_perm(wv[2], wv[3], 0x5410); b4.y = __byte_perm(wv[2], wv[3], 0x7632);
                    a4.z = __byte_perm(wv[4], wv[5], 0x5410); b4.z = __byte_perm(wv[4], wv[5], 0x7632);
                    a4.w = __byte_perm(wv[6], wv[7], 0x5410); b4.w = __byte_perm(wv[6], wv[7], 0x7632);
                    *reinterpret_cast<uint4*>(ob + C::B_VH + op_off(D, 2 * dp, kg)) = a4;
                    *reinterpret_cast<uint4*>(ob + C::B_VH + op_off(D, 2 * dp + 1, kg)) = b4;
                } else {  // fp32: split hi + lo
                    float a[8], bb[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        if (t * BKV + 8 * kg + e < nkeys) {
                            ld2(stV + (int64_t)(8 * kg + e) * D + 2 * dp, a[e], bb[e]);
                        } else {
                            a[e] = 0.f;
                            bb[e] = 0.f;
                        }
                    }
                    uint4 ah, al, bh, bl;
                    split8(a, ah, al);
                    split8(bb, bh, bl);
                    *reinterpret_cast<uint4*>(ob + C::B_VH + op_off(D, 2 * dp, kg)) = ah;
                    *reinterpret_cast<uint4*>(ob + C::B_VH + op_off(D, 2 * dp + 1, kg)) = bh;
                    *reinterpret_cast<uint4*>(ob + C::B_VL + op_off(D, 2 * dp, kg)) = al;
                    *reinterpret_cast<uint4*>(ob + C::B_VL + op_off(D, 2 * dp + 1, kg)) = bl;
                }
            }
            fence_proxy_async_shared();  // the operands -> visible to the tensor core
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.raw_empty);   // the staging may be refilled
                mbar_arrive(&sm.op_full[b]);  // the operands of tile t are ready
            }
        }
    } else if (warp == 8) {
        // ---------------- MMA issuer: S(t), then O += P V for tile t - 1
        if (lane == 0) {
            auto issue_pv = [&](int t) {
                const int b = t % NB;
                const uint8_t* ob = buf(b);
                const uint32_t ph = smem_u32(ob + C::B_PH);
                const uint32_t vh = smem_u32(ob + C::B_VH), vl = smem_u32(ob + C::B_VL);
                for (int kk = 0; kk < BKV / 16; kk++) {
                    const uint64_t dvh = op_desc(vh, D, kk);
                    const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
                    mma_f16(tmem + kOCol, op_desc(ph, BQ, kk), dvh, kIdO, acc);
                    if (C::SPLIT_KV) mma_f16(tmem + kOCol, op_desc(ph, BQ, kk), op_desc(vl, D, kk), kIdO, 1u);
                }
                mma_commit(&sm.op_free[b]);
            };
            // with one operand buffer the converters wait for P V(t - 1) before they fill it for tile t, so that
            // P V goes first; with two, S(t) goes first so that the softmax of tile t overlaps P V(t - 1)
            int t = 0;
            for (; t < ntiles; t++) {
                const int b = t % NB;
                if (NB == 1 && t > 0) {
                    if (!pwait1(&sm.p_full[(t - 1) & 1], ((t - 1) >> 1) & 1, sm, err)) break;
                    tc_fence_after();
                    issue_pv(t - 1);
                }
                if (!pwait1(&sm.op_full[b], (t / NB) & 1, sm, err)) break;
                tc_fence_after();
                const uint8_t* ob = buf(b);
                const uint32_t kh = smem_u32(ob + C::B_KH), kl = smem_u32(ob + C::B_KL);
                const uint32_t scol = tmem + (uint32_t)((t & 1) * BKV);
                for (int kk = 0; kk < D / 16; kk++) {
                    const uint64_t dkh = op_desc(kh, BKV, kk);
                    mma_f16(scol, op_desc(sbase + C::OFF_QH, BQ, kk), dkh, kIdS, kk > 0 ? 1u : 0u);
                    mma_f16(scol, op_desc(sbase + C::OFF_QL, BQ, kk), dkh, kIdS, 1u);
                    if (C::SPLIT_KV) mma_f16(scol, op_desc(sbase + C::OFF_QH, BQ, kk), op_desc(kl, BKV, kk), kIdS, 1u);
                }
                mma_commit(&sm.s_full[t & 1]);
                if (NB > 1 && t > 0) {  // the previous tile's P is ready: its P V
                    if (!pwait1(&sm.p_full[(t - 1) & 1], ((t - 1) >> 1) & 1, sm, err)) break;
                    tc_fence_after();
                    issue_pv(t - 1);
                }
            }
            if (t == ntiles && !sm.abort && pwait1(&sm.p_full[(t - 1) & 1], ((t - 1) >> 1) & 1, sm, err)) {
                tc_fence_after();
                issue_pv(t - 1);
            }
            mma_commit(&sm.done);  // always: also after a break, so the drain can wait on it
        }
    } else {
        // ---------------- softmax warps 0..3: TMEM lane = query vector
        const int v = warp * 32 + lane;
        const int rr = v % QT;
        const bool vrow = rr < nrows;
        const int qpos = pos0 + r0 + rr;
        float m_ref = -CUDART_INF_F, l = 0.f;
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        for (int t = 0; t < ntiles; t++) {
            const int b = t % NB, sb = t & 1;
            if (!pwait(&sm.s_full[sb], (t >> 1) & 1, sm, err)) break;
            tc_fence_after();
            float mt = -CUDART_INF_F;  // this tile's maximum of the row (S is read twice from TMEM: max, then p)
            // below the diagonal for every row of the warp: no mask (rows past the chunk see zero q: harmless)
            const bool whole = __all_sync(0xffffffffu, !vrow || t * BKV + BKV - 1 <= qpos);
#pragma unroll
            for (int c32 = 0; c32 < BKV / 32; c32++) {
                float s32[32];
                tmem_ld32(lane_addr + (uint32_t)(sb * BKV + c32 * 32), s32);
                if (whole) {
#pragma unroll
                    for (int e = 0; e < 32; e++) mt = fmaxf(mt, s32[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e++)
                        if (vrow && t * BKV + c32 * 32 + e <= qpos) mt = fmaxf(mt, s32[e]);
                }
            }
            // the reference maximum moves only when this tile exceeds it by more than kLazy
            const bool move = mt > m_ref + kLazy;
            if (__any_sync(0xffffffffu, move && t > 0)) {
                // O holds tiles < t: wait for the previous P V, then rescale this warp's rows (warp-collective)
                if (!pwait(&sm.op_free[(t - 1) % NB], ((t - 1) / NB) & 1, sm, err)) break;
                tc_fence_after();
                const float f = move ? ex2(m_ref - mt) : 1.f;
#pragma unroll
                for (int c32 = 0; c32 < D / 32; c32++) {
                    float o[32];
                    tmem_ld32(lane_addr + (uint32_t)(kOCol + c32 * 32), o);
                    uint32_t ou[32];
#pragma unroll
                    for (int e = 0; e < 32; e++) ou[e] = __float_as_uint(o[e] * f);
                    tmem_st32(lane_addr + (uint32_t)(kOCol + c32 * 32), ou);
                }
                tmem_st_wait();
                l *= f;
            }
            if (move) m_ref = mt;
            // P of tile t into buffer b (its previous P, of tile t - NBUF, was consumed: the converters waited on
            // that P V before writing this buffer's operands, and S(t) came after)
            uint8_t* ob = buf(b);
#pragma unroll
            for (int c32 = 0; c32 < BKV / 32; c32++) {
                float s32[32];
                tmem_ld32(lane_addr + (uint32_t)(sb * BKV + c32 * 32), s32);
#pragma unroll
                for (int q8 = 0; q8 < 4; q8++) {
                    float w[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const int key = t * BKV + c32 * 32 + q8 * 8 + e;
                        const float p = (whole || (vrow && key <= qpos)) ? ex2(s32[q8 * 8 + e] - m_ref) : 0.f;
                        l += p;
                        w[e] = p;
                    }
                    *reinterpret_cast<uint4*>(ob + C::B_PH + op_off(BQ, v, c32 * 4 + q8)) = pack8_f16(w);
                }
            }
            fence_proxy_async_shared();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full[sb]);
        }
        // ---- epilogue: O / l as fp16 hi + lo (whole warps load; lanes of valid rows store)
        if (__all_sync(0xffffffffu, !sm.abort) && pwait(&sm.done, 0, sm, err)) {
            tc_fence_after();
            const float inv = vrow ? 1.f / l : 0.f;
            const int64_t o0 = (int64_t)(r0 + rr) * ldo + (int64_t)(g * G + v / QT) * D;
#pragma unroll
            for (int c32 = 0; c32 < D / 32; c32++) {
                float o[32];
                tmem_ld32(lane_addr + (uint32_t)(kOCol + c32 * 32), o);
                if (vrow) {
#pragma unroll
                    for (int q8 = 0; q8 < 4; q8++) {
                        float w[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) w[e] = o[q8 * 8 + e] * inv;
                        uint4 hi, lo;
                        split8(w, hi, lo);
                        *reinterpret_cast<uint4*>(out_hi + o0 + c32 * 32 + q8 * 8) = hi;
                        *reinterpret_cast<uint4*>(out_lo + o0 + c32 * 32 + q8 * 8) = lo;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (sm.abort && tid == 0) {  // let the issued MMAs and the last staging fill issued finish before leaving
        mbar_wait_bounded(&sm.done, 0);
        if (sm.fills > 0) mbar_wait_bounded(&sm.raw_full, (unsigned)((sm.fills - 1) & 1));
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_free(tmem, kTmemCols);
    }
}

}  // namespace

namespace {

template <int D, int G, typename KT>
cudaError_t launch_pf(const float* q, int64_t ldq, const void* kc, const void* vc, int KVH, int max_ctx, int pos0,
                      int S, __half* out_hi, __half* out_lo, int64_t ldo, unsigned* err, cudaStream_t s) {
    constexpr int QT = BQ / G;
    auto k = attn_prefill_tc_kernel<D, G, KT>;
    const int smem = PCfg<D, KT>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((S + QT - 1) / QT, KVH);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, q, ldq, (const KT*)kc, (const KT*)vc, max_ctx, pos0, S, out_hi, out_lo, ldo,
                              err);
}

template <int D, int G>
cudaError_t dispatch_pf(const float* q, int64_t ldq, const void* kc, const void* vc, int kv_f16, int KVH,
                        int max_ctx, int pos0, int S, __half* out_hi, __half* out_lo, int64_t ldo, unsigned* err,
                        cudaStream_t s) {
    if (kv_f16) return launch_pf<D, G, __half>(q, ldq, kc, vc, KVH, max_ctx, pos0, S, out_hi, out_lo, ldo, err, s);
    return launch_pf<D, G, float>(q, ldq, kc, vc, KVH, max_ctx, pos0, S, out_hi, out_lo, ldo, err, s);
}

}  // namespace

cudaError_t launch_attn_prefill(const float* q, int64_t ldq, const void* kc, const void* vc, int kv_f16, int H,
                                int KVH, int D, int max_ctx, int pos0, int S, __half* out_hi, __half* out_lo,
                                int64_t ldo, unsigned* err, cudaStream_t s) {
    if (S < 1) return cudaSuccess;
    if (ldq % 4 || ldo % 8) return cudaErrorInvalidValue;  // vector loads of q, 16-byte stores of the output
    const int G = H / KVH;
    switch (D * 100 + G) {
        case 6401: return dispatch_pf<64, 1>(q, ldq, kc, vc, kv_f16, KVH, max_ctx, pos0, S, out_hi, out_lo, ldo, err, s);
        case 6402: return dispatch_pf<64, 2>(q, ldq, kc, vc, kv_f16, KVH, max_ctx, pos0, S, out_hi, out_lo, ldo, err, s);
        case 6404: return dispatch_pf<64, 4>(q, ldq, kc, vc, kv_f16, KVH, max_ctx, pos0, S, out_hi, out_lo, ldo, err, s);
        case 6408: return dispatch_pf<64, 8>(q, ldq, kc, vc, kv_f16, KVH, max_ctx, pos0, S, out_hi, out_lo, ldo, err, s);
        case 12801: return dispatch_pf<128, 1>(q, ldq, kc, vc, kv_f16, KVH, max_ctx, pos0, S, out_hi, out_lo, ldo, err, s);
        case 12802: return dispatch_pf<128, 2>(q, ldq, kc, vc, kv_f16, KVH, max_ctx, pos0, S, out_hi, out_lo, ldo, err, s);
        case 12804: return dispatch_pf<128, 4>(q, ldq, kc, vc, kv_f16, KVH, max_ctx, pos0, S, out_hi, out_lo, ldo, err, s);
        case 12808: return dispatch_pf<128, 8>(q, ldq, kc, vc, kv_f16, KVH, max_ctx, pos0, S, out_hi, out_lo, ldo, err, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace af
