// Causal GQA prefill attention on the 5th-generation tensor cores
// (Airframe "GPU_PIPELINE.md" per-layer ops: scores Q K^T / sqrt(head_dim),
// causal softmax over slots 0..t, weighted sum of V; dotLLM "GPU Inference",
// "Attention on GPU": GQA group = n_heads / n_kv_heads).
//
// CTA (query tile, kv head g): 128 query vectors = QT = 128/G rows x the G
// heads of the group (vector v = h * QT + row), so every K/V tile is used by
// all heads of the group.  Keys stream in tiles of BKV = 64 slots: one bulk
// copy each of the tile's raw K and V rows into a staging buffer, issued while
// the previous tile is multiplied, so the loads overlap the MMAs and the
// softmax.  Two passes over the keys:
//   pass A: S = Q_hi K_hi^T (one MMA per 16-wide K step) -> per-row maximum m;
//   pass B: S = Q K^T exactly (hi/lo split, below) -> p = exp(s - m) with the
//           causal mask, row sums l, P (fp16 hi + lo) written to shared memory,
//           O += P V accumulated in TMEM across all key tiles.
// With the maximum known before pass B nothing is ever rescaled; the output
// is O / l, written as the fp16 hi + lo planes the O-projection GEMM reads.
//
// Precision.  Q (scaled by 1/sqrt(D)) and P are split into fp16 hi + lo; an
// fp16 cache is exact in fp16, an fp32 cache is split too.  The products
// kept are A_hi B_hi + A_lo B_hi (+ A_hi B_lo for an fp32 cache), fp32
// accumulate: near-fp32 scores and outputs.
//
// Operands live in shared memory in the SWIZZLE_128B K-major layout, written
// by the CTA's threads (Q from the fp32 q rows; K rows as they are and V
// transposed, so that keys run along K of the P V product, both from the
// staging buffer).  One thread issues
// the MMAs; warps 0-3 own the 128 TMEM lanes (one query vector each) for the
// softmax and the epilogue (every tcgen05.ld is executed by whole warps under
// warp-uniform conditions).  Every wait on the MMA barrier is bounded.
#include <math_constants.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace af {

namespace {

constexpr int kPThreads = 256;
constexpr int BQ = 128;          // query vectors per CTA = TMEM lanes
constexpr int kTmemCols = 256;   // S at column 0 (BKV columns), O at column 128 (D columns)
constexpr int kOCol = 128;

template <int D, typename KT>
struct PCfg {
    static constexpr bool SPLIT_KV = sizeof(KT) == 4;  // fp32 cache: K and V need hi + lo
    static constexpr int BKV = 64;                     // keys per tile
    static constexpr int Q_BYTES = BQ * D * 2;         // one fp16 plane
    static constexpr int K_BYTES = BKV * D * 2;
    static constexpr int V_BYTES = D * BKV * 2;
    static constexpr int P_BYTES = BQ * BKV * 2;
    static constexpr int OFF_QH = 0;
    static constexpr int OFF_QL = OFF_QH + Q_BYTES;
    static constexpr int OFF_KH = OFF_QL + Q_BYTES;
    static constexpr int OFF_KL = OFF_KH + K_BYTES;
    static constexpr int OFF_VH = OFF_KL + (SPLIT_KV ? K_BYTES : 0);
    static constexpr int OFF_VL = OFF_VH + V_BYTES;
    static constexpr int OFF_PH = OFF_VL + (SPLIT_KV ? V_BYTES : 0);
    static constexpr int OFF_PL = OFF_PH + P_BYTES;
    static constexpr int RAW_BYTES = BKV * D * (int)sizeof(KT);  // one tile of raw cache rows
    static constexpr int OFF_RK = OFF_PL + P_BYTES;              // staging: raw K rows, then raw V rows
    static constexpr int OFF_RV = OFF_RK + RAW_BYTES;
    static constexpr int SMEM = OFF_RV + RAW_BYTES + 1024;       // + 1024-byte alignment slack
};

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
__device__ __forceinline__ void ld2(const __half* p, float& a, float& b) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(p));
    a = f.x;
    b = f.y;
}
__device__ __forceinline__ void ld2(const float* p, float& a, float& b) {
    const float2 f = *reinterpret_cast<const float2*>(p);
    a = f.x;
    b = f.y;
}

__device__ __forceinline__ uint4 pack8_f16(const float (&w)[8]) {  // exact for values that are fp16
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const __half2 hh = __floats2half2_rn(w[2 * i], w[2 * i + 1]);
        h[i] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

struct PSmem {
    uint64_t mma_bar;
    uint64_t raw_bar;  // staging filled (transaction bytes)
    uint32_t tmem_base;
    volatile int abort;
};

// Bounded wait on the MMA barrier (all threads); false after a timeout (recorded once).
__device__ __forceinline__ bool wait_mma(PSmem& sm, unsigned parity, unsigned* err) {
    if (mbar_wait_bounded(&sm.mma_bar, parity)) return true;
    sm.abort = 1;
    atomicExch(err, (unsigned)DEV_TIMEOUT);
    return false;
}

}  // namespace

namespace {

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

    if (tid == 0) {
        mbar_init(&sm.mma_bar, 1);
        mbar_init(&sm.raw_bar, 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    // ---- staging of raw cache rows: one bulk copy of the keys of tile t (K, and V in pass B), issued by one
    // thread; every wait is bounded, and the phase flips once per fill.
    const KT* stK = reinterpret_cast<const KT*>(smem + C::OFF_RK);
    const KT* stV = reinterpret_cast<const KT*>(smem + C::OFF_RV);
    unsigned raw_phase = 0;
    auto raw_issue = [&](int t, bool with_v) {  // thread 0 only
        const int keys = min(BKV, nkeys - t * BKV);
        const unsigned bytes = (unsigned)(keys * D * (int)sizeof(KT));
        mbar_arrive_expect_tx(&sm.raw_bar, with_v ? 2 * bytes : bytes);
        bulk_g2s(smem + C::OFF_RK, K + (int64_t)t * BKV * D, bytes, &sm.raw_bar);
        if (with_v) bulk_g2s(smem + C::OFF_RV, V + (int64_t)t * BKV * D, bytes, &sm.raw_bar);
    };
    auto raw_wait = [&]() {  // all threads; false after a timeout (the fill stays pending for the drain)
        const bool ok = mbar_wait_bounded(&sm.raw_bar, raw_phase);
        if (!ok) {
            sm.abort = 1;
            atomicExch(err, (unsigned)DEV_TIMEOUT);
            return false;
        }
        raw_phase ^= 1u;
        return true;
    };
    bool raw_pending = false;  // thread 0: a fill it issued has not been waited for (the drain on abort)
    if (tid == 0) {
        raw_issue(0, false);
        raw_pending = true;
    }

    // ---- Q tile: vector v = h * QT + row, scaled by 1/sqrt(D), split hi + lo
    {
        const float scale = rsqrtf((float)D);
        for (int i = tid; i < BQ * (D / 8); i += kPThreads) {
            const int v = i / (D / 8), c = i % (D / 8);
            const int h = v / QT, rr = v % QT;
            float w[8];
            if (rr < nrows) {
                ld8(q + (int64_t)(r0 + rr) * ldq + (int64_t)(g * G + h) * D + 8 * c, w);
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
    // K tile t: rows = keys, K axis = D
    auto load_k = [&](int t, bool with_lo) {
        for (int i = tid; i < BKV * (D / 8); i += kPThreads) {
            const int j = i / (D / 8), c = i % (D / 8);
            const int key = t * BKV + j;
            float w[8];
            if (key < nkeys) {
                ld8(stK + (int64_t)j * D + 8 * c, w);
            } else {
#pragma unroll
                for (int e = 0; e < 8; e++) w[e] = 0.f;
            }
            if (C::SPLIT_KV) {
                uint4 hi, lo;
                split8(w, hi, lo);
                *reinterpret_cast<uint4*>(smem + C::OFF_KH + op_off(BKV, j, c)) = hi;
                if (with_lo) *reinterpret_cast<uint4*>(smem + C::OFF_KL + op_off(BKV, j, c)) = lo;
            } else {
                *reinterpret_cast<uint4*>(smem + C::OFF_KH + op_off(BKV, j, c)) = pack8_f16(w);
            }
        }
    };
    // V tile t transposed: rows = d, K axis = keys (thread: dims 2dp, 2dp+1 of 8 keys)
    auto load_v = [&](int t) {
        for (int i = tid; i < (D / 2) * (BKV / 8); i += kPThreads) {
            const int dp = i % (D / 2), kg = i / (D / 2);
            float a[8], b[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const int key = t * BKV + 8 * kg + e;
                if (key < nkeys) {
                    ld2(stV + (int64_t)(8 * kg + e) * D + 2 * dp, a[e], b[e]);
                } else {
                    a[e] = 0.f;
                    b[e] = 0.f;
                }
            }
            if (C::SPLIT_KV) {
                uint4 ah, al, bh, bl;
                split8(a, ah, al);
                split8(b, bh, bl);
                *reinterpret_cast<uint4*>(smem + C::OFF_VH + op_off(D, 2 * dp, kg)) = ah;
                *reinterpret_cast<uint4*>(smem + C::OFF_VH + op_off(D, 2 * dp + 1, kg)) = bh;
                *reinterpret_cast<uint4*>(smem + C::OFF_VL + op_off(D, 2 * dp, kg)) = al;
                *reinterpret_cast<uint4*>(smem + C::OFF_VL + op_off(D, 2 * dp + 1, kg)) = bl;
            } else {
                *reinterpret_cast<uint4*>(smem + C::OFF_VH + op_off(D, 2 * dp, kg)) = pack8_f16(a);
                *reinterpret_cast<uint4*>(smem + C::OFF_VH + op_off(D, 2 * dp + 1, kg)) = pack8_f16(b);
            }
        }
    };
    // generic-proxy writes of the operands -> visible to the tensor core; then one thread issues
    auto publish = [&]() {
        fence_proxy_async_shared();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    // softmax state of this thread's query vector (warps 0..3: TMEM lane = vector)
    const int v = warp * 32 + lane;
    const int rr = v % QT;
    const bool vrow = warp < 4 && rr < nrows;
    const int qpos = pos0 + r0 + rr;
    float m = -CUDART_INF_F, l = 0.f;
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    unsigned phase = 0;

    // ---- pass A: row maxima from Q_hi K_hi^T
    for (int t = 0; t < ntiles && !sm.abort; t++) {
        if (__syncthreads_or(!raw_wait())) break;  // block-uniform
        raw_pending = false;
        load_k(t, false);
        publish();
        if (tid == 0 && !sm.abort) {  // the staging is free: the next tile (pass B starts over at tile 0 with V)
            fence_proxy_async_shared();
            if (t + 1 < ntiles) raw_issue(t + 1, false);
            else raw_issue(0, true);
            raw_pending = true;
        }
        if (tid == 0) {
            for (int kk = 0; kk < D / 16; kk++)
                mma_f16(tmem, op_desc(sbase + C::OFF_QH, BQ, kk), op_desc(sbase + C::OFF_KH, BKV, kk), kIdS,
                        kk > 0 ? 1u : 0u);
            mma_commit(&sm.mma_bar);
        }
        const bool ok = __all_sync(0xffffffffu, wait_mma(sm, phase, err));  // warp-uniform for tcgen05.ld
        phase ^= 1u;
        tc_fence_after();
        if (ok && warp < 4) {
#pragma unroll
            for (int c32 = 0; c32 < BKV / 32; c32++) {
                float s[32];
                tmem_ld32(lane_addr + (uint32_t)(c32 * 32), s);
#pragma unroll
                for (int e = 0; e < 32; e++) {
                    const int key = t * BKV + c32 * 32 + e;
                    if (key <= qpos) m = fmaxf(m, s[e]);
                }
            }
        }
        tc_fence_before();
        __syncthreads();
    }
    if (!vrow) m = 0.f;

    // ---- pass B: exact scores, P, O += P V
    for (int t = 0; t < ntiles && !sm.abort; t++) {
        if (__syncthreads_or(!raw_wait())) break;  // block-uniform
        raw_pending = false;
        load_k(t, true);
        load_v(t);
        publish();
        if (tid == 0 && !sm.abort && t + 1 < ntiles) {
            fence_proxy_async_shared();
            raw_issue(t + 1, true);
            raw_pending = true;
        }
        if (tid == 0) {
            for (int kk = 0; kk < D / 16; kk++) {
                const uint64_t kh = op_desc(sbase + C::OFF_KH, BKV, kk);
                mma_f16(tmem, op_desc(sbase + C::OFF_QH, BQ, kk), kh, kIdS, kk > 0 ? 1u : 0u);
                mma_f16(tmem, op_desc(sbase + C::OFF_QL, BQ, kk), kh, kIdS, 1u);
                if (C::SPLIT_KV)
                    mma_f16(tmem, op_desc(sbase + C::OFF_QH, BQ, kk), op_desc(sbase + C::OFF_KL, BKV, kk), kIdS, 1u);
            }
            mma_commit(&sm.mma_bar);
        }
        bool ok = __all_sync(0xffffffffu, wait_mma(sm, phase, err));
        phase ^= 1u;
        tc_fence_after();
        if (ok && warp < 4) {
#pragma unroll
            for (int c32 = 0; c32 < BKV / 32; c32++) {
                float s[32];
                tmem_ld32(lane_addr + (uint32_t)(c32 * 32), s);
#pragma unroll
                for (int q8 = 0; q8 < 4; q8++) {
                    float w[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const int key = t * BKV + c32 * 32 + q8 * 8 + e;
                        const float p = (vrow && key <= qpos) ? __expf(s[q8 * 8 + e] - m) : 0.f;
                        l += p;
                        w[e] = p;
                    }
                    uint4 hi, lo;
                    split8(w, hi, lo);
                    const int c = c32 * 4 + q8;  // 16-byte chunk along the keys
                    *reinterpret_cast<uint4*>(smem + C::OFF_PH + op_off(BQ, v, c)) = hi;
                    *reinterpret_cast<uint4*>(smem + C::OFF_PL + op_off(BQ, v, c)) = lo;
                }
            }
        }
        publish();
        if (sm.abort) break;
        if (tid == 0) {
            for (int kk = 0; kk < BKV / 16; kk++) {
                const uint64_t vh = op_desc(sbase + C::OFF_VH, D, kk);
                const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
                mma_f16(tmem + kOCol, op_desc(sbase + C::OFF_PH, BQ, kk), vh, kIdO, acc);
                mma_f16(tmem + kOCol, op_desc(sbase + C::OFF_PL, BQ, kk), vh, kIdO, 1u);
                if (C::SPLIT_KV)
                    mma_f16(tmem + kOCol, op_desc(sbase + C::OFF_PH, BQ, kk), op_desc(sbase + C::OFF_VL, D, kk),
                            kIdO, 1u);
            }
            mma_commit(&sm.mma_bar);
        }
        ok = __all_sync(0xffffffffu, wait_mma(sm, phase, err));
        phase ^= 1u;
        tc_fence_after();
        tc_fence_before();
        __syncthreads();  // P, K and V buffers are free for the next tile
    }

    // ---- epilogue: O / l as fp16 hi + lo.  tcgen05.ld is warp-collective: whole warps 0..3 load,
    // only the lanes of valid query rows store.
    if (!sm.abort && warp < 4) {
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
    tc_fence_before();
    __syncthreads();
    if (sm.abort && tid == 0) {
        mbar_wait_bounded(&sm.mma_bar, phase ^ 1u);  // let an issued MMA group finish
        if (raw_pending) mbar_wait_bounded(&sm.raw_bar, raw_phase);  // and a staging fill in flight
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_free(tmem, kTmemCols);
    }
}

template <int D, int G, typename KT>
cudaError_t launch_pf(const float* q, int64_t ldq, const void* kc, const void* vc, int KVH, int max_ctx, int pos0,
                      int S, __half* out_hi, __half* out_lo, int64_t ldo, unsigned* err, cudaStream_t s) {
    constexpr int QT = BQ / G;
    auto k = attn_prefill_tc_kernel<D, G, KT>;
    const int smem = PCfg<D, KT>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e) return e;
    dim3 grid((S + QT - 1) / QT, KVH);
    k<<<grid, kPThreads, smem, s>>>(q, ldq, (const KT*)kc, (const KT*)vc, max_ctx, pos0, S, out_hi, out_lo, ldo,
                                    err);
    return cudaGetLastError();
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
