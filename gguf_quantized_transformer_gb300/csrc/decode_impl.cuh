// Persistent decode step: one cooperative launch runs the whole token through
// every layer (Airframe "GPU_PIPELINE.md", "Decode loop" and per-layer ops;
// dotLLM "GPU Inference", "Forward Pass": embedding -> per layer
// [RMSNorm, Q/K/V, RoPE, KV write, attention, O + residual, RMSNorm,
// gate/up, SwiGLU, down + residual] -> final norm -> LM head).
//
// Structure.  One CTA per SM (16 warps).  The token's work is a sequence of
// phases separated by grid-wide barriers (bounded spins):
//   embed | per layer: QKV | attention | O | gate,up | down | LM head
// Every GEMV phase streams its weights through the CTA's shared-memory ring
// of bulk asynchronous copies exactly like the standalone GEMV (contiguous
// row range per CTA, last warp combines, fused epilogues).  The first stages
// of a GEMV phase do not depend on the previous phase, so they are issued
// before the barrier that precedes it: HBM keeps streaming while the grid
// synchronises.  Attention streams the CTA's slot range of the KV cache
// (K and V tiles per stage) through the same ring with an online softmax,
// and the last CTA of each kv head merges the split partials.
//
// Data produced by another CTA in this launch is read with ld.global.cg
// (L2), never through L1.  Every wait (mbarrier or grid barrier) is bounded:
// on a timeout the CTA records DEV_TIMEOUT, raises the global abort word,
// drains its copies and leaves; the host reports AF_ETIMEOUT.
#pragma once
#include <math_constants.h>

#include "common.cuh"
#include "gemv_common.cuh"
#include "tma.cuh"

namespace af {

namespace {

constexpr int kWarpsP = 16;
constexpr int kThreadsP = kWarpsP * 32;
constexpr int kSlotBytes = 40 * 1024;
constexpr int kSlots = 4;
constexpr int kRWMax = 4;
constexpr int kMaxRowsP = 512;
constexpr int kMaxSplitHeads = 1216;
constexpr int kMaxNormDim = 4096;  // largest n_embd the persistent kernel handles  // attention splits x query heads per kv head
constexpr unsigned kBarrierLimit = 1u << 24;  // polls of the grid barrier word (with nanosleep)

struct Shared {
    uint64_t full[kSlots];
    unsigned issues[kSlots];
    unsigned done_cnt[kSlots];
    float red[kSlots][kWarpsP][kRWMax];
    float ssum[kWarpsP];
    float xres[kMaxRowsP];
    float2 rope[64];
    unsigned long long amax;
    float att_s[64 * 8];   // scores / probabilities [T][G]
    float att_q[8 * 128];  // q of the kv head's query heads, scaled by 1/sqrt(D)
    float att_m[8], att_alpha[8], att_l[8];
    volatile int abort_cta;
    unsigned last;
    GemvTask task;  // the running GEMV phase's task (copied from global memory once per phase)
    uint64_t nw_bar;                  // completion of the norm-weight copy
    unsigned nw_issues;
    alignas(16) float nw[kMaxNormDim];  // RMSNorm weight of the next normalized GEMV phase (bulk-copy target)
    float att_w[2 * kMaxSplitHeads];  // merge (max, sum) then weights per (split, head)
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// ---------------------------------------------------------------- grid barrier
// The count starts at 0 each step (reset by the step-begin kernel).  Barrier i
// completes when the count reaches (i + 1) * gridDim.x: arrivals are release
// reductions, waiters poll the count with acquire loads (bounded).
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ bool grid_sync(const DecodePlan& p, unsigned& gen, Shared& sm) {
    __syncthreads();
    if (threadIdx.x == 0) {
        gen++;
        const unsigned target = gen * gridDim.x;
        red_release_add(p.bar_count, 1u);
        bool ok = true;
        unsigned it = 0;
        while ((int)(ld_acquire_u32(p.bar_count) - target) < 0) {
            if (++it > kBarrierLimit || ld_acquire_u32(p.abort) != 0u) {
                ok = false;
                break;
            }
            __nanosleep(32);
        }
        if (!ok) {
            atomicExch(p.err, (unsigned)DEV_TIMEOUT);
            atomicExch(p.abort, 1u);
            sm.abort_cta = 1;
        }
    }
    __syncthreads();
    return !sm.abort_cta;
}

// ---------------------------------------------------------------- ring
__device__ __forceinline__ void ring_issue(Shared& sm, uint8_t* ring, unsigned g, const void* src0, unsigned b0,
                                           const void* src1, unsigned b1, unsigned off1, uint64_t pol) {
    const int slot = (int)(g % kSlots);
    uint8_t* dst = ring + slot * kSlotBytes;
    sm.issues[slot]++;
    mbar_arrive_expect_tx(&sm.full[slot], b0 + b1);
    bulk_g2s_evict_first(dst, src0, b0, &sm.full[slot], pol);
    if (b1) bulk_g2s_evict_first(dst + off1, src1, b1, &sm.full[slot], pol);
}

// Bounded wait for global stage g; false (and abort raised) on timeout or abort.
__device__ __forceinline__ bool ring_wait(Shared& sm, const DecodePlan& p, unsigned g) {
    const int slot = (int)(g % kSlots);
    const unsigned par = (g / kSlots) & 1u;
    for (unsigned it = 0; it < kWaitLimit; it++) {
        if (mbar_try_wait(&sm.full[slot], par)) return true;
        if (sm.abort_cta) return false;
    }
    sm.abort_cta = 1;
    atomicExch(p.err, (unsigned)DEV_TIMEOUT);
    atomicExch(p.abort, 1u);
    return false;
}

// ---------------------------------------------------------------- GEMV phase
struct RowRange {
    int r0, nrows, nst;
};

__device__ __forceinline__ RowRange cta_rows(const GemvTask& t) {
    const int np = t.W.N / 2;
    const int pa = (int)((int64_t)np * blockIdx.x / gridDim.x), pb = (int)((int64_t)np * (blockIdx.x + 1) / gridDim.x);
    RowRange r;
    r.r0 = 2 * pa;
    r.nrows = 2 * (pb - pa);
    r.nst = (r.nrows + t.R - 1) / t.R;
    return r;
}

__device__ __forceinline__ void gemv_issue_stage(Shared& sm, uint8_t* ring, const GemvTask& t, const RowRange& rr,
                                                 unsigned base, int st, uint64_t pol) {
    const int64_t pitch = t.W.qs_pitch();
    const int ra = rr.r0 + st * t.R, nr = min(t.R, rr.r0 + rr.nrows - ra);
    ring_issue(sm, ring, base + st, t.W.qs + (int64_t)ra * pitch, (unsigned)(nr * pitch), nullptr, 0u, 0u, pol);
}

// Issue the first stages of a GEMV phase and the copy of its RMSNorm weight
// (thread 0); both only depend on the weights, not on the previous phase.
__device__ void gemv_prologue(Shared& sm, uint8_t* ring, const GemvTask& t, unsigned base, uint64_t pol) {
    if (threadIdx.x == 0) {
        if (t.nw) {  // first: the copy engine serves a CTA's copies in order
            const unsigned bytes = (unsigned)t.W.K * 4u;
            sm.nw_issues++;
            mbar_arrive_expect_tx(&sm.nw_bar, bytes);
            bulk_g2s(sm.nw, t.nw, bytes, &sm.nw_bar);
        }
        const RowRange rr = cta_rows(t);
        for (int st = 0; st < min(rr.nst, kSlots); st++) gemv_issue_stage(sm, ring, t, rr, base, st, pol);
    }
}

template <int RW>
__device__ __forceinline__ float reduce_rows(const float (&acc)[kRWMax], int lane) {
    float v[RW];
#pragma unroll
    for (int i = 0; i < RW; i++) v[i] = acc[i];
    return transpose_reduce<RW>(v, lane);
}

// Consume the phase's stages; returns the global stage index after the phase.
// `t` is the shared-memory copy of the task (never a reference into global memory,
// which the epilogue's stores could alias).
template <int WT, bool NORM, int UPL>
__device__ unsigned gemv_run(Shared& sm, uint8_t* ring, const DecodePlan& p, const GemvTask& t, unsigned base,
                             int pos, uint64_t pol) {
    constexpr int UW = Q<WT>::UW;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const Planes W = t.W;
    const int K = W.K;
    const int NC = W.Kp / (32 * UW);
    const int WK = t.WK, RS = kWarpsP / t.WK, RW = t.R / RS;
    const int rs = warp / WK, wk = warp % WK;
    const int64_t pitch = W.qs_pitch();
    const int scp = W.sc_pitch();
    const RowRange rr = cta_rows(t);
    const Epi& epi = t.epi;  // shared memory

    // prologue: this lane's x slices (one load round), epilogue inputs, RMS of x
    float xs[UPL][UW];
#pragma unroll
    for (int u = 0; u < UPL; u++) {
        const int c = wk + WK * u;
        const int k0 = (c * 32 + lane) * UW;
#pragma unroll
        for (int e = 0; e < UW; e += 4) {
            const float4 v = (c < NC && k0 < K) ? ldcg4(t.x + k0 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            xs[u][e] = v.x;
            xs[u][e + 1] = v.y;
            xs[u][e + 2] = v.z;
            xs[u][e + 3] = v.w;
        }
    }
    if (epi.kind == EPI_RESID)
        for (int i = tid; i < rr.nrows; i += kThreadsP) sm.xres[i] = __ldcg(epi.out + rr.r0 + i);
    if (epi.kind == EPI_QKV)
        for (int i = tid; i < epi.head_dim / 2; i += kThreadsP) sm.rope[i] = epi.rope[(int64_t)pos * (epi.head_dim / 2) + i];
    if (tid == 0) sm.amax = 0ull;
    float rstd = 1.f;
    if (NORM) {  // the lanes of row stream 0 hold every element of x exactly once
        float ss = 0.f;
        if (rs == 0) {
#pragma unroll
            for (int u = 0; u < UPL; u++)
#pragma unroll
                for (int e = 0; e < UW; e++) ss = fmaf(xs[u][e], xs[u][e], ss);
        }
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) sm.ssum[warp] = ss;
    }
    __syncthreads();
    if (NORM) {
        float tt = 0.f;
        for (int i = 0; i < WK; i++) tt += sm.ssum[i];  // warps 0..WK-1 form row stream 0
        rstd = rsqrtf(tt / (float)K + p.eps);
        // the norm weight copy was issued (first) with the phase's first stages
        bool okw = false;
        for (unsigned it = 0; it < kWaitLimit && !okw; it++) {
            okw = mbar_try_wait(&sm.nw_bar, (sm.nw_issues - 1u) & 1u);
            if (!okw && sm.abort_cta) break;
        }
        if (!okw && !sm.abort_cta) {
            sm.abort_cta = 1;
            atomicExch(p.err, (unsigned)DEV_TIMEOUT);
            atomicExch(p.abort, 1u);
        }
    }
    XUnit<UW / 4> xq[UPL];
#pragma unroll
    for (int u = 0; u < UPL; u++) {
        const int c = wk + WK * u;
        const int k0 = (c * 32 + lane) * UW;
        if (NORM && c < NC && k0 < K) {
#pragma unroll
            for (int e = 0; e < UW; e++) xs[u][e] = sm.nw[k0 + e] * (xs[u][e] * rstd);
        }
        quantize_unit<UW>(xs[u], xq[u]);
    }
    GemvEpiCtx ectx;
    ectx.xres = sm.xres;
    ectx.rope = sm.rope;
    ectx.amax = &sm.amax;
    ectx.r0 = rr.r0;
    ectx.pos = pos;

    for (int st = 0; st < rr.nst; st++) {
        const unsigned g = base + st;
        const int slot = (int)(g % kSlots);
        if (!ring_wait(sm, p, g)) break;
        const uint8_t* qsm = ring + slot * kSlotBytes;
        const unsigned short* ssm = reinterpret_cast<const unsigned short*>(qsm + W.sc_off());
        const int ra = rr.r0 + st * t.R, nr = min(t.R, rr.r0 + rr.nrows - ra);
        float acc[kRWMax];
#pragma unroll
        for (int i = 0; i < kRWMax; i++) {
            acc[i] = 0.f;
            const int j = rs + RS * i;
            if (i < RW && j < nr) {
#pragma unroll
                for (int u = 0; u < UPL; u++) {
                    const int c = wk + WK * u;
                    if (c < NC) {
                        const int unit = c * 32 + lane;
                        const uint4 q = *reinterpret_cast<const uint4*>(qsm + j * pitch + unit * 16);
                        const float d =
                            __half2float(__ushort_as_half(ssm[j * scp + (WT == AF_Q8_0 ? unit >> 1 : unit)]));
                        acc[i] = fmaf(d, Q<WT>::dot(q, xq[u]), acc[i]);
                    }
                }
            }
        }
        float r;
        switch (RW) {
            case 1: r = reduce_rows<1>(acc, lane); break;
            case 2: r = reduce_rows<2>(acc, lane); break;
            default: r = reduce_rows<4>(acc, lane); break;
        }
        if ((lane & (32 / RW - 1)) == 0) sm.red[slot][warp][lane / (32 / RW)] = r;
        __syncwarp();
        unsigned last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&sm.done_cnt[slot], 1u) == (unsigned)kWarpsP - 1u;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence_block();
            if (lane < nr / 2) {
                float y[2];
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int j = 2 * lane + h, jrs = j % RS, jt = j / RS;
                    float a = 0.f;
                    for (int w = 0; w < WK; w++) a += sm.red[slot][jrs * WK + w][jt];
                    y[h] = a;
                }
                gemv_epi(epi, ectx, ra + 2 * lane, y[0], y[1]);
            }
            __syncwarp();
            if (lane == 0) {
                sm.done_cnt[slot] = 0;
                if (st + kSlots < rr.nst) {
                    fence_proxy_async_shared();
                    gemv_issue_stage(sm, ring, t, rr, base, st + kSlots, pol);
                }
            }
        }
    }
    __syncthreads();
    if (epi.kind == EPI_LOGITS && tid == 0 && sm.amax) atomicMax(epi.argmax, sm.amax);
    return base + (unsigned)rr.nst;
}

template <int WT>
__device__ unsigned gemv_run_any(Shared& sm, uint8_t* ring, const DecodePlan& p, const GemvTask& tg, unsigned base,
                                 int pos, uint64_t pol) {
    {  // copy the task into shared memory (4-byte words, warp 0)
        static_assert(sizeof(GemvTask) % 4 == 0, "task size");
        const unsigned* src = reinterpret_cast<const unsigned*>(&tg);
        unsigned* dst = reinterpret_cast<unsigned*>(&sm.task);
        if (threadIdx.x < 32)
            for (int i = threadIdx.x; i < (int)(sizeof(GemvTask) / 4); i += 32) dst[i] = src[i];
        __syncthreads();
    }
    const GemvTask& t = sm.task;
    // chunk slots a lane needs: ceil(NC / WK); x slices for exactly that many stay in registers
    constexpr int UW = Q<WT>::UW;
    const int NC = t.W.Kp / (32 * UW);
    const int upl = (NC + t.WK - 1) / t.WK;
    if (upl <= 1)
        return t.nw ? gemv_run<WT, true, 1>(sm, ring, p, t, base, pos, pol)
                    : gemv_run<WT, false, 1>(sm, ring, p, t, base, pos, pol);
    return t.nw ? gemv_run<WT, true, 2>(sm, ring, p, t, base, pos, pol)
                : gemv_run<WT, false, 2>(sm, ring, p, t, base, pos, pol);
}

// ---------------------------------------------------------------- attention phase
// CTA b < KVH*S owns kv head b / S and split b % S of slots 0..pos.  Stage =
// T slots of K then T slots of V of that head (contiguous rows of the cache).
template <int D, typename KT>
__device__ unsigned attn_run(Shared& sm, uint8_t* ring, const DecodePlan& p, int layer, int pos, unsigned base,
                             uint64_t pol) {
    constexpr int T = (int)(kSlotBytes / (2 * D * sizeof(KT))) > 64 ? 64 : (int)(kSlotBytes / (2 * D * sizeof(KT)));
    constexpr int GMAX = 8;
    constexpr int NOUT = (GMAX * D + kThreadsP - 1) / kThreadsP;  // outputs per thread
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = p.attn_splits, KVH = p.KVH, G = p.H / p.KVH;
    const LayerPlan& L = p.layers[layer];
    const int b = blockIdx.x;
    if (b >= KVH * S) return base;
    const int kvh = b / S, s = b % S;
    const int n = pos + 1;
    const int chunk = (n + S - 1) / S;
    const int j0 = min(n, s * chunk), j1 = min(n, j0 + chunk);
    const int nst = (j1 - j0 + T - 1) / T;
    const KT* Kc = reinterpret_cast<const KT*>(L.kc) + (int64_t)kvh * p.max_ctx * D;
    const KT* Vc = reinterpret_cast<const KT*>(L.vc) + (int64_t)kvh * p.max_ctx * D;
    const unsigned tile = (unsigned)(T * D * sizeof(KT));

    auto issue = [&](int st) {
        const int a = j0 + st * T, na = min(T, j1 - a);
        ring_issue(sm, ring, base + st, Kc + (int64_t)a * D, (unsigned)(na * D * sizeof(KT)), Vc + (int64_t)a * D,
                   (unsigned)(na * D * sizeof(KT)), tile, pol);
    };
    if (tid == 0)
        for (int st = 0; st < min(nst, kSlots); st++) issue(st);

    // q of the G heads of this kv head, scaled by 1/sqrt(D)
    constexpr int DL = D / 32;
    const float scale = rsqrtf((float)D);
    for (int i = tid; i < G * D; i += kThreadsP) sm.att_q[i] = __ldcg(p.q + (int64_t)kvh * G * D + i) * scale;
    float acc[NOUT];
#pragma unroll
    for (int o = 0; o < NOUT; o++) acc[o] = 0.f;
    if (tid < G) {
        sm.att_m[tid] = -CUDART_INF_F;
        sm.att_l[tid] = 0.f;
    }
    __syncthreads();

    for (int st = 0; st < nst; st++) {
        const unsigned g = base + st;
        const int slot = (int)(g % kSlots);
        if (!__syncthreads_and(ring_wait(sm, p, g))) break;  // uniform: every thread leaves or none
        const KT* Kt = reinterpret_cast<const KT*>(ring + slot * kSlotBytes);
        const KT* Vt = reinterpret_cast<const KT*>(ring + slot * kSlotBytes + tile);
        const int na = min(T, j1 - (j0 + st * T));
        // scores: warp w takes slots w, w + 16, ...
        for (int t = warp; t < na; t += kWarpsP) {
            float kf[DL];
#pragma unroll
            for (int i = 0; i < DL; i++) kf[i] = (float)Kt[t * D + lane + 32 * i];
            for (int h = 0; h < G; h++) {  // warp-uniform
                {
                    float a = 0.f;
#pragma unroll
                    for (int i = 0; i < DL; i++) a = fmaf(sm.att_q[h * D + lane + 32 * i], kf[i], a);
#pragma unroll
                    for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                    if (lane == 0) sm.att_s[t * G + h] = a;
                }
            }
        }
        __syncthreads();
        if (warp < G) {  // warp h: running max, probabilities and sum of head h
            const int h = warp;
            const float s0 = lane < na ? sm.att_s[lane * G + h] : -CUDART_INF_F;
            const float s1 = lane + 32 < na ? sm.att_s[(lane + 32) * G + h] : -CUDART_INF_F;
            float mx = fmaxf(s0, s1);
#pragma unroll
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mold = sm.att_m[h];
            const float mnew = fmaxf(mold, mx);
            const float p0 = lane < na ? __expf(s0 - mnew) : 0.f;
            const float p1 = lane + 32 < na ? __expf(s1 - mnew) : 0.f;
            if (lane < na) sm.att_s[lane * G + h] = p0;
            if (lane + 32 < na) sm.att_s[(lane + 32) * G + h] = p1;
            float ps = p0 + p1;
#pragma unroll
            for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            if (lane == 0) {
                const float alpha = __expf(mold - mnew);
                sm.att_alpha[h] = alpha;
                sm.att_m[h] = mnew;
                sm.att_l[h] = sm.att_l[h] * alpha + ps;
            }
        }
        __syncthreads();
#pragma unroll
        for (int o = 0; o < NOUT; o++) {
            const int idx = tid + o * kThreadsP;
            if (idx < G * D) {
                const int h = idx / D, d = idx % D;
                float a = acc[o] * sm.att_alpha[h];
                for (int t = 0; t < na; t++) a = fmaf(sm.att_s[t * G + h], (float)Vt[t * D + d], a);
                acc[o] = a;
            }
        }
        __syncthreads();  // slot and scores free
        if (tid == 0 && st + kSlots < nst) {
            fence_proxy_async_shared();
            issue(st + kSlots);
        }
    }
    // partial of this split: part[((kvh*S + s)*G + h)*(D+2) + {0..D-1: o, D: max, D+1: sum}]
    float* my = p.attn_part + ((int64_t)(kvh * S + s) * G) * (D + 2);
#pragma unroll
    for (int o = 0; o < NOUT; o++) {
        const int idx = tid + o * kThreadsP;
        if (idx < G * D) my[(idx / D) * (D + 2) + idx % D] = acc[o];
    }
    if (tid < G) {
        my[tid * (D + 2) + D] = nst > 0 ? sm.att_m[tid] : -CUDART_INF_F;
        my[tid * (D + 2) + D + 1] = sm.att_l[tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.last = atomicAdd(&p.attn_cnt[kvh], 1u) == (unsigned)S - 1u;
    __syncthreads();
    if (sm.last) {  // merge the S splits of this kv head
        __threadfence();
        const float* pg = p.attn_part + ((int64_t)kvh * S * G) * (D + 2);
        for (int i = tid; i < S * G; i += kThreadsP) {  // (max, sum) of every split, in parallel
            const float* ps = pg + (int64_t)i * (D + 2);
            sm.att_w[2 * i] = __ldcg(ps + D);
            sm.att_w[2 * i + 1] = __ldcg(ps + D + 1);
        }
        __syncthreads();
        if (tid < G) {
            float M = -CUDART_INF_F;
            for (int ss2 = 0; ss2 < S; ss2++) M = fmaxf(M, sm.att_w[2 * (ss2 * G + tid)]);
            float den = 0.f;
            for (int ss2 = 0; ss2 < S; ss2++) {
                const float l = sm.att_w[2 * (ss2 * G + tid) + 1];
                if (l > 0.f) den = fmaf(__expf(sm.att_w[2 * (ss2 * G + tid)] - M), l, den);
            }
            sm.att_m[tid] = M;
            sm.att_l[tid] = 1.f / den;
        }
        __syncthreads();
        for (int i = tid; i < S * G; i += kThreadsP) {  // weight of split i / G for head i % G
            const float m = sm.att_w[2 * i], l = sm.att_w[2 * i + 1];
            sm.att_w[2 * i] = l > 0.f ? __expf(m - sm.att_m[i % G]) * sm.att_l[i % G] : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < G * D; idx += kThreadsP) {
            const int h = idx / D, d = idx % D;
            float a0 = 0.f, a1 = 0.f;
            int ss2 = 0;
            for (; ss2 + 2 <= S; ss2 += 2) {
                a0 = fmaf(sm.att_w[2 * (ss2 * G + h)], __ldcg(pg + ((int64_t)ss2 * G + h) * (D + 2) + d), a0);
                a1 = fmaf(sm.att_w[2 * ((ss2 + 1) * G + h)], __ldcg(pg + ((int64_t)(ss2 + 1) * G + h) * (D + 2) + d), a1);
            }
            if (ss2 < S) a0 = fmaf(sm.att_w[2 * (ss2 * G + h)], __ldcg(pg + ((int64_t)ss2 * G + h) * (D + 2) + d), a0);
            p.attn[(int64_t)(kvh * G + h) * D + d] = a0 + a1;
        }
        if (tid == 0) p.attn_cnt[kvh] = 0u;
    }
    __syncthreads();
    return base + (unsigned)nst;
}

// ---------------------------------------------------------------- the kernel
template <int WT, int D, typename KT>
__global__ void __launch_bounds__(kThreadsP, 1) decode_kernel(DecodePlan p) {
    extern __shared__ __align__(128) uint8_t ring[];
    // Shared's task member has default member initializers (Planes, Epi); shared memory is never
    // initialized, and every field is written before it is read
#pragma nv_diag_suppress 20054
    __shared__ Shared sm;
#pragma nv_diag_default 20054
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < kSlots; s++) {
            mbar_init(&sm.full[s], 1);
            sm.issues[s] = 0;
            sm.done_cnt[s] = 0;
        }
        sm.abort_cta = 0;
        mbar_init(&sm.nw_bar, 1);
        sm.nw_issues = 0;
        fence_mbar_init();
    }
    __syncthreads();
    unsigned gen = 0;  // barriers passed in this step (the count was reset by the step-begin kernel)
    int tr = 0;  // phase-boundary trace (CTA 0, thread 0)
    auto trace = [&]() {
        if (p.trace && blockIdx.x == 0 && tid == 0) {
            unsigned long long t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            p.trace[tr] = t;
        }
        tr++;
    };
    trace();
    const uint64_t pol = policy_evict_first();
    const int pos = p.st->pos;
    const int token = p.st->token;
    unsigned g = 0;  // global stage counter of this CTA's ring

    // layer 0's QKV weights start streaming now
    gemv_prologue(sm, ring, p.layers[0].qkv, g, pol);

    // embedding row of the token, split across CTAs
    {
        const Planes& emb = p.emb;
        const int row = (token >= 0 && token < emb.N) ? token : 0;
        const int E = emb.K;
        const int k0 = (int)((int64_t)E * blockIdx.x / gridDim.x), k1 = (int)((int64_t)E * (blockIdx.x + 1) / gridDim.x);
        for (int k = k0 + tid; k < k1; k += kThreadsP) {
            const int bk = k >> 5, e = k & 31;
            const float d = __half2float(emb.sc[(int64_t)row * emb.sc_pitch() + bk]);
            const uint8_t* q = emb.qs + (int64_t)row * emb.qs_pitch() + (int64_t)bk * emb.qb();
            float v;
            if (WT == AF_Q8_0) {
                v = d * (float)(int8_t)q[e];
            } else {
                const uint8_t byte = q[e & 15];
                v = d * (float)((e < 16 ? (byte & 15) : (byte >> 4)) - 8);
            }
            p.x[k] = v;
        }
    }
    bool ok = grid_sync(p, gen, sm);
    trace();
    auto capture = [&](int slot) {  // x is final once the barrier after a layer has passed
        if (!p.capture) return;
        const int E = p.emb.K;
        const int k0 = (int)((int64_t)E * blockIdx.x / gridDim.x), k1 = (int)((int64_t)E * (blockIdx.x + 1) / gridDim.x);
        for (int k = k0 + tid; k < k1; k += kThreadsP) p.capture[(int64_t)slot * E + k] = __ldcg(p.x + k);
    };
    if (ok) capture(0);

    for (int l = 0; l < p.n_layers && ok; l++) {
        const LayerPlan& L = p.layers[l];
        g = gemv_run_any<WT>(sm, ring, p, L.qkv, g, pos, pol);  // -> q, K/V cache at pos
        if (sm.abort_cta || !(ok = grid_sync(p, gen, sm))) break;
        trace();
        g = attn_run<D, KT>(sm, ring, p, l, pos, g, pol);  // -> attn
        gemv_prologue(sm, ring, L.o, g, pol);
        if (sm.abort_cta || !(ok = grid_sync(p, gen, sm))) break;
        trace();
        g = gemv_run_any<WT>(sm, ring, p, L.o, g, pos, pol);  // x += attn W_o^T
        gemv_prologue(sm, ring, L.gu, g, pol);
        if (sm.abort_cta || !(ok = grid_sync(p, gen, sm))) break;
        trace();
        g = gemv_run_any<WT>(sm, ring, p, L.gu, g, pos, pol);  // h = silu(gate) * up
        gemv_prologue(sm, ring, L.down, g, pol);
        if (sm.abort_cta || !(ok = grid_sync(p, gen, sm))) break;
        trace();
        g = gemv_run_any<WT>(sm, ring, p, L.down, g, pos, pol);  // x += h W_d^T
        gemv_prologue(sm, ring, l + 1 < p.n_layers ? p.layers[l + 1].qkv : p.head, g, pol);
        if (sm.abort_cta || !(ok = grid_sync(p, gen, sm))) break;
        trace();
        capture(l + 1);
    }
    if (ok && !sm.abort_cta) g = gemv_run_any<WT>(sm, ring, p, p.head, g, pos, pol);  // logits, argmax
    trace();

    __syncthreads();
    if (sm.abort_cta) {  // drain every copy still in flight before the CTA exits
        if (tid == 0)
            for (int s = 0; s < kSlots; s++)
                if (sm.issues[s]) mbar_wait_bounded(&sm.full[s], (sm.issues[s] - 1u) & 1u);
        if (tid == 0 && sm.nw_issues) mbar_wait_bounded(&sm.nw_bar, (sm.nw_issues - 1u) & 1u);
        __syncthreads();
    }
}

template <int WT, int D, typename KT>
cudaError_t launch_decode_t(const DecodePlan& p, cudaStream_t s, bool prepare) {
    auto kern = decode_kernel<WT, D, KT>;
    const size_t smem = (size_t)kSlots * kSlotBytes;
    if (prepare) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e) return e;
        int nb = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kThreadsP, smem);
        if (e) return e;
        return nb >= 1 ? cudaSuccess : cudaErrorCooperativeLaunchTooLarge;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms());
    cfg.blockDim = dim3(kThreadsP);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

// Launch (or, with prepare, opt in to shared memory and check residency) for one
// (weight type, head_dim) pair; defined by the decode_*.cu translation units.
template <int WT, int D>
cudaError_t decode_launch_for(const DecodePlan& p, cudaStream_t s, bool prepare) {
    return p.kv_f16 ? launch_decode_t<WT, D, __half>(p, s, prepare) : launch_decode_t<WT, D, float>(p, s, prepare);
}

}  // namespace af
