// Persistent streaming decode step: one cooperative launch runs the whole token
// through every layer (Airframe "GPU_PIPELINE.md", "Decode loop" and per-layer
// ops; dotLLM "GPU Inference", "Forward Pass": embedding -> per layer
// [RMSNorm, Q/K/V, RoPE, KV write, attention, O + residual, RMSNorm,
// gate/up, SwiGLU, down + residual] -> final norm -> LM head).
//
// Structure.  One CTA of 16 warps per SM.  The token is a sequence of phases
// separated by grid-wide barriers (bounded spins):
//   embed | per layer: QKV | attention | O | gate,up | down | LM head
// Every phase but the embedding streams data through shared-memory slots by
// bulk asynchronous copies: GEMV phases a stage of R whole weight rows of the
// CTA's contiguous row range, the attention phase a K tile and a V tile of T
// cache slots of the CTA's (kv head, split) range.  The CTA numbers all its
// stages of the token in phase order, g = 0, 1, ...; stage g lives in slot
// g mod nslot and belongs to warp g mod nslot, which waits for it, computes it
// and then issues stage g + nslot into the same slot, whatever phase that
// stage belongs to.  Weights and the cache slots before the current position
// depend on nothing computed in this launch, so the copies run ahead across
// phase boundaries: while the grid synchronises and the next phase's prologue
// runs, every slot is already filling with the next phase's data, and HBM
// keeps streaming.  The current position's K/V (written by this token's QKV
// phase) is read after the barrier instead of being streamed.
//
// GEMV phases: the prologue (all threads) converts the phase input (RMS-
// normalized where the op has a norm) to the 16-bit fixed-point block image
// in shared memory; a warp's stage is R rows x the whole K, dp4a units exactly
// as in the standalone decode GEMV, then a transpose-reduce and the fused
// epilogue (RoPE + q + KV write, residual add, SwiGLU, logits + argmax).
// Attention phase: CTA b < KVH * S owns kv head b / S and split b % S of the
// slots before the current position; each warp keeps an online softmax over
// its own stages (scores with the G query heads in registers, probabilities
// through shared memory), the CTA combines its warps, and the last CTA of a
// kv head (arrival counter) merges the S splits.
//
// Data produced by another CTA in this launch is read with ld.global.cg (L2),
// never through L1.  Every wait (mbarrier or grid barrier) is bounded: on a
// timeout the CTA records DEV_TIMEOUT, raises the global abort word, drains
// its copies and leaves; the host reports AF_ETIMEOUT.
#pragma once
#include <math_constants.h>

#include "common.cuh"
#include "gemv_common.cuh"
#include "tma.cuh"

namespace af {

namespace {

constexpr int kWarpsP = 16;
constexpr int kThreadsP = kWarpsP * 32;
constexpr int kMaxRowsP = 128;                // residual rows a CTA may own
constexpr unsigned kBarrierLimit = 1u << 24;  // polls of the grid barrier word
constexpr int kSubT = 16;                     // attention: slots per online-softmax step of a warp

struct SharedP {
    uint64_t full[kMaxSlotsP];
    unsigned issues[kMaxSlotsP];  // copies issued into the slot so far
    float ssum[kWarpsP];
    float xres[kMaxRowsP];
    float2 rope[64];
    float wm[kWarpsP][8], wl[kWarpsP][8];  // attention: warps' running maxima and sums per head
    float cw[kWarpsP][8];                  // attention: a warp's rescale factors of the current step
    unsigned long long amax;
    volatile int abort_cta;
    unsigned last;
    GemvTask task[2];  // the running GEMV phase's task and the next one's (copied from global memory)
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 8 consecutive cache values (16-byte aligned) as fp32
__device__ __forceinline__ void load_row8(const float* k, float* out) {
    const float4 a = *reinterpret_cast<const float4*>(k), b = *reinterpret_cast<const float4*>(k + 4);
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w; out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}
__device__ __forceinline__ void load_row8(const __half* k, float* out) {
    const uint4 raw = *reinterpret_cast<const uint4*>(k);
    const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const float2 f = __half22float2(h[e]);
        out[2 * e] = f.x;
        out[2 * e + 1] = f.y;
    }
}
// N (2 or 4) consecutive cache values as fp32; p aligned to N elements
template <int N>
__device__ __forceinline__ void load_small(const float* v, float* out) {
    if (N == 4) {
        const float4 a = *reinterpret_cast<const float4*>(v);
        out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    } else {
        const float2 a = *reinterpret_cast<const float2*>(v);
        out[0] = a.x; out[1] = a.y;
    }
}
template <int N>
__device__ __forceinline__ void load_small(const __half* v, float* out) {
    if (N == 4) {
        const uint2 raw = *reinterpret_cast<const uint2*>(v);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
    } else {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(v));
        out[0] = a.x; out[1] = a.y;
    }
}
// one cache value written earlier in this launch (through L2)
__device__ __forceinline__ float ldcg_kt(const float* v) { return __ldcg(v); }
__device__ __forceinline__ __half ldcg_kt(const __half* v) {
    return __ushort_as_half(__ldcg(reinterpret_cast<const unsigned short*>(v)));
}

__device__ __forceinline__ void raise_abort(const DecodePlan& p, SharedP& sm) {
    sm.abort_cta = 1;
    atomicExch(p.err, (unsigned)DEV_TIMEOUT);
    atomicExch(p.abort, 1u);
}

// ---------------------------------------------------------------- grid barrier
// The count starts at 0 each step (reset by the step-begin kernel).  Barrier i
// completes when the count reaches (i + 1) * gridDim.x: arrivals are release
// reductions, waiters poll the count with acquire loads (bounded).
__device__ bool grid_sync(const DecodePlan& p, unsigned& gen, SharedP& sm) {
    __syncthreads();
    if (threadIdx.x == 0) {
        gen++;
        const unsigned target = gen * gridDim.x;
        __threadfence();  // the CTA's writes (ordered before this thread by the barrier above) at gpu scope
        red_release_add(p.bar_count, 1u);
        bool ok = true;
        unsigned it = 0;
        while ((int)(ld_acquire_u32(p.bar_count) - target) < 0) {
            if (++it > kBarrierLimit || ld_acquire_u32(p.abort) != 0u) {
                ok = false;
                break;
            }
        }
        if (!ok) raise_abort(p, sm);
    }
    __syncthreads();
    return !sm.abort_cta;
}

// ---------------------------------------------------------------- the stage schedule
// Phase ph < 5 L: layer ph / 5, op ph % 5 (0 QKV, 1 attention, 2 O, 3 gate/up, 4 down); ph = 5 L: LM head.
struct RowRange {
    int r0, nrows;
};

__device__ __forceinline__ RowRange cta_rows(int N) {
    const int np = N / 2;
    const int pa = (int)((int64_t)np * blockIdx.x / gridDim.x), pb = (int)((int64_t)np * (blockIdx.x + 1) / gridDim.x);
    return {2 * pa, 2 * (pb - pa)};
}

// This CTA's attention range: slots [j0, j0 + len) of kv head kvh, before the current position.
struct AttnRange {
    int kvh, split, j0, len;
    bool holds_pos;  // the last split also takes the current position
};

__device__ __forceinline__ AttnRange cta_attn(const DecodePlan& p, int pos) {
    AttnRange a;
    const int S = p.attn_splits, b = blockIdx.x;
    a.kvh = b / S;
    a.split = b % S;
    a.j0 = 0;
    a.len = 0;
    a.holds_pos = false;
    if (b >= p.KVH * S) {
        a.kvh = -1;
        return a;
    }
    const int chunk = (pos + S - 1) / S;
    a.j0 = min(pos, a.split * chunk);
    a.len = min(chunk, pos - a.j0);
    a.holds_pos = a.split == S - 1;
    return a;
}

__device__ __forceinline__ const GemvTask& phase_task(const DecodePlan& p, int ph) {
    if (ph >= 5 * p.n_layers) return p.head;
    const LayerPlan& L = p.layers[ph / 5];
    switch (ph % 5) {
        case 0: return L.qkv;
        case 2: return L.o;
        case 3: return L.gu;
        default: return L.down;
    }
}

__device__ __forceinline__ bool is_attn_phase(const DecodePlan& p, int ph) { return ph < 5 * p.n_layers && ph % 5 == 1; }

// This CTA's stages of one phase, built once per launch into shared memory, so that issuing a stage reads no
// global memory: stage st copies `bytes` (`last` for the final stage) from a + st * stride, and for an
// attention phase as many from b + st * stride (the V tile) to the slot's second half.
struct PhaseDesc {
    const uint8_t* a;
    const uint8_t* b;
    unsigned stride, bytes, last;
    int nst;
};
static_assert(sizeof(PhaseDesc) == 32, "phase descriptor size");

template <typename KT>
__device__ PhaseDesc make_desc(const DecodePlan& p, int ph, int pos) {
    PhaseDesc d;
    d.b = nullptr;
    if (is_attn_phase(p, ph)) {
        const AttnRange a = cta_attn(p, pos);
        const LayerPlan& L = p.layers[ph / 5];
        const unsigned tile = (unsigned)(p.att_T * p.D * (int)sizeof(KT));
        d.nst = a.kvh < 0 ? 0 : (a.len + p.att_T - 1) / p.att_T;
        const int64_t off = ((int64_t)max(a.kvh, 0) * p.max_ctx + a.j0) * p.D * (int64_t)sizeof(KT);
        d.a = reinterpret_cast<const uint8_t*>(L.kc) + off;
        d.b = reinterpret_cast<const uint8_t*>(L.vc) + off;
        d.stride = d.bytes = tile;
        d.last = d.nst ? (unsigned)((a.len - (d.nst - 1) * p.att_T) * p.D * (int)sizeof(KT)) : 0u;
    } else {
        const GemvTask& t = phase_task(p, ph);
        const RowRange rr = cta_rows(t.W.N);
        const int64_t pitch = t.W.qs_pitch();
        d.nst = (rr.nrows + t.R - 1) / t.R;
        d.a = t.W.qs + (int64_t)rr.r0 * pitch;
        d.stride = d.bytes = (unsigned)(t.R * pitch);
        d.last = d.nst ? (unsigned)((rr.nrows - (d.nst - 1) * t.R) * pitch) : 0u;
    }
    return d;
}

// Walks the schedule forward: the phase holding global stage g (monotone in g for each caller).
struct Cursor {
    int ph, g0;  // phase, its first global stage
    __device__ __forceinline__ bool seek(const PhaseDesc* tab, int nph, int g) {
        while (ph < nph && g >= g0 + tab[ph].nst) {
            g0 += tab[ph].nst;
            ph++;
        }
        return ph < nph;
    }
};

// Issue global stage g (one thread) into its slot.
__device__ __forceinline__ void issue_stage(const DecodePlan& p, SharedP& sm, const PhaseDesc* tab, int nph,
                                            uint8_t* ring, Cursor& cur, int g, uint64_t pol) {
    if (!cur.seek(tab, nph, g)) return;
    const PhaseDesc& d = tab[cur.ph];
    const int slot = g % p.nslot, st = g - cur.g0;
    uint8_t* dst = ring + (size_t)slot * p.slot_bytes;
    const unsigned n = st == d.nst - 1 ? d.last : d.bytes;
    sm.issues[slot]++;
    mbar_arrive_expect_tx(&sm.full[slot], d.b ? 2u * n : n);
    bulk_g2s_evict_first(dst, d.a + (size_t)st * d.stride, n, &sm.full[slot], pol);
    if (d.b) bulk_g2s_evict_first(dst + d.stride, d.b + (size_t)st * d.stride, n, &sm.full[slot], pol);
}

// Copy the task of GEMV phase ph (global memory) into sm.task[ph & 1], one warp; the phase reads it there.
__device__ __forceinline__ void prefetch_task(const DecodePlan& p, SharedP& sm, int ph, int lane) {
    if (ph > 5 * p.n_layers || is_attn_phase(p, ph)) return;
    static_assert(sizeof(GemvTask) % 4 == 0, "task size");
    const unsigned* src = reinterpret_cast<const unsigned*>(&phase_task(p, ph));
    unsigned* dst = reinterpret_cast<unsigned*>(&sm.task[ph & 1]);
    for (int i = lane; i < (int)(sizeof(GemvTask) / 4); i += 32) dst[i] = src[i];
}

// Bounded wait (whole warp) for global stage g; false on a timeout or an abort.
__device__ __forceinline__ bool stage_wait(const DecodePlan& p, SharedP& sm, int g) {
    const int slot = g % p.nslot;
    const unsigned par = (unsigned)((g / p.nslot) & 1);
    bool ok = false;
    for (unsigned it = 0; it < kWaitLimit && !ok; it++) {
        ok = mbar_try_wait(&sm.full[slot], par);
        if (!ok && sm.abort_cta) break;
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0 && !sm.abort_cta) raise_abort(p, sm);
    return ok;
}

// ---------------------------------------------------------------- GEMV phase
// acc[r] += row r of the stage . x over the whole K (lane: unit l of every chunk).
template <int WT, int R, bool FULL>
__device__ __forceinline__ void gemv_rows(const uint8_t* stg, int pitch, int sc_off, int NC, int nr, const XBlk* xb,
                                          int lane, float (&acc)[R]) {
    for (int c = 0; c < NC; c++) {
        const int unit = c * 32 + lane;
        Unit<WT> xu;
        xu.load(xb, unit);
#pragma unroll
        for (int r = 0; r < R; r++)
            if (FULL || r < nr) acc[r] = xu.accumulate(stg + r * pitch, sc_off, unit, acc[r]);
    }
}

template <int WT, int R, typename Refill>
__device__ __forceinline__ void gemv_stage(const uint8_t* stg, const Planes& W, int nr, const XBlk* xb, int lane,
                                           const Epi& epi, const GemvEpiCtx& ectx, int ra, float rstd,
                                           Refill refill) {
    const int pitch = (int)W.qs_pitch(), sc_off = W.sc_off();
    const int NC = W.Kp / (32 * (WT == AF_Q8_0 ? 16 : 32));
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; r++) acc[r] = 0.f;
    if (nr == R)
        gemv_rows<WT, R, true>(stg, pitch, sc_off, NC, nr, xb, lane, acc);
    else
        gemv_rows<WT, R, false>(stg, pitch, sc_off, NC, nr, xb, lane, acc);
    __syncwarp();  // every lane is done reading the slot
    refill();
    // lanes (32/R)*t .. hold the sum of acc[t]; lane (64/R)*q applies row pair q
    const float v = transpose_reduce<R>(acc, lane);
    const float v1 = __shfl_down_sync(0xffffffffu, v, 32 / R);
    if (lane % (64 / R) == 0) {
        const int j0 = 2 * (lane / (64 / R));
        if (j0 < nr) gemv_epi(epi, ectx, ra + j0, v * rstd, v1 * rstd);
    }
}

// One GEMV phase: prologue (input image, RMS, epilogue inputs), then this warp's stages of the phase.
// The phase's task was copied to sm.task[ph & 1] before the barrier that precedes the phase.
template <int WT>
__device__ void gemv_phase(const DecodePlan& p, SharedP& sm, const PhaseDesc* tab, int nph, uint8_t* ximg,
                           uint8_t* ring, Cursor& cur, int ph, int gph, int& gnext, int pos, uint64_t pol) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const GemvTask& t = sm.task[ph & 1];
    const Planes W = t.W;
    const Epi epi = t.epi;
    const int R = t.R;
    const RowRange rr = cta_rows(W.N);
    const int nst = tab[ph].nst;
    XBlk* xb = reinterpret_cast<XBlk*>(ximg);
    const bool norm = t.nw != nullptr;
    // epilogue inputs first: their loads overlap the image's
    float xr = 0.f;
    float2 rp = make_float2(0.f, 0.f);
    if (epi.kind == EPI_RESID && tid < rr.nrows) xr = __ldcg(epi.out + rr.r0 + tid);
    if (epi.kind == EPI_QKV && tid < epi.head_dim / 2) rp = epi.rope[(int64_t)pos * (epi.head_dim / 2) + tid];
    float ss = norm ? quantize_x<true, kThreadsP, true>(t.x, t.nw, W.K, W.Kp / 32, xb, tid)
                    : quantize_x<false, kThreadsP, true>(t.x, nullptr, W.K, W.Kp / 32, xb, tid);
    if (norm) {
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) sm.ssum[warp] = ss;
    }
    if (epi.kind == EPI_RESID && tid < rr.nrows) sm.xres[tid] = xr;
    if (epi.kind == EPI_QKV && tid < epi.head_dim / 2) sm.rope[tid] = rp;
    if (tid == 0) sm.amax = 0ull;
    __syncthreads();
    if (warp == kWarpsP - 1) prefetch_task(p, sm, ph + 1, lane);  // ph + 1 is an attention phase or the next GEMV
    if (warp == kWarpsP - 1 && is_attn_phase(p, ph + 1)) prefetch_task(p, sm, ph + 2, lane);
    float rstd = 1.f;
    if (norm) {
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < kWarpsP; i++) a += sm.ssum[i];
        rstd = rsqrtf(a / (float)W.K + p.eps);
    }
    GemvEpiCtx ectx;
    ectx.xres = sm.xres;
    ectx.rope = sm.rope;
    ectx.amax = &sm.amax;
    ectx.r0 = rr.r0;
    ectx.pos = pos;
    if (warp < p.nslot) {
        int g = gnext;
        for (; g < gph + nst; g += p.nslot) {
            if (!stage_wait(p, sm, g)) break;
            const uint8_t* stg = ring + (size_t)(g % p.nslot) * p.slot_bytes;
            const int st = g - gph, ra = rr.r0 + st * R, nr = min(R, rr.r0 + rr.nrows - ra);
            const int gn = g + p.nslot;
            auto refill = [&]() {  // the slot's next stage, whatever phase it belongs to
                if (lane == 0) {
                    fence_proxy_async_shared();  // the warp's reads of the slot before the copy overwrites it
                    issue_stage(p, sm, tab, nph, ring, cur, gn, pol);
                }
            };
            switch (R) {
                case 2: gemv_stage<WT, 2>(stg, W, nr, xb, lane, epi, ectx, ra, rstd, refill); break;
                case 4: gemv_stage<WT, 4>(stg, W, nr, xb, lane, epi, ectx, ra, rstd, refill); break;
                default: gemv_stage<WT, 8>(stg, W, nr, xb, lane, epi, ectx, ra, rstd, refill); break;
            }
        }
        gnext = g;
    }
    __syncthreads();
    if (epi.kind == EPI_LOGITS && tid == 0 && sm.amax) atomicMax(epi.argmax, sm.amax);
}

// ---------------------------------------------------------------- attention phase
// One online-softmax step of a warp over `keys` (<= kSubT) cache slots: K rows kt[j*D..], V rows vt[j*D..].
//   scores: lanes (LPK = D / 8 per slot, 8 dims each) score KPW = 32 / LPK slots per step for all G heads;
//           a transpose-reduce leaves head li / LPH of the slot in lane li
//   P V:    probabilities through shared memory; lane l owns dims l*DV.. of all heads
template <int D, int G, typename KT>
__device__ __forceinline__ void attn_step(const KT* kt, const KT* vt, int keys, const float (&qv)[G][8], float& m_run,
                                          float& l_run, float (&acc)[G][D / 32], float* pw, float* cw, int lane) {
    constexpr int LPK = D / 8, KPW = 32 / LPK, LPH = LPK / G, STEPS = kSubT / KPW, DV = D / 32;
    const int li = lane % LPK, ks = lane / LPK, hl = li / LPH;
    float sreg[STEPS];
    float mt = -CUDART_INF_F;
#pragma unroll
    for (int st = 0; st < STEPS; st++) {
        const int j = st * KPW + ks;
        float kf[8];
        if (j < keys) {
            load_row8(kt + j * D + li * 8, kf);
        } else {
#pragma unroll
            for (int e = 0; e < 8; e++) kf[e] = 0.f;
        }
        float a[G];
#pragma unroll
        for (int h = 0; h < G; h++) {
            a[h] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; e++) a[h] = fmaf(qv[h][e], kf[e], a[h]);
        }
#pragma unroll
        for (int half = G / 2, bit = LPK / 2; half >= 1; half >>= 1, bit >>= 1) {
            const bool up = li & bit;
#pragma unroll
            for (int k = 0; k < half; k++) {
                const float send = up ? a[k] : a[k + half], keep = up ? a[k + half] : a[k];
                a[k] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
            }
        }
        float r = a[0];
#pragma unroll
        for (int bit = LPH / 2; bit >= 1; bit >>= 1) r += __shfl_xor_sync(0xffffffffu, r, bit);
        sreg[st] = j < keys ? r : -CUDART_INF_F;
        mt = fmaxf(mt, sreg[st]);
    }
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
    const float m_new = fmaxf(m_run, mt);
    const float corr = m_new == -CUDART_INF_F ? 1.f : __expf(m_run - m_new);
    float psum = 0.f;
#pragma unroll
    for (int st = 0; st < STEPS; st++) {
        const float pr = sreg[st] == -CUDART_INF_F ? 0.f : __expf(sreg[st] - m_new);
        psum += pr;
        if (li % LPH == 0) pw[(st * KPW + ks) * G + hl] = pr;
    }
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    l_run = fmaf(l_run, corr, psum);
    m_run = m_new;
    if (lane < LPK && li % LPH == 0) cw[hl] = corr;
    __syncwarp();
#pragma unroll
    for (int h = 0; h < G; h++) {
        const float c = cw[h];
#pragma unroll
        for (int e = 0; e < DV; e++) acc[h][e] *= c;
    }
    for (int j = 0; j < keys; j++) {
        float vf[DV];
        load_small<DV>(vt + j * D + lane * DV, vf);
#pragma unroll
        for (int h = 0; h < G; h++) {
            const float pj = pw[j * G + h];
#pragma unroll
            for (int e = 0; e < DV; e++) acc[h][e] = fmaf(pj, vf[e], acc[h][e]);
        }
    }
    __syncwarp();
}

// The attention phase of layer l.  Scratch in the image region: [warp][kSubT][G] probabilities, [warp][G][D]
// combine rows, the current position's K and V rows, and the merge weights [S][G].
template <int D, int G, typename KT>
__device__ void attn_phase(const DecodePlan& p, SharedP& sm, const PhaseDesc* tab, int nph, uint8_t* ximg,
                           uint8_t* ring, Cursor& cur, int l, int gph, int& gnext, int pos, uint64_t pol) {
    constexpr int DV = D / 32, LPK = D / 8, LPH = LPK / G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const LayerPlan& L = p.layers[l];
    const AttnRange a = cta_attn(p, pos);
    const int T = p.att_T;
    const int nst = tab[5 * l + 1].nst;
    float* pw_all = reinterpret_cast<float*>(ximg);                 // [kWarpsP][kSubT][G]
    float* red_o = pw_all + kWarpsP * kSubT * G;                    // [kWarpsP][G][D]
    KT* kv_pos = reinterpret_cast<KT*>(red_o + kWarpsP * G * D);    // [2][D]
    float* wts = reinterpret_cast<float*>(kv_pos + 2 * D);          // [S][G] merge weights
    float* pw = pw_all + warp * kSubT * G;
    const int li = lane % LPK, hl = li / LPH;

    float qv[G][8];
    if (a.kvh >= 0) {
        const float scale = rsqrtf((float)D);
#pragma unroll
        for (int h = 0; h < G; h++) {
            const float* qh = p.q + (int64_t)(a.kvh * G + h) * D + li * 8;
            const float4 x0 = __ldcg(reinterpret_cast<const float4*>(qh));
            const float4 x1 = __ldcg(reinterpret_cast<const float4*>(qh + 4));
            qv[h][0] = x0.x * scale; qv[h][1] = x0.y * scale; qv[h][2] = x0.z * scale; qv[h][3] = x0.w * scale;
            qv[h][4] = x1.x * scale; qv[h][5] = x1.y * scale; qv[h][6] = x1.z * scale; qv[h][7] = x1.w * scale;
        }
        if (a.holds_pos) {  // the current position's K and V, written by this token's QKV phase
            const int64_t off = ((int64_t)a.kvh * p.max_ctx + pos) * D;
            for (int i = tid; i < D; i += kThreadsP) {
                kv_pos[i] = ldcg_kt(reinterpret_cast<const KT*>(L.kc) + off + i);
                kv_pos[D + i] = ldcg_kt(reinterpret_cast<const KT*>(L.vc) + off + i);
            }
        }
    }
    __syncthreads();
    float m_run = -CUDART_INF_F, l_run = 0.f;
    float acc[G][DV];
#pragma unroll
    for (int h = 0; h < G; h++)
#pragma unroll
        for (int e = 0; e < DV; e++) acc[h][e] = 0.f;
    if (warp < p.nslot) {
        int g = gnext;
        for (; g < gph + nst; g += p.nslot) {
            if (!stage_wait(p, sm, g)) break;
            const uint8_t* stg = ring + (size_t)(g % p.nslot) * p.slot_bytes;
            const KT* kt = reinterpret_cast<const KT*>(stg);
            const KT* vt = reinterpret_cast<const KT*>(stg + (size_t)T * D * sizeof(KT));
            const int keys = min(T, a.len - (g - gph) * T);
            for (int j0 = 0; j0 < keys; j0 += kSubT)
                attn_step<D, G, KT>(kt + j0 * D, vt + j0 * D, min(kSubT, keys - j0), qv, m_run, l_run, acc, pw,
                                    sm.cw[warp], lane);
            if (lane == 0) {
                fence_proxy_async_shared();
                issue_stage(p, sm, tab, nph, ring, cur, g + p.nslot, pol);
            }
        }
        gnext = g;
    }
    if (a.kvh >= 0 && a.holds_pos && warp == kWarpsP - 1)
        attn_step<D, G, KT>(kv_pos, kv_pos + D, 1, qv, m_run, l_run, acc, pw, sm.cw[warp], lane);
    // combine the warps into the CTA's partial
#pragma unroll
    for (int h = 0; h < G; h++)
#pragma unroll
        for (int e = 0; e < DV; e++) red_o[(warp * G + h) * D + lane * DV + e] = acc[h][e];
    if (lane < LPK && li % LPH == 0) {
        sm.wm[warp][hl] = m_run;
        sm.wl[warp][hl] = l_run;
    }
    __syncthreads();
    if (a.kvh < 0) return;  // uniform per CTA
    const int S = p.attn_splits;
    constexpr int PST = D + 4;
    float* my = p.attn_part + ((int64_t)(a.kvh * S + a.split) * G) * PST;
    for (int t = tid; t < G * D; t += kThreadsP) {
        const int h = t / D, d = t % D;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarpsP; w++) M = fmaxf(M, sm.wm[w][h]);
        float o = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarpsP; w++) {
            const float e = sm.wm[w][h] == -CUDART_INF_F ? 0.f : __expf(sm.wm[w][h] - M);
            o = fmaf(e, red_o[(w * G + h) * D + d], o);
            lsum = fmaf(e, sm.wl[w][h], lsum);
        }
        my[h * PST + d] = o;
        if (d == 0) {
            my[h * PST + D] = M;
            my[h * PST + D + 1] = lsum;
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.last = atomicAdd(&p.attn_cnt[a.kvh], 1u) == (unsigned)S - 1u;
    __syncthreads();
    if (!sm.last) return;
    // the last split of this kv head merges all S:  o_h = sum_s exp(m_s - M) o_s / sum_s exp(m_s - M) l_s
    __threadfence();
    const float* pg = p.attn_part + ((int64_t)a.kvh * S * G) * PST;
    if (warp < G) {
        const int h = warp;
        float M = -CUDART_INF_F;
        for (int s = lane; s < S; s += 32) M = fmaxf(M, __ldcg(pg + ((int64_t)s * G + h) * PST + D));
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float den = 0.f;
        for (int s = lane; s < S; s += 32) {
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(pg + ((int64_t)s * G + h) * PST + D));
            const float e = ml.y > 0.f ? __expf(ml.x - M) : 0.f;
            wts[s * G + h] = e;
            den = fmaf(e, ml.y, den);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        const float inv = 1.f / den;
        for (int s = lane; s < S; s += 32) wts[s * G + h] *= inv;
    }
    __syncthreads();
    for (int t = tid; t < G * D; t += kThreadsP) {
        const int h = t / D, d = t % D;
        float o0 = 0.f, o1 = 0.f;
        int s = 0;
        for (; s + 2 <= S; s += 2) {
            o0 = fmaf(wts[s * G + h], __ldcg(pg + ((int64_t)s * G + h) * PST + d), o0);
            o1 = fmaf(wts[(s + 1) * G + h], __ldcg(pg + ((int64_t)(s + 1) * G + h) * PST + d), o1);
        }
        if (s < S) o0 = fmaf(wts[s * G + h], __ldcg(pg + ((int64_t)s * G + h) * PST + d), o0);
        p.attn[(int64_t)(a.kvh * G + h) * D + d] = o0 + o1;
    }
    if (tid == 0) p.attn_cnt[a.kvh] = 0u;
}

// ---------------------------------------------------------------- the kernel
template <int WT, int D, typename KT, int G>
__global__ void __launch_bounds__(kThreadsP, 1) decode_kernel(DecodePlan p) {
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ SharedP sm;
    // dynamic shared memory: [x image / attention scratch][phase table][slots]
    uint8_t* ximg = dsm;
    PhaseDesc* tab = reinterpret_cast<PhaseDesc*>(dsm + p.ximg_bytes);
    uint8_t* ring = dsm + p.ximg_bytes + p.tab_bytes;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nph = 5 * p.n_layers + 1;
    const int pos = p.st->pos;
    const int token = p.st->token;
    if (tid == 0) {
        for (int s = 0; s < p.nslot; s++) {
            mbar_init(&sm.full[s], 1);
            sm.issues[s] = 0;
        }
        sm.abort_cta = 0;
        fence_mbar_init();
    }
    // this CTA's schedule (one descriptor per phase); the first GEMV phase's task
    for (int ph = tid; ph < nph; ph += kThreadsP) tab[ph] = make_desc<KT>(p, ph, pos);
    if (warp == kWarpsP - 1) prefetch_task(p, sm, 0, lane);
    __syncthreads();
    unsigned gen = 0;  // barriers passed in this step (the count was reset by the step-begin kernel)
    int tr = 0;        // phase-boundary trace (CTA 0, thread 0)
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

    // every warp's issue cursor; thread 0 fills each slot with its first stage
    Cursor cur{0, 0};
    if (tid == 0)
        for (int g = 0; g < p.nslot; g++) issue_stage(p, sm, tab, nph, ring, cur, g, pol);

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

    int gnext = (tid >> 5);  // this warp's next global stage
    int gph = 0;             // first global stage of the running phase
    for (int l = 0; l < p.n_layers && ok; l++) {
        for (int op = 0; op < 5 && ok; op++) {
            const int ph = 5 * l + op;
            if (op == 1)
                attn_phase<D, G, KT>(p, sm, tab, nph, ximg, ring, cur, l, gph, gnext, pos, pol);
            else
                gemv_phase<WT>(p, sm, tab, nph, ximg, ring, cur, ph, gph, gnext, pos, pol);
            gph += tab[ph].nst;
            ok = !sm.abort_cta && grid_sync(p, gen, sm);
            trace();
        }
        if (ok) capture(l + 1);
    }
    if (ok) gemv_phase<WT>(p, sm, tab, nph, ximg, ring, cur, 5 * p.n_layers, gph, gnext, pos, pol);  // logits, argmax
    trace();

    __syncthreads();
    // copies of stages past the end are never issued; after an abort, drain the ones in flight
    if (sm.abort_cta) {
        if (tid == 0)
            for (int s = 0; s < p.nslot; s++)
                if (sm.issues[s]) mbar_wait_bounded(&sm.full[s], (sm.issues[s] - 1u) & 1u);
        __syncthreads();
    }
}

template <int WT, int D, typename KT, int G>
cudaError_t launch_decode_t(const DecodePlan& p, cudaStream_t s, bool prepare) {
    auto kern = decode_kernel<WT, D, KT, G>;
    const size_t smem = (size_t)p.ximg_bytes + (size_t)p.tab_bytes + (size_t)p.nslot * p.slot_bytes;
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

template <int WT, int D, typename KT>
cudaError_t launch_decode_g(const DecodePlan& p, cudaStream_t s, bool prepare) {
    switch (p.H / p.KVH) {
        case 2: return launch_decode_t<WT, D, KT, 2>(p, s, prepare);
        case 4: return launch_decode_t<WT, D, KT, 4>(p, s, prepare);
        case 8: return launch_decode_t<WT, D, KT, 8>(p, s, prepare);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Launch (or, with prepare, opt in to shared memory and check residency) for one
// (weight type, head_dim) pair; defined by the decode_*.cu translation units.
template <int WT, int D>
cudaError_t decode_launch_for(const DecodePlan& p, cudaStream_t s, bool prepare) {
    return p.kv_f16 ? launch_decode_g<WT, D, __half>(p, s, prepare) : launch_decode_g<WT, D, float>(p, s, prepare);
}

}  // namespace af
