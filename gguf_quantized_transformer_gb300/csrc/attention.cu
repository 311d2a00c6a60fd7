// Causal GQA attention over the KV cache (Airframe "GPU_PIPELINE.md": scores
// Q K^T / sqrt(head_dim), softmax over the sequence, weighted sum of V; the
// cache holds slots 0..t; dotLLM "Attention on GPU": GQA via
// group = n_heads / n_kv_heads, fp32 accumulation).
//
// Decode (one query row at position p): split-KV.  CTA (s, g) owns kv head g
// and the slot range s*chunk..: it serves all G query heads of the group, so
// each K/V byte is read once.  Within the CTA, pass 1 writes scores to shared
// memory, pass 2 exponentiates against the CTA maximum and accumulates P V.
// Each CTA stores (o, max, sum) for its range; the last CTA of a kv head to
// finish (acq_rel counter) merges the splits with the usual max-rescaling.
// For caches of up to kC * kClMaxSplit slots the kC = 8 splits of a kv head
// form a thread-block cluster instead and merge through distributed shared
// memory (attn_decode_kernel's CL path): no partials in global memory, no
// fence, counter or second round trip.
//
// Prefill attention runs on the tensor cores (attn_prefill_tc.cu).
#include <math_constants.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tma.cuh"

namespace af {

namespace {

template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float* out, int n);
template <>
__device__ __forceinline__ void load_vec<float>(const float* p, float* out, int n) {
    for (int i = 0; i < n; i += 4) {
        const float4 v = *reinterpret_cast<const float4*>(p + i);
        out[i] = v.x;
        out[i + 1] = v.y;
        out[i + 2] = v.z;
        out[i + 3] = v.w;
    }
}
template <>
__device__ __forceinline__ void load_vec<__half>(const __half* p, float* out, int n) {
    for (int i = 0; i < n; i += 8) {
        const uint4 raw = *reinterpret_cast<const uint4*>(p + i);
        const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float2 f = __half22float2(h[e]);
            out[i + 2 * e] = f.x;
            out[i + 2 * e + 1] = f.y;
        }
    }
}

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMinPerSplit = 64;  // positions per split before another split is used
constexpr int kRing = 64 * 1024;     // tile ring budget (two CTAs per SM)
constexpr int kRingCl = 176 * 1024;  // tile ring budget of the cluster path (one CTA per SM)
constexpr int kMaxStages = 12;
// Cluster path: the kC CTAs of one kv head form a thread-block cluster of one CTA per SM and merge through
// distributed shared memory; taken when every split has at most kClMaxSplit slots, i.e. for caches of up to
// 2048 slots, and when the device can schedule such clusters.  Longer caches take the split path: with few
// kv heads the clusters cover few SMs (measured: 16-CTA clusters of 16 warps took 18.6 us at position 4200 of
// an 8192-slot cache against 12.2 us for the split path, and 10.2 us against 6.2 us at position 128).
constexpr int kC = 8;
constexpr int kClMaxSplit = 256;
constexpr int kClWarps = 8;

// cache slots per pipeline tile: 16 KB of K (and 16 KB of V), one bulk copy each (smaller copies stream slower)
template <int D, typename KT>
__host__ __device__ constexpr int dec_tile() {
    return 16384 / (D * (int)sizeof(KT));
}
// stages (K tile + V tile) in the ring budget
template <int D, typename KT, bool CL>
__host__ __device__ constexpr int dec_stages() {
    return (CL ? kRingCl : kRing) / (2 * 16384) < kMaxStages ? (CL ? kRingCl : kRing) / (2 * 16384) : kMaxStages;
}

__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_dsmem(const float* local, uint32_t rank) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(dsmem_addr(local, rank)) : "memory");
    return v;
}
// every thread of every CTA of the cluster; release/acquire orders the shared-memory writes before it
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// n (2 or 4) consecutive cache values as fp32; p aligned to n elements.
template <int N>
__device__ __forceinline__ void load_small(const float* p, float* out) {
    if (N == 4) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    } else {
        const float2 v = *reinterpret_cast<const float2*>(p);
        out[0] = v.x; out[1] = v.y;
    }
}
template <int N>
__device__ __forceinline__ void load_small(const __half* p, float* out) {
    if (N == 4) {
        const uint2 raw = *reinterpret_cast<const uint2*>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        out[0] = a.x; out[1] = a.y; out[2] = b.x; out[3] = b.y;
    } else {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(p));
        out[0] = a.x; out[1] = a.y;
    }
}

// Splits of a sequence of n slots: ns_eff non-empty ranges of `chunk` slots (the last may be shorter).
__device__ __forceinline__ void dec_split(int n, int ns, int& ns_eff, int& chunk) {
    ns_eff = (n + kMinPerSplit - 1) / kMinPerSplit;
    ns_eff = ns_eff < ns ? ns_eff : ns;
    chunk = (n + ns_eff - 1) / ns_eff;
    ns_eff = (n + chunk - 1) / chunk;
}

// Offset of the merge's maxima / weights in a CTA's scratch: after the warps' combine buffer and after the
// merge's own per-thread float4 reduction area (which starts at the scratch base).
__host__ __device__ constexpr int merge_scratch_off(int combine_bytes, int nt) {
    return combine_bytes > nt * 16 ? combine_bytes : nt * 16;
}

// Merge of the ns_eff split partials of kv head g by the last CTA to finish (split path):
//   o_h = sum_s exp(m_s - M) o_s / sum_s exp(m_s - M) l_s.
// Each of the NT threads owns float4 f of the group's G x D outputs and the splits ph, ph + P, ..; it issues a
// batch of those partial-row loads into registers first, while warp h forms head h's weights with its lanes
// over the splits, so the partials and the weights arrive in about one L2 round trip.  scratch: shared memory
// for max(NT * 16, 2 * ns_eff * G * 4) bytes.
template <int D, int G, int NT>
__device__ __forceinline__ void merge_splits(const float* __restrict__ part, int g, int ns, int ns_eff,
                                             float* __restrict__ out, unsigned* __restrict__ cnt, uint8_t* red_smem,
                                             float* mm, int tid) {
    constexpr int PST = D + 4;
    constexpr int NF = G * D / 4;  // float4 outputs of the group
    constexpr int P = NT / NF;     // threads per output float4
    constexpr int kBatch = 16;     // partial loads in flight per thread
    static_assert(P >= 1 && P * NF == NT, "merge mapping");
    const int lane = tid & 31, warp = tid >> 5;
    const float* pg = part + ((int64_t)g * ns * G) * PST;
    float* ml = mm + ns_eff * G;  // [ns_eff][G] split maxima (then merge weights), sums
    const int f = tid % NF, ph = tid / NF, hf = (4 * f) / D, df = (4 * f) % D;
    float4 v[kBatch];
    auto load_batch = [&](int s0) {
#pragma unroll
        for (int i = 0; i < kBatch; i++) {
            const int ss = s0 + i * P;
            v[i] = ss < ns_eff ? __ldcg(reinterpret_cast<const float4*>(pg + ((int64_t)ss * G + hf) * PST + df))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    load_batch(ph);
    if (warp < G) {
        const int h = warp;
        float M = -CUDART_INF_F;
        for (int ss = lane; ss < ns_eff; ss += 32) {
            const float2 mlv = __ldcg(reinterpret_cast<const float2*>(pg + ((int64_t)ss * G + h) * PST + D));
            mm[ss * G + h] = mlv.x;
            ml[ss * G + h] = mlv.y;
            M = fmaxf(M, mlv.x);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float den = 0.f;
        for (int ss = lane; ss < ns_eff; ss += 32) den = fmaf(__expf(mm[ss * G + h] - M), ml[ss * G + h], den);
#pragma unroll
        for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        const float inv = 1.f / den;
        for (int ss = lane; ss < ns_eff; ss += 32) mm[ss * G + h] = __expf(mm[ss * G + h] - M) * inv;
    }
    __syncthreads();
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = ph; s0 < ns_eff; s0 += kBatch * P) {
        if (s0 != ph) load_batch(s0);
#pragma unroll
        for (int i = 0; i < kBatch; i++) {
            const int ss = s0 + i * P;
            if (ss < ns_eff) {
                const float w = mm[ss * G + hf];
                a.x = fmaf(w, v[i].x, a.x);
                a.y = fmaf(w, v[i].y, a.y);
                a.z = fmaf(w, v[i].z, a.z);
                a.w = fmaf(w, v[i].w, a.w);
            }
        }
    }
    // the P phases of an output, summed in a fixed order
    float4* red4 = reinterpret_cast<float4*>(red_smem);
    if (P > 1) {
        red4[ph * NF + f] = a;
        __syncthreads();
        if (ph == 0)
            for (int pp = 1; pp < P; pp++) {
                const float4 b = red4[pp * NF + f];
                a.x += b.x;
                a.y += b.y;
                a.z += b.z;
                a.w += b.w;
            }
    }
    if (ph == 0) {
        float* o = out + (int64_t)(g * G + hf) * D + df;
        o[0] = a.x;
        o[1] = a.y;
        o[2] = a.z;
        o[3] = a.w;
    }
    if (tid == 0) cnt[g] = 0u;
}

// Decode attention, CTA (s, g): kv head g, slots [s*chunk, ...) of the cache.
// The range streams through a ring of S stages; a stage is the K tile and the
// V tile (TS slots each, 16 KB) of the same slots, two bulk copies
// (cp.async.bulk) with an mbarrier each.  Every warp takes its own SPW = TS / 8
// slots of every stage and keeps an online softmax of its own (running
// maximum, running sum and the G x D output accumulator), so warps never wait
// for one another inside the loop: a stage is refilled by the last warp that
// is done with it (shared counter), and the only CTA barrier comes after the
// loop, where the warps' states are combined into the CTA's partial.
//   scores: lanes (LPK = D / 8 per slot, 8 dims each) score KPW = 32 / LPK
//           slots per warp step for all G heads (q pre-scaled by 1/sqrt(D) in
//           registers); a transpose-reduce leaves head li / LPH of the slot in
//           lane li, so each lane tracks the running maximum and sum of one head
//   P V:    the warp's probabilities go through shared memory; lane l owns
//           dims l*DV.. of all heads: acc = acc * corr + sum_j p_j V_j
// Split path (CL = false): two CTAs per SM where the registers allow, partials in global memory, merged by
// the last CTA of the kv head.  Cluster path (CL = true): the kC splits of a kv head are one cluster, one CTA
// per SM with a deeper ring; each keeps its partial in shared memory and, after a cluster barrier, CTA r
// merges output slice r from all of them through distributed shared memory (no counter, fence or atomic).
// Every mbarrier wait is bounded; a CTA that gives up records DEV_TIMEOUT, drains its copies and publishes a
// NaN weight, so the merged output of its kv head is NaN.
template <int D, int G, typename KT, bool CL>
__global__ void __launch_bounds__(CL ? kClWarps * 32 : kDecThreads, (!CL && G <= 4) ? 2 : 1)
    attn_decode_kernel(const float* __restrict__ q, const KT* __restrict__ kc, const KT* __restrict__ vc, int max_ctx,
                       const int* __restrict__ pos_dev, int pos_arg, float* __restrict__ part,
                       unsigned* __restrict__ cnt, float* __restrict__ out, unsigned* __restrict__ err) {
    constexpr int TS = dec_tile<D, KT>();            // slots per stage
    constexpr int TB = TS * D * (int)sizeof(KT);     // bytes of one K (or V) tile
    constexpr int S = dec_stages<D, KT, CL>();       // ring depth
    constexpr int NW = CL ? kClWarps : kDecWarps;    // warps
    constexpr int NT = NW * 32;
    constexpr int SPW = TS / NW;                     // slots of a warp per stage
    constexpr int LPK = D / 8;                       // scores: lanes per slot
    constexpr int KPW = 32 / LPK;                    // scores: slots per warp step
    constexpr int LPH = LPK / G;                     // lanes per head after the transpose-reduce
    constexpr int STEPS = SPW / KPW;                 // score steps per warp per stage
    constexpr int DV = D / 32;                       // P V: dims per lane
    static_assert(S >= 2 && S <= kMaxStages, "ring depth");
    static_assert(LPH >= 1 && STEPS >= 1 && SPW % KPW == 0, "lane mapping");
    extern __shared__ __align__(128) uint8_t dsm[];  // S x [K tile | V tile]; after the loop: combine scratch
    __shared__ uint64_t kfull[kMaxStages], vfull[kMaxStages];  // tile landed (transaction bytes)
    __shared__ unsigned issues[kMaxStages];  // copies issued into the stage slot so far
    __shared__ unsigned done[kMaxStages];    // warps done with the slot's current stage
    __shared__ __align__(16) float pw[NW][SPW][G];  // a warp's probabilities of the current stage
    __shared__ float cw[NW][G];                     // a warp's rescale factors of the current stage
    __shared__ float wm[NW][G], wl[NW][G];   // warps' running maxima and sums
    __shared__ unsigned last;
    __shared__ volatile int abort_f;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = blockIdx.y, s = blockIdx.x, ns = gridDim.x;
    pdl_launch_dependents();
    // the position word is written before the kernels of a step start; everything else the previous
    // kernel writes (q, the cache slot at pos) is read after griddepcontrol.wait
    const int pos = pos_dev ? __ldcg(pos_dev) : pos_arg;
    const int n = pos + 1;
    int ns_eff, chunk;
    dec_split(n, ns, ns_eff, chunk);
    const int j0 = s * chunk;
    const int nl = s < ns_eff ? min(n, j0 + chunk) - j0 : 0;
    const KT* K = kc + ((int64_t)g * max_ctx + j0) * D;
    const KT* V = vc + ((int64_t)g * max_ctx + j0) * D;
    constexpr int PST = D + 4;  // partial row: o[0..D-1], max, sum, 2 pad (16-byte rows)
    __shared__ __align__(16) float po[CL ? G * PST : 4];  // cluster path: this CTA's partial rows
    float* my = CL ? po : part + ((int64_t)(g * ns + s) * G) * PST;

    if (tid == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(&kfull[i], 1);
            mbar_init(&vfull[i], 1);
            issues[i] = 0;
            done[i] = 0;
        }
        abort_f = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int nst = (nl + TS - 1) / TS;
    auto issue = [&](int t) {  // one thread: K and V tiles of stage t into slot t % S
        const int keys = min(TS, nl - t * TS);
        const int slot = t % S;
        const unsigned bytes = (unsigned)(keys * D * (int)sizeof(KT));
        uint8_t* dst = dsm + slot * 2 * TB;
        issues[slot]++;
        mbar_arrive_expect_tx(&kfull[slot], bytes);
        bulk_g2s(dst, K + (int64_t)t * TS * D, bytes, &kfull[slot]);
        mbar_arrive_expect_tx(&vfull[slot], bytes);
        bulk_g2s(dst + TB, V + (int64_t)t * TS * D, bytes, &vfull[slot]);
    };
    // stages without slot pos stream in before waiting for the previous kernel
    if (tid == 0 && nst > 0) {
        const bool has_pos = j0 + nl == n;
        bool waited = false;
        for (int t = 0; t < min(S, nst); t++) {
            if (has_pos && !waited && t == nst - 1) {
                pdl_wait();
                waited = true;
            }
            issue(t);
        }
    }
    pdl_wait();

    const int li = lane % LPK, ks = lane / LPK, hl = li / LPH;
    float qv[G][8];
    {
        const float scale = rsqrtf((float)D);
#pragma unroll
        for (int h = 0; h < G; h++) {
            const float4 a = __ldcg(reinterpret_cast<const float4*>(q + (int64_t)(g * G + h) * D + li * 8));
            const float4 b = __ldcg(reinterpret_cast<const float4*>(q + (int64_t)(g * G + h) * D + li * 8 + 4));
            qv[h][0] = a.x * scale; qv[h][1] = a.y * scale; qv[h][2] = a.z * scale; qv[h][3] = a.w * scale;
            qv[h][4] = b.x * scale; qv[h][5] = b.y * scale; qv[h][6] = b.z * scale; qv[h][7] = b.w * scale;
        }
    }
    float m_run = -CUDART_INF_F, l_run = 0.f;  // head hl of this lane, over the warp's slots so far
    float acc[G][DV];
#pragma unroll
    for (int h = 0; h < G; h++)
#pragma unroll
        for (int e = 0; e < DV; e++) acc[h][e] = 0.f;

    auto wait_tile = [&](uint64_t* bar, unsigned par) {  // whole warp; false (uniformly) on a timeout or abort
        bool ok = false;
        for (unsigned it = 0; it < kWaitLimit && !ok; it++) {
            ok = mbar_try_wait(bar, par);
            if (!ok && abort_f) break;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0 && !abort_f) {
            abort_f = 1;
            atomicExch(err, (unsigned)DEV_TIMEOUT);
        }
        return ok;
    };

    for (int t = 0; t < nst; t++) {
        const int slot = t % S;
        const unsigned par = (unsigned)((t / S) & 1);
        const int keys = min(TS, nl - t * TS);
        if (!wait_tile(&kfull[slot], par)) break;
        const KT* kt = reinterpret_cast<const KT*>(dsm + slot * 2 * TB);
        const KT* vt = reinterpret_cast<const KT*>(dsm + slot * 2 * TB + TB);
        // ---- scores of the warp's slots: step st covers slots warp*SPW + st*KPW + (0..KPW-1)
        float sreg[STEPS];
        float mt = -CUDART_INF_F;
#pragma unroll
        for (int st = 0; st < STEPS; st++) {
            const int j = warp * SPW + st * KPW + ks;
            float kf[8];
            if (j < keys) {
                load_vec<KT>(kt + j * D + li * 8, kf, 8);
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
            // transpose-reduce over the slot's LPK lanes: each exchange halves the heads a lane keeps
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
        // ---- online softmax of head hl over this stage's slots of the warp (the KPW slot lanes share a head)
#pragma unroll
        for (int o = LPK; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
        const float m_new = fmaxf(m_run, mt);
        const float corr = m_new == -CUDART_INF_F ? 1.f : __expf(m_run - m_new);
        float psum = 0.f;
#pragma unroll
        for (int st = 0; st < STEPS; st++) {
            const float p = sreg[st] == -CUDART_INF_F ? 0.f : __expf(sreg[st] - m_new);
            psum += p;
            if (li % LPH == 0) pw[warp][st * KPW + ks][hl] = p;
        }
#pragma unroll
        for (int o = LPK; o < 32; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
        l_run = fmaf(l_run, corr, psum);
        m_run = m_new;
        if (lane < LPK && li % LPH == 0) cw[warp][hl] = corr;
        __syncwarp();
        // ---- P V over the warp's slots
        if (!wait_tile(&vfull[slot], par)) break;
#pragma unroll
        for (int h = 0; h < G; h++) {
            const float c = cw[warp][h];
#pragma unroll
            for (int e = 0; e < DV; e++) acc[h][e] *= c;
        }
#pragma unroll
        for (int jj = 0; jj < SPW; jj++) {
            const int j = warp * SPW + jj;
            if (j < keys) {
                float vf[DV];
                load_small<DV>(vt + j * D + lane * DV, vf);
                float p[G];
#pragma unroll
                for (int h = 0; h < G; h++) p[h] = pw[warp][jj][h];
#pragma unroll
                for (int h = 0; h < G; h++)
#pragma unroll
                    for (int e = 0; e < DV; e++) acc[h][e] = fmaf(p[h], vf[e], acc[h][e]);
            }
        }
        __syncwarp();
        // ---- the last warp done with this stage refills its slot
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&done[slot], 1u) == (unsigned)NW - 1u) {
                done[slot] = 0;
                if (t + S < nst) {
                    fence_proxy_async_shared();  // every warp's reads of the slot before the copies overwrite it
                    issue(t + S);
                }
            }
        }
    }
    __syncthreads();
    if (abort_f) {  // drain the copies still in flight before the ring is reused or the CTA exits
        if (tid == 0)
            for (int i = 0; i < S; i++)
                if (issues[i]) {
                    mbar_wait_bounded(&kfull[i], (issues[i] - 1u) & 1u);
                    mbar_wait_bounded(&vfull[i], (issues[i] - 1u) & 1u);
                }
        __syncthreads();
    }
    // ---- combine the warps' states into the CTA's partial (the ring is free now)
    float* red_o = reinterpret_cast<float*>(dsm);  // [warp][G][D]
#pragma unroll
    for (int h = 0; h < G; h++)
#pragma unroll
        for (int e = 0; e < DV; e++) red_o[(warp * G + h) * D + lane * DV + e] = acc[h][e];
    if (lane < LPK && li % LPH == 0) {
        wm[warp][hl] = m_run;
        wl[warp][hl] = l_run;
    }
    __syncthreads();
    if (nl > 0) {
        for (int t = tid; t < G * D; t += NT) {
            const int h = t / D, d = t % D;
            float M = -CUDART_INF_F;
#pragma unroll
            for (int w = 0; w < NW; w++) M = fmaxf(M, wm[w][h]);
            float o = 0.f, l = 0.f;
#pragma unroll
            for (int w = 0; w < NW; w++) {
                const float e = wm[w][h] == -CUDART_INF_F ? 0.f : __expf(wm[w][h] - M);
                o = fmaf(e, red_o[(w * G + h) * D + d], o);
                l = fmaf(e, wl[w][h], l);
            }
            my[h * PST + d] = o;
            if (d == 0) {  // an aborted split publishes a NaN weight, so the merged output of its kv head is NaN
                my[h * PST + D] = abort_f ? 0.f : M;
                my[h * PST + D + 1] = abort_f ? CUDART_NAN_F : l;
            }
        }
    } else if (CL) {  // an empty split: zero output, zero weight
        for (int t = tid; t < G * PST; t += NT) po[t] = (t % PST == D) ? -CUDART_INF_F : 0.f;
    }
    if constexpr (CL) {
        __shared__ float wc[kC][G];  // merge weights of the cluster's splits
        cluster_sync();              // every CTA's partial rows are written
        if (warp < G) {
            const int h = warp;
            float m = -CUDART_INF_F, l = 0.f;
            if (lane < kC) {
                m = ld_dsmem(&po[h * PST + D], lane);
                l = ld_dsmem(&po[h * PST + D + 1], lane);
            }
            float M = m;
#pragma unroll
            for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float e = m > -CUDART_INF_F ? __expf(m - M) : 0.f;
            float den = e * l;
#pragma unroll
            for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
            if (lane < kC) wc[lane][h] = e / den;
        }
        __syncthreads();
        // output slice of this CTA (cluster rank s): all kC partial values of each output in flight together
        constexpr int OPC = G * D / kC;
        for (int t = tid; t < OPC; t += NT) {
            const int o = s * OPC + t, h = o / D, d = o % D;
            float v[kC];
#pragma unroll
            for (int r = 0; r < kC; r++) v[r] = ld_dsmem(&po[h * PST + d], r);
            float acc2 = 0.f;
#pragma unroll
            for (int r = 0; r < kC; r++) acc2 = fmaf(wc[r][h], v[r], acc2);
            out[(int64_t)(g * G + h) * D + d] = acc2;
        }
        cluster_sync();  // no CTA leaves while another still reads its partial
        return;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned old = atomicAdd(&cnt[g], 1u);
        last = (old == (unsigned)ns - 1u);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    merge_splits<D, G, NT>(part, g, ns, ns_eff, out, cnt, dsm,
                           reinterpret_cast<float*>(dsm + merge_scratch_off(NW * G * D * 4, NT)), tid);
}

// ---------------------------------------------------------------------------------------------------------
// Decode attention over an fp16 cache on the tensor cores (split path).  Same split, stages, merge and
// per-warp online softmax as attn_decode_kernel, with the score and P V products as mma.sync m16n8k16 (fp16 in,
// fp32 accumulate) over 16-slot tiles of a warp's slots:
//   scores  S^T[16 slots][8] = K[16 slots][D] Qc^T[D][8], Qc = (q_hi of the G heads | q_lo of the G heads) with
//           1/sqrt(D) folded in; the score of head h is column h plus column 4 + h;
//   P V     O^T[D][8] += V^T[D][16 slots] Pc[16 slots][8], Pc = (p_hi | p_lo) per head, through shared memory.
// The fp16 cache is exact in fp16, so with q and p split into hi + lo the products keep near-fp32 precision.
// K and V tiles arrive by TMA (cp.async.bulk.tensor, SWIZZLE_128B, boxes of 64 dims), so the ldmatrix fragment
// loads (K as rows, V transposed) are free of bank conflicts.  Group sizes up to 4 (8 columns).
constexpr int kTcWarps = 4;

__device__ __forceinline__ void tma_load_tile(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// shared address of 16-byte chunk `chunk` (8 fp16 along D) of row `row` in a tile of `rows` rows stored as
// SWIZZLE_128B atoms of 64 dims (atom a at a * rows * 128 bytes); the tile base is 1024-byte aligned
__device__ __forceinline__ uint32_t sw_addr(uint32_t base, int rows, int row, int chunk) {
    return base + (uint32_t)((chunk >> 3) * rows * 128 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <int D, int G>
__global__ void __launch_bounds__(kTcWarps * 32, 2)
    attn_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const float* __restrict__ q, int max_ctx, const int* __restrict__ pos_dev, int pos_arg,
                          float* __restrict__ part, unsigned* __restrict__ cnt, float* __restrict__ out,
                          unsigned* __restrict__ err) {
    constexpr int NW = kTcWarps, NT = NW * 32;
    constexpr int TS = dec_tile<D, __half>();  // slots per stage (16 KB of K)
    constexpr int TB = TS * D * 2;
    constexpr int S = kRing / (2 * TB) < kMaxStages ? kRing / (2 * TB) : kMaxStages;
    constexpr int SPW = TS / NW;               // slots of a warp per stage
    constexpr int MT = SPW / 16;               // 16-slot MMA tiles of a warp per stage
    constexpr int KS = D / 16;                 // K steps of the score MMA
    constexpr int DT = D / 16;                 // 16-dim tiles of the P V MMA
    static_assert(G <= 4 && S >= 2 && MT >= 1 && SPW % 16 == 0, "shape");
    extern __shared__ __align__(128) uint8_t dsm[];  // S x [K tile | V tile] (aligned to 1024 below), 64-dim SW128 atoms
    __shared__ uint64_t kfull[kMaxStages], vfull[kMaxStages];
    __shared__ unsigned issues[kMaxStages], done[kMaxStages];
    __shared__ __align__(16) __half pc[NW][8][16];  // a warp's Pc tile, column-major: [col][slot]
    __shared__ float wm[NW][G], wl[NW][G];
    __shared__ __align__(16) float qs[G * D];      // q of the group's heads (one coalesced L2 read)
    __shared__ unsigned last;
    __shared__ volatile int abort_f;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = blockIdx.y, s = blockIdx.x, ns = gridDim.x;
    pdl_launch_dependents();
    if (tid == 0) {  // the tensor maps' descriptors, ahead of their first use
        asm volatile("prefetch.tensormap [%0];" ::"l"(&kmap) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&vmap) : "memory");
    }
    const int pos = pos_dev ? __ldcg(pos_dev) : pos_arg;
    const int n = pos + 1;
    int ns_eff, chunk;
    dec_split(n, ns, ns_eff, chunk);
    const int j0 = s * chunk;
    const int nl = s < ns_eff ? min(n, j0 + chunk) - j0 : 0;
    const int nst = (nl + TS - 1) / TS;
    const int row0 = g * max_ctx + j0;  // tensor-map row of the range's first slot
    constexpr int PST = D + 4;
    float* my = part + ((int64_t)(g * ns + s) * G) * PST;
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~(uintptr_t)1023);

    if (tid == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(&kfull[i], 1);
            mbar_init(&vfull[i], 1);
            issues[i] = 0;
            done[i] = 0;
        }
        abort_f = 0;
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int t) {  // one thread: K and V boxes of stage t into slot t % S (rows past the range are
                               // read too and masked; past the array they are zero-filled)
        const int slot = t % S;
        uint8_t* dst = ring + slot * 2 * TB;
        issues[slot]++;
        mbar_arrive_expect_tx(&kfull[slot], TB);
#pragma unroll
        for (int a = 0; a < D / 64; a++) tma_load_tile(dst + a * TS * 128, &kmap, 64 * a, row0 + t * TS, &kfull[slot]);
        mbar_arrive_expect_tx(&vfull[slot], TB);
#pragma unroll
        for (int a = 0; a < D / 64; a++)
            tma_load_tile(dst + TB + a * TS * 128, &vmap, 64 * a, row0 + t * TS, &vfull[slot]);
    };
    if (tid == 0 && nst > 0) {
        const bool has_pos = j0 + nl == n;
        bool waited = false;
        for (int t = 0; t < min(S, nst); t++) {
            if (has_pos && !waited && t == nst - 1) {
                pdl_wait();
                waited = true;
            }
            issue(t);
        }
    }
    pdl_wait();
    for (int i = tid; i < G * D / 4; i += NT)  // q was written by the previous kernel: through L2
        reinterpret_cast<float4*>(qs)[i] = __ldcg(reinterpret_cast<const float4*>(q + (int64_t)g * G * D) + i);
    __syncthreads();

    // B fragments of Qc (constant): thread holds column cn = lane / 4 (head cn % 4, hi if cn < 4) at K rows
    // 2 (lane % 4) + {0, 1} and + 8 of every K step
    const int quad = lane & 3, cn = lane >> 2;
    uint32_t qb[KS][2];
    {
        const int h = cn & 3;
        const float scale = rsqrtf((float)D);
        const float* qh = qs + (h < G ? h : 0) * D;
#pragma unroll
        for (int kk = 0; kk < KS; kk++) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int k = kk * 16 + 2 * quad + (e & 1) + 8 * (e >> 1);
                const float x = h < G ? qh[k] * scale : 0.f;
                const float hi = __half2float(__float2half_rn(x));
                v[e] = cn < 4 ? hi : x - hi;
            }
            qb[kk][0] = pack_h2(v[0], v[1]);
            qb[kk][1] = pack_h2(v[2], v[3]);
        }
    }
    // online softmax state: a lane with quad < 2 tracks heads 2 quad, 2 quad + 1 (columns of its score fragment)
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F}, l_run[2] = {0.f, 0.f};
    float oacc[DT][4];
#pragma unroll
    for (int d = 0; d < DT; d++)
#pragma unroll
        for (int e = 0; e < 4; e++) oacc[d][e] = 0.f;

    auto wait_tile = [&](uint64_t* bar, unsigned par) {
        bool ok = false;
        for (unsigned it = 0; it < kWaitLimit && !ok; it++) {
            ok = mbar_try_wait(bar, par);
            if (!ok && abort_f) break;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0 && !abort_f) {
            abort_f = 1;
            atomicExch(err, (unsigned)DEV_TIMEOUT);
        }
        return ok;
    };
    const uint32_t pcw = smem_u32(&pc[warp][0][0]);

    for (int t = 0; t < nst; t++) {
        const int slot = t % S;
        const unsigned par = (unsigned)((t / S) & 1);
        const int keys = min(TS, nl - t * TS);
        if (!wait_tile(&kfull[slot], par)) break;
        const uint32_t kt = smem_u32(ring + slot * 2 * TB), vt = kt + TB;
        bool vready = false;
#pragma unroll
        for (int mt = 0; mt < MT; mt++) {
            const int r0 = warp * SPW + mt * 16;  // first slot of this tile within the stage
            // ---- scores
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < KS; kk++) {
                uint32_t a[4];
                ldsm_x4(sw_addr(kt, TS, r0 + (lane & 15), 2 * kk + (lane >> 4)), a);
                mma16816(c, a, qb[kk][0], qb[kk][1]);
            }
            // c: rows r0 + cn, r0 + cn + 8; columns 2 quad, 2 quad + 1.  Score = hi column + lo column (quad ^ 2).
            float sc[4];
#pragma unroll
            for (int e = 0; e < 4; e++) sc[e] = c[e] + __shfl_xor_sync(0xffffffffu, c[e], 2);
            const bool v0 = r0 + cn < keys, v1 = r0 + cn + 8 < keys;
            if (!v0) sc[0] = sc[1] = -CUDART_INF_F;
            if (!v1) sc[2] = sc[3] = -CUDART_INF_F;
            float corr[2], p[4];
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {  // heads 2 quad + hh (meaningful for quad < 2)
                float mt2 = fmaxf(sc[hh], sc[2 + hh]);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) mt2 = fmaxf(mt2, __shfl_xor_sync(0xffffffffu, mt2, o));
                const float m_new = fmaxf(m_run[hh], mt2);
                corr[hh] = m_new == -CUDART_INF_F ? 1.f : __expf(m_run[hh] - m_new);
                p[hh] = sc[hh] == -CUDART_INF_F ? 0.f : __expf(sc[hh] - m_new);
                p[2 + hh] = sc[2 + hh] == -CUDART_INF_F ? 0.f : __expf(sc[2 + hh] - m_new);
                l_run[hh] = fmaf(l_run[hh], corr[hh], p[hh] + p[2 + hh]);
                m_run[hh] = m_new;
            }
            // Pc tile: column h = p_hi of head h, column 4 + h = p_lo; rows = the tile's 16 slots
            if (quad < 2) {
                __half* pw = &pc[warp][0][0];
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int h = 2 * quad + (e & 1), r = cn + 8 * (e >> 1);
                    const __half ph = __float2half_rn(p[e]);
                    pw[h * 16 + r] = ph;
                    pw[(4 + h) * 16 + r] = __float2half_rn(p[e] - __half2float(ph));
                }
            }
            __syncwarp();
            // the O^T accumulator's columns 2 quad, 2 quad + 1 are heads (2 quad) % 4.. (hi or lo): rescale both
            const float cr0 = __shfl_sync(0xffffffffu, corr[0], (lane & ~3) | (quad & 1));
            const float cr1 = __shfl_sync(0xffffffffu, corr[1], (lane & ~3) | (quad & 1));
#pragma unroll
            for (int d = 0; d < DT; d++) {
                oacc[d][0] *= cr0;
                oacc[d][1] *= cr1;
                oacc[d][2] *= cr0;
                oacc[d][3] *= cr1;
            }
            // ---- P V
            if (!vready) {
                if (!wait_tile(&vfull[slot], par)) break;
                vready = true;
            }
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&pc[warp][cn][2 * quad]);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&pc[warp][cn][2 * quad + 8]);
#pragma unroll
            for (int d = 0; d < DT; d++) {
                // V^T tile (dims 16 d.., slots r0..): matrices (dims 0-7 | 8-15) x (slots 0-7 | 8-15), transposed
                const int mq = lane >> 3;
                uint32_t a[4];
                ldsm_x4_t(sw_addr(vt, TS, r0 + (lane & 7) + 8 * (mq >> 1), 2 * d + (mq & 1)), a);
                mma16816(oacc[d], a, b0, b1);
            }
            __syncwarp();  // the Pc tile is reused by the next MMA tile
        }
        if (abort_f) break;
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&done[slot], 1u) == (unsigned)NW - 1u) {
                done[slot] = 0;
                if (t + S < nst) {
                    fence_proxy_async_shared();
                    issue(t + S);
                }
            }
        }
    }
    __syncthreads();
    if (abort_f) {
        if (tid == 0)
            for (int i = 0; i < S; i++)
                if (issues[i]) {
                    mbar_wait_bounded(&kfull[i], (issues[i] - 1u) & 1u);
                    mbar_wait_bounded(&vfull[i], (issues[i] - 1u) & 1u);
                }
        __syncthreads();
    }
    // ---- combine the warps: O = hi column + lo column; lanes with quad < 2 hold heads 2 quad, 2 quad + 1
    float* red_o = reinterpret_cast<float*>(ring);  // [warp][G][D]
#pragma unroll
    for (int d = 0; d < DT; d++) {
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; e++) o[e] = oacc[d][e] + __shfl_xor_sync(0xffffffffu, oacc[d][e], 2);
        if (quad < 2)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int h = 2 * quad + (e & 1), dim = 16 * d + cn + 8 * (e >> 1);
                if (h < G) red_o[(warp * G + h) * D + dim] = o[e];
            }
    }
    // l: per-lane partial sums over the lane's rows; reduce over the 8 lanes of each quad
#pragma unroll
    for (int hh = 0; hh < 2; hh++)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], o);
    if (lane < 2)
#pragma unroll
        for (int hh = 0; hh < 2; hh++)
            if (2 * lane + hh < G) {
                wm[warp][2 * lane + hh] = m_run[hh];
                wl[warp][2 * lane + hh] = l_run[hh];
            }
    __syncthreads();
    if (nl > 0)
        for (int t = tid; t < G * D; t += NT) {
            const int h = t / D, d = t % D;
            float M = -CUDART_INF_F;
#pragma unroll
            for (int w = 0; w < NW; w++) M = fmaxf(M, wm[w][h]);
            float o = 0.f, l = 0.f;
#pragma unroll
            for (int w = 0; w < NW; w++) {
                const float e = wm[w][h] == -CUDART_INF_F ? 0.f : __expf(wm[w][h] - M);
                o = fmaf(e, red_o[(w * G + h) * D + d], o);
                l = fmaf(e, wl[w][h], l);
            }
            my[h * PST + d] = o;
            if (d == 0) {
                my[h * PST + D] = abort_f ? 0.f : M;
                my[h * PST + D + 1] = abort_f ? CUDART_NAN_F : l;
            }
        }
    __threadfence();
    __syncthreads();
    if (tid == 0) last = (atomicAdd(&cnt[g], 1u) == (unsigned)ns - 1u);
    __syncthreads();
    if (!last) return;
    __threadfence();
    merge_splits<D, G, NT>(part, g, ns, ns_eff, out, cnt, ring,
                           reinterpret_cast<float*>(ring + merge_scratch_off(NW * G * D * 4, NT)), tid);
}

template <int D, int G>
cudaError_t launch_tc_t(const float* q, const void* kc, const void* vc, int max_ctx, const int* pos_dev, int pos,
                        const AttnScratch& scr, int ns, float* out, int KVH, cudaStream_t s) {
    constexpr int TS = dec_tile<D, __half>();
    constexpr int TB = TS * D * 2;
    constexpr int S = kRing / (2 * TB) < kMaxStages ? kRing / (2 * TB) : kMaxStages;
    const size_t smem = (size_t)S * 2 * TB + 1024;  // + alignment of the ring to 1024 bytes
    if ((size_t)merge_scratch_off(kTcWarps * G * D * 4, kTcWarps * 32) + (size_t)ns * G * 8 > (size_t)S * 2 * TB)
        return cudaErrorInvalidValue;
    CUtensorMap km, vm;
    if (!make_tmap_f16(&km, kc, (uint64_t)KVH * max_ctx, D, D, 64, TS) ||
        !make_tmap_f16(&vm, vc, (uint64_t)KVH * max_ctx, D, D, 64, TS))
        return cudaErrorInvalidValue;
    auto k = attn_decode_tc_kernel<D, G>;
    static int opened[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!opened[dev]) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e) return e;
            opened[dev] = 1;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ns, KVH);
    cfg.blockDim = dim3(kTcWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, km, vm, q, max_ctx, pos_dev, pos, scr.part, scr.cnt, out, scr.err);
}

// ---------------------------------------------------------------------------------------------------------
// Decode attention over a quantized cache (AF_KV_Q8_0 / AF_KV_Q4_0, split path): the slots that left the window
// (below cut = pos + 1 - window) are read from the quantized store, the window from the fp16 cache.  A CTA's
// range [j0, j0 + nl) (j0 a multiple of 4) is cut at `cut` into a store segment, streamed in stages of TQ slots
// (codes and scales of K, then of V: four bulk copies), and an fp16 segment, streamed as in attn_decode_kernel.
// The per-warp online softmax, the combine and the split merge are attn_decode_kernel's.

// One warp's share of one stage: scores of its slots, online-softmax update, P V.  ldk(j, li, kf) gives the 8
// K values of slot j at dims li*8.., ldv(j, lane, vf) the DV V values at dims lane*DV..; wait_v() waits for the
// stage's V data (false: give up).  Returns false if it gave up.
template <int D, int G, int SPW, class LoadK, class LoadV, class WaitV>
__device__ __forceinline__ bool warp_stage(const float (&qv)[G][8], int keys, int warp, int lane, LoadK ldk, LoadV ldv,
                                           WaitV wait_v, float& m_run, float& l_run, float (&acc)[G][D / 32],
                                           float (*pw)[G], float* cw) {
    constexpr int LPK = D / 8, KPW = 32 / LPK, LPH = LPK / G, STEPS = SPW / KPW, DV = D / 32;
    const int li = lane % LPK, ks = lane / LPK, hl = li / LPH;
    float sreg[STEPS];
    float mt = -CUDART_INF_F;
#pragma unroll
    for (int st = 0; st < STEPS; st++) {
        const int j = warp * SPW + st * KPW + ks;
        float kf[8];
        if (j < keys) {
            ldk(j, li, kf);
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
        const float p = sreg[st] == -CUDART_INF_F ? 0.f : __expf(sreg[st] - m_new);
        psum += p;
        if (li % LPH == 0) pw[st * KPW + ks][hl] = p;
    }
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    l_run = fmaf(l_run, corr, psum);
    m_run = m_new;
    if (lane < LPK && li % LPH == 0) cw[hl] = corr;
    __syncwarp();
    if (!wait_v()) return false;
#pragma unroll
    for (int h = 0; h < G; h++) {
        const float c = cw[h];
#pragma unroll
        for (int e = 0; e < DV; e++) acc[h][e] *= c;
    }
#pragma unroll
    for (int jj = 0; jj < SPW; jj++) {
        const int j = warp * SPW + jj;
        if (j < keys) {
            float vf[DV];
            ldv(j, lane, vf);
#pragma unroll
            for (int h = 0; h < G; h++) {
                const float p = pw[jj][h];
#pragma unroll
                for (int e = 0; e < DV; e++) acc[h][e] = fmaf(p, vf[e], acc[h][e]);
            }
        }
    }
    __syncwarp();
    return true;
}

constexpr int kQTile = 128;             // slots per store stage
constexpr int kRingQ = 104 * 1024;      // ring budget of the quantized-cache kernel (two CTAs per SM)

template <int D, int QT>
struct KvqCfg {
    static constexpr int TS = dec_tile<D, __half>();                      // fp16 stage slots
    static constexpr int CB = QT == AF_KV_Q8_0 ? D : D / 2;               // code bytes per slot
    static constexpr int SB = D / 32 * 2;                                 // scale bytes per slot
    static constexpr int QCODES = kQTile * CB, QSC = kQTile * SB;         // bytes of one K (or V) store tile
    static constexpr int FST = 2 * TS * D * 2;                            // fp16 stage
    static constexpr int QST = 2 * (QCODES + QSC);                        // store stage
    static constexpr int SLOT = ((FST > QST ? FST : QST) + 127) / 128 * 128;
    static constexpr int S = kRingQ / SLOT < kMaxStages ? kRingQ / SLOT : kMaxStages;
};

template <int D, int G, int QT>
__global__ void __launch_bounds__(kDecThreads, G <= 4 ? 2 : 1)
    attn_decode_kvq_kernel(const float* __restrict__ q, const __half* __restrict__ kc, const __half* __restrict__ vc,
                           KvLayerStore qs, int max_ctx, const int* __restrict__ pos_dev, int pos_arg,
                           float* __restrict__ part, unsigned* __restrict__ cnt, float* __restrict__ out,
                           unsigned* __restrict__ err) {
    using C = KvqCfg<D, QT>;
    constexpr int S = C::S, TS = C::TS, NW = kDecWarps, NT = kDecThreads;
    constexpr int LPK = D / 8, LPH = LPK / G, DV = D / 32;
    constexpr int SPWF = TS / NW, SPWQ = kQTile / NW, SPWM = SPWF > SPWQ ? SPWF : SPWQ;
    static_assert(S >= 2, "ring depth");
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ uint64_t kfull[kMaxStages], vfull[kMaxStages];
    __shared__ unsigned issues[kMaxStages], done[kMaxStages];
    __shared__ __align__(16) float pw[NW][SPWM][G];
    __shared__ float cw[NW][G];
    __shared__ float wm[NW][G], wl[NW][G];
    __shared__ unsigned last;
    __shared__ volatile int abort_f;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = blockIdx.y, s = blockIdx.x, ns = gridDim.x;
    pdl_launch_dependents();
    const int pos = pos_dev ? __ldcg(pos_dev) : pos_arg;
    const int n = pos + 1;
    const int cut = max(0, n - qs.window);  // slots below cut have retired (the newest, cut - 1, in this step)
    int ns_eff, chunk;
    dec_split(n, ns, ns_eff, chunk);
    chunk = (chunk + 3) & ~3;  // store tiles start on 4-slot boundaries (16-byte aligned scale copies)
    ns_eff = (n + chunk - 1) / chunk;
    const int j0 = s * chunk;
    const int nl = s < ns_eff ? min(n, j0 + chunk) - j0 : 0;
    const int qb = min(max(cut, j0), j0 + nl);  // store segment [j0, qb), fp16 segment [qb, j0 + nl)
    const int nstq = (qb - j0 + kQTile - 1) / kQTile;
    const int nst = nstq + (j0 + nl - qb + TS - 1) / TS;
    const int64_t rb = (int64_t)g * max_ctx;  // first slot row of this kv head in the layer
    constexpr int PST = D + 4;
    float* my = part + ((int64_t)(g * ns + s) * G) * PST;

    if (tid == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(&kfull[i], 1);
            mbar_init(&vfull[i], 1);
            issues[i] = 0;
            done[i] = 0;
        }
        abort_f = 0;
        fence_mbar_init();
    }
    __syncthreads();
    auto stage_keys = [&](int t) {
        return t < nstq ? min(kQTile, qb - j0 - t * kQTile) : min(TS, j0 + nl - qb - (t - nstq) * TS);
    };
    auto issue = [&](int t) {  // one thread: stage t into slot t % S
        const int slot = t % S, keys = stage_keys(t);
        uint8_t* dst = dsm + slot * C::SLOT;
        issues[slot]++;
        if (t < nstq) {
            const int64_t j = rb + j0 + (int64_t)t * kQTile;
            const int k4 = (keys + 3) & ~3;  // whole 4-slot groups (max_ctx is a multiple of 4)
            const unsigned cbytes = (unsigned)(k4 * C::CB), sbytes = (unsigned)(k4 * C::SB);
            mbar_arrive_expect_tx(&kfull[slot], cbytes + sbytes);
            bulk_g2s(dst, qs.kq + j * C::CB, cbytes, &kfull[slot]);
            bulk_g2s(dst + C::QCODES, reinterpret_cast<const uint8_t*>(qs.ks) + j * C::SB, sbytes, &kfull[slot]);
            mbar_arrive_expect_tx(&vfull[slot], cbytes + sbytes);
            bulk_g2s(dst + C::QCODES + C::QSC, qs.vq + j * C::CB, cbytes, &vfull[slot]);
            bulk_g2s(dst + 2 * C::QCODES + C::QSC, reinterpret_cast<const uint8_t*>(qs.vs) + j * C::SB, sbytes,
                     &vfull[slot]);
        } else {
            const int64_t j = rb + qb + (int64_t)(t - nstq) * TS;
            const unsigned bytes = (unsigned)(keys * D * 2);
            mbar_arrive_expect_tx(&kfull[slot], bytes);
            bulk_g2s(dst, kc + j * D, bytes, &kfull[slot]);
            mbar_arrive_expect_tx(&vfull[slot], bytes);
            bulk_g2s(dst + TS * D * 2, vc + j * D, bytes, &vfull[slot]);
        }
    };
    // stages holding slot pos (written by this step's QKV) or slot cut - 1 (retired in this step) wait for the
    // previous kernels; the rest stream in before
    if (tid == 0 && nst > 0) {
        bool waited = false;
        for (int t = 0; t < min(S, nst); t++) {
            const bool late = (t == nst - 1 && j0 + nl == n) || (t == nstq - 1 && qb == cut && cut > j0);
            if (late && !waited) {
                pdl_wait();
                waited = true;
            }
            issue(t);
        }
    }
    pdl_wait();

    const int li = lane % LPK, hl = li / LPH;
    float qv[G][8];
    {
        const float scale = rsqrtf((float)D);
#pragma unroll
        for (int h = 0; h < G; h++) {
            const float4 a = __ldcg(reinterpret_cast<const float4*>(q + (int64_t)(g * G + h) * D + li * 8));
            const float4 b = __ldcg(reinterpret_cast<const float4*>(q + (int64_t)(g * G + h) * D + li * 8 + 4));
            qv[h][0] = a.x * scale; qv[h][1] = a.y * scale; qv[h][2] = a.z * scale; qv[h][3] = a.w * scale;
            qv[h][4] = b.x * scale; qv[h][5] = b.y * scale; qv[h][6] = b.z * scale; qv[h][7] = b.w * scale;
        }
    }
    float m_run = -CUDART_INF_F, l_run = 0.f;
    float acc[G][DV];
#pragma unroll
    for (int h = 0; h < G; h++)
#pragma unroll
        for (int e = 0; e < DV; e++) acc[h][e] = 0.f;

    auto wait_tile = [&](uint64_t* bar, unsigned par) {
        bool ok = false;
        for (unsigned it = 0; it < kWaitLimit && !ok; it++) {
            ok = mbar_try_wait(bar, par);
            if (!ok && abort_f) break;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && lane == 0 && !abort_f) {
            abort_f = 1;
            atomicExch(err, (unsigned)DEV_TIMEOUT);
        }
        return ok;
    };

    for (int t = 0; t < nst; t++) {
        const int slot = t % S;
        const unsigned par = (unsigned)((t / S) & 1);
        const int keys = stage_keys(t);
        if (!wait_tile(&kfull[slot], par)) break;
        const uint8_t* base = dsm + slot * C::SLOT;
        auto wait_v = [&]() { return wait_tile(&vfull[slot], par); };
        bool ok;
        if (t < nstq) {
            const uint8_t* kq8 = base;
            const __half* ksc = reinterpret_cast<const __half*>(base + C::QCODES);
            const uint8_t* vq8 = base + C::QCODES + C::QSC;
            const __half* vsc = reinterpret_cast<const __half*>(base + 2 * C::QCODES + C::QSC);
            auto ldk = [&](int j, int l8, float (&kf)[8]) {
                const float d = __half2float(ksc[j * (D / 32) + l8 / 4]);
                if (QT == AF_KV_Q8_0) {
                    const uint2 w = *reinterpret_cast<const uint2*>(kq8 + j * C::CB + l8 * 8);
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        kf[e] = (float)(int)(signed char)(w.x >> (8 * e)) * d;
                        kf[4 + e] = (float)(int)(signed char)(w.y >> (8 * e)) * d;
                    }
                } else {
                    const unsigned w = *reinterpret_cast<const unsigned*>(kq8 + j * C::CB + l8 * 4);
#pragma unroll
                    for (int e = 0; e < 8; e++) kf[e] = (float)((int)((w >> (4 * e)) & 15u) - 8) * d;
                }
            };
            auto ldv = [&](int j, int ln, float (&vf)[DV]) {
                const float d = __half2float(vsc[j * (D / 32) + (ln * DV) / 32]);
                if (QT == AF_KV_Q8_0) {
                    if (DV == 4) {
                        const unsigned w = *reinterpret_cast<const unsigned*>(vq8 + j * C::CB + ln * 4);
#pragma unroll
                        for (int e = 0; e < DV; e++) vf[e] = (float)(int)(signed char)(w >> (8 * e)) * d;
                    } else {
                        const unsigned short w = *reinterpret_cast<const unsigned short*>(vq8 + j * C::CB + ln * 2);
#pragma unroll
                        for (int e = 0; e < DV; e++) vf[e] = (float)(int)(signed char)(w >> (8 * e)) * d;
                    }
                } else {
                    unsigned w;
                    if (DV == 4) w = *reinterpret_cast<const unsigned short*>(vq8 + j * C::CB + ln * 2);
                    else w = vq8[j * C::CB + ln];
#pragma unroll
                    for (int e = 0; e < DV; e++) vf[e] = (float)((int)((w >> (4 * e)) & 15u) - 8) * d;
                }
            };
            ok = warp_stage<D, G, SPWQ>(qv, keys, warp, lane, ldk, ldv, wait_v, m_run, l_run, acc,
                                        reinterpret_cast<float(*)[G]>(&pw[warp][0][0]), cw[warp]);
        } else {
            const __half* kt = reinterpret_cast<const __half*>(base);
            const __half* vt = reinterpret_cast<const __half*>(base + TS * D * 2);
            auto ldk = [&](int j, int l8, float (&kf)[8]) { load_vec<__half>(kt + j * D + l8 * 8, kf, 8); };
            auto ldv = [&](int j, int ln, float (&vf)[DV]) { load_small<DV>(vt + j * D + ln * DV, vf); };
            ok = warp_stage<D, G, SPWF>(qv, keys, warp, lane, ldk, ldv, wait_v, m_run, l_run, acc,
                                        reinterpret_cast<float(*)[G]>(&pw[warp][0][0]), cw[warp]);
        }
        if (!ok) break;
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&done[slot], 1u) == (unsigned)NW - 1u) {
                done[slot] = 0;
                if (t + S < nst) {
                    fence_proxy_async_shared();
                    issue(t + S);
                }
            }
        }
    }
    __syncthreads();
    if (abort_f) {
        if (tid == 0)
            for (int i = 0; i < S; i++)
                if (issues[i]) {
                    mbar_wait_bounded(&kfull[i], (issues[i] - 1u) & 1u);
                    mbar_wait_bounded(&vfull[i], (issues[i] - 1u) & 1u);
                }
        __syncthreads();
    }
    float* red_o = reinterpret_cast<float*>(dsm);  // [warp][G][D]
#pragma unroll
    for (int h = 0; h < G; h++)
#pragma unroll
        for (int e = 0; e < DV; e++) red_o[(warp * G + h) * D + lane * DV + e] = acc[h][e];
    if (lane < LPK && li % LPH == 0) {
        wm[warp][hl] = m_run;
        wl[warp][hl] = l_run;
    }
    __syncthreads();
    if (nl > 0)
        for (int t = tid; t < G * D; t += NT) {
            const int h = t / D, d = t % D;
            float M = -CUDART_INF_F;
#pragma unroll
            for (int w = 0; w < NW; w++) M = fmaxf(M, wm[w][h]);
            float o = 0.f, l = 0.f;
#pragma unroll
            for (int w = 0; w < NW; w++) {
                const float e = wm[w][h] == -CUDART_INF_F ? 0.f : __expf(wm[w][h] - M);
                o = fmaf(e, red_o[(w * G + h) * D + d], o);
                l = fmaf(e, wl[w][h], l);
            }
            my[h * PST + d] = o;
            if (d == 0) {
                my[h * PST + D] = abort_f ? 0.f : M;
                my[h * PST + D + 1] = abort_f ? CUDART_NAN_F : l;
            }
        }
    __threadfence();
    __syncthreads();
    if (tid == 0) last = (atomicAdd(&cnt[g], 1u) == (unsigned)ns - 1u);
    __syncthreads();
    if (!last) return;
    __threadfence();
    merge_splits<D, G, NT>(part, g, ns, ns_eff, out, cnt, dsm,
                           reinterpret_cast<float*>(dsm + merge_scratch_off(NW * G * D * 4, NT)), tid);
}

template <int D, int G, int QT>
cudaError_t launch_kvq_t(const float* q, const void* kc, const void* vc, const KvLayerStore& qs, int max_ctx,
                         const int* pos_dev, int pos, const AttnScratch& scr, int ns, float* out, int KVH,
                         cudaStream_t s) {
    using C = KvqCfg<D, QT>;
    const size_t smem = (size_t)C::S * C::SLOT;
    if ((size_t)merge_scratch_off(kDecWarps * G * D * 4, kDecThreads) + (size_t)ns * G * 8 > smem)
        return cudaErrorInvalidValue;
    auto k = attn_decode_kvq_kernel<D, G, QT>;
    static int opened[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!opened[dev]) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e) return e;
            opened[dev] = 1;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ns, KVH);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, q, (const __half*)kc, (const __half*)vc, qs, max_ctx, pos_dev, pos, scr.part,
                              scr.cnt, out, scr.err);
}

template <int D, int G>
cudaError_t dispatch_kvq(const float* q, const void* kc, const void* vc, const KvLayerStore& qs, int max_ctx,
                         const int* pos_dev, int pos, const AttnScratch& scr, int ns, float* out, int KVH,
                         cudaStream_t s) {
    if (qs.qtype == AF_KV_Q8_0)
        return launch_kvq_t<D, G, AF_KV_Q8_0>(q, kc, vc, qs, max_ctx, pos_dev, pos, scr, ns, out, KVH, s);
    return launch_kvq_t<D, G, AF_KV_Q4_0>(q, kc, vc, qs, max_ctx, pos_dev, pos, scr, ns, out, KVH, s);
}

template <int D, int G, typename KT, bool CL>
cudaError_t launch_decode_t(const float* q, const void* kc, const void* vc, int max_ctx, const int* pos_dev, int pos,
                            const AttnScratch& scr, int ns, float* out, int KVH, cudaStream_t s) {
    if (CL) ns = kC;
    const int nw = CL ? kClWarps : kDecWarps;
    // the ring; after the loop it holds the warps' outputs [nw][G][D], then the merge's [ns][G] maxima and sums
    const size_t smem = (size_t)dec_stages<D, KT, CL>() * 2 * dec_tile<D, KT>() * D * sizeof(KT);
    if ((size_t)merge_scratch_off(nw * G * D * 4, nw * 32) + (size_t)ns * G * 8 > smem) return cudaErrorInvalidValue;
    if (smem > 222 * 1024) return cudaErrorInvalidValue;  // with the static shared memory, within 227 KB
    auto k = attn_decode_kernel<D, G, KT, CL>;
    // the largest dynamic shared memory this instantiation was opened to, per device (set before a launch
    // that needs more; launches inside a stream capture reuse what was set before it)
    static int opened[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (opened[dev] < (int)smem) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (!e && CL) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e) return e;
            opened[dev] = (int)smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ns, KVH);
    cfg.blockDim = dim3(nw * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kC;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CL ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k, q, (const KT*)kc, (const KT*)vc, max_ctx, pos_dev, pos, scr.part, scr.cnt,
                              out, scr.err);
}

template <int D, int G>
cudaError_t dispatch_decode(const float* q, const void* kc, const void* vc, int kv_f16, int max_ctx,
                            const int* pos_dev, int pos, const AttnScratch& scr, int ns, float* out, int KVH,
                            bool cl, cudaStream_t s) {
    if (cl)
        return kv_f16 ? launch_decode_t<D, G, __half, true>(q, kc, vc, max_ctx, pos_dev, pos, scr, ns, out, KVH, s)
                      : launch_decode_t<D, G, float, true>(q, kc, vc, max_ctx, pos_dev, pos, scr, ns, out, KVH, s);
    return kv_f16 ? launch_decode_t<D, G, __half, false>(q, kc, vc, max_ctx, pos_dev, pos, scr, ns, out, KVH, s)
                  : launch_decode_t<D, G, float, false>(q, kc, vc, max_ctx, pos_dev, pos, scr, ns, out, KVH, s);
}

}  // namespace

// Whether this device can schedule the cluster path's clusters (kC CTAs of one SM's worth of shared memory);
// asked once per device.
bool cluster_path_available() {
    static int state[kMaxDevices] = {};  // 0 unknown, 1 yes, 2 no
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!state[dev]) {
        auto k = attn_decode_kernel<128, 4, __half, true>;
        const int smem = dec_stages<128, __half, true>() * 2 * 16384;
        int n = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kC, 8);
        cfg.blockDim = dim3(kClWarps * 32);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kC;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (!e) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (!e) e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
        if (e) cudaGetLastError();
        state[dev] = (!e && n > 0) ? 1 : 2;
    }
    return state[dev] == 1;
}

bool attn_decode_uses_cluster(int max_ctx) { return max_ctx <= kC * kClMaxSplit && cluster_path_available(); }

bool attn_supported(int H, int KVH, int D) {
    if (KVH <= 0 || H % KVH) return false;
    const int G = H / KVH;
    return (D == 64 || D == 128) && (G == 1 || G == 2 || G == 4 || G == 8);
}

int attn_decode_splits(int n_heads, int n_kv_heads, int max_ctx) {
    // two CTAs per SM over all kv heads (one wave)
    (void)n_heads;
    (void)max_ctx;
    const int ns = 2 * num_sms() / n_kv_heads;
    return ns < 1 ? 1 : ns;
}

size_t attn_decode_part_elems(int n_heads, int head_dim, int ns) { return (size_t)ns * n_heads * (head_dim + 4); }

#define AF_ATTN_DISPATCH(FN, ...)                                          \
    switch (D * 100 + G) {                                                 \
        case 6401: return FN<64, 1>(__VA_ARGS__);                          \
        case 6402: return FN<64, 2>(__VA_ARGS__);                          \
        case 6404: return FN<64, 4>(__VA_ARGS__);                          \
        case 6408: return FN<64, 8>(__VA_ARGS__);                          \
        case 12801: return FN<128, 1>(__VA_ARGS__);                        \
        case 12802: return FN<128, 2>(__VA_ARGS__);                        \
        case 12804: return FN<128, 4>(__VA_ARGS__);                        \
        case 12808: return FN<128, 8>(__VA_ARGS__);                        \
        default: return cudaErrorInvalidValue;                             \
    }

cudaError_t launch_attn_decode(const float* q, const void* kc, const void* vc, int kv_f16, int H, int KVH, int D,
                               int max_ctx, const int* pos_dev, int pos, const AttnScratch& scr, float* out,
                               cudaStream_t s, const KvLayerStore* qs) {
    const int G = H / KVH;
    if (qs && qs->qtype) {  // quantized cache: split path over the store and the fp16 window
        const int ns = attn_decode_splits(H, KVH, max_ctx);
        if (scr.ns < ns || max_ctx % 4) return cudaErrorInvalidValue;
        if ((reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc) | reinterpret_cast<uintptr_t>(qs->kq) |
             reinterpret_cast<uintptr_t>(qs->vq) | reinterpret_cast<uintptr_t>(qs->ks) |
             reinterpret_cast<uintptr_t>(qs->vs)) & 15)
            return cudaErrorInvalidValue;
        AF_ATTN_DISPATCH(dispatch_kvq, q, kc, vc, *qs, max_ctx, pos_dev, pos, scr, ns, out, KVH, s)
    }
    // the path depends on the cache size only (a captured decode step replays at every position)
    const bool cl = attn_decode_uses_cluster(max_ctx);
    const int ns = attn_decode_splits(H, KVH, max_ctx);
    if (!cl && scr.ns < ns) return cudaErrorInvalidValue;  // scratch sized for fewer splits
    if ((reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc)) & 15) return cudaErrorInvalidValue;
    if (!cl && kv_f16 && G <= 4) {  // fp16 cache on the split path: the tensor-core kernel
        switch (D * 100 + G) {
            case 6401: return launch_tc_t<64, 1>(q, kc, vc, max_ctx, pos_dev, pos, scr, ns, out, KVH, s);
            case 6402: return launch_tc_t<64, 2>(q, kc, vc, max_ctx, pos_dev, pos, scr, ns, out, KVH, s);
            case 6404: return launch_tc_t<64, 4>(q, kc, vc, max_ctx, pos_dev, pos, scr, ns, out, KVH, s);
            case 12801: return launch_tc_t<128, 1>(q, kc, vc, max_ctx, pos_dev, pos, scr, ns, out, KVH, s);
            case 12802: return launch_tc_t<128, 2>(q, kc, vc, max_ctx, pos_dev, pos, scr, ns, out, KVH, s);
            case 12804: return launch_tc_t<128, 4>(q, kc, vc, max_ctx, pos_dev, pos, scr, ns, out, KVH, s);
            default: break;
        }
    }
    AF_ATTN_DISPATCH(dispatch_decode, q, kc, vc, kv_f16, max_ctx, pos_dev, pos, scr, ns, out, KVH, cl, s)
}

}  // namespace af
