// On-device sampler chain after the logits (Airframe GPU pipeline, "sampling
// applies these transformations in order"): repetition penalty -> temperature
// -> softmax -> top-p -> sample.
//
// Readings (the same as the CPU reference):
//   - the penalty divides each distinct recent token's logit once;
//   - temperature 0 is greedy: argmax, lowest index on ties;
//   - the order is probability descending, then index ascending; the nucleus
//     is the shortest prefix whose mass reaches top_p, extended by every token
//     tied with its last one (top_p >= 1 keeps everything);
//   - the token drawn is the first of that order whose cumulative mass reaches
//     u times the nucleus mass (u: the caller's uniform draw in [0, 1)).
//
// No sort: the nucleus boundary and the drawn token are both "the key where
// the descending cumulative mass crosses a threshold", found by a radix select
// over the bits of the fp32 masses exp(z - max z) (non-negative floats order
// like their bits), one byte (256-bin mass histogram) per pass, most
// significant first.  The order is thus the fp32 mass descending, then index:
// logits whose fp32 masses round equal count as tied.
//
// One launch of one thread-block cluster of kCl CTAs.  CTA r holds the scaled
// logits of its contiguous vocabulary slice in shared memory for the whole
// call.  Each CTA pushes its partials (maximum and sum, pass histograms, tie
// masses) into every CTA's shared memory with distributed-shared-memory stores
// before a hardware cluster barrier; every CTA then sums them in the same order,
// so all of them take identical selections.  The draw's first pass reuses the
// nucleus boundary's first histogram, and so on while the two prefixes agree.
// There is no global scratch: calls on different streams are independent.
#include <math_constants.h>

#include <mutex>

#include "common.cuh"

namespace af {

namespace {

constexpr int kCl = 8;                          // CTAs in the cluster
constexpr int kT = 1024;                        // threads per CTA
constexpr int kW = kT / 32;
constexpr int kMaxVocab = 262144;
constexpr int kMaxChunk = kMaxVocab / kCl;      // 32768 logits per CTA
constexpr int kMaxRounds = kMaxChunk / kT;      // 32 strided rounds per slice
constexpr int kPasses = 8;                      // 4 bytes for the nucleus boundary, 4 for the draw
static_assert(kCl == 8 && kT == 1024, "the histogram fold pushes each bin from four threads to two CTAs each");

// fixed part of the dynamic shared memory, after the slice
struct SampShared {
    uint32_t lh[256 * 32];        // lane-private fixed-point histogram of the current pass: bin * 32 + lane (zero between passes)
    float gx[2][kCl][256];        // pushed by every CTA: its histogram, by exchange parity
    float ghs[kPasses][256];      // the cluster's histogram of each pass (the same in every CTA)
    float rw[kMaxRounds][kW];     // tie mass per strided round and warp
    float rt[kMaxRounds];         // tie mass per strided round
    float red[kW];
    unsigned long long redk[kW];
    float xs[kCl][4];             // pushed by every CTA: [0] slice maximum, [1] slice sum of exp(z - max), [2] tie mass
    unsigned long long xk[kCl];   // pushed by every CTA: greedy argmax key
    uint32_t prefix, pmask, kap;
    int reuse[2];
    float rem;
    int sel, found, last;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// all threads of all CTAs of the cluster; release/acquire orders the shared-memory writes before it
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

// stores into the same variable of CTA `rank` of the cluster (visible there after the next cluster_sync)
__device__ __forceinline__ void st_dsmem(float* local, uint32_t rank, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dsmem_addr(local, rank)), "f"(v) : "memory");
}

__device__ __forceinline__ void st_dsmem(unsigned long long* local, uint32_t rank, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(dsmem_addr(local, rank)), "l"(v) : "memory");
}

// Order-preserving key of a float: larger float -> larger unsigned key.
__device__ __forceinline__ uint32_t fkey(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float mass_of(float z, float M) { return z > -CUDART_INF_F ? __expf(z - M) : 0.f; }

// Fixed-point image of a mass (its bits k; masses are >= 0, so their bits order like the masses): all masses
// with the same top key byte t lie in [2^(2t-127), 2^(2t-125)), where (implicit one and mantissa) shifted by
// the low exponent bit and then right by 3 is mass * 2^(147 - 2t), an integer below 2^22 that is exact up to
// a relative 2^-20.  Masses below 2^-126 count as zero.  Integer shared-memory atomics then add them.
__device__ __forceinline__ uint32_t fixq(uint32_t k) {
    const uint32_t e = k >> 23;
    return e ? (((k & 0x7FFFFFu) | 0x800000u) << (e & 1u)) >> 3 : 0u;
}

struct Params {
    const float* logits;
    int V;
    const int* recent;
    int n_recent;
    float penalty, temperature, top_p, u;
    int* token_out;
};

// Byte selection of one pass from the cluster histogram (one warp): the bin where the descending mass,
// starting at `carried`, reaches `target`; updates carried (mass of keys above the selected bin) and
// returns the byte.  Lane l owns bins 255 - 8l down to 248 - 8l; the crossing lane is found from a scan of
// the lane sums and then scans its own eight bins.  If rounding leaves the target above the total, the
// lowest bin with mass is taken.
__device__ __forceinline__ int select_bin(const float* hist, float target, float& carried, float& bin_mass) {
    const int lane = threadIdx.x & 31;
    float m8[8], tot = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        m8[j] = hist[255 - 8 * lane - j];
        tot += m8[j];
    }
    float inc = tot;  // inclusive scan over lanes (descending bins)
    for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += x;
    }
    const float pre = carried + inc - tot;
    const unsigned cross = __ballot_sync(0xffffffffu, tot > 0.f && pre + tot >= target);
    const unsigned any = __ballot_sync(0xffffffffu, tot > 0.f);
    if (!any) {
        bin_mass = 0.f;
        return 0;
    }
    const int src = cross ? __ffs(cross) - 1 : 31 - __clz(any);
    int b = 0;
    float c_out = 0.f, m_out = 0.f;
    if (lane == src) {
        float c = pre, c_last = pre, m_last = 0.f;
        int last = 0;
        bool done = false;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const float m = m8[j];
            if (!done && m > 0.f) {
                if (cross && c + m >= target) {
                    b = 255 - 8 * lane - j;
                    c_out = c;
                    m_out = m;
                    done = true;
                } else {
                    last = 255 - 8 * lane - j;
                    c_last = c;
                    m_last = m;
                    c += m;
                }
            }
        }
        if (!done) {  // no single bin crossed (the lane total did, or nothing did): its lowest bin with mass
            b = last;
            c_out = c_last;
            m_out = m_last;
        }
    }
    b = __shfl_sync(0xffffffffu, b, src);
    carried = __shfl_sync(0xffffffffu, c_out, src);
    bin_mass = __shfl_sync(0xffffffffu, m_out, src);
    return b;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < kW; w++) t += red[w];
    __syncthreads();
    return t;
}

__device__ __forceinline__ float block_max(float v, float* red) {
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = red[0];
    for (int w = 1; w < kW; w++) t = fmaxf(t, red[w]);
    __syncthreads();
    return t;
}

__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kT, 1) samp_cluster_kernel(Params p) {
    extern __shared__ __align__(16) unsigned char dsm[];
    const int chunk = (p.V + kCl - 1) / kCl;
    const int chunk_pad = (chunk + 31) & ~31;
    float* z = reinterpret_cast<float*>(dsm);
    SampShared& sh = *reinterpret_cast<SampShared*>(dsm + (size_t)chunk_pad * 4);
    const uint32_t rank = cluster_rank();
    const int lo = (int)rank * chunk;
    const int n = max(0, min(chunk, p.V - lo));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool greedy = !(p.temperature > 0.f);

    for (int i = tid; i < 256 * 32; i += kT) sh.lh[i] = 0.f;  // once: every fold zeroes what it reads
    // the slice, penalized (each marked token rewritten from its own logit, so duplicates agree) and scaled
#pragma unroll 4
    for (int j = tid; j < n; j += kT) z[j] = p.logits[lo + j];
    __syncthreads();
    if (p.penalty > 1.f)
        for (int r = tid; r < p.n_recent; r += kT) {
            const int t = p.recent[r];
            if (t >= lo && t < lo + n) z[t - lo] = p.logits[t] / p.penalty;
        }
    __syncthreads();
    if (!greedy)
        for (int j = tid; j < n; j += kT) z[j] = z[j] / p.temperature;
    __syncthreads();

    if (greedy) {  // argmax, lowest index on ties
        unsigned long long best = 0ull;
        for (int j = tid; j < n; j += kT) {
            const unsigned long long k = ((unsigned long long)fkey(z[j]) << 32) | (0xFFFFFFFFu - (unsigned)(lo + j));
            best = k > best ? k : best;
        }
        for (int o = 16; o; o >>= 1) {
            const unsigned long long x = __shfl_xor_sync(0xffffffffu, best, o);
            best = x > best ? x : best;
        }
        if (lane == 0) sh.redk[warp] = best;
        __syncthreads();
        if (tid < kCl) {
            unsigned long long b = 0ull;
            for (int w = 0; w < kW; w++) b = sh.redk[w] > b ? sh.redk[w] : b;
            st_dsmem(&sh.xk[rank], tid, b);
        }
        cluster_sync();  // after it nothing touches another CTA's shared memory
        if (rank == 0 && tid == 0) {
            unsigned long long b = 0ull;
            for (int r = 0; r < kCl; r++) b = sh.xk[r] > b ? sh.xk[r] : b;
            *p.token_out = (int)(0xFFFFFFFFu - (unsigned)(b & 0xFFFFFFFFull));
        }
        return;
    }

    // softmax statistics: slice maximum and sum, pushed to every CTA, then the cluster's (same order everywhere)
    float m = -CUDART_INF_F;
    for (int j = tid; j < n; j += kT) m = fmaxf(m, z[j]);
    const float cm = block_max(m, sh.red);
    float t = 0.f;
    for (int j = tid; j < n; j += kT) t += mass_of(z[j], cm);
    const float cs = block_sum(t, sh.red);
    if (tid < kCl) {
        st_dsmem(&sh.xs[rank][0], tid, cm);
        st_dsmem(&sh.xs[rank][1], tid, cs);
    }
    if (tid == 0) {
        sh.prefix = 0u;
        sh.pmask = 0u;
        sh.reuse[0] = 0;
        sh.reuse[1] = 0;
    }
    cluster_sync();
    float M = -CUDART_INF_F, E = 0.f;
    for (int r = 0; r < kCl; r++) M = fmaxf(M, sh.xs[r][0]);
    for (int r = 0; r < kCl; r++)
        if (sh.xs[r][0] > -CUDART_INF_F) E += sh.xs[r][1] * __expf(sh.xs[r][0] - M);
    // from here on the slice holds the masses exp(z - M) (same thread-to-token map, so no barrier); the radix
    // keys are their bits, which order like the masses
    for (int j = tid; j < n; j += kT) z[j] = mass_of(z[j], M);

    // Radix passes; the selection state lives in warp 0.  Passes 4..7 select the draw; while its prefix
    // equals the nucleus boundary's, its histogram is that of the nucleus pass four earlier (pass 4 always).
    const bool cut = p.top_p < 1.f;
    uint32_t prefix = 0u, pmask = 0u, tau = 0u;
    float target = cut ? p.top_p * E : p.u * E, above = 0.f, bin_mass = 0.f, above_tau = 0.f, eq_tau = E;
    int ex = 0;  // exchanges so far (their buffers alternate)
    for (int q = cut ? 0 : 4; q < kPasses; q++) {
        const int shift = 24 - 8 * (q & 3);
        const float* hist = sh.ghs[q & 3];
        if (!sh.reuse[q & 1]) {  // uniform over the cluster: every CTA takes the same selections
            const uint32_t pre = sh.prefix, msk = sh.pmask;
            for (int j = tid; j < n; j += kT) {
                const uint32_t k = __float_as_uint(z[j]);
                if ((k & msk) == pre) atomicAdd(&sh.lh[((k >> shift) & 255u) * 32 + lane], fixq(k));
            }
            __syncthreads();
            {  // fold: bin b by four threads of eight lane copies each (rotated: no bank conflicts), then push
                const int b = tid >> 2, c = tid & 3;
                unsigned long long a = 0ull;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    uint32_t& x = sh.lh[b * 32 + 8 * c + ((i + b) & 7)];
                    a += x;
                    x = 0u;
                }
                a += __shfl_xor_sync(0xffffffffu, a, 1);
                a += __shfl_xor_sync(0xffffffffu, a, 2);
                // back to a mass: the scale is fixed by the top byte (the bin itself in a first-byte pass)
                const int top = (q & 3) ? (int)(pre >> 24) : b;
                const float v = ldexpf(__ull2float_rn(a), 2 * top - 147);
                st_dsmem(&sh.gx[ex & 1][rank][b], 2 * c, v);
                st_dsmem(&sh.gx[ex & 1][rank][b], 2 * c + 1, v);
            }
            cluster_sync();
            if (tid < 256) {
                float a = 0.f;
                for (int r = 0; r < kCl; r++) a += sh.gx[ex & 1][r][tid];
                sh.ghs[q][tid] = a;
            }
            __syncthreads();
            hist = sh.ghs[q];
            ex++;
        }
        if (warp == 0) {
            const int b = select_bin(hist, target, above, bin_mass);
            prefix |= (uint32_t)b << shift;
            pmask |= 255u << shift;
            if (q == 3) {  // the nucleus boundary is complete: record it and start the draw's select over
                tau = prefix;
                above_tau = above;
                eq_tau = bin_mass;
                target = p.u * (above_tau + eq_tau);
                prefix = 0u;
                pmask = 0u;
                above = 0.f;
            }
            if (tid == 0) {
                sh.prefix = prefix;
                sh.pmask = pmask;
                // the flag alternates by pass: a warp still reading this pass's flag never sees the next one
                sh.reuse[(q + 1) & 1] = cut && q >= 3 && q < kPasses - 1 && ((prefix ^ tau) & pmask) == 0u;
            }
        }
        __syncthreads();
    }

    // Ties at the drawn key kap, in index order.  Every CTA sums the same per-CTA tie masses in the same
    // order, so all agree on the one CTA holding the crossing (else the last CTA with tie mass); in it, the
    // strided round holding the crossing (else the last with mass), then the token in that round (else the
    // round's last token with mass).  A token is always written.
    if (tid == 0) {
        uint32_t kap = prefix;
        float tgt = target, abv = above;
        if (cut && kap < tau) {  // rounding between the two selects: stay in the nucleus
            kap = tau;
            abv = above_tau;
            tgt = above_tau + eq_tau;
        }
        sh.kap = kap;
        sh.rem = tgt - abv;
        sh.found = 0x7FFFFFFF;
        sh.last = -1;
    }
    __syncthreads();
    const uint32_t kap = sh.kap;
    const int rounds = (n + kT - 1) / kT;
    for (int k = 0; k < rounds; k++) {  // round k: tokens lo + k * kT .. lo + (k + 1) * kT - 1
        const int j = k * kT + tid;
        float tm = (j < n && __float_as_uint(z[j]) == kap) ? z[j] : 0.f;
        for (int o = 16; o; o >>= 1) tm += __shfl_xor_sync(0xffffffffu, tm, o);
        if (lane == 0) sh.rw[k][warp] = tm;
    }
    __syncthreads();
    if (tid < kMaxRounds) {
        float a = 0.f;
        if (tid < rounds)
            for (int w = 0; w < kW; w++) a += sh.rw[tid][w];
        sh.rt[tid] = a;
    }
    __syncthreads();
    if (tid < kCl) {
        float a = 0.f;
        for (int k = 0; k < kMaxRounds; k++) a += sh.rt[k];
        st_dsmem(&sh.xs[rank][2], tid, a);
    }
    cluster_sync();  // after it nothing touches another CTA's shared memory
    if (tid == 0) {
        const float rem_total = sh.rem;
        float cum = 0.f, cum_sel = 0.f, cum_last = 0.f;
        int sel = -1, last = -1;
        for (int r = 0; r < kCl; r++) {
            const float x = sh.xs[r][2];
            if (x > 0.f) {
                if (sel < 0 && cum + x >= rem_total) {
                    sel = r;
                    cum_sel = cum;
                }
                last = r;
                cum_last = cum;
            }
            cum += x;
        }
        if (sel < 0) {
            sel = last;
            cum_sel = cum_last;
        }
        sh.sel = sel == (int)rank;
        sh.rem = rem_total - cum_sel;
    }
    __syncthreads();
    if (!sh.sel) return;  // uniform over the CTA
    const float rem = sh.rem;
    float c = 0.f, c_last = 0.f;
    int kx = -1, k_last = -1;
    for (int k = 0; k < rounds; k++) {
        const float x = sh.rt[k];
        if (x > 0.f) {
            if (c + x >= rem) {
                kx = k;
                break;
            }
            k_last = k;
            c_last = c;
        }
        c += x;
    }
    if (kx < 0) {
        kx = k_last;
        c = c_last;
    }
    const int j = kx * kT + tid;
    const float tm = (kx >= 0 && j < n && __float_as_uint(z[j]) == kap) ? z[j] : 0.f;
    float inc = tm;
    for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += x;
    }
    if (lane == 31) sh.red[warp] = inc;
    __syncthreads();
    float wb = 0.f;
    for (int w = 0; w < warp; w++) wb += sh.red[w];
    if (tm > 0.f) {
        if (c + wb + inc >= rem) atomicMin(&sh.found, lo + j);
        atomicMax(&sh.last, lo + j);
    }
    __syncthreads();
    if (tid == 0) *p.token_out = sh.found != 0x7FFFFFFF ? sh.found : sh.last;
}

std::mutex g_mu;
bool g_attr[64] = {};

size_t smem_bytes(int V) {
    const int chunk = (V + kCl - 1) / kCl;
    return (size_t)((chunk + 31) & ~31) * 4 + sizeof(SampShared);
}

cudaError_t ensure_attr() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_attr[dev]) {
        e = cudaFuncSetAttribute(samp_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes(kMaxVocab));
        if (e) return e;
        g_attr[dev] = true;
    }
    return cudaSuccess;
}

}  // namespace

int sampler_max_vocab() { return kMaxVocab; }

cudaError_t launch_sample(const float* logits, int V, const int* recent, int n_recent, float penalty,
                          float temperature, float top_p, float u, int* token_out, cudaStream_t s) {
    if (V < 1 || V > kMaxVocab) return cudaErrorInvalidValue;
    cudaError_t e = ensure_attr();
    if (e) return e;
    Params p{logits, V, recent, n_recent, penalty, temperature, top_p, u, token_out};
    samp_cluster_kernel<<<kCl, kT, smem_bytes(V), s>>>(p);
    return cudaGetLastError();
}

}  // namespace af
