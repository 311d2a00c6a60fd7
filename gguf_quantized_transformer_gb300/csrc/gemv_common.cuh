// Building blocks of the quantized matrix-vector products (decode GEMV and the
// persistent decode kernel): 24-bit fixed-point activations, dp4a dot
// products over Q4_0 / Q8_0 sixteen-byte units, the warp transpose-reduce and
// the fused epilogue with its inputs preloaded into shared memory.
#pragma once
#include "common.cuh"

namespace af {

__device__ __forceinline__ int dp4a_uu(unsigned a, unsigned b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(unsigned a, unsigned b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_ss(unsigned a, unsigned b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(unsigned a, unsigned b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// One lane's x values for one 16-byte weight unit, in 24-bit fixed point:
// p[k][g] packs byte plane k (0 = low, 2 = signed top) of elements 4g..4g+3
// of the unit (Q4_0: groups 0..3 are elements 0..15, groups 4..7 are 16..31).
template <int G>
struct XUnit {
    unsigned p[3][G];
    float s;    // fixed-point scale
    float sx8;  // -8 * sum of the unit's x values (Q4_0 offset term)
};

template <int UW>
__device__ __forceinline__ void quantize_unit(const float (&xs)[UW], XUnit<UW / 4>& xu) {
    float m = 0.f, sum = 0.f;
#pragma unroll
    for (int e = 0; e < UW; e++) {
        m = fmaxf(m, fabsf(xs[e]));
        sum += xs[e];
    }
    // power-of-two scale: m = f 2^E with f in [0.5, 1) gives |x| / s < 2^23 and s * xi exact
    int E = 0;
    frexpf(m, &E);
    const float inv = m > 0.f ? ldexpf(1.f, 23 - E) : 0.f;
    xu.s = m > 0.f ? ldexpf(1.f, E - 23) : 0.f;
    xu.sx8 = -8.f * sum;
#pragma unroll
    for (int g = 0; g < UW / 4; g++) {
        unsigned w0 = 0, w1 = 0, w2 = 0;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            int q = __float2int_rn(xs[4 * g + i] * inv);
            q = max(-8388607, min(8388607, q));
            const unsigned u = (unsigned)q;
            w0 |= (u & 0xFFu) << (8 * i);
            w1 |= ((u >> 8) & 0xFFu) << (8 * i);
            w2 |= ((u >> 16) & 0xFFu) << (8 * i);
        }
        xu.p[0][g] = w0;
        xu.p[1][g] = w1;
        xu.p[2][g] = w2;
    }
}

template <int WT>
struct Q;
template <>
struct Q<AF_Q4_0> {
    static constexpr int UW = 32;  // weights per 16-byte unit
    // sum_j (n_j - 8) x_j over the block; byte j of the unit holds n_j (low) and n_{j+16} (high)
    static __device__ __forceinline__ float dot(uint4 q, const XUnit<8>& x) {
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
        int A = 0, B = 0, C = 0;
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const unsigned lo = w[t] & 0x0F0F0F0Fu, hi = (w[t] >> 4) & 0x0F0F0F0Fu;
            A = dp4a_us(lo, x.p[2][t], A);
            A = dp4a_us(hi, x.p[2][4 + t], A);
            B = dp4a_uu(lo, x.p[1][t], B);
            B = dp4a_uu(hi, x.p[1][4 + t], B);
            C = dp4a_uu(lo, x.p[0][t], C);
            C = dp4a_uu(hi, x.p[0][4 + t], C);
        }
        // |256 A + B| < 2^24: both conversions are exact
        const float v = fmaf(256.f, (float)(A * 256 + B), (float)C);
        return fmaf(x.s, v, x.sx8);
    }
};
template <>
struct Q<AF_Q8_0> {
    static constexpr int UW = 16;
    // sum_j q_j x_j over the half block
    static __device__ __forceinline__ float dot(uint4 q, const XUnit<4>& x) {
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
        int A = 0, B = 0, C = 0;
#pragma unroll
        for (int t = 0; t < 4; t++) {
            A = dp4a_ss(w[t], x.p[2][t], A);
            B = dp4a_su(w[t], x.p[1][t], B);
            C = dp4a_su(w[t], x.p[0][t], C);
        }
        const float v = fmaf(65536.f, (float)A, fmaf(256.f, (float)B, (float)C));
        return x.s * v;
    }
};

// Reduce v[0..RW-1] over the 32 lanes; afterwards lanes (32/RW)*t .. hold the sum of v[t].
template <int RW>
__device__ __forceinline__ float transpose_reduce(float (&v)[RW], int lane) {
#pragma unroll
    for (int half = RW / 2, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
        const bool up = lane & bit;
#pragma unroll
        for (int k = 0; k < half; k++) {
            const float send = up ? v[k] : v[k + half], keep = up ? v[k + half] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    float r = v[0];
#pragma unroll
    for (int bit = 16 / RW; bit >= 1; bit >>= 1) r += __shfl_xor_sync(0xffffffffu, r, bit);
    return r;
}

// Epilogue of the decode GEMV.  Everything it reads from global memory (the
// residual rows of this CTA, the RoPE row of the position) was preloaded into
// shared memory, so per-stage epilogues only store; the LM-head argmax is kept
// per CTA in shared memory and published with one atomic at the end.
struct GemvEpiCtx {
    const float* xres;       // shared: x[r0 + i] for EPI_RESID
    const float2* rope;      // shared: (cos, sin) of theta(pos, i) for EPI_QKV
    int pos;
    unsigned long long* amax;  // shared: CTA argmax key for EPI_LOGITS
    int r0;
};

__device__ __forceinline__ void gemv_epi(const Epi& e, const GemvEpiCtx& c, int n, float v0, float v1) {
    switch (e.kind) {
        case EPI_STORE:
            e.out[n] = v0;
            e.out[n + 1] = v1;
            break;
        case EPI_RESID:
            e.out[n] = c.xres[n - c.r0] + v0;
            e.out[n + 1] = c.xres[n - c.r0 + 1] + v1;
            break;
        case EPI_SWIGLU:
            e.out[n >> 1] = silu_f(v0) * v1;
            break;
        case EPI_LOGITS: {
            e.out[n] = v0;
            e.out[n + 1] = v1;
            const unsigned long long k0 = argmax_key(v0, n), k1 = argmax_key(v1, n + 1);
            atomicMax(c.amax, k0 > k1 ? k0 : k1);
        } break;
        case EPI_QKV: {
            const int D = e.head_dim;
            if (n < e.qd + e.kvd) {
                const int d = (n < e.qd ? n : n - e.qd) % D;
                const float2 cs = c.rope[d >> 1];
                const float r0 = v0 * cs.x - v1 * cs.y, r1 = v0 * cs.y + v1 * cs.x;
                v0 = r0;
                v1 = r1;
            }
            if (n < e.qd) {
                e.out[n] = v0;
                e.out[n + 1] = v1;
            } else {
                const bool isk = n < e.qd + e.kvd;
                const int cc = isk ? n - e.qd : n - e.qd - e.kvd;
                const int64_t idx = ((int64_t)(cc / D) * e.max_ctx + c.pos) * D + cc % D;
                void* base = isk ? e.kcache : e.vcache;
                if (e.kv_f16)
                    *reinterpret_cast<__half2*>((__half*)base + idx) = __floats2half2_rn(v0, v1);
                else
                    *reinterpret_cast<float2*>((float*)base + idx) = make_float2(v0, v1);
            }
        } break;
    }
}


}  // namespace af
