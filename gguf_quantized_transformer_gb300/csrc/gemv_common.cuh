// Building blocks of the quantized matrix-vector products (decode GEMV and the
// persistent decode kernel): 16-bit fixed-point images of the activations,
// dp4a dot products over the sixteen-byte weight units of every block type,
// the warp transpose-reduce and the fused epilogue with its inputs preloaded
// into shared memory.
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

constexpr int kXBlkBytes = 80;  // shared image of one 32-element x block

// Shared-memory image of 32 x values in 16-bit fixed point: hi[g] / lo[g] hold
// the high (signed) / low bytes of elements 4g..4g+3.
struct __align__(16) XBlk {
    unsigned hi[8];
    unsigned lo[8];
    float s;    // scale: x ~= s * xi
    float sx8;  // -8 * s * sum_j xi_j (the Q4_0 code offset)
    float sxa;  // s * sum of xi_j over elements 0..15 (K-quant mins and offsets), exact
    float sxb;  // the same over elements 16..31
};
static_assert(sizeof(XBlk) == kXBlkBytes, "x block image size");

template <int WT>
struct Unit;
// One lane's x for one 16-byte Q4_0 unit (= one block of 32 weights).
template <>
struct Unit<AF_Q4_0> {
    unsigned hi[8], lo[8];
    float s16, sx8;
    __device__ __forceinline__ void load(const XBlk* xb, int unit) {
        const XBlk& b = xb[unit];
        const uint4 h0 = *reinterpret_cast<const uint4*>(&b.hi[0]), h1 = *reinterpret_cast<const uint4*>(&b.hi[4]);
        const uint4 l0 = *reinterpret_cast<const uint4*>(&b.lo[0]), l1 = *reinterpret_cast<const uint4*>(&b.lo[4]);
        hi[0] = h0.x; hi[1] = h0.y; hi[2] = h0.z; hi[3] = h0.w; hi[4] = h1.x; hi[5] = h1.y; hi[6] = h1.z; hi[7] = h1.w;
        lo[0] = l0.x; lo[1] = l0.y; lo[2] = l0.z; lo[3] = l0.w; lo[4] = l1.x; lo[5] = l1.y; lo[6] = l1.z; lo[7] = l1.w;
        const float2 sv = *reinterpret_cast<const float2*>(&b.s);
        s16 = sv.x * (1.f / 16.f);
        sx8 = sv.y;
    }
    // sum_j (n_j - 8) x_j over the block; byte j of the unit holds n_j (low nibble) and n_{j+16} (high)
    __device__ __forceinline__ float dot(const uint4 q) const {
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
        int A = 0, B = 0, C = 0, D = 0;
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const unsigned l = w[t] & 0x0F0F0F0Fu, h = w[t] & 0xF0F0F0F0u;
            A = dp4a_us(l, hi[t], A);
            B = dp4a_uu(l, lo[t], B);
            C = dp4a_us(h, hi[4 + t], C);
            D = dp4a_uu(h, lo[4 + t], D);
        }
        // |16 A + C| < 2^20 and |16 B + D| < 2^21: the int32 sum is exact
        const int v = ((A * 16 + C) << 8) + (B * 16 + D);
        return fmaf(s16, (float)v, sx8);
    }
    // acc + d * (this unit's dot product with row `row` of a stage)
    __device__ __forceinline__ float accumulate(const uint8_t* row, int sc_off, int unit, float acc) const {
        const uint4 q = *reinterpret_cast<const uint4*>(row + unit * 16);
        const float d = __half2float(*reinterpret_cast<const __half*>(row + sc_off + unit * 2));
        return fmaf(d, dot(q), acc);
    }
};
// One lane's x for one 16-byte Q8_0 unit (= half a block: 16 weights).
template <>
struct Unit<AF_Q8_0> {
    unsigned hi[4], lo[4];
    float s;
    __device__ __forceinline__ void load(const XBlk* xb, int unit) {
        const XBlk& b = xb[unit >> 1];
        const int g = (unit & 1) * 4;
        const uint4 h = *reinterpret_cast<const uint4*>(&b.hi[g]);
        const uint4 l = *reinterpret_cast<const uint4*>(&b.lo[g]);
        hi[0] = h.x; hi[1] = h.y; hi[2] = h.z; hi[3] = h.w;
        lo[0] = l.x; lo[1] = l.y; lo[2] = l.z; lo[3] = l.w;
        s = b.s;
    }
    // sum_j q_j x_j over the half block
    __device__ __forceinline__ float dot(const uint4 q) const {
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
        int A = 0, B = 0;
#pragma unroll
        for (int t = 0; t < 4; t++) {
            A = dp4a_ss(w[t], hi[t], A);
            B = dp4a_su(w[t], lo[t], B);
        }
        return s * (float)(A * 256 + B);  // |256 A + B| < 2^25: exact in int32
    }
    __device__ __forceinline__ float accumulate(const uint8_t* row, int sc_off, int unit, float acc) const {
        const uint4 q = *reinterpret_cast<const uint4*>(row + unit * 16);
        const float d = __half2float(*reinterpret_cast<const __half*>(row + sc_off + (unit >> 1) * 2));
        return fmaf(d, dot(q), acc);
    }
};

// x planes of one 32-element unit, shared by the K-quant units
struct XPlanes {
    unsigned hi[8], lo[8];
    __device__ __forceinline__ void load(const XBlk& b) {
        const uint4 h0 = *reinterpret_cast<const uint4*>(&b.hi[0]), h1 = *reinterpret_cast<const uint4*>(&b.hi[4]);
        const uint4 l0 = *reinterpret_cast<const uint4*>(&b.lo[0]), l1 = *reinterpret_cast<const uint4*>(&b.lo[4]);
        hi[0] = h0.x; hi[1] = h0.y; hi[2] = h0.z; hi[3] = h0.w; hi[4] = h1.x; hi[5] = h1.y; hi[6] = h1.z; hi[7] = h1.w;
        lo[0] = l0.x; lo[1] = l0.y; lo[2] = l0.z; lo[3] = l0.w; lo[4] = l1.x; lo[5] = l1.y; lo[6] = l1.z; lo[7] = l1.w;
    }
};

// One lane's x for one Q4_K unit (32 weights = one sub-block j of a super-block).  Row value of the unit:
//   d s_j sum_e n_e x_e - dmin m_j sum_e x_e
// with (d, dmin) and the unpacked (s_j, m_j) from the row's super-block record.
template <>
struct Unit<AF_Q4_K> {
    XPlanes x;
    float s16, sx;  // s / 16; s * sum of the 32 xi
    __device__ __forceinline__ void load(const XBlk* xb, int unit) {
        const XBlk& b = xb[unit];
        x.load(b);
        s16 = b.s * (1.f / 16.f);
        sx = b.sxa + b.sxb;
    }
    __device__ __forceinline__ float accumulate(const uint8_t* row, int sc_off, int unit, float acc) const {
        const uint4 q = *reinterpret_cast<const uint4*>(row + unit * 16);
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
        int A = 0, B = 0, C = 0, D = 0;
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const unsigned l = w[t] & 0x0F0F0F0Fu, h = w[t] & 0xF0F0F0F0u;
            A = dp4a_us(l, x.hi[t], A);
            B = dp4a_uu(l, x.lo[t], B);
            C = dp4a_us(h, x.hi[4 + t], C);
            D = dp4a_uu(h, x.lo[4 + t], D);
        }
        const int v = ((A * 16 + C) << 8) + (B * 16 + D);  // 16 sum_e n_e xi_e, exact
        const uint8_t* rec = row + sc_off + (unit >> 3) * kQ4KRec;
        const float2 dm = __half22float2(*reinterpret_cast<const __half2*>(rec));      // (d, dmin)
        const unsigned smj = *reinterpret_cast<const unsigned short*>(rec + 4 + (unit & 7) * 2);
        const float ds = dm.x * (float)(smj & 255u), dmm = dm.y * (float)(smj >> 8);
        return fmaf(ds, s16 * (float)v, fmaf(-dmm, sx, acc));
    }
};

// One lane's x for one Q5_K unit (32 weights = sub-block j): 5-bit codes, nibble | high bit << 4, with the
// high bits in one word per unit (element 4t + i of half h at bit 8i + 4h + t).  Row value as Q4_K's:
//   d s_j sum_e q_e x_e - dmin m_j sum_e x_e
template <>
struct Unit<AF_Q5_K> {
    XPlanes x;
    float s, sx;  // s; s * sum of the 32 xi
    __device__ __forceinline__ void load(const XBlk* xb, int unit) {
        const XBlk& b = xb[unit];
        x.load(b);
        s = b.s;
        sx = b.sxa + b.sxb;
    }
    __device__ __forceinline__ float accumulate(const uint8_t* row, int sc_off, int hb_off, int unit,
                                                float acc) const {
        const uint4 q = *reinterpret_cast<const uint4*>(row + unit * 16);
        const unsigned hw = *reinterpret_cast<const unsigned*>(row + hb_off + unit * 4);
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
        int A = 0, B = 0, C = 0, D = 0;
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const unsigned qa = (w[t] & 0x0F0F0F0Fu) | ((hw >> t) << 4 & 0x10101010u);
            const unsigned qb = ((w[t] >> 4) & 0x0F0F0F0Fu) | ((hw >> t) & 0x10101010u);
            A = dp4a_us(qa, x.hi[t], A);
            B = dp4a_uu(qa, x.lo[t], B);
            C = dp4a_us(qb, x.hi[4 + t], C);
            D = dp4a_uu(qb, x.lo[4 + t], D);
        }
        const int v = (A + C) * 256 + (B + D);  // sum_e q_e xi_e, |.| < 2^26: exact
        const uint8_t* rec = row + sc_off + (unit >> 3) * kQ4KRec;
        const float2 dm = __half22float2(*reinterpret_cast<const __half2*>(rec));
        const unsigned smj = *reinterpret_cast<const unsigned short*>(rec + 4 + (unit & 7) * 2);
        const float ds = dm.x * (float)(smj & 255u), dmm = dm.y * (float)(smj >> 8);
        return fmaf(ds, s * (float)v, fmaf(-dmm, sx, acc));
    }
};

// One lane's x for one Q6_K unit (32 weights = sub-blocks 2g, 2g+1 of 16 weights).  Codes q in 0..63 are
// rebuilt from the low nibbles and the high-bit words (element 4t + i of a half at bits 8i + 2t); the value
// of a half with int8 scale c is d c (s sum_e q_e xi_e - 32 s sum_e xi_e).
template <>
struct Unit<AF_Q6_K> {
    XPlanes x;
    float s, sxa, sxb;
    __device__ __forceinline__ void load(const XBlk* xb, int unit) {
        const XBlk& b = xb[unit];
        x.load(b);
        s = b.s;
        sxa = b.sxa;
        sxb = b.sxb;
    }
    template <int T>
    static __device__ __forceinline__ unsigned high_bits(unsigned h) {  // bits 4-5 of each byte of group T
        return T <= 2 ? (h << (4 - 2 * T)) & 0x30303030u : (h >> (2 * T - 4)) & 0x30303030u;
    }
    __device__ __forceinline__ float accumulate(const uint8_t* row, int sc_off, int hb_off, int unit,
                                                float acc) const {
        const uint4 q = *reinterpret_cast<const uint4*>(row + unit * 16);
        const uint2 hw = *reinterpret_cast<const uint2*>(row + hb_off + unit * 8);
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
        int A = 0, B = 0, C = 0, D = 0;
#pragma unroll
        for (int t = 0; t < 4; t++) {
            unsigned ha, hb;
            switch (t) {
                case 0: ha = high_bits<0>(hw.x); hb = high_bits<0>(hw.y); break;
                case 1: ha = high_bits<1>(hw.x); hb = high_bits<1>(hw.y); break;
                case 2: ha = high_bits<2>(hw.x); hb = high_bits<2>(hw.y); break;
                default: ha = high_bits<3>(hw.x); hb = high_bits<3>(hw.y); break;
            }
            const unsigned qa = (w[t] & 0x0F0F0F0Fu) | ha, qb = ((w[t] >> 4) & 0x0F0F0F0Fu) | hb;
            A = dp4a_us(qa, x.hi[t], A);
            B = dp4a_uu(qa, x.lo[t], B);
            C = dp4a_us(qb, x.hi[4 + t], C);
            D = dp4a_uu(qb, x.lo[4 + t], D);
        }
        const int va = A * 256 + B, vb = C * 256 + D;  // sum q xi over each half, |.| < 2^26: exact in int32
        const uint8_t* rec = row + sc_off + (unit >> 3) * kQ6KRec;
        const float d = __half2float(*reinterpret_cast<const __half*>(rec));
        const unsigned sc = *reinterpret_cast<const unsigned short*>(rec + 2 + (unit & 7) * 2);
        const float da = d * (float)(int)(signed char)(sc & 255u), db = d * (float)(int)(signed char)(sc >> 8);
        return fmaf(da, fmaf(s, (float)va, -32.f * sxa), fmaf(db, fmaf(s, (float)vb, -32.f * sxb), acc));
    }
};


// Convert x (optionally RMS-normalized) to the fixed-point block images.
// Eight lanes per block, lane g of the group holds elements 4g..4g+3.
// With NORM the images hold w (.) x (the RMS factor is a scalar, applied to each row's dot product in the
// epilogue) and the return value is this thread's part of sum(x^2), from the same loads.
// NT: threads taking part; CG: read x through L2 only (x was written by other CTAs of the same launch).
template <bool NORM, int NT = 512, bool CG = false>
__device__ __forceinline__ float quantize_x(const float* __restrict__ x, const float* __restrict__ nw, int K,
                                            int nblk, XBlk* xb, int tid) {
    float ss = 0.f;
    constexpr int kBlkPerRound = NT / 8;
    constexpr int kBatch = 8;  // rounds whose global loads are in flight together (K <= 8 * NT * 4 in one batch)
    const int g = tid & 7;
    const int nround = (nblk + kBlkPerRound - 1) / kBlkPerRound;
    for (int r0 = 0; r0 < nround; r0 += kBatch) {
        float v[kBatch][4];
#pragma unroll
        for (int i = 0; i < kBatch; i++) {
            const int b = (r0 + i) * kBlkPerRound + (tid >> 3);
            const int k = b * 32 + g * 4;
            v[i][0] = v[i][1] = v[i][2] = v[i][3] = 0.f;
            if (r0 + i < nround && b < nblk && k < K) {  // K % 32 == 0: the 4 elements are all in range
                const float4 xv = CG ? __ldcg(reinterpret_cast<const float4*>(x + k))
                                     : *reinterpret_cast<const float4*>(x + k);
                v[i][0] = xv.x; v[i][1] = xv.y; v[i][2] = xv.z; v[i][3] = xv.w;
                if (NORM) {
                    ss = fmaf(xv.x, xv.x, fmaf(xv.y, xv.y, fmaf(xv.z, xv.z, fmaf(xv.w, xv.w, ss))));
                    const float4 w = *reinterpret_cast<const float4*>(nw + k);
                    v[i][0] *= w.x; v[i][1] *= w.y; v[i][2] *= w.z; v[i][3] *= w.w;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; i++) {
            // uniform per warp: every lane takes part in the shuffles
            if (r0 + i >= nround) break;
            const int b = (r0 + i) * kBlkPerRound + (tid >> 3);
            float m = fmaxf(fmaxf(fabsf(v[i][0]), fabsf(v[i][1])), fmaxf(fabsf(v[i][2]), fabsf(v[i][3])));
#pragma unroll
            for (int o = 4; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            // power-of-two scale: m = f 2^E with f in [0.5, 1) gives |x| / s <= 2^15 and s * xi exact
            int E = 0;
            frexpf(m, &E);
            const float inv = m > 0.f ? ldexpf(1.f, 15 - E) : 0.f;
            const float sc = m > 0.f ? ldexpf(1.f, E - 15) : 0.f;
            int xi[4];
            int sum = 0;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                xi[e] = max(-32767, min(32767, __float2int_rn(v[i][e] * inv)));
                sum += xi[e];
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            const int half = sum;  // elements 0..15 in lanes g < 4, 16..31 in lanes g >= 4
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            // byte planes: lo = byte 0 of each element, hi = byte 1
            const unsigned a01 = __byte_perm((unsigned)xi[0], (unsigned)xi[1], 0x5410);  // (x0.lo16, x1.lo16)
            const unsigned a23 = __byte_perm((unsigned)xi[2], (unsigned)xi[3], 0x5410);
            const unsigned lo = __byte_perm(a01, a23, 0x6420);  // bytes 0 of x0, x1, x2, x3
            const unsigned hi = __byte_perm(a01, a23, 0x7531);  // bytes 1
            if (b < nblk) {
                xb[b].hi[g] = hi;
                xb[b].lo[g] = lo;
                if (g == 0) {
                    xb[b].s = sc;
                    xb[b].sx8 = -8.f * sc * (float)sum;
                    xb[b].sxa = sc * (float)half;
                }
                if (g == 4) xb[b].sxb = sc * (float)half;
            }
        }
    }
    return ss;
}

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
