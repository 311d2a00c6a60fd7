// Small kernels of the forward pass: weight repack, RoPE table, embedding
// lookup, row RMSNorm, fp32->fp16 conversion and decode-step bookkeeping.
#include <cmath>

#include "common.cuh"
#include "tma.cuh"

namespace af {

int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

// GGUF AoS blocks -> per-row records (see Planes).  One thread per destination 32-weight unit (per 32-weight
// block for Q4_0 / Q8_0); units past K are zero.  The first unit of a K-quant super-block also writes the
// super-block's record.  Source row r goes to destination row row0 + r * step.
// qs_off: byte offset of the nibbles in the source block (16 for Q4_K, 48 for Q5_K)
__device__ void repack_q4_k_unit(const uint8_t* blk, int j, uint8_t* dq, uint8_t* rec, int qs_off = 16) {
    // codes of sub-block j: elements 32 j + i live in qs[32 (j / 2) + i], low nibble for even j
    const uint8_t* qs = blk + qs_off + 32 * (j >> 1);
    const int sh = (j & 1) * 4;
    for (int t = 0; t < 16; t++)
        dq[t] = (uint8_t)(((qs[t] >> sh) & 15) | (((qs[t + 16] >> sh) & 15) << 4));
    if (j == 0) {  // record: d, dmin, then the unpacked (scale, min) of every sub-block
        for (int i = 0; i < 4; i++) rec[i] = blk[i];
        const uint8_t* sc = blk + 4;
        for (int k = 0; k < 8; k++) {
            int sk, mk;
            if (k < 4) {
                sk = sc[k] & 63;
                mk = sc[k + 4] & 63;
            } else {
                sk = (sc[k + 4] & 15) | ((sc[k - 4] >> 6) << 4);
                mk = (sc[k + 4] >> 4) | ((sc[k] >> 6) << 4);
            }
            rec[4 + 2 * k] = (uint8_t)sk;
            rec[5 + 2 * k] = (uint8_t)mk;
        }
    }
}

// Q5_K: Q4_K's nibbles and record, plus the high bits of sub-block j (bit j of qh[i] for element i) as one
// word: element 4t + b of half h at bit 8b + 4h + t
__device__ void repack_q5_k_unit(const uint8_t* blk, int j, uint8_t* dq, uint8_t* dh, uint8_t* rec) {
    repack_q4_k_unit(blk, j, dq, rec, 48);
    const uint8_t* qh = blk + 16;
    uint32_t hw = 0u;
    for (int e = 0; e < 32; e++) {
        const int h = e >> 4, i = e & 15;
        hw |= (uint32_t)((qh[e] >> j) & 1) << (8 * (i & 3) + 4 * h + (i >> 2));
    }
    for (int b = 0; b < 4; b++) dh[b] = (uint8_t)(hw >> (8 * b));
}

__device__ void repack_q6_k_unit(const uint8_t* blk, int g, uint8_t* dq, uint8_t* dh, uint8_t* rec) {
    // code of element e = 32 g + i of the super-block: low 4 bits in ql, high 2 bits in qh
    auto code = [&](int e) {
        const int h = e >> 7, k = (e & 127) >> 5, l = e & 31;
        const uint8_t lo = blk[64 * h + 32 * (k & 1) + l];
        return ((k < 2 ? lo : lo >> 4) & 15) | (((blk[128 + 32 * h + l] >> (2 * k)) & 3) << 4);
    };
    uint32_t hw[2] = {0u, 0u};
    for (int t = 0; t < 16; t++) {
        const int c0 = code(32 * g + t), c1 = code(32 * g + t + 16);
        dq[t] = (uint8_t)((c0 & 15) | ((c1 & 15) << 4));
        // element 4 tt + i of a half at bits 8 i + 2 tt of that half's word
        const int tt = t >> 2, i = t & 3;
        hw[0] |= (uint32_t)(c0 >> 4) << (8 * i + 2 * tt);
        hw[1] |= (uint32_t)(c1 >> 4) << (8 * i + 2 * tt);
    }
    for (int b = 0; b < 8; b++) dh[b] = (uint8_t)(hw[b >> 2] >> (8 * (b & 3)));
    if (g == 0) {  // record: d, then the 16 scales
        rec[0] = blk[208];
        rec[1] = blk[209];
        for (int k = 0; k < 16; k++) rec[2 + k] = blk[192 + k];
    }
}

__global__ void repack_kernel(const uint8_t* __restrict__ src, Planes P, int N, int row0, int step) {
    const int nbp = P.Kp / 32, nb = P.K / 32;  // destination units per row, source units per row
    int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)N * nbp) return;
    const int r = (int)(t / nbp), b = (int)(t % nbp);
    const int64_t pitch = P.qs_pitch();
    uint8_t* row = const_cast<uint8_t*>(P.qs) + ((int64_t)row0 + (int64_t)r * step) * pitch;
    if (is_kquant(P.wtype)) {
        const int sb = b / 8, u = b % 8;
        const int bb = P.wtype == AF_Q4_K ? 144 : P.wtype == AF_Q5_K ? 176 : 210;
        const int rec_bytes = P.wtype == AF_Q6_K ? kQ6KRec : kQ4KRec;
        const int hbu = P.wtype == AF_Q6_K ? 8 : 4;  // high-bit bytes per unit (Q5_K, Q6_K)
        uint8_t* dq = row + (int64_t)b * 16;
        uint8_t* rec = row + P.sc_off() + (int64_t)sb * rec_bytes;
        uint8_t* dh = row + P.hb_off() + (int64_t)b * hbu;
        if (b < nb) {
            const uint8_t* blk = src + ((int64_t)r * (nb / 8) + sb) * bb;
            if (P.wtype == AF_Q4_K) repack_q4_k_unit(blk, u, dq, rec);
            else if (P.wtype == AF_Q5_K) repack_q5_k_unit(blk, u, dq, dh, rec);
            else repack_q6_k_unit(blk, u, dq, dh, rec);
        } else {
            for (int j = 0; j < 16; j++) dq[j] = 0;
            if (P.wtype != AF_Q4_K)
                for (int j = 0; j < hbu; j++) dh[j] = 0;
            if (u == 0)
                for (int j = 0; j < rec_bytes; j++) rec[j] = 0;
        }
        if (b == nbp - 1)  // the row's padding up to its 16-byte pitch
            for (int64_t j = P.sc_off() + (int64_t)(nbp / 8) * rec_bytes; j < pitch; j++) row[j] = 0;
        return;
    }
    const int qb = P.qb(), bb = qb + 2;
    uint8_t* dq = row + (int64_t)b * qb;
    __half* dsc = reinterpret_cast<__half*>(row + P.sc_off()) + b;
    if (b < nb) {
        const uint8_t* s = src + ((int64_t)r * nb + b) * bb;
        unsigned short bits = (unsigned short)(s[0] | (s[1] << 8));
        *dsc = __ushort_as_half(bits);
        for (int j = 0; j < qb; j++) dq[j] = s[2 + j];
    } else {
        *dsc = __ushort_as_half(0);
        for (int j = 0; j < qb; j++) dq[j] = 0;
    }
}

cudaError_t launch_repack(const uint8_t* src, const Planes& P, int N, int row0, int step, cudaStream_t s) {
    int64_t n = (int64_t)N * (P.Kp / 32);
    int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    repack_kernel<<<(unsigned)blocks, threads, 0, s>>>(src, P, N, row0, step);
    return cudaGetLastError();
}

// RoPE table: tab[t][i] = (cos, sin) of theta(t, i) = (t / yarn_scale) / base^(2i / head_dim),
// evaluated in fp64 and rounded once to fp32.
__global__ void rope_table_kernel(float2* tab, int max_ctx, int half_d, int head_dim, double base, double ys) {
    int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)max_ctx * half_d) return;
    int pos = (int)(t / half_d), i = (int)(t % half_d);
    double theta = ((double)pos / ys) / pow(base, (2.0 * i) / (double)head_dim);
    double sn, cs;
    sincos(theta, &sn, &cs);
    tab[t] = make_float2((float)cs, (float)sn);
}

cudaError_t launch_rope_table(float2* tab, int max_ctx, int head_dim, double base, double ys, cudaStream_t s) {
    int64_t n = (int64_t)max_ctx * (head_dim / 2);
    rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(tab, max_ctx, head_dim / 2, head_dim, base, ys);
    return cudaGetLastError();
}

// Value of weight k of row `row` of repacked planes (the embedding table), in fp32.
__device__ float plane_weight(const Planes& P, int row, int k) {
    const uint8_t* base = P.qs + (int64_t)row * P.qs_pitch();
    const int u = k >> 5, e = k & 31;
    if (is_kquant(P.wtype)) {
        const uint8_t byte = base[(int64_t)u * 16 + (e & 15)];
        const int lo4 = e < 16 ? (byte & 15) : (byte >> 4);
        if (P.wtype != AF_Q6_K) {
            int q = lo4;
            if (P.wtype == AF_Q5_K) {  // high bit: element 4t + b of half h at bit 8b + 4h + t of the unit's word
                const uint8_t* hb = base + P.hb_off() + (int64_t)u * 4;
                const uint32_t hw = (uint32_t)hb[0] | ((uint32_t)hb[1] << 8) | ((uint32_t)hb[2] << 16) | ((uint32_t)hb[3] << 24);
                const int i = e & 15;
                q |= (int)((hw >> (8 * (i & 3) + 4 * (e >> 4) + (i >> 2))) & 1u) << 4;
            }
            const uint8_t* rec = base + P.sc_off() + (int64_t)(u >> 3) * kQ4KRec;
            const float d = __half2float(__ushort_as_half((unsigned short)(rec[0] | (rec[1] << 8))));
            const float dmin = __half2float(__ushort_as_half((unsigned short)(rec[2] | (rec[3] << 8))));
            const int j = u & 7;
            return d * (float)rec[4 + 2 * j] * (float)q - dmin * (float)rec[5 + 2 * j];
        }
        const uint8_t* hb = base + P.hb_off() + (int64_t)u * 8 + (e >> 4) * 4;
        const uint32_t hw = (uint32_t)hb[0] | ((uint32_t)hb[1] << 8) | ((uint32_t)hb[2] << 16) | ((uint32_t)hb[3] << 24);
        const int i = e & 15;
        const int q = lo4 | (int)((hw >> (8 * (i & 3) + 2 * (i >> 2))) & 3u) << 4;
        const uint8_t* rec = base + P.sc_off() + (int64_t)(u >> 3) * kQ6KRec;
        const float d = __half2float(__ushort_as_half((unsigned short)(rec[0] | (rec[1] << 8))));
        const int sc = (int8_t)rec[2 + 2 * (u & 7) + (e >> 4)];
        return d * (float)sc * (float)(q - 32);
    }
    const float d = __half2float(P.sc[(int64_t)row * P.sc_pitch() + u]);
    const uint8_t* q = base + (int64_t)u * P.qb();
    if (P.wtype == AF_Q8_0) return d * (float)(int8_t)q[e];
    const uint8_t byte = q[e & 15];
    return d * (float)((e < 16 ? (byte & 15) : (byte >> 4)) - 8);
}

// x[r][:] = dequantized row tok[r] of the embedding table.
__global__ void embed_kernel(Planes emb, const int* __restrict__ tok, int E, float* __restrict__ x, int64_t ldx) {
    const int r = blockIdx.y;
    int row = tok[r];
    if (row < 0 || row >= emb.N) row = 0;  // ids are validated on the host; never read outside the table
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < E; k += gridDim.x * blockDim.x)
        x[(int64_t)r * ldx + k] = plane_weight(emb, row, k);
}

cudaError_t launch_embed(const Planes& emb, const int* tok_dev, int n, float* x, int64_t ldx, cudaStream_t s) {
    dim3 grid((emb.K + 255) / 256, n);
    embed_kernel<<<grid, 256, 0, s>>>(emb, tok_dev, emb.K, x, ldx);
    return cudaGetLastError();
}

__device__ __forceinline__ float block_sum(float v, float* red) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < nw; i++) t += red[i];  // same order in every thread
    return t;
}

// y = w * x / sqrt(mean(x^2) + eps) for each of n rows (one CTA per row), as fp16 hi + lo.  Rows of up to
// kRmsMaxV * 4 * 256 elements (E % 4 == 0) stay in registers between the sum of squares and the scaling; the
// norm weights are read before griddepcontrol.wait (they do not depend on the previous kernel).
constexpr int kRmsThreads = 256;
constexpr int kRmsMaxV = 8;  // float4 per thread
__global__ void __launch_bounds__(kRmsThreads) rmsnorm_rows_kernel(const float* __restrict__ x, int E,
                                                                   const float* __restrict__ w, float eps,
                                                                   __half* __restrict__ y_hi,
                                                                   __half* __restrict__ y_lo) {
    __shared__ float red[32];
    pdl_launch_dependents();
    const int nv = E / 4, tid = threadIdx.x;
    const float4* w4 = reinterpret_cast<const float4*>(w);
    float4 wv[kRmsMaxV], xv[kRmsMaxV];
#pragma unroll
    for (int j = 0; j < kRmsMaxV; j++) {
        const int i = tid + j * kRmsThreads;
        wv[j] = i < nv ? w4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_wait();  // x is written by an earlier kernel: read through L2 (the note above epi_pair)
    const float4* x4 = reinterpret_cast<const float4*>(x + (int64_t)blockIdx.x * E);
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kRmsMaxV; j++) {
        const int i = tid + j * kRmsThreads;
        xv[j] = i < nv ? __ldcg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        ss = fmaf(xv[j].x, xv[j].x, fmaf(xv[j].y, xv[j].y, fmaf(xv[j].z, xv[j].z, fmaf(xv[j].w, xv[j].w, ss))));
    }
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / (float)E + eps);
    uint2* yh = reinterpret_cast<uint2*>(y_hi + (int64_t)blockIdx.x * E);
    uint2* yl = reinterpret_cast<uint2*>(y_lo + (int64_t)blockIdx.x * E);
#pragma unroll
    for (int j = 0; j < kRmsMaxV; j++) {
        const int i = tid + j * kRmsThreads;
        if (i < nv) {
            const float v[4] = {wv[j].x * (xv[j].x * inv), wv[j].y * (xv[j].y * inv), wv[j].z * (xv[j].z * inv),
                                wv[j].w * (xv[j].w * inv)};
            __half h[4], l[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                h[e] = __float2half_rn(v[e]);
                l[e] = __float2half_rn(v[e] - __half2float(h[e]));
            }
            uint2 ph, pl;
            ph.x = (unsigned)__half_as_ushort(h[0]) | ((unsigned)__half_as_ushort(h[1]) << 16);
            ph.y = (unsigned)__half_as_ushort(h[2]) | ((unsigned)__half_as_ushort(h[3]) << 16);
            pl.x = (unsigned)__half_as_ushort(l[0]) | ((unsigned)__half_as_ushort(l[1]) << 16);
            pl.y = (unsigned)__half_as_ushort(l[2]) | ((unsigned)__half_as_ushort(l[3]) << 16);
            yh[i] = ph;
            yl[i] = pl;
        }
    }
}

cudaError_t launch_rmsnorm_rows(const float* x, int n, int E, const float* w, float eps, __half* y_hi, __half* y_lo,
                                cudaStream_t s) {
    if (E % 4 || E > kRmsMaxV * 4 * kRmsThreads) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n);
    cfg.blockDim = dim3(kRmsThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rmsnorm_rows_kernel, x, E, w, eps, y_hi, y_lo);
}

__global__ void split_f16_kernel(const float* __restrict__ x, __half* __restrict__ hi, __half* __restrict__ lo,
                                 int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = x[i];
        const __half h = __float2half_rn(v);
        hi[i] = h;
        lo[i] = __float2half_rn(v - __half2float(h));
    }
}

cudaError_t launch_split_f16(const float* x, __half* hi, __half* lo, int64_t n, cudaStream_t s) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) blocks = 1;
    split_f16_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, hi, lo, n);
    return cudaGetLastError();
}

__global__ void join_f16_kernel(const __half* __restrict__ hi, const __half* __restrict__ lo, float* __restrict__ out,
                                int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = __half2float(hi[i]) + __half2float(lo[i]);
}

cudaError_t launch_join_f16(const __half* hi, const __half* lo, float* out, int64_t n, cudaStream_t s) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) blocks = 1;
    join_f16_kernel<<<(unsigned)blocks, 256, 0, s>>>(hi, lo, out, n);
    return cudaGetLastError();
}

__global__ void step_begin_kernel(StepState* st, int token, int pos, unsigned* bar_count) {
    st->token = token >= 0 ? token : st->next_token;
    st->pos = pos;
    st->argmax = 0ull;
    if (bar_count) *bar_count = 0u;  // grid barrier of the persistent decode kernel starts over
}

__global__ void step_end_kernel(StepState* st) {
    // no key recorded (all logits NaN) -> token 0, so a device-fed next step stays in range
    st->next_token = st->argmax ? (int)(0xFFFFFFFFu - (unsigned)(st->argmax & 0xFFFFFFFFull)) : 0;
}

cudaError_t launch_step_begin(StepState* st, int token, int pos, cudaStream_t s, unsigned* bar_count) {
    step_begin_kernel<<<1, 1, 0, s>>>(st, token, pos, bar_count);
    return cudaGetLastError();
}

cudaError_t launch_step_end(StepState* st, cudaStream_t s) {
    step_end_kernel<<<1, 1, 0, s>>>(st);
    return cudaGetLastError();
}

}  // namespace af
