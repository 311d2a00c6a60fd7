// Quantized KV cache: retiring slots that left the fp16 window (dotLLM, "CUDA components": "Q8_0/Q4_0 + FP16
// window").  A retired slot's K and V rows are replaced, per 32 values along head_dim, by their Q8_0 / Q4_0
// quantization (block format of "Shimmy v2.0 Architecture", Quantization), with every decision taken in fp32
// on the fp16 values:
//   Q8_0: d = fp16(max|v| / 127), q = clamp(round-half-away(v / d), -127, 127)
//   Q4_0: m = the value of largest magnitude (first on ties), d = fp16(m / -8), n = clamp(floor(v / d + 8.5), 0, 15)
// (a zero d gives zero codes).  The codes and d go to the quantized store (decode attention reads retired
// slots there); fp16(d q) is written back into the fp16 cache, which prefill attention reads.
#include "common.cuh"

namespace af {

namespace {

// one thread per 32-value block of one row (layer, kv head, K or V, slot)
__global__ void kv_retire_kernel(KvStore st, __half* __restrict__ kc, __half* __restrict__ vc, int L, int KVH,
                                 int max_ctx, int D, const int* __restrict__ pos_dev, int first, int count) {
    if (pos_dev) first = __ldcg(pos_dev) - st.window;
    const int nb = D / 32;
    const int64_t total = (int64_t)count * L * KVH * 2 * nb;
    const int cb = kv_code_bytes(st.qtype, D);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = i;
        const int b = (int)(r % nb);
        r /= nb;
        const int isv = (int)(r % 2);
        r /= 2;
        const int64_t row = r % ((int64_t)L * KVH);  // layer * KVH + kv head
        const int slot = first + (int)(r / ((int64_t)L * KVH));
        if (slot < 0 || slot >= max_ctx) continue;
        const int64_t srow = row * max_ctx + slot;  // [layer][kv head][slot]
        __half* h = (isv ? vc : kc) + srow * D + b * 32;
        float x[32];
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const uint4 raw = *reinterpret_cast<const uint4*>(h + 8 * c);
            const __half2* hp = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float2 f = __half22float2(hp[e]);
                x[8 * c + 2 * e] = f.x;
                x[8 * c + 2 * e + 1] = f.y;
            }
        }
        int q[32];
        __half dh;
        if (st.qtype == AF_KV_Q8_0) {
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < 32; j++) amax = fmaxf(amax, fabsf(x[j]));
            dh = __float2half_rn(amax / 127.f);
            const float df = __half2float(dh);
#pragma unroll
            for (int j = 0; j < 32; j++) {
                int v = 0;
                if (df != 0.f) {
                    const float t = x[j] / df;
                    v = (int)(t >= 0.f ? floorf(t + 0.5f) : -floorf(-t + 0.5f));
                    v = v < -127 ? -127 : (v > 127 ? 127 : v);
                }
                q[j] = v;
            }
        } else {
            float mx = 0.f, amax = 0.f;
#pragma unroll
            for (int j = 0; j < 32; j++)
                if (fabsf(x[j]) > amax) {
                    amax = fabsf(x[j]);
                    mx = x[j];
                }
            dh = __float2half_rn(mx / -8.f);
            const float df = __half2float(dh);
#pragma unroll
            for (int j = 0; j < 32; j++) {
                int n = 8;
                if (df != 0.f) {
                    n = (int)floorf(x[j] / df + 8.5f);
                    n = n < 0 ? 0 : (n > 15 ? 15 : n);
                }
                q[j] = n - 8;
            }
        }
        // store: codes and scale
        uint8_t* code = (isv ? st.vq : st.kq) + srow * cb + (st.qtype == AF_KV_Q8_0 ? b * 32 : b * 16);
        if (st.qtype == AF_KV_Q8_0) {
#pragma unroll
            for (int c = 0; c < 2; c++) {
                unsigned w[4];
#pragma unroll
                for (int k = 0; k < 4; k++)
                    w[k] = (unsigned)(q[16 * c + 4 * k] & 255) | (unsigned)(q[16 * c + 4 * k + 1] & 255) << 8 |
                           (unsigned)(q[16 * c + 4 * k + 2] & 255) << 16 | (unsigned)(q[16 * c + 4 * k + 3] & 255) << 24;
                *reinterpret_cast<uint4*>(code + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
            unsigned w[4];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                unsigned v = 0;
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int j = 8 * k + 2 * e;
                    v |= (unsigned)((q[j] + 8) | (q[j + 1] + 8) << 4) << (8 * e);
                }
                w[k] = v;
            }
            *reinterpret_cast<uint4*>(code) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        (isv ? st.vs : st.ks)[srow * (D / 32) + b] = dh;
        // the fp16 cache's copy of the slot: fp16(d q)
        const float df = __half2float(dh);
#pragma unroll
        for (int c = 0; c < 4; c++) {
            __half2 o[4];
#pragma unroll
            for (int e = 0; e < 4; e++)
                o[e] = __floats2half2_rn(df * (float)q[8 * c + 2 * e], df * (float)q[8 * c + 2 * e + 1]);
            *reinterpret_cast<uint4*>(h + 8 * c) = *reinterpret_cast<const uint4*>(o);
        }
    }
}

}  // namespace

cudaError_t launch_kv_retire(const KvStore& st, __half* kc, __half* vc, int L, int KVH, int max_ctx, int D,
                             const int* pos_dev, int first, int count, cudaStream_t s) {
    if (!st.qtype || count < 1) return cudaSuccess;
    const int64_t total = (int64_t)count * L * KVH * 2 * (D / 32);
    int64_t blocks = (total + 127) / 128;
    if (blocks > 8 * 152) blocks = 8 * 152;
    kv_retire_kernel<<<(unsigned)blocks, 128, 0, s>>>(st, kc, vc, L, KVH, max_ctx, D, pos_dev, first, count);
    return cudaGetLastError();
}

}  // namespace af
