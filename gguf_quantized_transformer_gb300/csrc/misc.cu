// Small kernels of the forward pass: weight repack, RoPE table, embedding
// lookup, row RMSNorm, fp32->fp16 conversion and decode-step bookkeeping.
#include <cmath>

#include "common.cuh"

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

// GGUF AoS blocks -> per-row records of quants then scales (see Planes).  One thread per
// destination block; blocks past K/32 are zero.
__global__ void repack_kernel(const uint8_t* __restrict__ src, int wtype, int N, int nb, uint8_t* __restrict__ qs,
                              __half* __restrict__ sc, int nbp, int row0, int step) {
    int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)N * nbp) return;
    int r = (int)(t / nbp), b = (int)(t % nbp);
    const int qb = wtype == AF_Q8_0 ? 32 : 16, bb = qb + 2;
    const int64_t pitch = (int64_t)nbp * bb;  // bytes per destination row (quants, then scales)
    int64_t dr = (int64_t)row0 + (int64_t)r * step;
    uint8_t* dq = qs + dr * pitch + (int64_t)b * qb;
    __half* dsc = sc + dr * (pitch / 2) + b;
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

cudaError_t launch_repack(const uint8_t* src, int wtype, int N, int K, uint8_t* qs, __half* sc, int Kp, int row0,
                          int step, cudaStream_t s) {
    int64_t n = (int64_t)N * (Kp / 32);
    int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    repack_kernel<<<(unsigned)blocks, threads, 0, s>>>(src, wtype, N, K / 32, qs, sc, Kp / 32, row0, step);
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

// x[r][:] = dequantized row tok[r] of the embedding table.
__global__ void embed_kernel(Planes emb, const int* __restrict__ tok, int E, float* __restrict__ x, int64_t ldx) {
    const int r = blockIdx.y;
    int row = tok[r];
    if (row < 0 || row >= emb.N) row = 0;  // ids are validated on the host; never read outside the table
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < E; k += gridDim.x * blockDim.x) {
        const int b = k >> 5, e = k & 31;
        const float d = __half2float(emb.sc[(int64_t)row * emb.sc_pitch() + b]);
        const uint8_t* q = emb.qs + (int64_t)row * emb.qs_pitch() + (int64_t)b * emb.qb();
        float v;
        if (emb.wtype == AF_Q8_0) {
            v = d * (float)(int8_t)q[e];
        } else {
            const uint8_t byte = q[e & 15];
            v = d * (float)((e < 16 ? (byte & 15) : (byte >> 4)) - 8);
        }
        x[(int64_t)r * ldx + k] = v;
    }
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

// y = w * x / sqrt(mean(x^2) + eps) for each of n rows (one CTA per row), as fp16 hi + lo.
__global__ void rmsnorm_rows_kernel(const float* __restrict__ x, int E, const float* __restrict__ w, float eps,
                                    __half* __restrict__ y_hi, __half* __restrict__ y_lo) {
    __shared__ float red[32];
    const float* xr = x + (int64_t)blockIdx.x * E;
    float ss = 0.f;
    for (int k = threadIdx.x; k < E; k += blockDim.x) ss += xr[k] * xr[k];
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / (float)E + eps);
    for (int k = threadIdx.x; k < E; k += blockDim.x) {
        const float v = w[k] * (xr[k] * inv);
        const __half h = __float2half_rn(v);
        y_hi[(int64_t)blockIdx.x * E + k] = h;
        y_lo[(int64_t)blockIdx.x * E + k] = __float2half_rn(v - __half2float(h));
    }
}

cudaError_t launch_rmsnorm_rows(const float* x, int n, int E, const float* w, float eps, __half* y_hi, __half* y_lo,
                                cudaStream_t s) {
    rmsnorm_rows_kernel<<<n, 256, 0, s>>>(x, E, w, eps, y_hi, y_lo);
    return cudaGetLastError();
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
