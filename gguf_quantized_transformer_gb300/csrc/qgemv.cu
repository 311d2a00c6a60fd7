// Decode GEMV: y = W x over repacked Q4_0 / Q8_0 planes, with an optional
// RMSNorm prologue and a fused epilogue (Airframe "GPU_PIPELINE.md" per-layer
// ops: "Dequantization happens inline ... No separate dequantize-then-multiply
// step"; decode is bound by reading the weights, "Decode loop").
//
// Work split.  A row of Kp weights is NC chunks of 32 sixteen-byte units
// (Q4_0: one unit = one 32-weight block; Q8_0: half a block).  The N*NC
// (chunk, row) items, ordered chunk-major, are divided evenly over all warps of
// the grid, so every warp streams the same number of bytes (+-1 item)
// whatever N and K are.  Lane l of a warp owns unit l of the chunk, keeps that
// unit's x slice in registers and walks down the rows, issuing one 128-bit
// streaming load per row, 8 rows at a time.
//
// Reduction.  The 8 per-lane row partials are reduced across the warp with a
// transpose-reduce (3 exchange steps + 2 butterfly steps), leaving row j's
// chunk sum in lanes 4j..4j+3.  It is stored to part[c][row]; an acq_rel
// counter per row pair counts arrivals, and the lane that completes a pair
// sums its NC partials in chunk order (deterministic) and applies the fused
// epilogue to the pair, then re-zeroes the counter for the next launch.
//
// Dequantization in registers.
//   Q4_0: byte_perm places a nibble n in bits 16..19 under exponent 0x3F0,
//         giving the float 0.5 + n/256 in one instruction.  With S the FMA sum
//         of those floats times x over the block and sx = sum(x):
//           sum_j (n_j - 8) x_j = 256 S - 136 sx,   block value = d * that.
//   Q8_0: byte_perm places (q + 128) under 0x4B00 00.., i.e. 2^23 + q + 128,
//         and one FADD recovers q exactly.
#include "common.cuh"

namespace af {

namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ float ld_relaxed(const float* p) {
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}

template <int WT>
struct Q;
template <>
struct Q<AF_Q4_0> {
    static constexpr int UW = 32;  // weights per 16-byte unit
    static __device__ __forceinline__ float dot(uint4 q, const float* xv, float sx) {
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const unsigned lo = w[t] & 0x0F0F0F0Fu, hi = (w[t] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
            for (int b = 0; b < 4; b++) {
                const unsigned sel = 0x7044u | ((unsigned)b << 8);
                s0 = fmaf(__uint_as_float(__byte_perm(lo, 0x3F000000u, sel)), xv[4 * t + b], s0);
                s1 = fmaf(__uint_as_float(__byte_perm(hi, 0x3F000000u, sel)), xv[16 + 4 * t + b], s1);
            }
        }
        return 256.f * (s0 + s1) - 136.f * sx;
    }
};
template <>
struct Q<AF_Q8_0> {
    static constexpr int UW = 16;
    static __device__ __forceinline__ float dot(uint4 q, const float* xv, float) {
        const unsigned w[4] = {q.x ^ 0x80808080u, q.y ^ 0x80808080u, q.z ^ 0x80808080u, q.w ^ 0x80808080u};
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int t = 0; t < 4; t++) {
#pragma unroll
            for (int b = 0; b < 4; b += 2) {
                const float q0 = __uint_as_float(__byte_perm(w[t], 0x4B000000u, 0x7440u | b)) - 8388736.f;
                const float q1 = __uint_as_float(__byte_perm(w[t], 0x4B000000u, 0x7440u | (b + 1))) - 8388736.f;
                s0 = fmaf(q0, xv[4 * t + b], s0);
                s1 = fmaf(q1, xv[4 * t + b + 1], s1);
            }
        }
        return s0 + s1;
    }
};

// Reduce v[0..7] over the 32 lanes; afterwards lanes 4j..4j+3 hold sum of v[j].
__device__ __forceinline__ float transpose_reduce8(float v[8], int lane) {
    {
        const bool up = lane & 16;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float send = up ? v[k] : v[k + 4], keep = up ? v[k + 4] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    {
        const bool up = lane & 8;
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const float send = up ? v[k] : v[k + 2], keep = up ? v[k + 2] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
    {
        const bool up = lane & 4;
        const float send = up ? v[0] : v[1], keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float r = v[0];
    r += __shfl_xor_sync(0xffffffffu, r, 2);
    r += __shfl_xor_sync(0xffffffffu, r, 1);
    return r;
}

template <int WT, bool NORM>
__global__ void __launch_bounds__(kWarps * 32, 2)
    qgemv_kernel(Planes W, const float* __restrict__ x, const float* __restrict__ nw, float eps, Epi epi,
                 float* __restrict__ part, unsigned* __restrict__ cnt) {
    constexpr int UW = Q<WT>::UW;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int N = W.N, K = W.K;
    const int NC = W.Kp / (32 * UW);

    float rstd = 1.f;
    if (NORM) {  // RMSNorm prologue: every CTA reduces sum(x^2) over the whole input
        __shared__ float red[kWarps];
        float ss = 0.f;
        const float4* x4 = reinterpret_cast<const float4*>(x);
        for (int k = threadIdx.x; k < K / 4; k += blockDim.x) {
            const float4 v = x4[k];
            ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
        }
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < kWarps; i++) t += red[i];
        rstd = rsqrtf(t / (float)K + eps);
    }

    const int64_t T = (int64_t)NC * N;
    const int64_t Wt = (int64_t)gridDim.x * kWarps, wg = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t i0 = T * wg / Wt, i1 = T * (wg + 1) / Wt;
    const int64_t pitch = W.qs_pitch();
    const int scp = W.sc_pitch();

    float xv[UW];
    float sx = 0.f;
    int cur_c = -1;
    for (int64_t i = i0; i < i1;) {
        const int c = (int)(i / N);
        const int r = (int)(i - (int64_t)c * N);
        int rows = N - r;
        if (rows > 8) rows = 8;
        if ((int64_t)rows > i1 - i) rows = (int)(i1 - i);
        const int unit = c * 32 + lane;  // this lane's unit within the row
        if (c != cur_c) {                // (re)load the x slice for this chunk
            const int k0 = unit * UW;
            sx = 0.f;
            if (k0 < K) {
                const float4* xp = reinterpret_cast<const float4*>(x + k0);
#pragma unroll
                for (int e = 0; e < UW / 4; e++) {
                    float4 v = xp[e];
                    if (NORM) {
                        const float4 g = reinterpret_cast<const float4*>(nw + k0)[e];
                        v.x = g.x * (v.x * rstd);
                        v.y = g.y * (v.y * rstd);
                        v.z = g.z * (v.z * rstd);
                        v.w = g.w * (v.w * rstd);
                    }
                    xv[4 * e] = v.x;
                    xv[4 * e + 1] = v.y;
                    xv[4 * e + 2] = v.z;
                    xv[4 * e + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < UW; e++) xv[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < UW; e++) sx += xv[e];
            cur_c = c;
        }
        const uint8_t* qrow = W.qs + (int64_t)r * pitch + (int64_t)unit * 16;
        const __half* srow = W.sc + (int64_t)r * scp + (WT == AF_Q8_0 ? unit >> 1 : unit);
        uint4 q[8];
        float d[8];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            if (j < rows) {
                q[j] = ld_stream(qrow + (int64_t)j * pitch);
                d[j] = __half2float(srow[(int64_t)j * scp]);
            }
        }
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] = (j < rows) ? d[j] * Q<WT>::dot(q[j], xv, sx) : 0.f;
        const float s = transpose_reduce8(v, lane);
        const int jr = lane >> 2;
        if ((lane & 3) == 0 && jr < rows) {
            const int row = r + jr;
            part[(int64_t)c * N + row] = s;
            const unsigned old = atom_add_acq_rel(&cnt[row >> 1], 1u);
            if (old == 2u * (unsigned)NC - 1u) {  // this lane completed the pair
                const int r0 = row & ~1;
                float y0 = 0.f, y1 = 0.f;
                for (int cc = 0; cc < NC; cc++) {
                    y0 += ld_relaxed(part + (int64_t)cc * N + r0);
                    y1 += ld_relaxed(part + (int64_t)cc * N + r0 + 1);
                }
                epi_pair(epi, 0, r0, y0, y1);
                cnt[row >> 1] = 0u;
            }
        }
        i += rows;
    }
}

}  // namespace

size_t qgemv_part_elems(const Planes& W) { return (size_t)(W.Kp / chunk_weights(W.wtype)) * (size_t)W.N; }

cudaError_t launch_qgemv(const Planes& W, const float* x, const float* norm_w, float eps, const Epi& epi,
                         const GemvScratch& scr, cudaStream_t s) {
    const int grid = 2 * num_sms();
    const int threads = kWarps * 32;
    if (W.wtype == AF_Q4_0) {
        if (norm_w)
            qgemv_kernel<AF_Q4_0, true><<<grid, threads, 0, s>>>(W, x, norm_w, eps, epi, scr.part, scr.cnt);
        else
            qgemv_kernel<AF_Q4_0, false><<<grid, threads, 0, s>>>(W, x, norm_w, eps, epi, scr.part, scr.cnt);
    } else {
        if (norm_w)
            qgemv_kernel<AF_Q8_0, true><<<grid, threads, 0, s>>>(W, x, norm_w, eps, epi, scr.part, scr.cnt);
        else
            qgemv_kernel<AF_Q8_0, false><<<grid, threads, 0, s>>>(W, x, norm_w, eps, epi, scr.part, scr.cnt);
    }
    return cudaGetLastError();
}

}  // namespace af
