// Prefill GEMM, CUDA-core version: Y[m][n] = sum_k X[m][k] W[n][k] with the
// quantized W dequantized into shared memory one 32-weight block column at a
// time (dotLLM "GPU Inference", "Weight Strategy", approach 1: dequantized
// values never touch device memory) and the fused epilogue applied per column
// pair.  X and the dequantized weights are exact fp32 operands; products
// accumulate in fp32.
#include "common.cuh"

namespace af {

namespace {

constexpr int BM = 64, BN = 64, BK = 32;

__global__ void __launch_bounds__(256) qgemm_simt_kernel(Planes W, const float* __restrict__ X, int64_t ldx, int M,
                                                         Epi epi) {
    __shared__ float Xs[BK][BM + 4];
    __shared__ float Ws[BK][BN + 4];
    const int tid = threadIdx.x;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int tx = tid & 15, ty = tid >> 4;  // 16 x 16 threads, 4 x 4 outputs each
    float acc[4][4] = {};
    const int nkb = W.K / 32;
    for (int kb = 0; kb < nkb; kb++) {
        {  // X tile: 64 rows x 32 floats, 8 per thread
            const int r = tid >> 2, q = tid & 3;
            const int m = m0 + r;
            float v[8];
            if (m < M) {
                const float4* xp = reinterpret_cast<const float4*>(X + (int64_t)m * ldx + kb * 32 + q * 8);
                const float4 a = xp[0], b = xp[1];
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; e++) v[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; e++) Xs[q * 8 + e][r] = v[e];
        }
        {  // W tile: 64 rows x one block, 8 weights per thread
            const int r = tid >> 2, q = tid & 3;
            const int n = n0 + r;
            float v[8];
            if (n < W.N) {
                const float d = __half2float(W.sc[(int64_t)n * W.sc_pitch() + kb]);
                const uint8_t* qp = W.qs + (int64_t)n * W.qs_pitch() + (int64_t)kb * W.qb();
                if (W.wtype == AF_Q8_0) {
#pragma unroll
                    for (int e = 0; e < 8; e++) v[e] = d * (float)(int8_t)qp[q * 8 + e];
                } else {
                    // elements 8q..8q+7: low nibbles of bytes 8q.. (q < 2), high nibbles of bytes 8(q-2).. (q >= 2)
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const int el = q * 8 + e;
                        const uint8_t b = qp[el & 15];
                        v[e] = d * (float)((el < 16 ? (b & 15) : (b >> 4)) - 8);
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; e++) v[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; e++) Ws[q * 8 + e][r] = v[e];
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < BK; k++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = Xs[k][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = Ws[k][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            const int n = n0 + tx * 4 + j;
            if (n < W.N) epi_pair(epi, m, n, acc[i][j], acc[i][j + 1]);
        }
    }
}

}  // namespace

cudaError_t launch_qgemm(const Planes& W, const float* X, int64_t ldx, int M, const Epi& epi, cudaStream_t s) {
    dim3 grid((W.N + BN - 1) / BN, (M + BM - 1) / BM);
    qgemm_simt_kernel<<<grid, 256, 0, s>>>(W, X, ldx, M, epi);
    return cudaGetLastError();
}

}  // namespace af
