// Prefill GEMM on the 5th-generation tensor cores: Y[m][n] = sum_k X[m][k] W[n][k]
// with W in Q4_0 / Q8_0 planes, dequantized tile by tile into shared memory
// and multiplied with tcgen05.mma into a TMEM accumulator (dotLLM "GPU
// Inference", "Weight Strategy", approach 1: fused dequantize-in-kernel feeding
// the tensor cores; dequantized values never touch device memory).
//
// Precision.  A single fp16 product would round X and W to 11 significant
// bits.  X arrives split as X_hi + X_lo (two fp16 planes written by the
// producing kernel) and each weight w = d * (n - 8) (or d * q) is split as
// w_hi + w_lo in fp16 while dequantizing; three MMAs per K step accumulate
//   X_hi W_hi + X_lo W_hi + X_hi W_lo
// in fp32 (the dropped X_lo W_lo term is ~2^-22 relative).
//
// Tile 128 (rows of X) x 256 (rows of W) x 64 (K), two stages in shared
// memory, SWIZZLE_128B K-major operand layout:
//   warp 0      : TMA producer for the X_hi / X_lo tiles (cp.async.bulk.tensor.2d)
//   warp 1      : TMEM allocation; one lane issues the MMAs and commits
//   warps 2..9  : dequantize the W tile (one weight row per thread) into the
//                 W_hi / W_lo tiles; warps 2..5 then run the fused epilogue
//                 from TMEM (tcgen05.ld, 32 columns at a time).
// Every mbarrier wait is bounded; on a timeout the CTA records DEV_TIMEOUT,
// drains what it issued and frees its TMEM before returning.
#include <cuda.h>

#include "common.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace af {

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 2;
constexpr int kATile = BM * BK * 2;  // 16 KB per fp16 plane
constexpr int kBTile = BN * BK * 2;  // 32 KB per fp16 plane
constexpr int kStageBytes = 2 * kATile + 2 * kBTile;
constexpr int kThreads = 10 * 32;
constexpr int kDequantThreads = 8 * 32;  // == BN: one weight row per thread
constexpr int kTmemCols = 256;           // fp32 accumulator, BN columns
constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack

static_assert(kDequantThreads == BN, "one dequant thread per weight row");

// Instruction descriptor of this GEMM's tile.
constexpr uint32_t kIdesc = idesc_f16(BM, BN);

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

struct TcSmem {
    uint64_t full_a[kStages];  // X tiles landed (TMA transaction bytes)
    uint64_t full_b[kStages];  // W tiles written (kDequantThreads arrivals)
    uint64_t empty[kStages];   // MMAs reading the stage finished (commit)
    uint64_t done;             // all MMAs finished (commit)
    uint32_t tmem_base;
    volatile int abort;
    int issued_a;  // X tile loads issued so far
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, unsigned parity, TcSmem& sm, unsigned* err) {
    for (unsigned i = 0; i < kWaitLimit; i++) {
        if (mbar_try_wait(bar, parity)) return true;
        if (sm.abort) return false;
    }
    sm.abort = 1;
    atomicExch(err, (unsigned)DEV_TIMEOUT);
    return false;
}

template <int WT>
__global__ void __launch_bounds__(kThreads, 1)
    qgemm_tc_kernel(const __grid_constant__ CUtensorMap map_hi, const __grid_constant__ CUtensorMap map_lo, Planes W,
                    int M, Epi epi, unsigned* err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ TcSmem sm;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int nk = (W.K + BK - 1) / BK;

    if (tid == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&sm.full_a[s], 1);
            mbar_init(&sm.full_b[s], kDequantThreads);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.done, 1);
        sm.abort = 0;
        sm.issued_a = 0;
        fence_mbar_init();
    }
    if (warp == 1) {  // TMEM accumulator (whole warp)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    auto a_hi = [&](int s) { return smem + s * kStageBytes; };
    auto a_lo = [&](int s) { return smem + s * kStageBytes + kATile; };
    auto b_hi = [&](int s) { return smem + s * kStageBytes + 2 * kATile; };
    auto b_lo = [&](int s) { return smem + s * kStageBytes + 2 * kATile + kBTile; };

    if (warp == 0) {
        // ---------------- TMA producer: X_hi, X_lo tiles
        if (lane == 0) {
            for (int ks = 0; ks < nk; ks++) {
                const int s = ks % kStages, u = ks / kStages;
                if (u > 0 && !wait_or_abort(&sm.empty[s], (u - 1) & 1, sm, err)) break;
                mbar_arrive_expect_tx(&sm.full_a[s], 2 * kATile);
                tma_load_2d(a_hi(s), &map_hi, ks * BK, m0, &sm.full_a[s]);
                tma_load_2d(a_lo(s), &map_lo, ks * BK, m0, &sm.full_a[s]);
                sm.issued_a = ks + 1;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            for (int ks = 0; ks < nk; ks++) {
                const int s = ks % kStages, u = ks / kStages;
                if (!wait_or_abort(&sm.full_a[s], u & 1, sm, err)) break;
                if (!wait_or_abort(&sm.full_b[s], u & 1, sm, err)) break;
                tc_fence_after();
                const uint32_t ah = smem_u32(a_hi(s)), al = smem_u32(a_lo(s));
                const uint32_t bh = smem_u32(b_hi(s)), bl = smem_u32(b_lo(s));
#pragma unroll
                for (int kk = 0; kk < BK / 16; kk++) {  // 16 fp16 = 32 bytes along K per MMA
                    const uint32_t off = kk * 32;
                    const uint32_t acc = (ks > 0 || kk > 0) ? 1u : 0u;
                    mma_f16(tmem, umma_desc_sw128(ah + off), umma_desc_sw128(bh + off), kIdesc, acc);
                    mma_f16(tmem, umma_desc_sw128(al + off), umma_desc_sw128(bh + off), kIdesc, 1u);
                    mma_f16(tmem, umma_desc_sw128(ah + off), umma_desc_sw128(bl + off), kIdesc, 1u);
                }
                mma_commit(&sm.empty[s]);  // frees the stage when these MMAs complete
            }
            mma_commit(&sm.done);  // always: also after a break, so the drain can wait on it
        }
    } else {
        // ---------------- dequantize W rows into the fp16 hi / lo tiles
        const int r = tid - 64;  // 0..255: weight row n0 + r
        const int n = n0 + r;
        const int64_t pitch = W.qs_pitch();
        const int scp = W.sc_pitch();
        for (int ks = 0; ks < nk; ks++) {
            const int s = ks % kStages, u = ks / kStages;
            if (u > 0 && !wait_or_abort(&sm.empty[s], (u - 1) & 1, sm, err)) break;
            float w[64];
            if (n < W.N) {
                const int kb = ks * 2;  // two 32-weight blocks per K step
#pragma unroll
                for (int b = 0; b < 2; b++) {
                    const float d = __half2float(W.sc[(int64_t)n * scp + kb + b]);
                    const uint8_t* q = W.qs + (int64_t)n * pitch + (int64_t)(kb + b) * W.qb();
                    if (WT == AF_Q8_0) {
                        const uint4 q0 = *reinterpret_cast<const uint4*>(q);
                        const uint4 q1 = *reinterpret_cast<const uint4*>(q + 16);
                        const uint32_t ws[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                        for (int j = 0; j < 32; j++) w[b * 32 + j] = d * (float)(int8_t)((ws[j >> 2] >> (8 * (j & 3))) & 0xFF);
                    } else {
                        const uint4 q0 = *reinterpret_cast<const uint4*>(q);
                        const uint32_t ws[4] = {q0.x, q0.y, q0.z, q0.w};
#pragma unroll
                        for (int j = 0; j < 16; j++) {
                            const uint32_t byte = (ws[j >> 2] >> (8 * (j & 3))) & 0xFF;
                            w[b * 32 + j] = d * (float)((int)(byte & 15) - 8);
                            w[b * 32 + 16 + j] = d * (float)((int)(byte >> 4) - 8);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 64; j++) w[j] = 0.f;
            }
#pragma unroll
            for (int c = 0; c < 8; c++) {
                float w8[8];
#pragma unroll
                for (int e = 0; e < 8; e++) w8[e] = w[8 * c + e];
                uint4 hi, lo;
                split8(w8, hi, lo);
                *reinterpret_cast<uint4*>(b_hi(s) + sw128(r, c)) = hi;
                *reinterpret_cast<uint4*>(b_lo(s) + sw128(r, c)) = lo;
            }
            fence_proxy_async_shared();  // generic-proxy writes -> visible to the tensor core
            mbar_arrive(&sm.full_b[s]);
        }
        // ---------------- epilogue (warps 2..5: TMEM lane quadrant = warp % 4)
        if (warp < 6) {
            // tcgen05.ld below is warp-collective: the whole warp takes the same branch
            if (__all_sync(0xffffffffu, wait_or_abort(&sm.done, 0, sm, err))) {
                tc_fence_after();
                const int quad = warp & 3;
                const int m = m0 + quad * 32 + lane;
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)c0, v);
                    if (m < M) {
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const int nn = n0 + c0 + j;
                            if (nn < W.N) epi_pair(epi, m, nn, v[j], v[j + 1]);
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (sm.abort && tid == 0) {  // let every MMA and copy that was issued finish before leaving
        mbar_wait_bounded(&sm.done, 0);
        // loads older than the last kStages were consumed by the MMA issuer, i.e. complete
        for (int ks = max(0, sm.issued_a - kStages); ks < sm.issued_a; ks++)
            mbar_wait_bounded(&sm.full_a[ks % kStages], (ks / kStages) & 1);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D map over an fp16 [rows][ld] plane, box 64 (K) x 128 (rows), SWIZZLE_128B, zero fill out of bounds.
bool make_map(CUtensorMap* map, const __half* base, int rows, int cols, int64_t ld) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {BK, BM};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t qgemm_prepare() {
    cudaError_t e = cudaFuncSetAttribute(qgemm_tc_kernel<AF_Q4_0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (!e)
        e = cudaFuncSetAttribute(qgemm_tc_kernel<AF_Q8_0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    return e;
}

cudaError_t launch_qgemm(const Planes& W, const __half* X_hi, const __half* X_lo, int64_t ldx, int M, const Epi& epi,
                         unsigned* err, cudaStream_t s) {
    if (M < 1) return cudaSuccess;
    if (ldx % 8 || (reinterpret_cast<uintptr_t>(X_hi) & 15) || (reinterpret_cast<uintptr_t>(X_lo) & 15))
        return cudaErrorInvalidValue;  // TMA: 16-byte aligned base and row stride
    CUtensorMap mh, ml;
    if (!make_map(&mh, X_hi, M, W.K, ldx) || !make_map(&ml, X_lo, M, W.K, ldx)) return cudaErrorInvalidValue;
    dim3 grid((W.N + BN - 1) / BN, (M + BM - 1) / BM);
    if (W.wtype == AF_Q4_0)
        qgemm_tc_kernel<AF_Q4_0><<<grid, kThreads, kSmemBytes, s>>>(mh, ml, W, M, epi, err);
    else
        qgemm_tc_kernel<AF_Q8_0><<<grid, kThreads, kSmemBytes, s>>>(mh, ml, W, M, epi, err);
    return cudaGetLastError();
}

}  // namespace af
