// Decode GEMV: y = W x over repacked Q4_0 / Q8_0 planes, with an optional
// RMSNorm prologue and a fused epilogue (Airframe "GPU_PIPELINE.md" per-layer
// ops: "Dequantization happens inline ... No separate dequantize-then-multiply
// step"; decode is bound by reading the weights, "Decode loop").
//
// Streaming.  One CTA per SM owns a contiguous, even-aligned range of rows
// (N/#SM rows +-2).  Rows are contiguous in the quant and scale planes, so a
// stage of R whole rows is two bulk asynchronous copies (cp.async.bulk,
// mbarrier completion, L2 evict-first) into a shared-memory ring of a few
// stages; one thread keeps the ring full while all warps compute.  The first
// stages are issued before griddepcontrol.wait (the weights do not depend on
// the previous kernel), and the ring is small enough (<= 96 KB, <= 128
// registers/thread) for the next kernel's CTA to be resident and pre-fill
// its own ring while this one drains.
//
// Compute.  Each lane keeps its slice of x (RMS-normalized in the prologue)
// in registers for the whole kernel: the K axis of a row is NC chunks of 32
// sixteen-byte units and warp (rs, wk) owns chunks wk, wk+WK, ... of the rows
// of row stream rs, lane l unit l of each.  Per stage a warp dequantizes its
// units straight from shared memory and reduces its row partials with a
// transpose-reduce; the WK partials of each row are summed in a fixed order
// (deterministic) and the fused epilogue is applied per row pair.
//
// Dot products in integer arithmetic.  In the prologue each lane converts the
// x values of each of its 32-element units (16 for Q8_0) to 24-bit fixed
// point with a per-unit power-of-two scale s (max|x| / s in [2^22, 2^23)):
// x ~= s * xi, error <= s/2, the same order as fp32 rounding of the products
// (and exact for values that fit, e.g. a one-hot x reads a weight exactly).  xi is kept as
// three byte planes (top byte signed), four elements per register, so the
// products with the weight codes are dp4a instructions (3 per 4 weights):
//   Q4_0: code n in 0..15 (nibbles unpacked with 1 LOP3 per 4),
//         sum_j (n_j - 8) x_j = s * (65536 A + 256 B + C) - 8 sum_j x_j
//   Q8_0: code q in -127..127,  sum_j q_j x_j = s * (65536 A + 256 B + C)
// with A, B, C the int32 dp4a sums over the top, middle and low byte planes.
// The block value is d * that, accumulated in fp32 per row.
//
// Every mbarrier wait is bounded; on a timeout the kernel records DEV_TIMEOUT
// in its error word, drains its outstanding copies (bounded) and returns.
#include "common.cuh"
#include "gemv_common.cuh"
#include "tma.cuh"

namespace af {

namespace {

constexpr int kWarps = 16;
constexpr int kMaxCtaRows = 512;  // residual rows a CTA may own (x preloaded to shared memory)






constexpr int kMaxRing = 8;
constexpr int kRingBytes = 160 * 1024;  // stage ring budget (one CTA per SM)

template <int WT, bool NORM, int R, int WK>
__global__ void __launch_bounds__(kWarps * 32, 1)
    qgemv_kernel(Planes W, const float* __restrict__ x, const float* __restrict__ nw, float eps, Epi epi,
                 int ring, unsigned* __restrict__ err) {
    constexpr int UW = Q<WT>::UW;
    constexpr int RS = kWarps / WK;                 // row streams (rows j, j + RS, ... of a stage)
    constexpr int RW = R / RS;                      // rows per warp per stage
    constexpr int UPL = WT == AF_Q4_0 ? 2 : 4;      // chunk slots per warp (NC <= WK * UPL)
    static_assert(RW >= 1 && RS * RW == R, "R must be a multiple of the row streams");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kMaxRing];
    __shared__ unsigned done_cnt[kMaxRing];    // warps finished with the slot's current stage
    __shared__ unsigned issues[kMaxRing];      // copies issued into the slot so far
    __shared__ float red[kMaxRing][kWarps][RW];
    __shared__ float ssum[kWarps];
    __shared__ float xres[kMaxCtaRows];
    __shared__ float2 rope_s[64];
    __shared__ unsigned long long amax_s;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rs = warp / WK, wk = warp % WK;
    const int N = W.N, K = W.K;
    const int NC = W.Kp / (32 * UW);
    const int64_t pitch = W.qs_pitch();
    const int scp = W.sc_pitch();
    const int qstage = R * (int)pitch;
    const int stage_bytes = (qstage + R * scp * 2 + 127) & ~127;
    const int np = N / 2;
    const int pa = (int)((int64_t)np * blockIdx.x / gridDim.x), pb = (int)((int64_t)np * (blockIdx.x + 1) / gridDim.x);
    const int r0 = 2 * pa, nrows = 2 * (pb - pa);
    const int nst = (nrows + R - 1) / R;

    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < ring; s++) {
            mbar_init(&full[s], 1);
            done_cnt[s] = 0;
            issues[s] = 0;
        }
        abort_flag = 0;
        amax_s = 0ull;
        fence_mbar_init();
    }
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int st) {  // one thread: stage st (rows r0 + st*R ..) into its slot
        const int slot = st % ring;
        const int ra = r0 + st * R, nr = min(R, r0 + nrows - ra);
        const unsigned qb = (unsigned)(nr * pitch), sb = (unsigned)(nr * scp * 2);
        uint8_t* dst = smem + slot * stage_bytes;
        issues[slot]++;
        mbar_arrive_expect_tx(&full[slot], qb + sb);
        bulk_g2s_evict_first(dst, W.qs + (int64_t)ra * pitch, qb, &full[slot], pol);
        bulk_g2s_evict_first(dst + qstage, W.sc + (int64_t)ra * scp, sb, &full[slot], pol);
    };
    if (tid == 0)
        for (int st = 0; st < min(nst, ring); st++) issue(st);

    pdl_wait();  // x (and the residual rows) are written by the previous kernel

    float rstd = 1.f;
    if (NORM) {  // RMSNorm prologue: every CTA reduces sum(x^2) over the whole input
        float ss = 0.f;
        const float4* x4 = reinterpret_cast<const float4*>(x);
        for (int k4 = tid; k4 < K / 4; k4 += kWarps * 32) {
            const float4 v = x4[k4];
            ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
        }
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) ssum[warp] = ss;
    }
    // epilogue inputs into shared memory
    if (epi.kind == EPI_RESID)
        for (int i = tid; i < nrows; i += kWarps * 32) xres[i] = epi.out[r0 + i];
    GemvEpiCtx ectx;
    ectx.xres = xres;
    ectx.rope = rope_s;
    ectx.amax = &amax_s;
    ectx.r0 = r0;
    ectx.pos = 0;
    if (epi.kind == EPI_QKV) {
        ectx.pos = epi.pos_dev ? *epi.pos_dev : epi.pos0;
        for (int i = tid; i < epi.head_dim / 2; i += kWarps * 32)
            rope_s[i] = epi.rope[(int64_t)ectx.pos * (epi.head_dim / 2) + i];
    }
    __syncthreads();
    if (NORM) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < kWarps; i++) t += ssum[i];
        rstd = rsqrtf(t / (float)K + eps);
    }

    // this lane's x slices (chunk wk + WK*u, unit lane) in 24-bit fixed point
    XUnit<UW / 4> xq[UPL];
#pragma unroll
    for (int u = 0; u < UPL; u++) {
        const int c = wk + WK * u;
        const int k0 = (c * 32 + lane) * UW;
        float xs[UW];
        if (c < NC && k0 < K) {
#pragma unroll
            for (int e = 0; e < UW; e += 4) {
                float4 v = *reinterpret_cast<const float4*>(x + k0 + e);
                if (NORM) {
                    const float4 g = *reinterpret_cast<const float4*>(nw + k0 + e);
                    v = make_float4(g.x * (v.x * rstd), g.y * (v.y * rstd), g.z * (v.z * rstd), g.w * (v.w * rstd));
                }
                xs[e] = v.x;
                xs[e + 1] = v.y;
                xs[e + 2] = v.z;
                xs[e + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < UW; e++) xs[e] = 0.f;
        }
        quantize_unit<UW>(xs, xq[u]);
    }

    // main loop: warps run independently; the last warp to finish a stage combines
    // the row partials, applies the epilogue and refills the slot
    for (int st = 0; st < nst; st++) {
        const int slot = st % ring;
        const unsigned par = (unsigned)((st / ring) & 1);
        bool ok = false;
        for (unsigned it = 0; it < kWaitLimit && !ok; it++) {
            ok = mbar_try_wait(&full[slot], par);
            if (!ok && abort_flag) break;
        }
        if (!ok) {
            if (lane == 0) {
                abort_flag = 1;
                atomicExch(err, (unsigned)DEV_TIMEOUT);
            }
            break;
        }
        const uint8_t* qsm = smem + slot * stage_bytes;
        const unsigned short* ssm = reinterpret_cast<const unsigned short*>(qsm + qstage);
        const int ra = r0 + st * R, nr = min(R, r0 + nrows - ra);
        float acc[RW];
#pragma unroll
        for (int t = 0; t < RW; t++) {
            const int j = rs + RS * t;
            acc[t] = 0.f;
            if (j < nr) {
#pragma unroll
                for (int u = 0; u < UPL; u++) {
                    const int c = wk + WK * u;
                    if (c < NC) {
                        const int unit = c * 32 + lane;
                        const uint4 q = *reinterpret_cast<const uint4*>(qsm + j * pitch + unit * 16);
                        const float d = __half2float(__ushort_as_half(ssm[j * scp + (WT == AF_Q8_0 ? unit >> 1 : unit)]));
                        acc[t] = fmaf(d, Q<WT>::dot(q, xq[u]), acc[t]);
                    }
                }
            }
        }
        const float r = transpose_reduce<RW>(acc, lane);
        if ((lane & (32 / RW - 1)) == 0) red[slot][warp][lane / (32 / RW)] = r;
        __syncwarp();
        unsigned last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&done_cnt[slot], 1u) == (unsigned)kWarps - 1u;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {  // every warp is done with this slot
            __threadfence_block();
            if (lane < nr / 2) {  // rows (2 lane, 2 lane + 1) of the stage
                float y[2];
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int j = 2 * lane + h, jrs = j % RS, jt = j / RS;
                    float a = 0.f;
#pragma unroll
                    for (int w = 0; w < WK; w++) a += red[slot][jrs * WK + w][jt];
                    y[h] = a;
                }
                gemv_epi(epi, ectx, ra + 2 * lane, y[0], y[1]);
            }
            __syncwarp();
            if (lane == 0) {
                done_cnt[slot] = 0;
                if (st + ring < nst) {
                    fence_proxy_async_shared();
                    issue(st + ring);
                }
            }
        }
    }
    __syncthreads();
    if (abort_flag) {  // drain every copy still in flight before the CTA exits
        if (tid == 0)
            for (int s = 0; s < ring; s++)
                if (issues[s]) mbar_wait_bounded(&full[s], (issues[s] - 1u) & 1u);
        __syncthreads();
        return;
    }
    if (epi.kind == EPI_LOGITS && tid == 0 && amax_s) atomicMax(epi.argmax, amax_s);
}

struct Shape {
    int R, WK, ring, stage_bytes;
};

Shape pick_shape(const Planes& W) {
    const int UW = W.wtype == AF_Q8_0 ? 16 : 32;
    const int NC = W.Kp / (32 * UW);
    Shape s;
    s.WK = NC >= 8 ? 8 : (NC > 4 ? 8 : (NC > 2 ? 4 : NC));
    const int RS = kWarps / s.WK;
    const int row_bytes = (int)W.qs_pitch() + W.sc_pitch() * 2;
    s.R = 32;
    while (s.R > RS && s.R * row_bytes > 40 * 1024) s.R /= 2;
    s.stage_bytes = (s.R * (int)W.qs_pitch() + s.R * W.sc_pitch() * 2 + 127) & ~127;
    s.ring = kRingBytes / s.stage_bytes;
    s.ring = s.ring < 2 ? 2 : (s.ring > kMaxRing ? kMaxRing : s.ring);
    return s;
}

template <int WT, bool NORM, int R, int WK>
cudaError_t launch_t(const Planes& W, const float* x, const float* nw, float eps, const Epi& epi, const Shape& sh,
                     unsigned* err, cudaStream_t s) {
    auto kern = qgemv_kernel<WT, NORM, R, WK>;
    const size_t smem = (size_t)sh.ring * sh.stage_bytes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms());
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, W, x, nw, eps, epi, sh.ring, err);
}

template <int WT, bool NORM>
cudaError_t dispatch(const Planes& W, const float* x, const float* nw, float eps, const Epi& epi, unsigned* err,
                     cudaStream_t s) {
    const Shape sh = pick_shape(W);
#define AF_GEMV_CASE(RR, WW) \
    if (sh.R == RR && sh.WK == WW) return launch_t<WT, NORM, RR, WW>(W, x, nw, eps, epi, sh, err, s);
    AF_GEMV_CASE(16, 1)
    AF_GEMV_CASE(32, 1)
    AF_GEMV_CASE(8, 2)
    AF_GEMV_CASE(16, 2)
    AF_GEMV_CASE(32, 2)
    AF_GEMV_CASE(4, 4)
    AF_GEMV_CASE(8, 4)
    AF_GEMV_CASE(16, 4)
    AF_GEMV_CASE(32, 4)
    AF_GEMV_CASE(2, 8)
    AF_GEMV_CASE(4, 8)
    AF_GEMV_CASE(8, 8)
    AF_GEMV_CASE(16, 8)
    AF_GEMV_CASE(32, 8)
#undef AF_GEMV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t qgemv_prepare() {
    // every instantiation may use up to kRingBytes of dynamic shared memory (its stage ring); done once,
    // outside any stream capture
    static bool done = false;
    if (done) return cudaSuccess;
    const int smem = kRingBytes;
    cudaError_t e = cudaSuccess;
#define AF_GEMV_ATTR(WT, NORM, RR, WW) \
    if (!e) e = cudaFuncSetAttribute(qgemv_kernel<WT, NORM, RR, WW>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
#define AF_GEMV_ATTR4(RR, WW)                 \
    AF_GEMV_ATTR(AF_Q4_0, true, RR, WW)       \
    AF_GEMV_ATTR(AF_Q4_0, false, RR, WW)      \
    AF_GEMV_ATTR(AF_Q8_0, true, RR, WW)       \
    AF_GEMV_ATTR(AF_Q8_0, false, RR, WW)
    AF_GEMV_ATTR4(16, 1)
    AF_GEMV_ATTR4(32, 1)
    AF_GEMV_ATTR4(8, 2)
    AF_GEMV_ATTR4(16, 2)
    AF_GEMV_ATTR4(32, 2)
    AF_GEMV_ATTR4(4, 4)
    AF_GEMV_ATTR4(8, 4)
    AF_GEMV_ATTR4(16, 4)
    AF_GEMV_ATTR4(32, 4)
    AF_GEMV_ATTR4(2, 8)
    AF_GEMV_ATTR4(4, 8)
    AF_GEMV_ATTR4(8, 8)
    AF_GEMV_ATTR4(16, 8)
    AF_GEMV_ATTR4(32, 8)
#undef AF_GEMV_ATTR4
#undef AF_GEMV_ATTR
    if (!e) done = true;
    return e;
}

int qgemv_max_chunks() { return 32; }


cudaError_t launch_qgemv(const Planes& W, const float* x, const float* norm_w, float eps, const Epi& epi,
                         const GemvScratch& scr, cudaStream_t s) {
    if (W.wtype == AF_Q4_0)
        return norm_w ? dispatch<AF_Q4_0, true>(W, x, norm_w, eps, epi, scr.err, s)
                      : dispatch<AF_Q4_0, false>(W, x, norm_w, eps, epi, scr.err, s);
    return norm_w ? dispatch<AF_Q8_0, true>(W, x, norm_w, eps, epi, scr.err, s)
                  : dispatch<AF_Q8_0, false>(W, x, norm_w, eps, epi, scr.err, s);
}

}  // namespace af
