// Decode GEMV: y = W x over repacked Q4_0 / Q8_0 / Q4_K / Q5_K / Q6_K rows, with an optional
// RMSNorm prologue and a fused epilogue (Airframe "GPU_PIPELINE.md" per-layer
// ops: dequantization happens inside the matmul, no separate dequantize pass;
// decode is bound by reading the weights, "Decode loop").
//
// Streaming.  One CTA of 16 warps per SM owns a contiguous, even-aligned range
// of rows.  Rows are contiguous in the quant and scale planes, so a stage of R
// whole rows (scales included) is one bulk asynchronous copy (cp.async.bulk, mbarrier
// completion, L2 evict-first) into a shared-memory ring; the warp that
// finishes a stage last refills its slot.  The first stages are issued before
// griddepcontrol.wait (weights do not depend on the previous kernel), so the
// ring (up to 112 KB, so that the CTAs of the kernels before and after it can
// be resident on the same SM) fills while the prologue runs.
//
// Activations.  The prologue (all threads) reads x once: it reduces sum(x^2)
// for the optional RMSNorm and converts w (.) x (the norm weight times x; the
// scalar RMS factor is applied to each row's result), 32 elements at a time,
// to 16-bit fixed point with a
// power-of-two scale per block: x_j ~= s * xi_j, |xi_j| <= 32767 (relative
// error <= 2^-16 of the block maximum).  The integers are stored in shared
// memory as two byte planes (high byte signed, low byte unsigned; four
// elements per word), and each lane copies the planes of the units it owns
// into registers once.
//
// Compute.  The K axis of a row is NC chunks of 32 sixteen-byte units; all 16
// warps work on every stage: warp (rs, wk) owns chunks wk, wk+WK, ... of the
// row pairs rs, rs+RS, ... (RS x WK = 16), lane l unit l of each chunk.
// Products with the weight codes are dp4a instructions:
//   Q4_0: code n in 0..15; lo = w & 0x0F0F0F0F, hi = w & 0xF0F0F0F0 (= 16 n),
//         sum_j n_j xi_j = (4096 A + 256 C + 16 B + D) / 16 over the byte planes,
//         sum_j (n_j - 8) x_j = s * that - 8 s sum_j xi_j
//   Q8_0: code q in -127..127, sum_j q_j x_j = s * (256 A + B)
//   Q4_K / Q5_K / Q6_K: 4-, 5- or 6-bit codes (nibble, or nibble | high bits << 4)
//         per 32-weight unit, with the sub-block scale (and min) from the row's
//         super-block record applied in fp32 (the Unit specializations below)
// accumulated exactly in int32 per unit; the unit value times the block's
// scale is accumulated in fp32 per row.  Row partials are reduced over
// the lanes with a transpose-reduce; with WK > 1 the WK partials of a row are
// summed in a fixed order (deterministic) by the last warp of the stage.
//
// Shared memory.  Stages of about 24 KB (the rows that make it), several in
// flight; the x images live in the last ring slots, which are filled only
// after every lane has copied its x units into registers.
//
// A second kernel, qgemv_pw_kernel, serves the shapes where it measured faster
// (few rows per CTA that all fit in shared memory, and the LM head): each
// stage of R whole rows belongs to one warp, in a slot that warp owns; the warp
// waits for it, computes its R rows over the whole K with the x units read from
// the shared image, refills the slot and applies the epilogue, with no
// cross-warp reduction.
//
// Every mbarrier wait is bounded; on a timeout the kernel records DEV_TIMEOUT
// in its error word, drains its outstanding copies (bounded) and returns.
#pragma once
#include "common.cuh"
#include "gemv_common.cuh"
#include "tma.cuh"

namespace af {

// per-type entry points, one translation unit each (qgemv_<type>.cu)
template <int WT>
cudaError_t qgemv_dispatch(const Planes& W, const float* x, const float* norm_w, float eps, const Epi& epi,
                           unsigned* err, cudaStream_t s);
template <int WT>
cudaError_t qgemv_set_attrs();

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxCtaRows = 512;        // residual rows a CTA may own (preloaded to shared memory)
constexpr int kMaxRing = 12;
constexpr int kRingBudget = 112 * 1024;  // ring, x images inside: room beside it for the neighbouring kernels' CTAs
constexpr int kMinStage = 24 * 1024;     // stage size target: enough work per warp between waits
constexpr int kMaxStage = 64 * 1024;     // largest stage that still leaves three in the ring
constexpr int kMaxGemvSmem = 208 * 1024;
// per-warp kernel (qgemv_pw_kernel)
constexpr int kPwMaxSlots = 2 * kWarps;
constexpr int kPwSlotMax = 24 * 1024;      // stage size bound for streamed matrices (16-24 KB copies)
constexpr int kPwMaxSmem = 216 * 1024;     // x image + slots (one CTA per SM)

__host__ __device__ constexpr int pw_ximage_bytes(int Kp) { return ((Kp / 32) * kXBlkBytes + 127) & ~127; }

template <int WT>
__host__ __device__ constexpr int units_per_lane() { return WT == AF_Q8_0 ? 8 : 4; }


template <int WT, bool NORM, int WK, int PPW>
__global__ void __launch_bounds__(kThreads, 1)
    qgemv_kernel(Planes W, const float* __restrict__ x, const float* __restrict__ nw, float eps, Epi epi, int ring,
                 int xslot, unsigned* __restrict__ err) {
    constexpr int UPL = units_per_lane<WT>();
    constexpr int RS = kWarps / WK;  // row-pair streams
    constexpr int RW = 2 * PPW;      // rows per warp per stage (PPW row pairs)
    constexpr int R = RS * RW;       // rows per stage
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kMaxRing];
    __shared__ unsigned done_cnt[kMaxRing];  // warps finished with the slot's current stage
    __shared__ unsigned issues[kMaxRing];    // copies issued into the slot so far
    __shared__ float red[kMaxRing][kWarps][RW];
    __shared__ float ssum[kWarps];
    __shared__ float xres[kMaxCtaRows];
    __shared__ float2 rope_s[64];
    __shared__ unsigned long long amax_s;
    __shared__ volatile int abort_flag;
    __shared__ uint64_t never;  // an mbarrier nothing arrives on (the error path's test hook, below)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rs = warp / WK, wk = warp % WK;
    const int N = W.N, K = W.K;
    const int UW = WT == AF_Q8_0 ? 16 : 32;  // weights per unit
    const int NC = W.Kp / (32 * UW);
    const int64_t pitch = W.qs_pitch();
    const int sc_off = W.sc_off(), hb_off = W.hb_off();
    const int stage_bytes = (R * (int)pitch + 127) & ~127;
    // x images at the end of the ring: slots xslot.. are filled after the prologue
    const int xbytes = (W.Kp / 32) * kXBlkBytes;
    XBlk* xb = reinterpret_cast<XBlk*>(smem + ((ring * stage_bytes - xbytes) & ~127));
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
        mbar_init(&never, 1);
        fence_mbar_init();
    }
    // err[1] != 0 (test instrumentation): the first stage wait polls `never` that many times, gives up and takes
    // the timeout path (error code, drain of the copies in flight, early return) exactly as a real timeout would
    const unsigned stall = err[1];
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int st) {  // one thread: stage st (rows r0 + st*R ..) into its slot
        const int slot = st % ring;
        const int ra = r0 + st * R, nr = min(R, r0 + nrows - ra);
        const unsigned bytes = (unsigned)(nr * pitch);  // rows ra.. with their scales: one range
        uint8_t* dst = smem + slot * stage_bytes;
        issues[slot]++;
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s_evict_first(dst, W.qs + (int64_t)ra * pitch, bytes, &full[slot], pol);
    };
    if (tid == 0)
        for (int st = 0; st < min(nst, xslot); st++) issue(st);
    // the position word is written before the step's first kernel starts and the RoPE table never: both are
    // read before waiting for the previous kernel
    int qpos = 0;
    if (epi.kind == EPI_QKV) {
        qpos = epi.pos_dev ? __ldcg(epi.pos_dev) : epi.pos0;
        for (int i = tid; i < epi.head_dim / 2; i += kThreads) rope_s[i] = epi.rope[(int64_t)qpos * (epi.head_dim / 2) + i];
    }

    pdl_wait();  // x (and the residual rows) are written by the previous kernel

    // RMSNorm prologue: every CTA reduces sum(x^2) over the whole input while it converts w (.) x
    float ss = quantize_x<NORM, kThreads, true>(x, nw, K, W.Kp / 32, xb, tid);
    if (NORM) {
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) ssum[warp] = ss;
    }
    // epilogue inputs into shared memory
    if (epi.kind == EPI_RESID)
        for (int i = tid; i < nrows; i += kThreads) xres[i] = __ldcg(epi.out + r0 + i);
    GemvEpiCtx ectx;
    ectx.xres = xres;
    ectx.rope = rope_s;
    ectx.amax = &amax_s;
    ectx.r0 = r0;
    ectx.pos = 0;
    ectx.pos = qpos;
    __syncthreads();

    float rstd = 1.f;  // applied to each row's dot product (the images hold w (.) x)
    if (NORM) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < kWarps; i++) t += ssum[i];
        rstd = rsqrtf(t / (float)K + eps);
    }
    // this lane's x units: chunk wk + WK*u, unit lane
    Unit<WT> xr[UPL];
#pragma unroll
    for (int u = 0; u < UPL; u++) {
        const int c = wk + WK * u;
        if (c < NC) xr[u].load(xb, c * 32 + lane);
    }
    __syncthreads();  // the x images are dead: their slots take stages now
    if (tid == 0) {
        fence_proxy_async_shared();  // generic-proxy accesses of those bytes before the copies overwrite them
        for (int st = xslot; st < min(nst, ring); st++) issue(st);
    }

    for (int st = 0; st < nst; st++) {
        const int slot = st % ring;
        const unsigned par = (unsigned)((st / ring) & 1);
        bool ok = false;
        uint64_t* bar = (stall && st == 0) ? &never : &full[slot];
        const unsigned lim = (stall && st == 0) ? stall : kWaitLimit;
        for (unsigned it = 0; it < lim && !ok; it++) {
            ok = mbar_try_wait(bar, par);
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
        const int ra = r0 + st * R, nr = min(R, r0 + nrows - ra);
        float acc[RW];
#pragma unroll
        for (int t = 0; t < RW; t++) acc[t] = 0.f;
#pragma unroll
        for (int p = 0; p < PPW; p++) {
            const int j0 = 2 * (rs + RS * p);  // rows j0, j0 + 1 of the stage
            if (j0 < nr) {
#pragma unroll
                for (int u = 0; u < UPL; u++) {
                    const int c = wk + WK * u;
                    if (c < NC) {
                        const int unit = c * 32 + lane;
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            const uint8_t* row = qsm + (j0 + h) * pitch;
                            if constexpr (WT == AF_Q5_K || WT == AF_Q6_K)
                                acc[2 * p + h] = xr[u].accumulate(row, sc_off, hb_off, unit, acc[2 * p + h]);
                            else
                                acc[2 * p + h] = xr[u].accumulate(row, sc_off, unit, acc[2 * p + h]);
                        }
                    }
                }
            }
        }
        // lanes (32/RW)*t .. hold the sum of acc[t]
        const float r = transpose_reduce<RW>(acc, lane);
        if (WK == 1) {
            const float r1 = __shfl_down_sync(0xffffffffu, r, 32 / RW);
            if (lane % (64 / RW) == 0) {
                const int p = lane / (64 / RW), j0 = 2 * (rs + RS * p);
                if (j0 < nr) gemv_epi(epi, ectx, ra + j0, r * rstd, r1 * rstd);
            }
        } else {
            if ((lane & (32 / RW - 1)) == 0) red[slot][warp][lane / (32 / RW)] = r;
        }
        __syncwarp();
        unsigned last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&done_cnt[slot], 1u) == (unsigned)kWarps - 1u;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {  // every warp is done with this slot
            __threadfence_block();
            if (WK > 1 && lane < nr / 2) {  // row pair `lane` of the stage
                const int prs = lane % RS, pp = lane / RS;
                float y[2];
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    float a = 0.f;
#pragma unroll
                    for (int w = 0; w < WK; w++) a += red[slot][prs * WK + w][2 * pp + h];
                    y[h] = a;
                }
                gemv_epi(epi, ectx, ra + 2 * lane, y[0] * rstd, y[1] * rstd);
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

// ---------------------------------------------------------------- per-warp kernel
template <int WT, bool NORM, int R>
__global__ void __launch_bounds__(kThreads, 1)
    qgemv_pw_kernel(Planes W, const float* __restrict__ x, const float* __restrict__ nw, float eps, Epi epi, int nslot,
                 int slot_bytes, unsigned* __restrict__ err) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[kPwMaxSlots];
    __shared__ unsigned issues[kPwMaxSlots];  // copies issued into the slot so far
    __shared__ float ssum[kWarps];
    __shared__ float xres[kMaxCtaRows];
    __shared__ float2 rope_s[64];
    __shared__ unsigned long long amax_s;
    __shared__ volatile int abort_flag;
    __shared__ uint64_t never;  // an mbarrier nothing arrives on (the error path's test hook, below)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = W.N, K = W.K;
    constexpr int UW = WT == AF_Q8_0 ? 16 : 32;  // weights per unit
    const int NC = W.Kp / (32 * UW);              // chunks of 32 units (one per lane)
    const int64_t pitch = W.qs_pitch();
    const int sc_off = W.sc_off(), hb_off = W.hb_off();
    // x image first, then the slots
    XBlk* xb = reinterpret_cast<XBlk*>(smem);
    uint8_t* ring = smem + pw_ximage_bytes(W.Kp);
    const int np = N / 2;
    const int pa = (int)((int64_t)np * blockIdx.x / gridDim.x), pb = (int)((int64_t)np * (blockIdx.x + 1) / gridDim.x);
    const int r0 = 2 * pa, nrows = 2 * (pb - pa);
    const int nst = (nrows + R - 1) / R;
    // consumer warps and slots per warp: stage s belongs to warp s % WC; its i-th stage (s = warp + WC i) lives
    // in slot warp + WC (i % S), so every slot has one owner, which waits its phases in order and refills it
    const int WC = nslot < kWarps ? nslot : kWarps;
    const int S = nslot / WC;

    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < nslot; s++) {
            mbar_init(&full[s], 1);
            issues[s] = 0;
        }
        abort_flag = 0;
        amax_s = 0ull;
        mbar_init(&never, 1);
        fence_mbar_init();
    }
    // err[1] != 0 (test instrumentation): warp 0's first stage wait polls `never` that many times, gives up and
    // takes the timeout path (error code, drain of the copies in flight, early return) exactly as a real timeout
    const unsigned stall = err[1];
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int st, int slot) {  // one thread: rows r0 + st*R .. with their scales, one range
        const int ra = r0 + st * R, nr = min(R, r0 + nrows - ra);
        const unsigned bytes = (unsigned)(nr * pitch);
        issues[slot]++;
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s_evict_first(ring + (size_t)slot * slot_bytes, W.qs + (int64_t)ra * pitch, bytes, &full[slot], pol);
    };
    // the first stage of every slot: weights do not depend on the previous kernel
    if (tid == 0)
        for (int st = 0; st < min(nst, nslot); st++) issue(st, st);
    // the position word is written before the step's first kernel starts and the RoPE table never: both are
    // read before waiting for the previous kernel
    int qpos = 0;
    if (epi.kind == EPI_QKV) {
        qpos = epi.pos_dev ? __ldcg(epi.pos_dev) : epi.pos0;
        for (int i = tid; i < epi.head_dim / 2; i += kThreads) rope_s[i] = epi.rope[(int64_t)qpos * (epi.head_dim / 2) + i];
    }

    pdl_wait();  // x (and the residual rows) are written by the previous kernel

    // RMSNorm prologue: every CTA reduces sum(x^2) over the whole input while it converts w (.) x
    float ss = quantize_x<NORM, kThreads, true>(x, nw, K, W.Kp / 32, xb, tid);
    if (NORM) {
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) ssum[warp] = ss;
    }
    // epilogue inputs into shared memory
    if (epi.kind == EPI_RESID)
        for (int i = tid; i < nrows; i += kThreads) xres[i] = __ldcg(epi.out + r0 + i);
    GemvEpiCtx ectx;
    ectx.xres = xres;
    ectx.rope = rope_s;
    ectx.amax = &amax_s;
    ectx.r0 = r0;
    ectx.pos = 0;
    ectx.pos = qpos;
    __syncthreads();

    float rstd = 1.f;  // applied to each row's dot product (the image holds w (.) x)
    if (NORM) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < kWarps; i++) t += ssum[i];
        rstd = rsqrtf(t / (float)K + eps);
    }

    if (warp < WC) {
        for (int i = 0;; i++) {
            const int st = warp + WC * i;
            if (st >= nst) break;
            const int slot = warp + WC * (i % S);
            const unsigned par = (unsigned)((i / S) & 1);
            bool ok = false;
            uint64_t* bar = (stall && warp == 0 && i == 0) ? &never : &full[slot];
            const unsigned lim = (stall && warp == 0 && i == 0) ? stall : kWaitLimit;
            for (unsigned it = 0; it < lim && !ok; it++) {
                ok = mbar_try_wait(bar, par);
                if (!ok && abort_flag) break;
            }
            if (!ok) {
                if (lane == 0) {
                    abort_flag = 1;
                    atomicExch(err, (unsigned)DEV_TIMEOUT);
                }
                break;
            }
            const uint8_t* sm = ring + (size_t)slot * slot_bytes;
            const int ra = r0 + st * R, nr = min(R, r0 + nrows - ra);
            float acc[R];
#pragma unroll
            for (int r = 0; r < R; r++) acc[r] = 0.f;
            for (int c = 0; c < NC; c++) {
                const int unit = c * 32 + lane;
                Unit<WT> xu;
                xu.load(xb, unit);
#pragma unroll
                for (int r = 0; r < R; r++) {
                    if (r < nr) {  // warp-uniform
                        if constexpr (WT == AF_Q5_K || WT == AF_Q6_K)
                            acc[r] = xu.accumulate(sm + r * pitch, sc_off, hb_off, unit, acc[r]);
                        else
                            acc[r] = xu.accumulate(sm + r * pitch, sc_off, unit, acc[r]);
                    }
                }
            }
            __syncwarp();  // every lane is done reading the slot
            if (lane == 0 && st + WC * S < nst) {
                fence_proxy_async_shared();  // generic-proxy reads of the slot before the copy overwrites it
                issue(st + WC * S, slot);
            }
            // lanes (32/R)*t .. hold the sum of acc[t]; lane (64/R)*p applies row pair p
            const float rv = transpose_reduce<R>(acc, lane);
            const float rv1 = __shfl_down_sync(0xffffffffu, rv, 32 / R);
            if (lane % (64 / R) == 0) {
                const int j0 = 2 * (lane / (64 / R));
                if (j0 < nr) gemv_epi(epi, ectx, ra + j0, rv * rstd, rv1 * rstd);
            }
        }
    }
    __syncthreads();
    if (abort_flag) {  // drain every copy still in flight before the CTA exits
        if (tid == 0)
            for (int s = 0; s < nslot; s++)
                if (issues[s]) mbar_wait_bounded(&full[s], (issues[s] - 1u) & 1u);
        __syncthreads();
        return;
    }
    if (epi.kind == EPI_LOGITS && tid == 0 && amax_s) atomicMax(epi.argmax, amax_s);
}

struct PwShape {
    int R, nslot, slot_bytes, smem;
};

// Rows per stage R (2, 4 or 8) and slots of the per-warp kernel.  When one CTA's rows fit in shared memory at once
// (the QKV and O shapes), R spreads them over about all warps and every stage is issued before the previous kernel
// ends; otherwise (the LM head's hundreds of rows per CTA) stages of 16-24 KB stream through as many slots as fit.
PwShape pw_pick_shape(const Planes& W, int grid) {
    const int pitch = (int)W.qs_pitch();
    const int xbytes = pw_ximage_bytes(W.Kp);
    const int budget = kPwMaxSmem - xbytes;
    const int cta_rows = 2 * ((W.N / 2 + grid - 1) / grid);
    PwShape s;
    if ((int64_t)cta_rows * pitch + kWarps * 128 <= budget) {
        s.R = 2;
        while (s.R < 8 && (cta_rows + s.R - 1) / s.R > kWarps) s.R *= 2;
    } else {
        s.R = 8;
        while (s.R > 2 && s.R * pitch > kPwSlotMax) s.R /= 2;
    }
    s.slot_bytes = (s.R * pitch + 127) & ~127;
    s.nslot = budget / s.slot_bytes;
    if (s.nslot > kWarps) s.nslot = s.nslot >= 2 * kWarps ? 2 * kWarps : kWarps;  // a multiple of the warps
    // rows that fit at once: only the slots their stages take, so the neighbouring kernels of the decode chain
    // (attention, about 100 KB) can be resident on the same SM and start their own copies early
    const int nst = (cta_rows + s.R - 1) / s.R;
    if ((int64_t)cta_rows * pitch + kWarps * 128 <= budget && nst < s.nslot) s.nslot = nst;
    s.smem = xbytes + s.nslot * s.slot_bytes;
    return s;
}

// The per-warp kernel for matrices where it measured faster: few rows per CTA that all fit in shared memory
// (QKV 6144 x 4096: 5.45 against 6.44 us; O 4096 x 4096: equal) and the LM head's many rows per CTA (128256 x
// 4096: 50.8 against 57.5 us).  The ring kernel stays for gate/up (16.1 against 17.1 us) and down (11.2 / 13.3).
bool use_pw(const Planes& W, int grid) {
    const int cta_rows = 2 * ((W.N / 2 + grid - 1) / grid);
    if (cta_rows >= 512) return true;
    return cta_rows <= 64 && (int64_t)cta_rows * W.qs_pitch() + kWarps * 128 <= kPwMaxSmem - pw_ximage_bytes(W.Kp);
}

template <int WT, bool NORM, int R>
cudaError_t pw_launch_t(const Planes& W, const float* x, const float* nw, float eps, const Epi& epi,
                        const PwShape& sh, unsigned* err, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qgemv_pw_kernel<WT, NORM, R>, W, x, nw, eps, epi, sh.nslot, sh.slot_bytes, err);
}

template <int WT, bool NORM>
cudaError_t pw_dispatch(const Planes& W, const float* x, const float* nw, float eps, const Epi& epi, unsigned* err,
                        cudaStream_t s) {
    const PwShape sh = pw_pick_shape(W, num_sms());
    if (sh.nslot < 1 || sh.smem > kPwMaxSmem) return cudaErrorInvalidValue;
    if (epi.kind == EPI_RESID && 2 * ((W.N / 2 + num_sms() - 1) / num_sms()) > kMaxCtaRows) return cudaErrorInvalidValue;
    switch (sh.R) {
        case 2: return pw_launch_t<WT, NORM, 2>(W, x, nw, eps, epi, sh, err, s);
        case 4: return pw_launch_t<WT, NORM, 4>(W, x, nw, eps, epi, sh, err, s);
        default: return pw_launch_t<WT, NORM, 8>(W, x, nw, eps, epi, sh, err, s);
    }
}

struct Shape {
    int WK, PPW, ring, xslot, stage_bytes, smem;
};

Shape pick_shape(const Planes& W) {
    const int UW = W.wtype == AF_Q8_0 ? 16 : 32;
    const int UPL = W.wtype == AF_Q8_0 ? units_per_lane<AF_Q8_0>() : units_per_lane<AF_Q4_0>();
    const int NC = W.Kp / (32 * UW);
    const int row_bytes = (int)W.qs_pitch();
    const int pairs = (kMinStage + 2 * row_bytes - 1) / (2 * row_bytes);  // row pairs for a >= kMinStage stage
    const int xbytes = (W.Kp / 32) * kXBlkBytes;
    int wk_min = 1;  // fewest warps per row that keep a lane's x units within UPL
    while (wk_min < kWarps && NC > wk_min * UPL) wk_min *= 2;
    int RS = 1;
    while (RS < pairs && RS < kWarps / wk_min) RS *= 2;
    if (2 * (kWarps / wk_min) * row_bytes <= kMaxStage) RS = kWarps / wk_min;  // more work per warp per stage
    Shape s;
    s.WK = kWarps / RS;
    s.PPW = 1;
    while (s.PPW < 4 && RS == kWarps && RS * s.PPW < pairs) s.PPW *= 2;
    const int R = 2 * RS * s.PPW;
    s.stage_bytes = (R * row_bytes + 127) & ~127;
    s.ring = kRingBudget / s.stage_bytes;
    s.ring = s.ring > kMaxRing ? kMaxRing : (s.ring < 2 ? 2 : s.ring);
    // at least one slot before the x images (they may push the ring above the budget)
    while (((s.ring * s.stage_bytes - xbytes) & ~127) < s.stage_bytes) s.ring++;
    s.xslot = ((s.ring * s.stage_bytes - xbytes) & ~127) / s.stage_bytes;
    s.smem = s.ring * s.stage_bytes;
    return s;
}

template <int WT, bool NORM, int WK, int PPW>
cudaError_t launch_t(const Planes& W, const float* x, const float* nw, float eps, const Epi& epi, const Shape& sh,
                     unsigned* err, cudaStream_t s) {
    auto kern = qgemv_kernel<WT, NORM, WK, PPW>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, W, x, nw, eps, epi, sh.ring, sh.xslot, err);
}

// (WK, PPW) shapes pick_shape can return (row-pair streams RS = 16 / WK; PPW > 1 only with WK = 1)
#define AF_GEMV_SHAPES(X) X(1, 1) X(1, 2) X(1, 4) X(2, 1) X(4, 1) X(8, 1) X(16, 1)

template <int WT, bool NORM>
cudaError_t dispatch(const Planes& W, const float* x, const float* nw, float eps, const Epi& epi, unsigned* err,
                     cudaStream_t s) {
    if (use_pw(W, num_sms())) return pw_dispatch<WT, NORM>(W, x, nw, eps, epi, err, s);
    const Shape sh = pick_shape(W);
    if (sh.smem > kMaxGemvSmem || sh.ring > kMaxRing) return cudaErrorInvalidValue;
#define AF_GEMV_CASE(WW, PP) \
    if (sh.WK == WW && sh.PPW == PP) return launch_t<WT, NORM, WW, PP>(W, x, nw, eps, epi, sh, err, s);
    AF_GEMV_SHAPES(AF_GEMV_CASE)
#undef AF_GEMV_CASE
    return cudaErrorInvalidValue;
}

#define AF_GEMV_ATTR(WT, NORM, WW, PP)                                                                    \
    if (!e)                                                                                                \
        e = cudaFuncSetAttribute(qgemv_kernel<WT, NORM, WW, PP>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 kMaxGemvSmem);

// every instantiation may use up to kMaxGemvSmem of dynamic shared memory
template <int WT>
cudaError_t set_attrs_t() {
    cudaError_t e = cudaSuccess;
#define AF_GEMV_ATTR2(WW, PP) AF_GEMV_ATTR(WT, true, WW, PP) AF_GEMV_ATTR(WT, false, WW, PP)
    AF_GEMV_SHAPES(AF_GEMV_ATTR2)
#undef AF_GEMV_ATTR2
#define AF_PW_ATTR(NORM, RR) \
    if (!e) e = cudaFuncSetAttribute(qgemv_pw_kernel<WT, NORM, RR>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPwMaxSmem);
    AF_PW_ATTR(true, 2) AF_PW_ATTR(true, 4) AF_PW_ATTR(true, 8) AF_PW_ATTR(false, 2) AF_PW_ATTR(false, 4) AF_PW_ATTR(false, 8)
#undef AF_PW_ATTR
    return e;
}
#undef AF_GEMV_ATTR

template <int WT>
cudaError_t dispatch_t(const Planes& W, const float* x, const float* nw, float eps, const Epi& epi, unsigned* err,
                       cudaStream_t s) {
    return nw ? dispatch<WT, true>(W, x, nw, eps, epi, err, s) : dispatch<WT, false>(W, x, nw, eps, epi, err, s);
}

}  // namespace

// Defines the entry points of type WT in the including translation unit.
#define AF_QGEMV_INSTANTIATE(WT)                                                                              \
    template <>                                                                                             \
    cudaError_t qgemv_dispatch<WT>(const Planes& W, const float* x, const float* nw, float eps, const Epi& epi, \
                                   unsigned* err, cudaStream_t s) {                                           \
        return dispatch_t<WT>(W, x, nw, eps, epi, err, s);                                                    \
    }                                                                                                       \
    template <>                                                                                             \
    cudaError_t qgemv_set_attrs<WT>() {                                                                     \
        return set_attrs_t<WT>();                                                                           \
    }

}  // namespace af
