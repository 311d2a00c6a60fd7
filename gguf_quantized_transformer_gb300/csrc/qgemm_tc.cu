// Prefill GEMM on the 5th-generation tensor cores: Y[m][n] = sum_k X[m][k] W[n][k]
// with W in Q4_0 / Q8_0 / Q4_K / Q5_K / Q6_K planes, dequantized tile by tile
// and multiplied with tcgen05.mma into a TMEM accumulator (dotLLM "GPU
// Inference", "Weight Strategy", approach 1: fused dequantize-in-kernel feeding
// the tensor cores; dequantized values never touch device memory).
//
// Operands.  The MMA computes D[n][m] = sum_k W[n][k] X[m][k]: A is the
// dequantized weight tile (128 rows of W = the 128 TMEM lanes), written by the
// dequantizing warps straight from registers into tensor memory (tcgen05.st),
// so it costs no shared-memory bandwidth; B is the X tile (BT = 128 or 256
// rows of X), loaded by TMA into shared memory in the SWIZZLE_128B K-major
// layout.  The accumulator holds one W row per TMEM lane and one X row per
// column, so the epilogue's stores of a token run along n (coalesced).
//
// Precision.  A single fp16 product would round X and W to 11 significant
// bits.  X arrives split as X_hi + X_lo (two fp16 planes written by the
// producing kernel) and each weight is split as w_hi + w_lo in fp16 while
// dequantizing: exactly for Q4_0 / Q8_0 (w_hi = d * c by HMUL2 on the exact
// integer code c, w_lo = fma(d, c, -w_hi) by HFMA2), and from an fp32 value
// for the K-quants (formed from the unpacked sub-block scale and min).  Three
// MMAs per K step accumulate
//   W_hi X_hi + W_hi X_lo + W_lo X_hi
// in fp32 (the dropped W_lo X_lo term is ~2^-22 relative); see kProducts for the
// measured cost of dropping W_lo X_hi.
//
// Tile 128 (W rows) x BT (X rows) x 64 (K), S stages of the X tile in shared
// memory and of the W tile in tensor memory:
//   warp 0      : TMA producer for the X_hi / X_lo tiles (cp.async.bulk.tensor.2d)
//   warp 1      : TMEM allocation; one lane issues the MMAs and commits
//   warps 2..9  : two groups of four warps (one per TMEM lane quadrant) take
//                 alternate K steps: load the raw blocks of their 32 rows two
//                 steps ahead into registers, dequantize, split and store the
//                 W_hi / W_lo tile into the stage's TMEM columns;
//                 warps 2..5 then run the fused epilogue from TMEM
//                 (tcgen05.ld, 32 columns at a time).
// Split K.  A GEMM with few output tiles (small N) leaves SMs idle; it then runs
// ksplit CTAs per tile, each over a contiguous range of the K steps.  Each CTA
// stores its fp32 partial tile (column-major, coalesced) in a workspace; the last of a tile's CTAs to
// arrive (arrival counter, no waiting) adds the ksplit partials in split order,
// its own taken from TMEM, and runs the fused epilogue, so the result does not
// depend on the arrival order.
// Every mbarrier wait is bounded; on a timeout the CTA records DEV_TIMEOUT,
// drains what it issued and frees its TMEM before returning.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace af {

namespace {

constexpr int BW = 128, BK = 64;   // W rows (MMA M, TMEM lanes) and K per step
constexpr int kThreads = 10 * 32;
constexpr int kMaxStages = 4;
constexpr int kTmemCols = 512;

// Every weight keeps its fp16 remainder W_lo as a third product W_lo X_hi.  Rounding W to fp16 alone (two MMAs)
// measured 17.3k against 15.4k prefill tok/s on the 8B Q4_0 shape with the previous tile layout, but its worst
// layer error on a 17-token prompt was 1.67e-2 of the 2e-2 RMS bar (5.6e-3 with the third product), and the bar is
// a maximum over all elements: a 4096-token prompt has ~240x more of them, which puts the expected maximum near
// 2.05e-2.  The 8B Q4_K_M model reached 2.05e-2 already on the short prompt.
constexpr int kProducts = 3;

template <int BT>
struct TcCfg {
    static constexpr int kXTile = BT * BK * 2;                    // one fp16 plane of the X tile
    static constexpr int kStageBytes = 2 * kXTile;                // X_hi, X_lo
    static constexpr int kStages = BT == 256 ? 3 : 4;             // 192 / 128 KB of X stages
    static constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
    static constexpr int kACol = BT;                              // W stages: 64 TMEM columns each after D
    static_assert(kACol + 64 * kStages <= kTmemCols, "TMEM columns");
    static constexpr uint32_t kIdesc = idesc_f16(BW, BT);
};

// One 32-weight block as loaded from the weight rows: quant bytes and the fp16 scale bits.
template <int WT>
struct RawBlk;
template <>
struct RawBlk<AF_Q4_0> {
    uint4 q;
    unsigned short d;
};
template <>
struct RawBlk<AF_Q8_0> {
    uint4 q0, q1;
    unsigned short d;
};

template <>
struct RawBlk<AF_Q4_K> {
    uint4 q;
    unsigned dm;         // fp16 d, dmin of the super-block
    unsigned short smj;  // unpacked (s_j, m_j) of this sub-block
};
template <>
struct RawBlk<AF_Q5_K> {
    uint4 q;
    unsigned h;          // high bits: element 4t + i of half hh at bit 8i + 4hh + t
    unsigned dm;
    unsigned short smj;
};
template <>
struct RawBlk<AF_Q6_K> {
    uint4 q;             // low 4 bits of the codes
    uint2 h;             // high 2 bits (element 4t + i of a half at bits 8i + 2t of that half's word)
    unsigned short d;    // fp16 d of the super-block
    unsigned short sc;   // int8 scales of the two 16-weight halves
};

__device__ __forceinline__ void load_blk(const Planes& W, int n, int blk, RawBlk<AF_Q4_K>& b) {
    const uint8_t* row = W.qs + (int64_t)n * W.qs_pitch();
    b.q = *reinterpret_cast<const uint4*>(row + (int64_t)blk * 16);
    const uint8_t* rec = row + W.sc_off() + (int64_t)(blk >> 3) * kQ4KRec;
    b.dm = *reinterpret_cast<const unsigned*>(rec);
    b.smj = *reinterpret_cast<const unsigned short*>(rec + 4 + (blk & 7) * 2);
}
__device__ __forceinline__ void load_blk(const Planes& W, int n, int blk, RawBlk<AF_Q5_K>& b) {
    const uint8_t* row = W.qs + (int64_t)n * W.qs_pitch();
    b.q = *reinterpret_cast<const uint4*>(row + (int64_t)blk * 16);
    b.h = *reinterpret_cast<const unsigned*>(row + W.hb_off() + (int64_t)blk * 4);
    const uint8_t* rec = row + W.sc_off() + (int64_t)(blk >> 3) * kQ4KRec;
    b.dm = *reinterpret_cast<const unsigned*>(rec);
    b.smj = *reinterpret_cast<const unsigned short*>(rec + 4 + (blk & 7) * 2);
}
__device__ __forceinline__ void zero_blk(RawBlk<AF_Q5_K>& b) {
    b.q = make_uint4(0, 0, 0, 0);
    b.h = 0;
    b.dm = 0;
    b.smj = 0;
}
__device__ __forceinline__ void load_blk(const Planes& W, int n, int blk, RawBlk<AF_Q6_K>& b) {
    const uint8_t* row = W.qs + (int64_t)n * W.qs_pitch();
    b.q = *reinterpret_cast<const uint4*>(row + (int64_t)blk * 16);
    b.h = *reinterpret_cast<const uint2*>(row + W.hb_off() + (int64_t)blk * 8);
    const uint8_t* rec = row + W.sc_off() + (int64_t)(blk >> 3) * kQ6KRec;
    b.d = *reinterpret_cast<const unsigned short*>(rec);
    b.sc = *reinterpret_cast<const unsigned short*>(rec + 2 + (blk & 7) * 2);
}
__device__ __forceinline__ void zero_blk(RawBlk<AF_Q4_K>& b) {
    b.q = make_uint4(0, 0, 0, 0);
    b.dm = 0;
    b.smj = 0;
}
__device__ __forceinline__ void zero_blk(RawBlk<AF_Q6_K>& b) {
    b.q = make_uint4(0, 0, 0, 0);
    b.h = make_uint2(0, 0);
    b.d = 0;
    b.sc = 0;
}

__device__ __forceinline__ void load_blk(const Planes& W, int n, int blk, RawBlk<AF_Q4_0>& b) {
    b.q = *reinterpret_cast<const uint4*>(W.qs + (int64_t)n * W.qs_pitch() + (int64_t)blk * 16);
    b.d = __half_as_ushort(W.sc[(int64_t)n * W.sc_pitch() + blk]);
}
__device__ __forceinline__ void load_blk(const Planes& W, int n, int blk, RawBlk<AF_Q8_0>& b) {
    const uint8_t* q = W.qs + (int64_t)n * W.qs_pitch() + (int64_t)blk * 32;
    b.q0 = *reinterpret_cast<const uint4*>(q);
    b.q1 = *reinterpret_cast<const uint4*>(q + 16);
    b.d = __half_as_ushort(W.sc[(int64_t)n * W.sc_pitch() + blk]);
}
__device__ __forceinline__ void zero_blk(RawBlk<AF_Q4_0>& b) { b.q = make_uint4(0, 0, 0, 0); b.d = 0; }
__device__ __forceinline__ void zero_blk(RawBlk<AF_Q8_0>& b) {
    b.q0 = make_uint4(0, 0, 0, 0);
    b.q1 = b.q0;
    b.d = 0;
}

__device__ __forceinline__ __half2 u2h(unsigned v) { return *reinterpret_cast<const __half2*>(&v); }
__device__ __forceinline__ unsigned h2u(__half2 v) { return *reinterpret_cast<const unsigned*>(&v); }

// codes c (fp16, exact) times d -> exact split hi + lo
__device__ __forceinline__ void split_pair(__half2 c, __half2 d2, unsigned& hi, unsigned& lo) {
    const __half2 h = __hmul2(c, d2);
    hi = h2u(h);
    lo = h2u(__hfma2(c, d2, __hneg2(h)));
}

// 32 weights of a block -> 4 chunks (8 weights each, block order) of fp16 hi and lo
__device__ __forceinline__ void deq_blk(const RawBlk<AF_Q4_0>& b, uint4 (&hi)[4], uint4 (&lo)[4]) {
    const __half2 d2 = __half2half2(__ushort_as_half(b.d));
    const __half2 k1032 = __float2half2_rn(1032.f);
    const unsigned w[4] = {b.q.x, b.q.y, b.q.z, b.q.w};
    unsigned h[16], l[16];  // h[4*i + t]: i = 0,1 low-nibble pairs (x, y), i = 2,3 high-nibble pairs, word t
#pragma unroll
    for (int t = 0; t < 4; t++) {
        const unsigned x = __byte_perm(w[t], 0u, 0x4140);  // bytes b0, 0, b1, 0
        const unsigned y = __byte_perm(w[t], 0u, 0x4342);  // bytes b2, 0, b3, 0
        const unsigned c[4] = {(x & 0x000F000Fu) | 0x64006400u, (y & 0x000F000Fu) | 0x64006400u,
                               ((x >> 4) & 0x000F000Fu) | 0x64006400u, ((y >> 4) & 0x000F000Fu) | 0x64006400u};
#pragma unroll
        for (int i = 0; i < 4; i++) split_pair(__hsub2(u2h(c[i]), k1032), d2, h[4 * i + t], l[4 * i + t]);
    }
    // chunk 0: elements 0..7 = low nibbles of words 0, 1; chunk 1: words 2, 3; chunks 2, 3: high nibbles
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const int i0 = q < 2 ? 0 : 2, t0 = (q & 1) * 2;
        hi[q] = make_uint4(h[4 * i0 + t0], h[4 * (i0 + 1) + t0], h[4 * i0 + t0 + 1], h[4 * (i0 + 1) + t0 + 1]);
        lo[q] = make_uint4(l[4 * i0 + t0], l[4 * (i0 + 1) + t0], l[4 * i0 + t0 + 1], l[4 * (i0 + 1) + t0 + 1]);
    }
}
__device__ __forceinline__ void deq_blk(const RawBlk<AF_Q8_0>& b, uint4 (&hi)[4], uint4 (&lo)[4]) {
    const __half2 d2 = __half2half2(__ushort_as_half(b.d));
    const __half2 k1152 = __float2half2_rn(1152.f);
    const unsigned w[8] = {b.q0.x, b.q0.y, b.q0.z, b.q0.w, b.q1.x, b.q1.y, b.q1.z, b.q1.w};
    unsigned h[16], l[16];
#pragma unroll
    for (int t = 0; t < 8; t++) {
        const unsigned u = w[t] ^ 0x80808080u;  // q + 128 in 0..255
        split_pair(__hsub2(u2h(__byte_perm(u, 0x64646464u, 0x5140)), k1152), d2, h[2 * t], l[2 * t]);
        split_pair(__hsub2(u2h(__byte_perm(u, 0x64646464u, 0x5342)), k1152), d2, h[2 * t + 1], l[2 * t + 1]);
    }
#pragma unroll
    for (int q = 0; q < 4; q++) {
        hi[q] = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
        lo[q] = make_uint4(l[4 * q], l[4 * q + 1], l[4 * q + 2], l[4 * q + 3]);
    }
}

// fp32 weights (w0, w1) -> fp16 hi pair and the fp16 rounding of the remainders (relative error ~2^-22)
__device__ __forceinline__ void split_f32_pair(float w0, float w1, unsigned& hi, unsigned& lo) {
    const __half2 h = __floats2half2_rn(w0, w1);
    const float2 hf = __half22float2(h);
    hi = h2u(h);
    lo = h2u(__floats2half2_rn(w0 - hf.x, w1 - hf.y));
}

// exact float of a small unsigned integer v < 2^23
__device__ __forceinline__ float u2f_small(unsigned v) { return __uint_as_float(0x4B000000u | v) - 8388608.f; }

// Q4_K: w_e = (d s_j) n_e - dmin m_j, formed in fp32 (d s_j and dmin m_j are exact products), then split.
// Chunk c holds elements 8c..8c+7: low nibbles of bytes 8c.. (c < 2), high nibbles of bytes 8(c-2).. (c >= 2).
__device__ __forceinline__ void deq_blk(const RawBlk<AF_Q4_K>& b, uint4 (&hi)[4], uint4 (&lo)[4]) {
    const float2 dm = __half22float2(u2h(b.dm));
    const float A = dm.x * (float)(b.smj & 255u), B = dm.y * (float)(b.smj >> 8);
    const unsigned w[4] = {b.q.x, b.q.y, b.q.z, b.q.w};
#pragma unroll
    for (int c = 0; c < 4; c++) {
        unsigned hv[4], lv[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {  // elements 8c + 2k, 8c + 2k + 1
            const unsigned word = w[2 * (c & 1) + (k >> 1)] >> (c < 2 ? 0 : 4);
            const int sh = 16 * (k & 1);
            const float n0 = u2f_small((word >> sh) & 15u), n1 = u2f_small((word >> (sh + 8)) & 15u);
            split_f32_pair(fmaf(A, n0, -B), fmaf(A, n1, -B), hv[k], lv[k]);
        }
        hi[c] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        lo[c] = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    }
}

// Q5_K: as Q4_K with the 5-bit code nibble + 16 * high bit.
__device__ __forceinline__ void deq_blk(const RawBlk<AF_Q5_K>& b, uint4 (&hi)[4], uint4 (&lo)[4]) {
    const float2 dm = __half22float2(u2h(b.dm));
    const float A = dm.x * (float)(b.smj & 255u), B = dm.y * (float)(b.smj >> 8);
    const unsigned w[4] = {b.q.x, b.q.y, b.q.z, b.q.w};
#pragma unroll
    for (int c = 0; c < 4; c++) {
        unsigned hv[4], lv[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            float v[2];
#pragma unroll
            for (int e2 = 0; e2 < 2; e2++) {
                const int i = 8 * (c & 1) + 2 * k + e2;  // index within the half c / 2
                const unsigned nib = (w[i >> 2] >> (8 * (i & 3) + (c < 2 ? 0 : 4))) & 15u;
                const unsigned h1 = (b.h >> (8 * (i & 3) + 4 * (c >> 1) + (i >> 2))) & 1u;
                v[e2] = fmaf(A, u2f_small(nib | (h1 << 4)), -B);
            }
            split_f32_pair(v[0], v[1], hv[k], lv[k]);
        }
        hi[c] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        lo[c] = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    }
}

// Q6_K: w_e = (d c_half) (q_e - 32), exact in fp32 (at most 24 significant bits), then split.
__device__ __forceinline__ void deq_blk(const RawBlk<AF_Q6_K>& b, uint4 (&hi)[4], uint4 (&lo)[4]) {
    const float d = __half2float(__ushort_as_half(b.d));
    const float da = d * (float)(int)(signed char)(b.sc & 255u), db = d * (float)(int)(signed char)(b.sc >> 8);
    const unsigned w[4] = {b.q.x, b.q.y, b.q.z, b.q.w};
#pragma unroll
    for (int c = 0; c < 4; c++) {
        // elements 8c..8c+7 lie in half c / 2; their index within the half is i = 8 (c & 1) + ..
        const unsigned hw = c < 2 ? b.h.x : b.h.y;
        const float dh = c < 2 ? da : db;
        unsigned hv[4], lv[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            float v[2];
#pragma unroll
            for (int e2 = 0; e2 < 2; e2++) {
                const int i = 8 * (c & 1) + 2 * k + e2;  // index within the half, 0..15
                const unsigned nib = (w[i >> 2] >> (8 * (i & 3) + (c < 2 ? 0 : 4))) & 15u;
                const unsigned h2 = (hw >> (8 * (i & 3) + 2 * (i >> 2))) & 3u;
                v[e2] = dh * (u2f_small(nib | (h2 << 4)) - 32.f);
            }
            split_f32_pair(v[0], v[1], hv[k], lv[k]);
        }
        hi[c] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        lo[c] = make_uint4(lv[0], lv[1], lv[2], lv[3]);
    }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

struct TcSmem {
    uint64_t xfull[kMaxStages];  // X tiles landed (TMA transaction bytes)
    uint64_t afull[kMaxStages];  // W tile stored in TMEM (one arrival per quadrant warp)
    uint64_t empty[kMaxStages];  // MMAs reading the stage finished (commit)
    uint64_t done;               // all MMAs finished (commit)
    uint32_t tmem_base;
    volatile int abort;
    int issued_x;  // X tile loads issued so far
    int last;      // split K: this CTA is the last of its tile to arrive
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

// Epilogue of one quadrant warp: lane l holds W row n (= n0 + 32 quad + l) of the accumulator, i.e. output
// column n for every X row of the tile.  The fused epilogues take adjacent column pairs (n, n + 1) of one output
// row, so lanes 2p and 2p + 1 trade halves: for tokens j (even) and j + 1, lane 2p gets row 2p + 1's value of
// token j and lane 2p + 1 gets row 2p's value of token j + 1; each lane then applies the pair of one token.
// Per 32 tokens, every value the epilogue reads (the residual, the RoPE rows) is loaded before any of its stores:
// the compiler cannot reorder a load above a store that may alias it, so an interleaved load-store sequence would
// pay one L2 round trip per pair.
template <int KIND>
__device__ __forceinline__ void epi_chunk(const Epi& e, const float (&v)[32], int lane, int n, int N, int mb, int M) {
    const int np = n & ~1;  // the pair's first column
    const bool odd = lane & 1;
    float a0[16], a1[16];
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float got = __shfl_xor_sync(0xffffffffu, odd ? v[j] : v[j + 1], 1);
        a0[j / 2] = odd ? got : v[j];
        a1[j / 2] = odd ? v[j + 1] : got;
    }
    const int m1 = mb + (odd ? 1 : 0);  // token of pair i: m1 + 2 i
    if (np >= N) return;
    if (KIND == EPI_RESID) {
        float2 old[16];
#pragma unroll
        for (int i = 0; i < 16; i++)
            old[i] = m1 + 2 * i < M ? __ldcg(reinterpret_cast<const float2*>(e.out + (int64_t)(m1 + 2 * i) * e.ld + np))
                                    : make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; i++)
            if (m1 + 2 * i < M)
                *reinterpret_cast<float2*>(e.out + (int64_t)(m1 + 2 * i) * e.ld + np) =
                    make_float2(old[i].x + a0[i], old[i].y + a1[i]);
    } else if (KIND == EPI_QKV) {
        const int D = e.head_dim;
        const bool rot = np < e.qd + e.kvd;  // q or k: rotate the pair (2i, 2i+1) by theta(pos, i)
        const int d = (np < e.qd ? np : np - e.qd) % D;
        const int pos1 = (e.pos_dev ? __ldcg(e.pos_dev) : e.pos0) + m1;
        float2 cs[16];
#pragma unroll
        for (int i = 0; i < 16; i++)
            cs[i] = rot && m1 + 2 * i < M ? e.rope[(int64_t)(pos1 + 2 * i) * (D / 2) + (d >> 1)] : make_float2(1.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const int m = m1 + 2 * i;
            if (m >= M) continue;
            float v0 = a0[i], v1 = a1[i];
            if (rot) {
                const float r0 = v0 * cs[i].x - v1 * cs[i].y, r1 = v0 * cs[i].y + v1 * cs[i].x;
                v0 = r0;
                v1 = r1;
            }
            if (np < e.qd) {
                if (e.out) *reinterpret_cast<float2*>(e.out + (int64_t)m * e.ld + np) = make_float2(v0, v1);
            } else {
                const bool isk = np < e.qd + e.kvd;
                const int c = isk ? np - e.qd : np - e.qd - e.kvd;
                const int64_t idx = ((int64_t)(c / D) * e.max_ctx + pos1 + 2 * i) * D + c % D;
                void* base = isk ? e.kcache : e.vcache;
                if (e.kv_f16)
                    *reinterpret_cast<__half2*>((__half*)base + idx) = __floats2half2_rn(v0, v1);
                else
                    *reinterpret_cast<float2*>((float*)base + idx) = make_float2(v0, v1);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; i++) {
            if (m1 + 2 * i < M) {
                Epi k = e;
                k.kind = KIND;  // constant: the switch in epi_pair folds away
                epi_pair(k, m1 + 2 * i, np, a0[i], a1[i]);
            }
        }
    }
}

template <int KIND, int BT>
__device__ __forceinline__ void epilogue(const Epi& epi, uint32_t lane_base, int lane, int n, int N, int m0, int M) {
    for (int c0 = 0; c0 < BT; c0 += 32) {
        float v[32];
        tmem_ld32(lane_base + (uint32_t)c0, v);
        epi_chunk<KIND>(epi, v, lane, n, N, m0 + c0, M);
    }
}

// Named barrier of the four epilogue warps (warps 2..5).
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Split K: store this CTA's partial tile, column-major ([BT columns][BW rows] fp32): lane r of a quadrant warp holds
// W row r, so each of its stores is one contiguous 128-byte line per warp.
template <int BT>
__device__ __forceinline__ void store_partial(float* part, uint32_t lane_base, int r) {
    for (int c0 = 0; c0 < BT; c0 += 32) {
        float v[32];
        tmem_ld32(lane_base + (uint32_t)c0, v);
#pragma unroll
        for (int j = 0; j < 32; j++) part[(size_t)(c0 + j) * BW + r] = v[j];
    }
}

// Split K, last CTA of the tile: sum the ksplit partials of row r in split order (its own from TMEM) and apply
// the epilogue as `epilogue` does; the 32 loads of a partial's chunk are in flight together.
template <int KIND, int BT>
__device__ __forceinline__ void epilogue_split(const Epi& epi, uint32_t lane_base, int lane, int n, int N, int m0,
                                               int M, const float* tile_ws, int ksplit, int kz, int r) {
    for (int c0 = 0; c0 < BT; c0 += 32) {
        float own[32], v[32];
        tmem_ld32(lane_base + (uint32_t)c0, own);
#pragma unroll
        for (int j = 0; j < 32; j++) v[j] = 0.f;
        for (int z = 0; z < ksplit; z++) {
            if (z == kz) {
#pragma unroll
                for (int j = 0; j < 32; j++) v[j] += own[j];
            } else {
                const float* src = tile_ws + (size_t)z * BW * BT + (size_t)c0 * BW + r;
                float w[32];
#pragma unroll
                for (int j = 0; j < 32; j++) w[j] = __ldcg(src + (size_t)j * BW);
#pragma unroll
                for (int j = 0; j < 32; j++) v[j] += w[j];
            }
        }
        epi_chunk<KIND>(epi, v, lane, n, N, m0 + c0, M);
    }
}

template <int BT>
__device__ __forceinline__ void run_epilogue(const Epi& epi, uint32_t lane_base, int lane, int n, int N, int m0,
                                             int M) {
    switch (epi.kind) {  // one loop per kind, so the loop body has no dispatch
        case EPI_RESID: epilogue<EPI_RESID, BT>(epi, lane_base, lane, n, N, m0, M); break;
        case EPI_QKV: epilogue<EPI_QKV, BT>(epi, lane_base, lane, n, N, m0, M); break;
        case EPI_SWIGLU: epilogue<EPI_SWIGLU, BT>(epi, lane_base, lane, n, N, m0, M); break;
        default: epilogue<EPI_STORE, BT>(epi, lane_base, lane, n, N, m0, M); break;
    }
}

template <int BT>
__device__ __forceinline__ void run_epilogue_split(const Epi& epi, uint32_t lane_base, int lane, int n, int N, int m0,
                                                   int M, const float* tile_ws, int ksplit, int kz, int r) {
    switch (epi.kind) {
        case EPI_RESID: epilogue_split<EPI_RESID, BT>(epi, lane_base, lane, n, N, m0, M, tile_ws, ksplit, kz, r); break;
        case EPI_QKV: epilogue_split<EPI_QKV, BT>(epi, lane_base, lane, n, N, m0, M, tile_ws, ksplit, kz, r); break;
        case EPI_SWIGLU: epilogue_split<EPI_SWIGLU, BT>(epi, lane_base, lane, n, N, m0, M, tile_ws, ksplit, kz, r); break;
        default: epilogue_split<EPI_STORE, BT>(epi, lane_base, lane, n, N, m0, M, tile_ws, ksplit, kz, r); break;
    }
}

template <int WT, int BT>
__global__ void __launch_bounds__(kThreads, 1)
    qgemm_tc_kernel(const __grid_constant__ CUtensorMap map_hi, const __grid_constant__ CUtensorMap map_lo, Planes W,
                    int M, Epi epi, unsigned* err, int ksplit, float* __restrict__ ws, unsigned* __restrict__ cnt) {
    using C = TcCfg<BT>;
    constexpr int kStages = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    __shared__ TcSmem sm;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // grid (M tiles, N tiles, splits): the M tiles of one weight tile are adjacent in launch order, so the weight
    // rows come from DRAM once and from L2 for the other M tiles
    const int n0 = blockIdx.y * BW, m0 = blockIdx.x * BT;
    const int nk_all = (W.K + BK - 1) / BK;
    const int kz = blockIdx.z;  // this CTA's K steps: [k_lo, k_lo + nk)
    const int k_lo = (int)((int64_t)nk_all * kz / ksplit);
    const int nk = (int)((int64_t)nk_all * (kz + 1) / ksplit) - k_lo;

    // programmatic dependent launch: the next kernel may start its own prologue; this one reads X (and writes
    // its outputs) only after griddepcontrol.wait, while the weight tiles, which do not depend on the previous
    // kernel, are fetched and dequantized before it
    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&sm.xfull[s], 1);
            mbar_init(&sm.afull[s], 4);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.done, 1);
        sm.abort = 0;
        sm.issued_x = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    auto x_hi = [&](int s) { return smem + s * C::kStageBytes; };
    auto x_lo = [&](int s) { return smem + s * C::kStageBytes + C::kXTile; };

    if (warp == 0) {
        // ---------------- TMA producer: X_hi, X_lo tiles
        if (lane == 0) {
            pdl_wait();  // X is written by the previous kernel
            for (int ks = 0; ks < nk; ks++) {
                const int s = ks % kStages, u = ks / kStages;
                if (u > 0 && !wait_or_abort(&sm.empty[s], (u - 1) & 1, sm, err)) break;
                mbar_arrive_expect_tx(&sm.xfull[s], 2 * C::kXTile);
                tma_load_2d(x_hi(s), &map_hi, (k_lo + ks) * BK, m0, &sm.xfull[s]);
                tma_load_2d(x_lo(s), &map_lo, (k_lo + ks) * BK, m0, &sm.xfull[s]);
                sm.issued_x = ks + 1;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            for (int ks = 0; ks < nk; ks++) {
                const int s = ks % kStages, u = ks / kStages;
                if (!wait_or_abort(&sm.xfull[s], u & 1, sm, err)) break;
                if (!wait_or_abort(&sm.afull[s], u & 1, sm, err)) break;
                tc_fence_after();
                const uint32_t bh = smem_u32(x_hi(s)), bl = smem_u32(x_lo(s));
                const uint32_t ah = tmem + (uint32_t)(C::kACol + 64 * s), al = ah + 32;
#pragma unroll
                for (int kk = 0; kk < BK / 16; kk++) {  // 16 fp16 along K per MMA: 8 TMEM columns, 32 bytes of B
                    const uint32_t acc = (ks > 0 || kk > 0) ? 1u : 0u;
                    const uint64_t dh = umma_desc_sw128(bh + kk * 32), dl = umma_desc_sw128(bl + kk * 32);
                    mma_f16_ts(tmem, ah + kk * 8, dh, C::kIdesc, acc);
                    mma_f16_ts(tmem, ah + kk * 8, dl, C::kIdesc, 1u);
                    if (kProducts == 3) mma_f16_ts(tmem, al + kk * 8, dh, C::kIdesc, 1u);
                }
                mma_commit(&sm.empty[s]);  // frees the stage (X smem and W TMEM) when these MMAs complete
            }
            mma_commit(&sm.done);  // always: also after a break, so the drain can wait on it
        }
    } else {
        // ---------------- dequantize W rows into the stage's TMEM columns
        const int quad = warp & 3;            // TMEM lanes this warp may access
        const int grp = (warp - 2) >> 2;      // K steps grp, grp + 2, ...
        const int r = quad * 32 + lane;       // weight row n0 + r = TMEM lane
        const int n = n0 + r;
        const bool valid = n < W.N;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        // the raw blocks of this group's next two K steps are in flight while one is converted (weights mostly
        // come from DRAM: about four K steps of MMA time hide that latency)
        RawBlk<WT> cur[2], nxt[2], nxt2[2];
        auto fetch = [&](int ks, RawBlk<WT> (&b)[2]) {
#pragma unroll
            for (int i = 0; i < 2; i++) {
                if (valid && ks < nk) load_blk(W, n, (k_lo + ks) * 2 + i, b[i]);
                else zero_blk(b[i]);
            }
        };
        fetch(grp, cur);
        fetch(grp + 2, nxt);
        for (int ks = grp; ks < nk; ks += 2) {
            const int s = ks % kStages, u = ks / kStages;
            fetch(ks + 4, nxt2);
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int i = 0; i < 2; i++) {
                uint4 h4[4], l4[4];
                deq_blk(cur[i], h4, l4);
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    hi[16 * i + 4 * q + 0] = h4[q].x; hi[16 * i + 4 * q + 1] = h4[q].y;
                    hi[16 * i + 4 * q + 2] = h4[q].z; hi[16 * i + 4 * q + 3] = h4[q].w;
                    lo[16 * i + 4 * q + 0] = l4[q].x; lo[16 * i + 4 * q + 1] = l4[q].y;
                    lo[16 * i + 4 * q + 2] = l4[q].z; lo[16 * i + 4 * q + 3] = l4[q].w;
                }
            }
            // the stage's previous MMAs must be done before its W columns are overwritten (warp-uniform wait)
            if (u > 0 && !__all_sync(0xffffffffu, wait_or_abort(&sm.empty[s], (u - 1) & 1, sm, err))) break;
            tc_fence_after();
            const uint32_t col = (uint32_t)(C::kACol + 64 * s);
            tmem_st32(lane_base + col, hi);
            if (kProducts == 3) tmem_st32(lane_base + col + 32, lo);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.afull[s]);
#pragma unroll
            for (int i = 0; i < 2; i++) {
                cur[i] = nxt[i];
                nxt[i] = nxt2[i];
            }
        }
        // ---------------- epilogue (warps 2..5: TMEM lane quadrant = warp % 4)
        if (warp < 6) {
            pdl_wait();  // (already satisfied: the MMAs consumed X) before the epilogue's reads and writes
            // tcgen05.ld is warp-collective: the whole warp takes the same branch
            const bool ok = __all_sync(0xffffffffu, wait_or_abort(&sm.done, 0, sm, err));
            if (ok) tc_fence_after();
            if (ksplit == 1) {
                if (ok) run_epilogue<BT>(epi, lane_base, lane, n, W.N, m0, M);
            } else {
                // every CTA of the tile arrives, also after a timeout (the counter must return to zero)
                const int tile = blockIdx.y * gridDim.x + blockIdx.x;
                float* tile_ws = ws + (size_t)tile * ksplit * BW * BT;
                if (ok) store_partial<BT>(tile_ws + (size_t)kz * BW * BT, lane_base, r);
                __threadfence();
                epi_bar();
                if (warp == 2 && lane == 0) sm.last = atomicAdd(&cnt[tile], 1u) == (unsigned)ksplit - 1u;
                epi_bar();
                if (sm.last) {
                    __threadfence();
                    if (ok) run_epilogue_split<BT>(epi, lane_base, lane, n, W.N, m0, M, tile_ws, ksplit, kz, r);
                    if (warp == 2 && lane == 0) cnt[tile] = 0u;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (sm.abort && tid == 0) {  // let every MMA and copy that was issued finish before leaving
        mbar_wait_bounded(&sm.done, 0);
        // loads older than the last kStages were consumed by the MMA issuer, i.e. complete
        for (int ks = max(0, sm.issued_x - kStages); ks < sm.issued_x; ks++)
            mbar_wait_bounded(&sm.xfull[ks % kStages], (ks / kStages) & 1);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_free(tmem, kTmemCols);
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

// 2-D map over an fp16 [rows][ld] plane, box 64 (K) x box_rows, SWIZZLE_128B, zero fill out of bounds.
bool make_map(CUtensorMap* map, const __half* base, int rows, int cols, int64_t ld, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_tmap_f16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_cols,
                   uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
std::mutex g_prep_mu;
bool g_prepared[kMaxDevices] = {};
}  // namespace

cudaError_t qgemm_prepare() {
    // once per device (kernel attributes are per device), outside any stream capture
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_prep_mu);
    if (g_prepared[dev]) return cudaSuccess;
#define AF_QGEMM_ATTR(WT, BT)                                                                                  \
    if (!e) e = cudaFuncSetAttribute(qgemm_tc_kernel<WT, BT>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                     TcCfg<BT>::kSmemBytes);
    AF_QGEMM_ATTR(AF_Q4_0, 256)
    AF_QGEMM_ATTR(AF_Q4_0, 128)
    AF_QGEMM_ATTR(AF_Q8_0, 256)
    AF_QGEMM_ATTR(AF_Q8_0, 128)
    AF_QGEMM_ATTR(AF_Q4_K, 256)
    AF_QGEMM_ATTR(AF_Q4_K, 128)
    AF_QGEMM_ATTR(AF_Q5_K, 256)
    AF_QGEMM_ATTR(AF_Q5_K, 128)
    AF_QGEMM_ATTR(AF_Q6_K, 256)
    AF_QGEMM_ATTR(AF_Q6_K, 128)
#undef AF_QGEMM_ATTR
    if (!e) g_prepared[dev] = true;
    return e;
}

namespace {
// Tile width BT and K split for an N x K weight at M rows: the least estimated time, waves of CTAs x the time of
// one CTA.  The per-CTA times are fitted to measurements of this kernel on the 8B and 1B Q4_0 shapes at M = 512
// (every (BT, split) pair timed, weights streamed from DRAM): K steps x 1.05 us + 8 us at BT = 256, x 0.83 us +
// 12 us at BT = 128; a split CTA also stores its partial and the last one sums them, which measured as a fixed
// 20 us (BT = 256) or 13 us (BT = 128).  A split keeps at least 8 K steps per CTA and fits the workspace and the counters.
struct GemmShape {
    int BT, ksplit;
};
GemmShape pick_gemm(int N, int K, int M, size_t ws_bytes, int cnt_n) {
    constexpr int kMaxSplit = 4;
    const int sms = num_sms();
    const int nk = (K + BK - 1) / BK, nt = (N + BW - 1) / BW;
    GemmShape best{128, 1};
    double best_t = 1e30;
    for (int BT : {256, 128}) {
        const int mt = (M + BT - 1) / BT;
        const double step = BT == 256 ? 1.05 : 0.83;
        for (int ks = 1; ks <= kMaxSplit; ks++) {
            if (ks > 1 && (nk / ks < 8 || (size_t)nt * mt * ks * BW * BT * 4 > ws_bytes || nt * mt > cnt_n)) break;
            const double fixed = ks == 1 ? (BT == 256 ? 8.0 : 12.0) : (BT == 256 ? 20.0 : 13.0);
            const int ctas = nt * mt * ks;
            const double t = (double)((ctas + sms - 1) / sms) * ((double)nk / ks * step + fixed);
            if (t < best_t - 1e-9) {
                best_t = t;
                best = {BT, ks};
            }
        }
    }
    return best;
}
}  // namespace

size_t qgemm_ws_bytes(int N, int K, int M) {
    const GemmShape g = pick_gemm(N, K, M, (size_t)-1, 1 << 30);
    if (g.ksplit == 1) return 0;
    const size_t tiles = (size_t)((N + BW - 1) / BW) * ((M + g.BT - 1) / g.BT);
    return tiles * g.ksplit * BW * g.BT * 4;
}

int qgemm_tiles(int N, int M) { return ((N + BW - 1) / BW) * ((M + 127) / 128); }

cudaError_t launch_qgemm(const Planes& W, const __half* X_hi, const __half* X_lo, int64_t ldx, int M, const Epi& epi,
                         unsigned* err, cudaStream_t s, const GemmSplit* split) {
    if (M < 1) return cudaSuccess;
    if (ldx % 8 || (reinterpret_cast<uintptr_t>(X_hi) & 15) || (reinterpret_cast<uintptr_t>(X_lo) & 15))
        return cudaErrorInvalidValue;  // TMA: 16-byte aligned base and row stride
    const int nt = (W.N + BW - 1) / BW;
    const GemmShape g = split ? pick_gemm(W.N, W.K, M, split->ws_bytes, split->cnt_n) : pick_gemm(W.N, W.K, M, 0, 0);
    const int BT = g.BT;
    float* ws = g.ksplit > 1 ? split->ws : nullptr;
    unsigned* cnt = g.ksplit > 1 ? split->cnt : nullptr;
    CUtensorMap mh, ml;
    if (!make_map(&mh, X_hi, M, W.K, ldx, BT) || !make_map(&ml, X_lo, M, W.K, ldx, BT)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((M + BT - 1) / BT, nt, g.ksplit);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t le = cudaSuccess;
#define AF_QGEMM_LAUNCH(WT, BTV)                                                                                \
    cfg.dynamicSmemBytes = TcCfg<BTV>::kSmemBytes;                                                             \
    le = cudaLaunchKernelEx(&cfg, qgemm_tc_kernel<WT, BTV>, mh, ml, W, M, epi, err, g.ksplit, ws, cnt)
#define AF_QGEMM_TYPES(BTV)                                         \
    switch (W.wtype) {                                              \
        case AF_Q4_0: AF_QGEMM_LAUNCH(AF_Q4_0, BTV); break;         \
        case AF_Q8_0: AF_QGEMM_LAUNCH(AF_Q8_0, BTV); break;         \
        case AF_Q4_K: AF_QGEMM_LAUNCH(AF_Q4_K, BTV); break;         \
        case AF_Q5_K: AF_QGEMM_LAUNCH(AF_Q5_K, BTV); break;         \
        case AF_Q6_K: AF_QGEMM_LAUNCH(AF_Q6_K, BTV); break;         \
        default: return cudaErrorInvalidValue;                      \
    }
    if (BT == 256) {
        AF_QGEMM_TYPES(256)
    } else {
        AF_QGEMM_TYPES(128)
    }
#undef AF_QGEMM_TYPES
#undef AF_QGEMM_LAUNCH
    return le;
}

}  // namespace af
