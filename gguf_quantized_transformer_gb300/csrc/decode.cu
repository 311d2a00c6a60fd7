// Host side of the persistent decode step (see decode_impl.cuh): stage shapes,
// slot sizing, split counts and dispatch to the per-(weight type, head_dim) kernels.
#include <algorithm>

#include "common.cuh"

namespace af {

template <int WT, int D>
cudaError_t decode_launch_for(const DecodePlan& p, cudaStream_t s, bool prepare);

namespace {
constexpr int kWarpsP = 16;
constexpr int kMaxRowsP = 128;
constexpr int kSubT = 16;                      // attention slots per online-softmax step (decode_impl.cuh)
constexpr int kSlotTarget = 20 * 1024;         // stage size: bulk copies of 16-20 KB stream at full rate
constexpr int kSmemBudgetP = 222 * 1024;       // dynamic shared memory (image region, schedule, slots)
constexpr int kXBlkBytesP = 80;                // x image bytes per 32-element block

int ximage_bytes_p(int Kp) { return ((Kp / 32) * kXBlkBytesP + 127) & ~127; }

cudaError_t dispatch(const DecodePlan& p, cudaStream_t s, bool prepare) {
    const int G = p.KVH > 0 ? p.H / p.KVH : 0;
    if (p.H % p.KVH || (G != 2 && G != 4 && G != 8)) return cudaErrorInvalidValue;
    if (p.wtype == AF_Q4_0 && p.D == 64) return decode_launch_for<AF_Q4_0, 64>(p, s, prepare);
    if (p.wtype == AF_Q4_0 && p.D == 128) return decode_launch_for<AF_Q4_0, 128>(p, s, prepare);
    if (p.wtype == AF_Q8_0 && p.D == 64) return decode_launch_for<AF_Q8_0, 64>(p, s, prepare);
    if (p.wtype == AF_Q8_0 && p.D == 128) return decode_launch_for<AF_Q8_0, 128>(p, s, prepare);
    return cudaErrorInvalidValue;
}
}  // namespace

// Rows per stage: the largest of 8, 4, 2 whose stage stays within the target (at least 2: epilogue pairs).
bool decode_gemv_task(const Planes& W, GemvTask& t) {
    if (W.wtype != AF_Q4_0 && W.wtype != AF_Q8_0) return false;  // the persistent kernel decodes Q4_0 / Q8_0
    t.W = W;
    const int64_t pitch = W.qs_pitch();
    t.R = 8;
    while (t.R > 2 && t.R * pitch > kSlotTarget) t.R /= 2;
    return true;
}

int decode_attn_splits(int n_kv_heads) {
    int s = num_sms() / n_kv_heads;
    return s < 1 ? 1 : s;
}

int decode_max_cta_rows() { return kMaxRowsP; }

bool decode_configure(DecodePlan& p, const LayerPlan& l0) {
    if (p.KVH < 1 || p.H % p.KVH || (p.D != 64 && p.D != 128)) return false;
    const int G = p.H / p.KVH;
    const int kvb = p.kv_f16 ? 2 : 4;
    int64_t slot = 0, ximg = 0;
    const GemvTask* tasks[5] = {&l0.qkv, &l0.o, &l0.gu, &l0.down, &p.head};  // every layer has layer 0's shapes
    for (const GemvTask* t : tasks) {
        slot = std::max<int64_t>(slot, t->R * t->W.qs_pitch());
        ximg = std::max<int64_t>(ximg, ximage_bytes_p(t->W.Kp));
    }
    // attention: T cache slots of K and of V per stage, a multiple of the softmax step
    int T = (int)(slot / (2 * p.D * kvb)) / kSubT * kSubT;
    T = T < kSubT ? kSubT : (T > 64 ? 64 : T);
    slot = std::max<int64_t>(slot, 2 * T * p.D * kvb);
    // attention scratch in the image region: probabilities, combine rows, the current K/V, merge weights
    const int64_t scratch = (int64_t)kWarpsP * kSubT * G * 4 + (int64_t)kWarpsP * G * p.D * 4 + 2 * p.D * kvb +
                            (int64_t)p.attn_splits * G * 4;
    ximg = std::max<int64_t>(ximg, scratch);
    slot = (slot + 127) & ~(int64_t)127;
    ximg = (ximg + 127) & ~(int64_t)127;
    const int64_t tab = ((int64_t)(5 * p.n_layers + 1) * 32 + 127) & ~(int64_t)127;  // one descriptor per phase
    const int64_t n = (kSmemBudgetP - ximg - tab) / slot;
    if (n < 2) return false;
    p.nslot = (int)std::min<int64_t>(n, kMaxSlotsP);
    p.slot_bytes = (int)slot;
    p.att_T = T;
    p.ximg_bytes = (int)ximg;
    p.tab_bytes = (int)tab;
    return true;
}

cudaError_t decode_prepare(const DecodePlan& p) { return dispatch(p, nullptr, true); }

cudaError_t launch_decode(const DecodePlan& p, cudaStream_t s) { return dispatch(p, s, false); }

}  // namespace af
