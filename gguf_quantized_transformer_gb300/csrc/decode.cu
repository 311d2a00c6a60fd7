// Host side of the persistent decode step (see decode_impl.cuh): stage shapes,
// split counts and dispatch to the per-(weight type, head_dim) kernels.
#include "common.cuh"

namespace af {

template <int WT, int D>
cudaError_t decode_launch_for(const DecodePlan& p, cudaStream_t s, bool prepare);

namespace {
constexpr int kWarpsP = 16;
constexpr int kSlotBytes = 40 * 1024;
constexpr int kRWMax = 4;
constexpr int kMaxRowsP = 512;

cudaError_t dispatch(const DecodePlan& p, cudaStream_t s, bool prepare) {
    const int G = p.KVH > 0 ? p.H / p.KVH : 0;
    if (G < 1 || G > 8 || p.H % p.KVH) return cudaErrorInvalidValue;
    if (p.wtype == AF_Q4_0 && p.D == 64) return decode_launch_for<AF_Q4_0, 64>(p, s, prepare);
    if (p.wtype == AF_Q4_0 && p.D == 128) return decode_launch_for<AF_Q4_0, 128>(p, s, prepare);
    if (p.wtype == AF_Q8_0 && p.D == 64) return decode_launch_for<AF_Q8_0, 64>(p, s, prepare);
    if (p.wtype == AF_Q8_0 && p.D == 128) return decode_launch_for<AF_Q8_0, 128>(p, s, prepare);
    return cudaErrorInvalidValue;
}
}  // namespace

// Shapes of a GEMV phase: R rows per stage within one ring slot, WK chunk warps.
bool decode_gemv_task(const Planes& W, GemvTask& t) {
    if (is_kquant(W.wtype)) return false;  // the persistent kernel is built for Q4_0 / Q8_0 only
    const int UW = W.wtype == AF_Q8_0 ? 16 : 32;
    const int NC = W.Kp / (32 * UW);
    const int UPL = 2;  // x slots per lane the kernel is instantiated for
    t.W = W;
    t.WK = NC > 8 ? 16 : (NC > 4 ? 8 : (NC > 2 ? 4 : NC));  // 16 warps split long rows: one slot per lane
    if (NC > t.WK * UPL) return false;
    const int RS = kWarpsP / t.WK;
    const int row_bytes = (int)W.qs_pitch();  // quants and scales of a row
    t.R = kRWMax * RS < 32 ? kRWMax * RS : 32;
    while (t.R > RS && t.R * row_bytes > kSlotBytes) t.R /= 2;
    if (t.R * row_bytes > kSlotBytes) return false;
    if (t.R / RS > kRWMax) return false;
    return true;
}

int decode_attn_splits(int n_kv_heads) {
    int s = num_sms() / n_kv_heads;
    return s < 1 ? 1 : s;
}

int decode_max_cta_rows() { return kMaxRowsP; }

cudaError_t decode_prepare(const DecodePlan& p) { return dispatch(p, nullptr, true); }

cudaError_t launch_decode(const DecodePlan& p, cudaStream_t s) { return dispatch(p, s, false); }

}  // namespace af
