// Decode GEMV entry points: the kernel is in qgemv_impl.cuh and each weight type's instantiations live in
// their own translation unit (qgemv_<type>.cu), so they compile in parallel.
#include <mutex>

#include "qgemv_impl.cuh"

namespace af {

namespace {
std::mutex g_prep_mu;
bool g_prepared[kMaxDevices] = {};
}  // namespace

cudaError_t qgemv_prepare() {
    // once per device (kernel attributes are per device), outside any stream capture
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_prep_mu);
    if (g_prepared[dev]) return cudaSuccess;
    e = qgemv_set_attrs<AF_Q4_0>();
    if (!e) e = qgemv_set_attrs<AF_Q8_0>();
    if (!e) e = qgemv_set_attrs<AF_Q4_K>();
    if (!e) e = qgemv_set_attrs<AF_Q5_K>();
    if (!e) e = qgemv_set_attrs<AF_Q6_K>();
    if (!e) g_prepared[dev] = true;
    return e;
}

int qgemv_max_chunks() { return 32; }

cudaError_t launch_qgemv(const Planes& W, const float* x, const float* norm_w, float eps, const Epi& epi,
                         const GemvScratch& scr, cudaStream_t s) {
    switch (W.wtype) {
        case AF_Q4_0: return qgemv_dispatch<AF_Q4_0>(W, x, norm_w, eps, epi, scr.err, s);
        case AF_Q8_0: return qgemv_dispatch<AF_Q8_0>(W, x, norm_w, eps, epi, scr.err, s);
        case AF_Q4_K: return qgemv_dispatch<AF_Q4_K>(W, x, norm_w, eps, epi, scr.err, s);
        case AF_Q5_K: return qgemv_dispatch<AF_Q5_K>(W, x, norm_w, eps, epi, scr.err, s);
        case AF_Q6_K: return qgemv_dispatch<AF_Q6_K>(W, x, norm_w, eps, epi, scr.err, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace af
