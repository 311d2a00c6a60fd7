// Fixed, allocation-free scratch for the decode attention entry point that
// must not allocate (af_attention_decode_static).
//
// The split-KV decode attention needs two scratch areas: the per-split
// partials (output row, running max, running sum for every query head of a
// split) and one arrival counter per kv head.  Here both live in one
// file-scope device array, so a call needs no cudaMalloc / cudaFree.
//
// Layout of g_attn_static:
//   [0, kStaticAttnMaxKVH * 4)          arrival counters (unsigned)
//   word kStaticAttnMaxKVH              error word (a bounded device wait gave up)
//   [kStaticAttnCntBytes, end)          split partials (float)
// The counters are zero when the module is loaded and every call that runs
// to completion leaves them zero again (the last CTA of each kv head resets
// its counter).  The partials need no initial value: a call reads only the
// partials it wrote itself.
#include <mutex>

#include "common.cuh"

namespace af {

namespace {

constexpr size_t kStaticAttnCntBytes = ((size_t)kStaticAttnMaxKVH + 64) * sizeof(unsigned);
constexpr size_t kStaticAttnBytes = kStaticAttnCntBytes + kStaticAttnPartFloats * sizeof(float);
static_assert(kStaticAttnCntBytes % 256 == 0, "partials start 256-byte aligned");

static __device__ __align__(256) unsigned char g_attn_static[kStaticAttnBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

}  // namespace

cudaError_t attn_static_scratch(float** part, unsigned** cnt, unsigned** err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {  // once per device, with that device current
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_static);
        if (e) return e;
        g_addr[dev] = p;
    }
    *cnt = reinterpret_cast<unsigned*>(g_addr[dev]);
    *err = *cnt + kStaticAttnMaxKVH;
    *part = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(g_addr[dev]) + kStaticAttnCntBytes);
    return cudaSuccess;
}

}  // namespace af
