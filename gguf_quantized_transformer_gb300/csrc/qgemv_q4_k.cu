// Decode GEMV instantiations for Q4_K weights (kernel in qgemv_impl.cuh).
#include "qgemv_impl.cuh"

namespace af {
AF_QGEMV_INSTANTIATE(AF_Q4_K)
}  // namespace af
