// Decode GEMV instantiations for Q5_K weights (kernel in qgemv_impl.cuh).
#include "qgemv_impl.cuh"

namespace af {
AF_QGEMV_INSTANTIATE(AF_Q5_K)
}  // namespace af
