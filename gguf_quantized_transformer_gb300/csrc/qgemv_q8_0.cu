// Decode GEMV instantiations for Q8_0 weights (kernel in qgemv_impl.cuh).
#include "qgemv_impl.cuh"

namespace af {
AF_QGEMV_INSTANTIATE(AF_Q8_0)
}  // namespace af
