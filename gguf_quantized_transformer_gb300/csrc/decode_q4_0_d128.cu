// Persistent decode kernel instantiated for Q4_0 weights and head_dim 128.
#include "decode_impl.cuh"

namespace af {
template cudaError_t decode_launch_for<AF_Q4_0, 128>(const DecodePlan& p, cudaStream_t s, bool prepare);
}  // namespace af
