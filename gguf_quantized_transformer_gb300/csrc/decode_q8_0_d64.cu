// Persistent decode kernel instantiated for Q8_0 weights and head_dim 64.
#include "decode_impl.cuh"

namespace af {
template cudaError_t decode_launch_for<AF_Q8_0, 64>(const DecodePlan& p, cudaStream_t s, bool prepare);
}  // namespace af
