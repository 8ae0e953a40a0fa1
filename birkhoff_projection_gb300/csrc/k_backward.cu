// Backward pass instantiations: from a stored P, and with P recomputed.
#include "b4_launch.cuh"

namespace b4 {
template cudaError_t launch<Mode::Backward, float, float>(const LaunchArgs&, cudaStream_t);
template cudaError_t launch<Mode::Backward, bf16_t, bf16_t>(const LaunchArgs&, cudaStream_t);
template cudaError_t launch<Mode::Recompute, float, float>(const LaunchArgs&, cudaStream_t);
template cudaError_t launch<Mode::Recompute, bf16_t, bf16_t>(const LaunchArgs&, cudaStream_t);
}  // namespace b4
