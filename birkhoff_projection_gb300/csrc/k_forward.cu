// Forward pass instantiations (X -> P), all dtype pairs.
#include "b4_launch.cuh"

namespace b4 {
template cudaError_t launch<Mode::Forward, float, float>(const LaunchArgs&, cudaStream_t);
template cudaError_t launch<Mode::Forward, bf16_t, bf16_t>(const LaunchArgs&, cudaStream_t);
template cudaError_t launch<Mode::Forward, bf16_t, float>(const LaunchArgs&, cudaStream_t);
template cudaError_t launch<Mode::Forward, float, bf16_t>(const LaunchArgs&, cudaStream_t);
}  // namespace b4
