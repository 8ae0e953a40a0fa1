// Fused forward + backward instantiations ((X, G) -> (P, dX)).
#include "b4_launch.cuh"

namespace b4 {
template cudaError_t launch<Mode::Fused, float, float>(const LaunchArgs&, cudaStream_t);
template cudaError_t launch<Mode::Fused, bf16_t, bf16_t>(const LaunchArgs&, cudaStream_t);
}  // namespace b4
