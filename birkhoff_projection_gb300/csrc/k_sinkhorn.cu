// Fixed-iteration Sinkhorn-Knopp reference instantiations.
#include "b4_launch.cuh"

namespace b4 {
template cudaError_t launch<Mode::Sinkhorn, float, float>(const LaunchArgs&, cudaStream_t);
template cudaError_t launch<Mode::Sinkhorn, bf16_t, bf16_t>(const LaunchArgs&, cudaStream_t);
}  // namespace b4
