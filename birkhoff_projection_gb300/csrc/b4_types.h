// b4_types.h -- types shared by the host launch code, the kernels and the
// C ABI layer; no device code.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace b4 {

// Passes over a token stream.
enum class Mode : int {
  Forward = 0,    // X -> P (+ b, statistics)
  Backward = 1,   // (P, G) -> dX
  Recompute = 2,  // (X, G) -> dX, P recomputed in registers
  Fused = 3,      // (X, G) -> (P, dX)
  Sinkhorn = 4,   // X -> P, fixed iterations
};

// How the Newton passes assign tokens to threads (birkhoff4_opts.schedule).
enum class Schedule : int {
  Default = 0,  // the measured fastest (Queue)
  Queue = 1,    // one thread per token, slow tokens compacted into resume rounds
  Lane = 2,     // one thread per token for its whole solve
  Lanes4 = 3,   // four lanes per token, one row each (fp32 forward only)
};

// Stopping rule of the Newton forward.
struct NewtonCfg {
  int max_evals;  // cap on evaluations of P (>= 1)
  float tol;      // residual tolerance on max_j |colsum_j - 1|
};

// Storage type of a bf16 element (bit pattern); arithmetic is fp32.
struct bf16_t {
  uint16_t bits;
};

struct LaunchArgs {
  const void* in[2];            // inputs in pass order (X | P, then G)
  void* out[2];                 // outputs in pass order (P | dX, then dX)
  float* b;                     // Forward: optional [T,4] dual
  int32_t* evals_out;           // optional [T] evaluation counts
  unsigned long long* nonconv;  // optional counter
  int64_t T;
  NewtonCfg cfg;
  int32_t iters;                // Sinkhorn iterations
  unsigned int* fault;          // device fault latch
  Schedule schedule;            // Newton passes: token schedule
};

// Enqueue one pass (defined in b4_launch.cuh, instantiated per pass in the
// k_*.cu translation units).
template <Mode M, class TIn, class TOut>
cudaError_t launch(const LaunchArgs& la, cudaStream_t stream);

}  // namespace b4
