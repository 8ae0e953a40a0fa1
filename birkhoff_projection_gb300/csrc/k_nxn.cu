// n x n kernels (2 <= n <= 8) and their C ABI entry points
// birkhoff4_forward_nxn / birkhoff4_backward_nxn (declared in birkhoff4.h).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "b4_launch.cuh"
#include "b4_nxn.cuh"
#include "birkhoff4.h"

namespace b4 {

int record_cuda_error(cudaError_t e);  // birkhoff4_api.cu

namespace {

template <int N, int TILE, bool FWD>
cudaError_t launch_nxn(const NxnParams& p, cudaStream_t stream) {
  using S = NxnShape<N>;
  constexpr int SMEM = (FWD ? 1 : 2) * TILE * S::STRIDE * static_cast<int>(sizeof(float));
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int nsm = sm_count(dev);
  if (nsm <= 0) return cudaErrorInvalidDevice;
  auto kern = nxn_kernel<N, TILE, FWD>;
  static std::atomic<int> cap_cache[64];
  int cap = dev < 64 ? cap_cache[dev].load(std::memory_order_acquire) : 0;
  if (cap == 0) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (err != cudaSuccess) return err;
    int occ = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, TILE, SMEM);
    if (err != cudaSuccess) return err;
    cap = nsm * std::max(occ, 1);
    if (dev < 64) cap_cache[dev].store(cap, std::memory_order_release);
  }
  const int64_t tiles = (p.T + TILE - 1) / TILE;
  const int grid = static_cast<int>(std::min<int64_t>(tiles, cap));
  kern<<<grid, TILE, SMEM, stream>>>(p);
  return cudaGetLastError();
}

template <bool FWD>
cudaError_t dispatch_nxn(int n, const NxnParams& p, cudaStream_t s) {
  constexpr int TF = 128, TB = 64;
  switch (n) {
    case 2: return FWD ? launch_nxn<2, TF, true>(p, s) : launch_nxn<2, TB, false>(p, s);
    case 3: return FWD ? launch_nxn<3, TF, true>(p, s) : launch_nxn<3, TB, false>(p, s);
    case 4: return FWD ? launch_nxn<4, TF, true>(p, s) : launch_nxn<4, TB, false>(p, s);
    case 5: return FWD ? launch_nxn<5, TF, true>(p, s) : launch_nxn<5, TB, false>(p, s);
    case 6: return FWD ? launch_nxn<6, TF, true>(p, s) : launch_nxn<6, TB, false>(p, s);
    case 7: return FWD ? launch_nxn<7, TF, true>(p, s) : launch_nxn<7, TB, false>(p, s);
    case 8: return FWD ? launch_nxn<8, TF, true>(p, s) : launch_nxn<8, TB, false>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace b4

extern "C" int birkhoff4_forward_nxn(const float* X, float* P, float* b, int32_t n, int64_t T,
                                     birkhoff4_stream_t stream) {
  if (T < 0 || n < 2 || n > 8) return B4_EINVAL;
  if (T == 0) return B4_OK;
  if (X == nullptr || P == nullptr) return B4_EINVAL;
  b4::NxnParams p;
  p.in0 = X;
  p.in1 = nullptr;
  p.out = P;
  p.b = b;
  p.T = T;
  p.cfg.max_evals = 48;
  p.cfg.tol = 1e-6f;
  return b4::record_cuda_error(b4::dispatch_nxn<true>(n, p, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" int birkhoff4_backward_nxn(const float* P, const float* dP, float* dX, int32_t n,
                                      int64_t T, birkhoff4_stream_t stream) {
  if (T < 0 || n < 2 || n > 8) return B4_EINVAL;
  if (T == 0) return B4_OK;
  if (P == nullptr || dP == nullptr || dX == nullptr) return B4_EINVAL;
  b4::NxnParams p;
  p.in0 = P;
  p.in1 = dP;
  p.out = dX;
  p.b = nullptr;
  p.T = T;
  p.cfg.max_evals = 48;
  p.cfg.tol = 1e-6f;
  return b4::record_cuda_error(b4::dispatch_nxn<false>(n, p, reinterpret_cast<cudaStream_t>(stream)));
}
