// b4_launch.cuh -- host-side launch of the token-stream kernels: TMA tensor
// maps, tile configuration per pass, persistent grid sizing, chunking of very
// long token arrays.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "b4_kernels.cuh"
#include "b4_lanes4.cuh"
#include "b4_queue.cuh"

namespace b4 {

// Tile shape per pass: tokens per CTA step, input stages, output stages,
// minimum resident CTAs per SM (register budget).  Compute-heavy passes
// (Newton forward, fused, recompute) trade stages for resident warps;
// streaming passes keep more bytes in flight.
#ifndef B4_FWD_TILE
#define B4_FWD_TILE 128
#endif
#ifndef B4_FWD_NSTAGE
#define B4_FWD_NSTAGE 2
#endif
#ifndef B4_FWD_NOSTAGE
#define B4_FWD_NOSTAGE 1
#endif
#ifndef B4_FWD_MINB
#define B4_FWD_MINB 1
#endif
#ifndef B4_FUSED_MINB
#define B4_FUSED_MINB 6
#endif
#ifndef B4_BWD_TILE
#define B4_BWD_TILE 256
#endif
#ifndef B4_BWD_NSTAGE
#define B4_BWD_NSTAGE 2
#endif
#ifndef B4_BWD_NOSTAGE
#define B4_BWD_NOSTAGE 3
#endif
#ifndef B4_BWD_MINB
#define B4_BWD_MINB 1
#endif
// Compacting schedule of the Newton passes (b4_queue.cuh): warps per CTA,
// TMA stages, queue entries per warp, evaluations of a fresh round and of a
// resume round, minimum resident CTAs per SM.
#ifndef B4_Q_WARPS
#define B4_Q_WARPS 4
#endif
#ifndef B4_Q_NSTAGE
#define B4_Q_NSTAGE 2
#endif
#ifndef B4_Q_QC
#define B4_Q_QC 64
#endif
// Fresh-round length per pass, swept on GB300 at 2^26 N(0,10^2) tokens
// (K1 = 6 / 7 / 8 / 9 / 10): forward 2.928 / 2.840 / 2.911 / 3.079 /
// 3.279 ms; fused 4.529 / 4.143 / 3.971 / 4.006 / 4.149 ms; recompute
// 4.088 / 3.790 / 3.738 / 3.854 / 4.031 ms; N(0,1) unchanged (every token is
// solved within 5 evaluations).  A resume re-reads X (and, for the passes
// with a backward, dP) after it may have left L2, so the passes with a
// backward prefer the longer round.
#ifndef B4_Q_K1_FWD
#define B4_Q_K1_FWD 7
#endif
#ifndef B4_Q_K1_BWD
#define B4_Q_K1_BWD 8
#endif
#ifndef B4_Q_K2
#define B4_Q_K2 2
#endif
#ifndef B4_Q_MINB_FWD
#define B4_Q_MINB_FWD 8
#endif
#ifndef B4_Q_MINB_FUSED
#define B4_Q_MINB_FUSED 5
#endif
#ifndef B4_Q_MINB_RECOMPUTE
#define B4_Q_MINB_RECOMPUTE 7
#endif
#ifndef B4_Q_MINB_BF16
#define B4_Q_MINB_BF16 8
#endif

template <Mode M, class TIn>
struct TileCfg {
  static constexpr bool STREAMING = (M == Mode::Backward);
  static constexpr int TILE = STREAMING ? B4_BWD_TILE : B4_FWD_TILE;
  static constexpr int NSTAGE = STREAMING ? B4_BWD_NSTAGE : B4_FWD_NSTAGE;
  static constexpr int NOSTAGE = STREAMING ? B4_BWD_NOSTAGE : B4_FWD_NOSTAGE;
  static constexpr int MINB = STREAMING ? B4_BWD_MINB : (M == Mode::Forward ? B4_FWD_MINB : B4_FUSED_MINB);
};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Tensor map of a [T, 16] row array (one token per row), box [16, tile].
template <class T>
inline bool encode_rows(CUtensorMap* map, const void* ptr, int64_t ntok, int tile) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {16, static_cast<cuuint64_t>(ntok)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(TileIO<T>::ROW_BYTES)};
  const cuuint32_t box[2] = {16, static_cast<cuuint32_t>(tile)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, TileIO<T>::TMA_TYPE, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, TileIO<T>::TMA_SWIZZLE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int sm_count(int dev) {
  static std::atomic<int> cache[64];
  if (dev < 0 || dev >= 64) return 0;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kChunkTokens = int64_t(1) << 30;  // TMA row coordinates stay in int32

template <class T>
inline const void* advance(const void* p, int64_t tokens) {
  return p == nullptr ? nullptr
                      : static_cast<const void*>(static_cast<const unsigned char*>(p) +
                                                 tokens * TileIO<T>::ROW_BYTES);
}
template <class T>
inline void* advance(void* p, int64_t tokens) {
  return p == nullptr ? nullptr : static_cast<void*>(static_cast<unsigned char*>(p) + tokens * TileIO<T>::ROW_BYTES);
}

// The Newton passes with compaction of slow tokens (queue_kernel): X by TMA
// tiles of B4_Q_WARPS x 32 tokens, results stored directly.
template <Mode M, class TIn, class TOut>
cudaError_t launch_queue(const LaunchArgs& la, cudaStream_t stream, int dev, int nsm) {
  using Q = QueueShape<M, TIn, TOut, B4_Q_WARPS, B4_Q_NSTAGE, B4_Q_QC>;
  // Register caps, swept on GB300: the fp32 fused pass (256 B per token,
  // close to HBM) is fastest with 5 CTAs per SM, the compute-heavier bf16
  // passes and the recompute pass with more.
  constexpr bool BF16 = std::is_same<TIn, bf16_t>::value;
  constexpr int MINB = M == Mode::Forward ? B4_Q_MINB_FWD
                       : BF16             ? B4_Q_MINB_BF16
                       : M == Mode::Fused ? B4_Q_MINB_FUSED
                                          : B4_Q_MINB_RECOMPUTE;
  constexpr int K1 = M == Mode::Forward ? B4_Q_K1_FWD : B4_Q_K1_BWD;
  auto kern = queue_kernel<M, TIn, TOut, B4_Q_WARPS, B4_Q_NSTAGE, B4_Q_QC, K1, B4_Q_K2, MINB>;
  static std::atomic<int> cap_cache[64];
  int grid_cap = dev < 64 ? cap_cache[dev].load(std::memory_order_acquire) : 0;
  cudaError_t err;
  if (grid_cap == 0) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Q::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    int occ = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Q::TILE, Q::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    grid_cap = nsm * std::max(occ, 1);
    if (dev < 64) cap_cache[dev].store(grid_cap, std::memory_order_release);
  }
  constexpr int NIN = ModeTraits<M>::NIN;
  constexpr int NOUT = ModeTraits<M>::NOUT;
  for (int64_t done = 0; done < la.T; done += kChunkTokens) {
    const int64_t n = std::min(la.T - done, kChunkTokens);
    KParams p;
    memset(&p, 0, sizeof(p));
    for (int k = 0; k < NIN; ++k) p.gin[k] = advance<TIn>(la.in[k], done);
    for (int k = 0; k < NOUT; ++k) p.gout[k] = advance<TOut>(la.out[k], done);
    p.b = la.b ? la.b + 4 * done : nullptr;
    p.b_vec = aligned16(la.b) ? 1 : 0;
    p.evals_out = la.evals_out ? la.evals_out + done : nullptr;
    p.nonconv = la.nonconv;
    p.fault = la.fault;
    p.T = n;
    p.cfg = la.cfg;
    if (!encode_rows<TIn>(&p.in[0], p.gin[0], n, Q::TILE)) return cudaErrorInvalidValue;
    p.ntiles = static_cast<int32_t>((n + Q::TILE - 1) / Q::TILE);
    const int grid = static_cast<int>(std::min<int64_t>(p.ntiles, grid_cap));
    kern<<<grid, Q::TILE, Q::SMEM_BYTES, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

// The fp32 forward with four lanes per token (lanes4_kernel): 256-thread CTAs,
// a persistent grid, tokens read and written as contiguous 16-byte rows.
inline cudaError_t launch_lanes4(const LaunchArgs& la, cudaStream_t stream, int dev, int nsm) {
  auto kern = lanes4_kernel<float, float>;
  static std::atomic<int> cap_cache[64];
  int grid_cap = dev < 64 ? cap_cache[dev].load(std::memory_order_acquire) : 0;
  cudaError_t err;
  if (grid_cap == 0) {
    int occ = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 256, 0);
    if (err != cudaSuccess) return err;
    grid_cap = nsm * std::max(occ, 1);
    if (dev < 64) cap_cache[dev].store(grid_cap, std::memory_order_release);
  }
  for (int64_t done = 0; done < la.T; done += kChunkTokens) {
    const int64_t n = std::min(la.T - done, kChunkTokens);
    KParams p;
    memset(&p, 0, sizeof(p));
    p.gin[0] = advance<float>(la.in[0], done);
    p.gout[0] = advance<float>(la.out[0], done);
    p.b = la.b ? la.b + 4 * done : nullptr;
    p.b_vec = aligned16(la.b) ? 1 : 0;
    p.evals_out = la.evals_out ? la.evals_out + done : nullptr;
    p.nonconv = la.nonconv;
    p.fault = la.fault;
    p.T = n;
    p.cfg = la.cfg;
    const int grid = static_cast<int>(std::min<int64_t>((n + 63) / 64, grid_cap));
    kern<<<grid, 256, 0, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

// Enqueue one pass over la.T tokens on `stream`.  Returns the CUDA error of
// the preparation or launch (cudaSuccess if everything was enqueued).
template <Mode M, class TIn, class TOut>
cudaError_t launch(const LaunchArgs& la, cudaStream_t stream) {
  constexpr int NIN = ModeTraits<M>::NIN;
  constexpr int NOUT = ModeTraits<M>::NOUT;
  using C = TileCfg<M, TIn>;
  using S = StreamShape<M, TIn, TOut, C::TILE, C::NSTAGE, C::NOSTAGE>;

  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int nsm = sm_count(dev);
  if (nsm <= 0) return cudaErrorInvalidDevice;

  bool aligned = true;
  for (int k = 0; k < NIN; ++k) aligned = aligned && aligned16(la.in[k]);
  for (int k = 0; k < NOUT; ++k) aligned = aligned && aligned16(la.out[k]);

  // four lanes per token: the fp32 forward (16-byte aligned tokens)
  if constexpr (M == Mode::Forward && std::is_same<TIn, float>::value && std::is_same<TOut, float>::value) {
    if (aligned && la.schedule == Schedule::Lanes4) return launch_lanes4(la, stream, dev, nsm);
  }
  // the compacting schedule for the Newton passes (16-byte aligned tokens)
  constexpr bool NEWTON = (M == Mode::Forward || M == Mode::Fused || M == Mode::Recompute);
  if constexpr (NEWTON) {
    if (aligned && (la.schedule == Schedule::Default || la.schedule == Schedule::Queue))
      return launch_queue<M, TIn, TOut>(la, stream, dev, nsm);
  }

  auto kern = stream_kernel<M, TIn, TOut, C::TILE, C::NSTAGE, C::NOSTAGE, C::MINB>;
  const int smem_bytes = S::SMEM_BYTES;
  const int box_rows = C::TILE;
  // Persistent grid size (SMs x resident CTAs), worked out once per device
  // for this kernel: the shared-memory opt-in and the occupancy query are
  // host calls that would otherwise dominate small launches.
  static std::atomic<int> cap_cache[64];
  int grid_cap = 0;
  if (aligned) {
    grid_cap = dev < 64 ? cap_cache[dev].load(std::memory_order_acquire) : 0;
    if (grid_cap == 0) {
      err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
      if (err != cudaSuccess) return err;
      int occ = 0;
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::TILE, smem_bytes);
      if (err != cudaSuccess) return err;
      grid_cap = nsm * std::max(occ, 1);
      if (dev < 64) cap_cache[dev].store(grid_cap, std::memory_order_release);
    }
  }

  for (int64_t done = 0; done < la.T; done += kChunkTokens) {
    const int64_t n = std::min(la.T - done, kChunkTokens);
    KParams p;
    memset(&p, 0, sizeof(p));
    for (int k = 0; k < NIN; ++k) p.gin[k] = advance<TIn>(la.in[k], done);
    for (int k = 0; k < NOUT; ++k) p.gout[k] = advance<TOut>(la.out[k], done);
    p.b = la.b ? la.b + 4 * done : nullptr;
    p.b_vec = aligned16(la.b) ? 1 : 0;
    p.evals_out = la.evals_out ? la.evals_out + done : nullptr;
    p.nonconv = la.nonconv;
    p.fault = la.fault;
    p.T = n;
    p.cfg = la.cfg;
    p.iters = la.iters;
    bool use_tma = aligned;
    if (use_tma) {
      for (int k = 0; k < NIN && use_tma; ++k) use_tma = encode_rows<TIn>(&p.in[k], p.gin[k], n, box_rows);
      for (int k = 0; k < NOUT && use_tma; ++k) use_tma = encode_rows<TOut>(&p.out[k], p.gout[k], n, box_rows);
    }
    if (use_tma) {
      p.ntiles = static_cast<int32_t>((n + box_rows - 1) / box_rows);
      const int grid = static_cast<int>(std::min<int64_t>(p.ntiles, grid_cap));
      kern<<<grid, C::TILE, smem_bytes, stream>>>(p);
    } else {
      const int64_t blocks = (n + 255) / 256;
      const int grid = static_cast<int>(std::min<int64_t>(blocks, int64_t(nsm) * 8));
      plain_kernel<M, TIn, TOut><<<grid, 256, 0, stream>>>(p);
    }
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace b4
