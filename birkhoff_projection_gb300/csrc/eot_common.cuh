// eot_common.cuh -- pieces shared by the streaming entropic-OT kernels
// (eot_stream.cu: the potential update; eot_transport.cu: the transport
// application): tile constants, the bounded mbarrier wait, 2-D tensor-map
// encoding of packed point arrays, and the launchers of the packing and
// key-bias kernels (defined in eot_stream.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "b4_device.cuh"
#include "b4_launch.cuh"

namespace eot {

constexpr int BM = 128;        // query rows per CTA tile = MMA M = TMEM lanes
constexpr int KC = 32;         // fp32 elements per K chunk (one 128-byte swizzle row)
constexpr int ROW_PAD = 256;   // point counts are padded to this multiple
constexpr int KSTEP = 8;       // K of one kind::tf32 MMA
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr unsigned int kFaultEot = 4u;
constexpr int64_t kMaxPoints = (int64_t(1) << 31) - 512;

// mbarrier wait bounded in time and abandoned when another role of the CTA
// has given up (shared abort flag); a wait that runs out sets the abort flag
// and bit 2 of the fault latch.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* fault) {
  if (b4::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = b4::global_ns();
  for (;;) {
    if (b4::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (b4::global_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      if (fault != nullptr) atomicOr(fault, kFaultEot);
      return false;
    }
  }
}

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
inline size_t align_bytes(size_t v) { return (v + 1023) & ~static_cast<size_t>(1023); }

// Tensor map of a row-major fp32 array [outer rows, inner columns] (inner a
// multiple of 32, so rows are multiples of 128 bytes), box {32 columns,
// box_rows rows}, 128-byte swizzle: the K-major operand layout of tcgen05.
inline bool encode_rows128(CUtensorMap* map, const float* base, int64_t outer, int64_t inner,
                           int box_rows) {
  b4::EncodeTiledFn fn = b4::encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(KC), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Pack `rows` points of dimension d into [rows_pad, d_pad] (zero padding,
// rounded to TF32; `lo`, if not NULL, receives the TF32 remainder) with
// their fp32 squared norms (eot_stream.cu).
cudaError_t pack(const float* src, int64_t rows, int32_t d, int64_t rows_pad, int32_t d_pad,
                 float* hi, float* lo, float* norm, cudaStream_t s);

// Key bias in log2 units, (h_j - knorm_j) log2(e)/eps + log2(w_j), and -inf
// for the padding keys j >= nk (eot_stream.cu).
cudaError_t bias(const float* h, const float* log_w, const float* knorm, int64_t nk, int64_t nk_pad,
                 float eps, float* kb, cudaStream_t s);

}  // namespace eot
