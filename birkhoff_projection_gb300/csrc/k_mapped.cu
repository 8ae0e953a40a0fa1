// k_mapped.cu -- the fused forward + backward pass on tokens that stay in
// page-locked host memory, read and written by the kernel itself over the
// host link (zero copy): birkhoff4_forward_backward_mapped, declared in
// birkhoff4.h.  On a GPU whose host memory is coherently attached (GB300:
// NVLink-C2C), loads and stores issued by the SMs can move more bytes per
// second than the copy engines behind cudaMemcpyAsync, and no device
// staging buffer is needed.  Each CTA stages 128 tokens through shared
// memory so that every warp access to host memory is a contiguous 128-byte
// run; the per-token arithmetic is the same as the device passes'.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "b4_kernels.cuh"
#include "birkhoff4.h"

namespace b4 {

int record_cuda_error(cudaError_t e);              // birkhoff4_api.cu
unsigned int* device_fault_latch(cudaError_t* e);  // birkhoff4_api.cu

namespace {

constexpr int MT = 128;  // tokens per CTA tile

// 32-bit words per token and the conversions between a token's words and
// its registers, per storage type.
template <class T>
struct Words;
template <>
struct Words<float> {
  static constexpr int N = 16;
  __device__ __forceinline__ static void unpack(const uint32_t* w, Tok& t) {
#pragma unroll
    for (int k = 0; k < 8; ++k) t.v[k] = make_float2(__uint_as_float(w[2 * k]), __uint_as_float(w[2 * k + 1]));
  }
  __device__ __forceinline__ static void pack(const Tok& t, uint32_t* w) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      w[2 * k] = __float_as_uint(t.v[k].x);
      w[2 * k + 1] = __float_as_uint(t.v[k].y);
    }
  }
};
template <>
struct Words<bf16_t> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint32_t* w, Tok& t) {
#pragma unroll
    for (int k = 0; k < 8; ++k) t.v[k] = make_float2(bf16lo(w[k]), bf16hi(w[k]));
  }
  __device__ __forceinline__ static void pack(const Tok& t, uint32_t* w) {
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = pack_bf16(t.v[k].x, t.v[k].y);
  }
};

// Persistent over 128-token tiles: coalesced word loads of X and dP into
// shared memory (rows padded to an odd stride: conflict-free per-token
// access), the fused per-token pass, coalesced word stores of P (unless
// NULL) and dX.
template <class T>
__global__ void __launch_bounds__(MT) mapped_fused_kernel(const __grid_constant__ KParams a) {
  constexpr int W = Words<T>::N;
  constexpr int S = W + 1;
  __shared__ uint32_t s0[MT * S], s1[MT * S];
  const int tid = threadIdx.x;
  const uint32_t* gx = static_cast<const uint32_t*>(a.gin[0]);
  const uint32_t* gg = static_cast<const uint32_t*>(a.gin[1]);
  uint32_t* gp = static_cast<uint32_t*>(a.gout[0]);
  uint32_t* gd = static_cast<uint32_t*>(a.gout[1]);
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * MT; base < a.T;
       base += static_cast<int64_t>(gridDim.x) * MT) {
    const int64_t left = a.T - base;
    const int ntok = left < MT ? static_cast<int>(left) : MT;
    const int nw = ntok * W;
    const int64_t w0 = base * W;
    for (int i = tid; i < nw; i += MT) {
      s0[(i / W) * S + i % W] = __ldg(gx + w0 + i);
      s1[(i / W) * S + i % W] = __ldg(gg + w0 + i);
    }
    __syncthreads();
    if (tid < ntok) {
      Tok in0, in1, out0, out1;
      Words<T>::unpack(s0 + tid * S, in0);
      Words<T>::unpack(s1 + tid * S, in1);
      token_compute<Mode::Fused, T>(a, base + tid, true, in0, in1, out0, out1);
      Words<T>::pack(out0, s0 + tid * S);
      Words<T>::pack(out1, s1 + tid * S);
    }
    __syncthreads();
    for (int i = tid; i < nw; i += MT) {
      if (gp != nullptr) gp[w0 + i] = s0[(i / W) * S + i % W];
      gd[w0 + i] = s1[(i / W) * S + i % W];
    }
    __syncthreads();
  }
}

// Device address of a page-locked, mapped host buffer (NULL stays NULL).
cudaError_t device_view(const void* h, void** d) {
  *d = nullptr;
  if (h == nullptr) return cudaSuccess;
  return cudaHostGetDevicePointer(d, const_cast<void*>(h), 0);
}

template <class T>
int mapped_impl(const void* X_h, const void* dP_h, void* P_h, void* dX_h, int64_t n,
                cudaStream_t stream) {
  void *x = nullptr, *g = nullptr, *p = nullptr, *dx = nullptr;
  cudaError_t e = device_view(X_h, &x);
  if (e == cudaSuccess) e = device_view(dP_h, &g);
  if (e == cudaSuccess) e = device_view(P_h, &p);
  if (e == cudaSuccess) e = device_view(dX_h, &dx);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return B4_EINVAL;  // not page-locked (and mapped) host memory
  }
  int dev = 0;
  e = cudaGetDevice(&dev);
  int nsm = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return record_cuda_error(e);
  KParams a;
  memset(&a, 0, sizeof(a));
  a.gin[0] = x;
  a.gin[1] = g;
  a.gout[0] = p;
  a.gout[1] = dx;
  a.T = n;
  a.cfg.max_evals = 48;
  a.cfg.tol = 1e-6f;
  a.fault = device_fault_latch(&e);
  if (e != cudaSuccess) return record_cuda_error(e);
  const int64_t tiles = (n + MT - 1) / MT;
  const int grid = static_cast<int>(std::min<int64_t>(tiles, static_cast<int64_t>(nsm) * 16));
  mapped_fused_kernel<T><<<grid, MT, 0, stream>>>(a);
  return record_cuda_error(cudaGetLastError());
}

}  // namespace
}  // namespace b4

extern "C" int birkhoff4_forward_backward_mapped(const void* X_h, const void* dP_h, void* P_h,
                                                 void* dX_h, int64_t T, int32_t dtype,
                                                 birkhoff4_stream_t stream) {
  if (T < 0 || (dtype != B4_F32 && dtype != B4_BF16)) return B4_EINVAL;
  if (T == 0) return B4_OK;
  if (X_h == nullptr || dP_h == nullptr || dX_h == nullptr) return B4_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == B4_F32) return b4::mapped_impl<float>(X_h, dP_h, P_h, dX_h, T, s);
  return b4::mapped_impl<b4::bf16_t>(X_h, dP_h, P_h, dX_h, T, s);
}
