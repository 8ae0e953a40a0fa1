// birkhoff4_api.cu -- the extern "C" boundary of libbirkhoff4.so (declared
// and documented in include/birkhoff4.h): argument checks on the host, dtype
// dispatch to the pass launchers, diagnostics.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "b4_context.cuh"
#include "b4_device.cuh"
#include "b4_types.h"
#include "birkhoff4.h"

namespace b4 {

// Device-side fault latch, one per device the library is loaded on.  Host
// code only ever uses the address obtained from cudaGetSymbolAddress.
__device__ unsigned int g_fault_latch;

namespace {

thread_local int t_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return B4_OK;
  t_last_cuda_error = static_cast<int>(e);
  return B4_ECUDA;
}

// Device address of g_fault_latch on the current device (cached per device
// and context).
unsigned int* fault_latch(cudaError_t* err) {
  static SymbolCache cache;
  return static_cast<unsigned int*>(cached_symbol_address(
      cache, [](void** q) { return cudaGetSymbolAddress(q, g_fault_latch); }, err));
}

bool dtype_ok(int32_t d) { return d == B4_F32 || d == B4_BF16; }

NewtonCfg newton_cfg(const birkhoff4_opts* o) {
  NewtonCfg c;
  c.max_evals = (o != nullptr && o->max_evals > 0) ? o->max_evals : 48;
  c.tol = (o != nullptr && o->tol > 0.0f) ? o->tol : 1e-6f;
  return c;
}

template <Mode M, class TIn, class TOut>
int run(LaunchArgs la, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  la.fault = fault_latch(&e);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch<M, TIn, TOut>(la, s));
}

LaunchArgs blank(int64_t T) {
  LaunchArgs la;
  la.in[0] = la.in[1] = nullptr;
  la.out[0] = la.out[1] = nullptr;
  la.b = nullptr;
  la.evals_out = nullptr;
  la.nonconv = nullptr;
  la.T = T;
  la.cfg = newton_cfg(nullptr);
  la.iters = 0;
  la.fault = nullptr;
  la.schedule = Schedule::Default;
  return la;
}

// Options common to the Newton entry points: checks, then copied into la.
int apply_opts(const birkhoff4_opts* o, LaunchArgs* la) {
  if (o->max_evals < 0 || o->max_evals > 1024) return B4_EINVAL;
  if (!(o->tol >= 0.0f) || std::isinf(o->tol)) return B4_EINVAL;
  if (o->schedule < B4_SCHED_DEFAULT || o->schedule > B4_SCHED_LANES4) return B4_EINVAL;
  la->evals_out = o->evals_out;
  la->nonconv = o->nonconv_count;
  la->cfg = newton_cfg(o);
  la->schedule = static_cast<Schedule>(o->schedule);
  return B4_OK;
}

int forward_impl(const void* X, void* P, float* b, int64_t T, const birkhoff4_opts* o,
                 cudaStream_t s) {
  if (T < 0 || o == nullptr) return B4_EINVAL;
  if (!dtype_ok(o->in_dtype) || !dtype_ok(o->out_dtype)) return B4_EINVAL;
  LaunchArgs la = blank(T);
  const int st = apply_opts(o, &la);
  if (st != B4_OK) return st;
  if (o->schedule == B4_SCHED_LANES4 && (o->in_dtype != B4_F32 || o->out_dtype != B4_F32))
    return B4_ENOTIMPL;
  if (T == 0) return B4_OK;
  if (X == nullptr || P == nullptr) return B4_EINVAL;
  la.in[0] = X;
  la.out[0] = P;
  la.b = b;
  const bool fin = o->in_dtype == B4_F32, fout = o->out_dtype == B4_F32;
  if (fin && fout) return run<Mode::Forward, float, float>(la, s);
  if (!fin && !fout) return run<Mode::Forward, bf16_t, bf16_t>(la, s);
  if (!fin && fout) return run<Mode::Forward, bf16_t, float>(la, s);
  return run<Mode::Forward, float, bf16_t>(la, s);
}

template <class T>
int backward_impl(const void* X, const void* P, const void* dP, void* dX, int64_t n,
                  cudaStream_t s) {
  if (n < 0) return B4_EINVAL;
  if (n == 0) return B4_OK;
  if (dP == nullptr || dX == nullptr || (P == nullptr && X == nullptr)) return B4_EINVAL;
  LaunchArgs la = blank(n);
  la.in[1] = dP;
  la.out[0] = dX;
  if (P != nullptr) {
    la.in[0] = P;
    return run<Mode::Backward, T, T>(la, s);
  }
  la.in[0] = X;
  return run<Mode::Recompute, T, T>(la, s);
}

template <class T>
int fused_impl(const void* X, const void* dP, void* P, void* dX, int64_t n, cudaStream_t s,
               const birkhoff4_opts* o = nullptr) {
  if (n < 0) return B4_EINVAL;
  LaunchArgs la = blank(n);
  if (o != nullptr) {
    const int st = apply_opts(o, &la);
    if (st != B4_OK) return st;
    if (o->schedule == B4_SCHED_LANES4) return B4_ENOTIMPL;  // forward only
  }
  if (n == 0) return B4_OK;
  if (X == nullptr || dP == nullptr || dX == nullptr) return B4_EINVAL;
  la.in[0] = X;
  la.in[1] = dP;
  if (P == nullptr) {
    la.out[0] = dX;
    return run<Mode::Recompute, T, T>(la, s);
  }
  la.out[0] = P;
  la.out[1] = dX;
  return run<Mode::Fused, T, T>(la, s);
}

template <class T>
int sinkhorn_impl(const void* X, void* P, int iters, int64_t n, cudaStream_t s) {
  if (n < 0 || iters < 0) return B4_EINVAL;
  if (n == 0) return B4_OK;
  if (X == nullptr || P == nullptr) return B4_EINVAL;
  LaunchArgs la = blank(n);
  la.in[0] = X;
  la.out[0] = P;
  la.iters = iters;
  return run<Mode::Sinkhorn, T, T>(la, s);
}

// Chunked host <-> device streaming of the fused pass over caller streams.
template <class T>
int host_stream_impl(const void* X_h, const void* dP_h, void* P_h, void* dX_h, int64_t n,
                     unsigned char* ws, size_t chunk, const birkhoff4_stream_t* streams,
                     int nstreams) {
  const size_t rb = TileIO<T>::ROW_BYTES;
  for (int64_t c0 = 0, ci = 0; c0 < n; c0 += static_cast<int64_t>(chunk), ++ci) {
    const int64_t m = std::min<int64_t>(static_cast<int64_t>(chunk), n - c0);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(streams[ci % nstreams]);
    unsigned char* slot = ws + static_cast<size_t>(ci % nstreams) * 4 * chunk * rb;
    unsigned char* dx = slot;
    unsigned char* dg = slot + chunk * rb;
    unsigned char* dp = slot + 2 * chunk * rb;
    unsigned char* dd = slot + 3 * chunk * rb;
    const size_t off = static_cast<size_t>(c0) * rb, bytes = static_cast<size_t>(m) * rb;
    cudaError_t e = cudaMemcpyAsync(dx, static_cast<const unsigned char*>(X_h) + off, bytes,
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dg, static_cast<const unsigned char*>(dP_h) + off, bytes,
                          cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_status(e);
    const int st = fused_impl<T>(dx, dg, P_h ? dp : nullptr, dd, m, s);
    if (st != B4_OK) return st;
    if (P_h != nullptr) {
      e = cudaMemcpyAsync(static_cast<unsigned char*>(P_h) + off, dp, bytes, cudaMemcpyDeviceToHost, s);
      if (e != cudaSuccess) return cuda_status(e);
    }
    e = cudaMemcpyAsync(static_cast<unsigned char*>(dX_h) + off, dd, bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return B4_OK;
}

int host_stream_check(const void* X_h, const void* dP_h, const void* dX_h, int64_t n, int32_t dtype,
                      const void* ws, size_t ws_bytes, const birkhoff4_stream_t* streams,
                      int nstreams, size_t* chunk) {
  if (n < 0 || !dtype_ok(dtype) || nstreams < 1 || nstreams > 16) return B4_EINVAL;
  if (n == 0) return B4_OK;
  if (X_h == nullptr || dP_h == nullptr || dX_h == nullptr || ws == nullptr || streams == nullptr)
    return B4_EINVAL;
  const size_t rb = dtype == B4_F32 ? 64 : 32;
  *chunk = ws_bytes / (static_cast<size_t>(nstreams) * 4 * rb);
  if (*chunk < 1) return B4_EINVAL;
  return B4_OK;
}

// Throughput probe of MUFU ex2: eight independent recurrences a <- 2^-a per
// thread (each stays in [0.5, 1]), so the MUFU pipe, not latency, limits it.
__global__ void __launch_bounds__(256) mufu_probe_kernel(float* sink, int iters) {
  float a0 = 0.50f + threadIdx.x * 1e-6f, a1 = 0.55f, a2 = 0.60f, a3 = 0.65f;
  float a4 = 0.70f, a5 = 0.75f, a6 = 0.80f, a7 = 0.85f;
  for (int i = 0; i < iters; ++i) {
    a0 = ex2(-a0);
    a1 = ex2(-a1);
    a2 = ex2(-a2);
    a3 = ex2(-a3);
    a4 = ex2(-a4);
    a5 = ex2(-a5);
    a6 = ex2(-a6);
    a7 = ex2(-a7);
  }
  const float s = ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
  if (s < 0.0f && sink != nullptr) sink[blockIdx.x] = s;  // keeps the loop alive; never true
}

// One CTA waits on an mbarrier that nothing completes, with a time limit.
__global__ void selftest_wait_kernel(unsigned int* fault, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0u, limit_ns);
  const int timed_out = __syncthreads_or(!ok);
  if (timed_out && threadIdx.x == 0) atomicOr(fault, 2u);
}

}  // namespace

// Records a CUDA error for birkhoff4_last_cuda_error (for other translation
// units of the library) and returns B4_ECUDA (B4_OK for cudaSuccess).
int record_cuda_error(cudaError_t e) { return cuda_status(e); }

// The fault latch's device address for kernels launched from other
// translation units (bounded waits that run out set bits in it).
unsigned int* device_fault_latch(cudaError_t* err) { return fault_latch(err); }

}  // namespace b4

using namespace b4;

extern "C" {

int birkhoff4_version(void) { return BIRKHOFF4_VERSION; }

const char* birkhoff4_strerror(int code) {
  switch (code) {
    case B4_OK:
      return "success";
    case B4_EINVAL:
      return "invalid argument (NULL pointer with T > 0, T < 0, bad option or iters < 0)";
    case B4_ECUDA:
      return "CUDA error while preparing or launching a kernel";
    case B4_ENOTIMPL:
      return "not implemented in this build";
    case B4_ESCRATCH:
      return "chunk does not fit the library's static scratch (B4_STATIC_SCRATCH_BYTES)";
    default:
      return "unknown status code";
  }
}

int birkhoff4_last_cuda_error(void) { return t_last_cuda_error; }

int birkhoff4_forward(const float* X, float* P, float* b, int64_t T, birkhoff4_stream_t stream) {
  birkhoff4_opts o = {};
  o.in_dtype = B4_F32;
  o.out_dtype = B4_F32;
  return forward_impl(X, P, b, T, &o, reinterpret_cast<cudaStream_t>(stream));
}

int birkhoff4_forward_bf16(const uint16_t* X, uint16_t* P, float* b, int64_t T,
                           birkhoff4_stream_t stream) {
  birkhoff4_opts o = {};
  o.in_dtype = B4_BF16;
  o.out_dtype = B4_BF16;
  return forward_impl(X, P, b, T, &o, reinterpret_cast<cudaStream_t>(stream));
}

int birkhoff4_forward_ex(const void* X, void* P, float* b, int64_t T, const birkhoff4_opts* opts,
                         birkhoff4_stream_t stream) {
  return forward_impl(X, P, b, T, opts, reinterpret_cast<cudaStream_t>(stream));
}

int birkhoff4_backward(const float* X, const float* P, const float* dP, float* dX, int64_t T,
                       birkhoff4_stream_t stream) {
  return backward_impl<float>(X, P, dP, dX, T, reinterpret_cast<cudaStream_t>(stream));
}

int birkhoff4_backward_bf16(const uint16_t* X, const uint16_t* P, const uint16_t* dP, uint16_t* dX,
                            int64_t T, birkhoff4_stream_t stream) {
  return backward_impl<bf16_t>(X, P, dP, dX, T, reinterpret_cast<cudaStream_t>(stream));
}

int birkhoff4_forward_backward(const float* X, const float* dP, float* P, float* dX, int64_t T,
                               birkhoff4_stream_t stream) {
  return fused_impl<float>(X, dP, P, dX, T, reinterpret_cast<cudaStream_t>(stream));
}

int birkhoff4_forward_backward_bf16(const uint16_t* X, const uint16_t* dP, uint16_t* P,
                                    uint16_t* dX, int64_t T, birkhoff4_stream_t stream) {
  return fused_impl<bf16_t>(X, dP, P, dX, T, reinterpret_cast<cudaStream_t>(stream));
}

int birkhoff4_forward_backward_ex(const void* X, const void* dP, void* P, void* dX, int64_t T,
                                  const birkhoff4_opts* opts, birkhoff4_stream_t stream) {
  if (opts == nullptr || !dtype_ok(opts->in_dtype) || opts->out_dtype != opts->in_dtype)
    return B4_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (opts->in_dtype == B4_F32) return fused_impl<float>(X, dP, P, dX, T, s, opts);
  return fused_impl<bf16_t>(X, dP, P, dX, T, s, opts);
}

int birkhoff4_forward_backward_host(const void* X_h, const void* dP_h, void* P_h, void* dX_h,
                                    int64_t T, int32_t dtype, void* workspace,
                                    size_t workspace_bytes, const birkhoff4_stream_t* streams,
                                    int32_t nstreams) {
  size_t chunk = 0;
  const int st = host_stream_check(X_h, dP_h, dX_h, T, dtype, workspace, workspace_bytes, streams,
                                   nstreams, &chunk);
  if (st != B4_OK || T == 0) return st;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  if (dtype == B4_F32)
    return host_stream_impl<float>(X_h, dP_h, P_h, dX_h, T, ws, chunk, streams, nstreams);
  return host_stream_impl<bf16_t>(X_h, dP_h, P_h, dX_h, T, ws, chunk, streams, nstreams);
}

int birkhoff4_sinkhorn(const float* X, float* P, int iters, int64_t T, birkhoff4_stream_t stream) {
  return sinkhorn_impl<float>(X, P, iters, T, reinterpret_cast<cudaStream_t>(stream));
}

int birkhoff4_sinkhorn_bf16(const uint16_t* X, uint16_t* P, int iters, int64_t T,
                            birkhoff4_stream_t stream) {
  return sinkhorn_impl<bf16_t>(X, P, iters, T, reinterpret_cast<cudaStream_t>(stream));
}

int birkhoff4_device_status(unsigned int* out, int clear) {
  if (out == nullptr) return B4_EINVAL;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e);
  unsigned int* latch = fault_latch(&e);
  if (latch == nullptr) return cuda_status(e);
  e = cudaMemcpy(out, latch, sizeof(unsigned int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  if (clear) {
    e = cudaMemset(latch, 0, sizeof(unsigned int));
    if (e != cudaSuccess) return cuda_status(e);
    e = cudaDeviceSynchronize();
  }
  return cuda_status(e);
}

int birkhoff4_selftest_wait_timeout(int64_t limit_ns) {
  if (limit_ns < 1 || limit_ns > 1000000000) return B4_EINVAL;
  cudaError_t e = cudaSuccess;
  unsigned int* latch = fault_latch(&e);
  if (latch == nullptr) return cuda_status(e);
  selftest_wait_kernel<<<1, 32>>>(latch, static_cast<uint64_t>(limit_ns));
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(cudaDeviceSynchronize());
}

int birkhoff4_mufu_probe(float* out_host, int n_blocks, int iters, birkhoff4_stream_t stream) {
  if (out_host == nullptr || n_blocks < 1 || iters < 1) return B4_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaEvent_t e0, e1;
  cudaError_t e = cudaEventCreate(&e0);
  if (e != cudaSuccess) return cuda_status(e);
  e = cudaEventCreate(&e1);
  if (e != cudaSuccess) {
    cudaEventDestroy(e0);
    return cuda_status(e);
  }
  cudaEventRecord(e0, s);
  mufu_probe_kernel<<<n_blocks, 256, 0, s>>>(nullptr, iters);
  e = cudaGetLastError();
  cudaEventRecord(e1, s);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return cuda_status(e);
  out_host[0] = ms;
  out_host[1] = static_cast<float>(static_cast<double>(n_blocks) * 256.0 * iters * 8.0);
  return B4_OK;
}

}  // extern "C"
