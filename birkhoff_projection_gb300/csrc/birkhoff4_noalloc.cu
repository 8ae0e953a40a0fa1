// birkhoff4_noalloc.cu -- birkhoff4_forward_backward_host_static: the
// host-streaming forward + backward with its device staging area in a
// file-scope static device array instead of caller-allocated memory.
//
// The pages have no counterpart to this entry point; it is a deployment
// variant.  For callers that cannot allocate device memory: code that must not call
// cudaMalloc because it synchronises the device (latency-critical loops), code
// whose device memory belongs to another framework's allocator or pool, and
// plugins or sandboxed hosts where creating device allocations is not
// allowed.  The array belongs to this library's module.  With CUDA's lazy
// module loading the module is loaded on a device by the first call there,
// which reserves the array (and may synchronise); it then stays reserved
// until the process exits.
#include <cuda_runtime.h>

#include <cstdint>

#include "b4_context.cuh"
#include "birkhoff4.h"

namespace b4 {

int record_cuda_error(cudaError_t e);  // birkhoff4_api.cu

// The staging area (B4_STATIC_SCRATCH_BYTES per GPU).  Host code must not use
// this name as an address: on the host it is only a stand-in for the symbol,
// and its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[B4_STATIC_SCRATCH_BYTES];

namespace {

// Device address of g_static_scratch on the current device, looked up with
// that device current and cached per device and context (a reset or another
// context makes it look the address up again).
unsigned char* static_scratch_address(cudaError_t* err) {
  static SymbolCache cache;
  return static_cast<unsigned char*>(cached_symbol_address(
      cache, [](void** q) { return cudaGetSymbolAddress(q, g_static_scratch); }, err));
}

}  // namespace
}  // namespace b4

extern "C" int birkhoff4_forward_backward_host_static(const void* X_h, const void* dP_h, void* P_h,
                                                      void* dX_h, int64_t T, int32_t dtype,
                                                      int64_t chunk_tokens,
                                                      const birkhoff4_stream_t* streams,
                                                      int32_t nstreams) {
  if (T < 0 || chunk_tokens < 0 || nstreams < 1 || nstreams > 16) return B4_EINVAL;
  if (dtype != B4_F32 && dtype != B4_BF16) return B4_EINVAL;
  const uint64_t row_bytes = dtype == B4_F32 ? 64 : 32;
  const uint64_t per_token = static_cast<uint64_t>(nstreams) * 4 * row_bytes;
  const uint64_t fit = B4_STATIC_SCRATCH_BYTES / per_token;
  const uint64_t chunk = chunk_tokens > 0 ? static_cast<uint64_t>(chunk_tokens) : fit;
  if (chunk < 1 || chunk > fit) return B4_ESCRATCH;
  if (T == 0) return B4_OK;
  if (X_h == nullptr || dP_h == nullptr || dX_h == nullptr || streams == nullptr) return B4_EINVAL;
  // Every stream must belong to the current device, whose array is used:
  // checked before anything is enqueued.
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return b4::record_cuda_error(err);
  for (int32_t k = 0; k < nstreams; ++k) {
    int sdev = -1;
    err = cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(streams[k]), &sdev);
    if (err != cudaSuccess) return b4::record_cuda_error(err);
    if (sdev != dev) return B4_EINVAL;
  }
  unsigned char* scratch = b4::static_scratch_address(&err);
  if (scratch == nullptr) return b4::record_cuda_error(err);
  // The staging slots are written in full by the copies in before anything
  // reads them, so nothing left by an earlier call needs clearing.
  return birkhoff4_forward_backward_host(X_h, dP_h, P_h, dX_h, T, dtype, scratch,
                                         static_cast<size_t>(chunk * per_token), streams, nstreams);
}
