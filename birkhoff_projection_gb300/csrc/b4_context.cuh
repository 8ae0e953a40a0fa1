// b4_context.cuh -- device addresses of the library's file-scope device
// symbols, cached per device and keyed on the CUDA context they were looked
// up in.
//
// A __device__ variable lives in the module that the current context loaded.
// After cudaDeviceReset (or with another context made current) the module is
// loaded again and the variable may sit at another address, so a cached
// address is reused only while the context that produced it, identified by
// its unique id (cuCtxGetId), is still the current one.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace b4 {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context, 0 if there is none or
// the driver does not provide the query.
inline unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Per-device cache of one symbol's address.
struct SymbolCache {
  static constexpr int kDevices = 64;
  std::mutex mu;
  unsigned long long ctx_id[kDevices] = {};
  void* addr[kDevices] = {};
};

// Device address of a symbol on the current device.  `lookup(void**)` calls
// cudaGetSymbolAddress for the symbol (it may load the library's module on
// this device, which reserves its static device memory and can synchronise).
// The looked-up address is cached with the id of the context it came from;
// it is looked up again whenever another context is current.  Returns
// nullptr and sets *err on failure.
template <class Lookup>
void* cached_symbol_address(SymbolCache& c, Lookup&& lookup, cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= SymbolCache::kDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> guard(c.mu);
  const unsigned long long id = current_context_id();
  if (id != 0 && c.ctx_id[dev] == id && c.addr[dev] != nullptr) return c.addr[dev];
  void* p = nullptr;
  *err = lookup(&p);
  if (*err == cudaSuccess && p == nullptr) *err = cudaErrorInvalidSymbol;
  if (*err != cudaSuccess) return nullptr;
  // the lookup makes the primary context current if nothing was
  c.ctx_id[dev] = current_context_id();
  c.addr[dev] = p;
  return p;
}

}  // namespace b4
