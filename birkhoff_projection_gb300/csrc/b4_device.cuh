// b4_device.cuh -- sm_103a device primitives for the 4x4 Birkhoff kernels:
// inline PTX for the MUFU approximations, mbarrier waits with a time limit,
// 2-D TMA tile loads/stores, and the swizzled shared-memory layout of a tile
// of tokens.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "b4_types.h"

namespace b4 {

// ---------------------------------------------------------------------------
// Scalar helpers (hardware approximations, called through PTX)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rsqrt(float x) {
  float y;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Three-input maximum (sm_100+).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// log2(e) and ln(2): the natural-log dual b and the base-2 dual beta used in
// the kernels are related by beta = b * LOG2E.
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// bf16 <-> fp32
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// Round two floats to bf16 (nearest even) and pack: lo at the lower address.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// Shared memory, mbarriers, TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for phase `parity` of `bar` to complete, for at most limit_ns.
// Returns false if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// Load the box at (x, y) of a 2-D tensor map into shared memory; completion
// is signalled on `bar` (complete_tx of the box bytes).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}
// Store shared memory to the box at (x, y); rows past the tensor end are
// dropped by the copy engine.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x,
                                             int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::
                   "l"(map),
               "r"(x), "r"(y), "r"(smem_addr(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Prefetch [addr, addr + bytes) of global memory into L2 (addr 16-byte
// aligned, bytes a multiple of 16); nothing waits for it.
__device__ __forceinline__ void prefetch_l2_bulk(const void* addr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(addr), "r"(bytes) : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the TMA
// (async proxy) before a bulk store reads them.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Token tiles in shared memory.
//
// A tile is TILE consecutive tokens, one 16-element row each, written by a
// 2-D TMA box [16 elements, TILE rows] with the tensor map's swizzle:
//   fp32 (64-byte rows): SWIZZLE_64B, 16-byte chunk k of row t lands at
//                        chunk k ^ ((t >> 1) & 3);
//   bf16 (32-byte rows): SWIZZLE_32B, chunk k of row t lands at
//                        chunk k ^ ((t >> 2) & 1).
// With one thread per token these patterns make the 128-bit shared loads and
// stores of a warp conflict-free.  Tile buffers are 1024-byte aligned so the
// pattern is the same relative to the buffer as in absolute addresses.
// ---------------------------------------------------------------------------
template <class T>
struct TileIO;


template <>
struct TileIO<float> {
  static constexpr int ROW_BYTES = 64;
  static constexpr CUtensorMapDataType TMA_TYPE = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  static constexpr CUtensorMapSwizzle TMA_SWIZZLE = CU_TENSOR_MAP_SWIZZLE_64B;
  // chunk k of the row = matrix row k
  __device__ __forceinline__ static void load(const unsigned char* tile, int t, float2 v[8]) {
    const unsigned char* row = tile + t * 64;
    const int sw = (t >> 1) & 3;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 c = *reinterpret_cast<const float4*>(row + 16 * (k ^ sw));
      v[2 * k] = make_float2(c.x, c.y);
      v[2 * k + 1] = make_float2(c.z, c.w);
    }
  }
  __device__ __forceinline__ static void store(unsigned char* tile, int t, const float2 v[8]) {
    unsigned char* row = tile + t * 64;
    const int sw = (t >> 1) & 3;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      *reinterpret_cast<float4*>(row + 16 * (k ^ sw)) =
          make_float4(v[2 * k].x, v[2 * k].y, v[2 * k + 1].x, v[2 * k + 1].y);
  }
  // One row from / to global memory with 16-byte accesses (base 16-byte
  // aligned; rows are 64 bytes).
  __device__ __forceinline__ static void gload_vec(const void* base, int64_t t, float2 v[8]) {
    const float4* p = static_cast<const float4*>(base) + 4 * t;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 c = __ldg(p + k);
      v[2 * k] = make_float2(c.x, c.y);
      v[2 * k + 1] = make_float2(c.z, c.w);
    }
  }
  __device__ __forceinline__ static void gstore_vec(void* base, int64_t t, const float2 v[8]) {
    float4* p = static_cast<float4*>(base) + 4 * t;
#pragma unroll
    for (int k = 0; k < 4; ++k) p[k] = make_float4(v[2 * k].x, v[2 * k].y, v[2 * k + 1].x, v[2 * k + 1].y);
  }
  // Unaligned global fallback: plain element loads/stores.
  __device__ __forceinline__ static void gload(const void* base, int64_t t, float2 v[8]) {
    const float* p = static_cast<const float*>(base) + 16 * t;
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = make_float2(__ldg(p + 2 * k), __ldg(p + 2 * k + 1));
  }
  __device__ __forceinline__ static void gstore(void* base, int64_t t, const float2 v[8]) {
    float* p = static_cast<float*>(base) + 16 * t;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      p[2 * k] = v[k].x;
      p[2 * k + 1] = v[k].y;
    }
  }
};

template <>
struct TileIO<bf16_t> {
  static constexpr int ROW_BYTES = 32;
  static constexpr CUtensorMapDataType TMA_TYPE = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  static constexpr CUtensorMapSwizzle TMA_SWIZZLE = CU_TENSOR_MAP_SWIZZLE_32B;
  // chunk k of the row = matrix rows 2k and 2k+1
  __device__ __forceinline__ static void load(const unsigned char* tile, int t, float2 v[8]) {
    const unsigned char* row = tile + t * 32;
    const int sw = (t >> 2) & 1;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 c = *reinterpret_cast<const uint4*>(row + 16 * (k ^ sw));
      v[4 * k + 0] = make_float2(bf16lo(c.x), bf16hi(c.x));
      v[4 * k + 1] = make_float2(bf16lo(c.y), bf16hi(c.y));
      v[4 * k + 2] = make_float2(bf16lo(c.z), bf16hi(c.z));
      v[4 * k + 3] = make_float2(bf16lo(c.w), bf16hi(c.w));
    }
  }
  __device__ __forceinline__ static void store(unsigned char* tile, int t, const float2 v[8]) {
    unsigned char* row = tile + t * 32;
    const int sw = (t >> 2) & 1;
#pragma unroll
    for (int k = 0; k < 2; ++k)
      *reinterpret_cast<uint4*>(row + 16 * (k ^ sw)) =
          make_uint4(pack_bf16(v[4 * k].x, v[4 * k].y), pack_bf16(v[4 * k + 1].x, v[4 * k + 1].y),
                     pack_bf16(v[4 * k + 2].x, v[4 * k + 2].y), pack_bf16(v[4 * k + 3].x, v[4 * k + 3].y));
  }
  // One row from / to global memory with 16-byte accesses (base 16-byte
  // aligned; rows are 32 bytes).
  __device__ __forceinline__ static void gload_vec(const void* base, int64_t t, float2 v[8]) {
    const uint4* p = static_cast<const uint4*>(base) + 2 * t;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 c = __ldg(p + k);
      v[4 * k + 0] = make_float2(bf16lo(c.x), bf16hi(c.x));
      v[4 * k + 1] = make_float2(bf16lo(c.y), bf16hi(c.y));
      v[4 * k + 2] = make_float2(bf16lo(c.z), bf16hi(c.z));
      v[4 * k + 3] = make_float2(bf16lo(c.w), bf16hi(c.w));
    }
  }
  __device__ __forceinline__ static void gstore_vec(void* base, int64_t t, const float2 v[8]) {
    uint4* p = static_cast<uint4*>(base) + 2 * t;
#pragma unroll
    for (int k = 0; k < 2; ++k)
      p[k] = make_uint4(pack_bf16(v[4 * k].x, v[4 * k].y), pack_bf16(v[4 * k + 1].x, v[4 * k + 1].y),
                        pack_bf16(v[4 * k + 2].x, v[4 * k + 2].y), pack_bf16(v[4 * k + 3].x, v[4 * k + 3].y));
  }
  __device__ __forceinline__ static void gload(const void* base, int64_t t, float2 v[8]) {
    const unsigned short* p = static_cast<const unsigned short*>(base) + 16 * t;
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = make_float2(bf16lo(__ldg(p + 2 * k)), bf16lo(__ldg(p + 2 * k + 1)));
  }
  __device__ __forceinline__ static void gstore(void* base, int64_t t, const float2 v[8]) {
    unsigned short* p = static_cast<unsigned short*>(base) + 16 * t;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t w = pack_bf16(v[k].x, v[k].y);
      p[2 * k] = static_cast<unsigned short>(w & 0xffffu);
      p[2 * k + 1] = static_cast<unsigned short>(w >> 16);
    }
  }
};

}  // namespace b4
