// b4_kernels.cuh -- the token-stream kernels.
//
// Every pass of the projection is a stream of independent tokens
// ("Accelerating the Birkhoff Projection for Manifold-Constrained
// Hyper-Connections", s2.3: many 4x4 matrices processed in one batch), so all
// passes share one persistent kernel shape:
//   * one thread per token, TILE tokens per CTA step, one CTA per
//     (SM x resident slot), CTAs striding over tiles;
//   * input tiles arrive by 2-D TMA into an NSTAGE-deep ring of shared-memory
//     stages (mbarrier complete_tx), prefetched NSTAGE tiles ahead;
//   * each thread reads its token from the swizzled tile, computes in
//     registers, writes its result into a swizzled output stage, and one
//     thread stores the tile back with a TMA bulk store (double-buffered);
//   * the partial last tile needs no special case: TMA zero-fills rows past T
//     on load and drops them on store.
// A plain-load kernel with the same arithmetic serves base addresses that are
// not 16-byte aligned.
#pragma once

#include "b4_device.cuh"
#include "b4_math.cuh"
#include "b4_types.h"

namespace b4 {

template <Mode M>
struct ModeTraits {
  static constexpr int NIN = (M == Mode::Forward || M == Mode::Sinkhorn) ? 1 : 2;
  static constexpr int NOUT = (M == Mode::Fused) ? 2 : 1;
};

struct KParams {
  CUtensorMap in[2];    // TMA maps of the inputs (unused by the plain kernel)
  CUtensorMap out[2];   // TMA maps of the outputs
  const void* gin[2];   // raw input pointers (plain kernel)
  void* gout[2];        // raw output pointers (plain kernel)
  float* b;             // Forward: optional [T,4] natural-log dual
  int32_t* evals_out;   // optional [T] evaluation counts
  unsigned long long* nonconv;  // optional counter of tokens above tol
  int64_t T;
  int32_t ntiles;
  int32_t b_vec;        // b is 16-byte aligned
  NewtonCfg cfg;
  int32_t iters;        // Sinkhorn iterations
  unsigned int* fault;  // device fault latch (bit 0: a TMA wait ran out)
};

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Per-token work of each mode; `valid` is false for the zero-filled rows of
// a partial last tile (their results are dropped).
template <Mode M, class TIn>
__device__ __forceinline__ void token_compute(const KParams& a, int64_t tok, bool valid,
                                              const Tok& in0, const Tok& in1, Tok& out0,
                                              Tok& out1) {
  if constexpr (M == Mode::Sinkhorn) {
    sinkhorn_fixed(in0, out0, a.iters);
  } else if constexpr (M == Mode::Backward) {
    implicit_backward(in0, in1, out0);
  } else {
    float beta[3];
    int evals;
    Tok& p = (M == Mode::Recompute) ? out1 : out0;  // out1 is scratch there
    // the periodic refresh re-reads X from global memory (the zero rows of a
    // partial tile converge at once and never refresh)
    auto reload = [&](Tok& xr) {
      if (valid) {
        TileIO<TIn>::gload(a.gin[0], tok, xr.v);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) xr.v[k] = make_float2(0.0f, 0.0f);
      }
    };
    const bool ok = newton_forward(in0, p, beta, evals, a.cfg, reload);
    if constexpr (M == Mode::Forward) {
      if (a.b != nullptr && valid) {
        const float b0 = beta[0] * LN2, b1 = beta[1] * LN2, b2 = beta[2] * LN2;
        float* bp = a.b + 4 * tok;
        if (a.b_vec) {
          *reinterpret_cast<float4*>(bp) = make_float4(b0, b1, b2, 0.0f);
        } else {
          bp[0] = b0;
          bp[1] = b1;
          bp[2] = b2;
          bp[3] = 0.0f;
        }
      }
    }
    if (a.evals_out != nullptr && valid) a.evals_out[tok] = evals;
    if (a.nonconv != nullptr) {
      const unsigned miss = __ballot_sync(0xffffffffu, valid && !ok);
      if ((threadIdx.x & 31) == 0 && miss != 0u) atomicAdd(a.nonconv, (unsigned long long)__popc(miss));
    }
    if constexpr (M == Mode::Recompute) implicit_backward<false>(p, in1, out0);
    if constexpr (M == Mode::Fused) implicit_backward<false>(out0, in1, out1);
  }
}

template <Mode M, class TIn, class TOut, int TILE, int NSTAGE, int NOSTAGE>
struct StreamShape {
  static constexpr int NIN = ModeTraits<M>::NIN;
  static constexpr int NOUT = ModeTraits<M>::NOUT;
  static constexpr int IN_BYTES = TILE * TileIO<TIn>::ROW_BYTES;    // one input, one tile
  static constexpr int OUT_BYTES = TILE * TileIO<TOut>::ROW_BYTES;  // one output, one tile
  static constexpr int STAGE_BYTES = NIN * IN_BYTES;
  static constexpr int OSTAGE_BYTES = NOUT * OUT_BYTES;
  static constexpr int BAR_OFFSET = NSTAGE * STAGE_BYTES + NOSTAGE * OSTAGE_BYTES;
  // + 1024 so the base can be rounded up to a 1024-byte boundary
  static constexpr int SMEM_BYTES = BAR_OFFSET + 8 * NSTAGE + 1024;
  static_assert(IN_BYTES % 1024 == 0 && OUT_BYTES % 1024 == 0, "tile buffers stay 1024-aligned");
  static_assert(TILE <= 256, "TMA box rows <= 256");
};

template <Mode M, class TIn, class TOut, int TILE, int NSTAGE, int NOSTAGE, int MINB>
__global__ void __launch_bounds__(TILE, MINB) stream_kernel(const __grid_constant__ KParams a) {
  using S = StreamShape<M, TIn, TOut, TILE, NSTAGE, NOSTAGE>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* in_stage = smem;
  unsigned char* out_stage = smem + NSTAGE * S::STAGE_BYTES;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::BAR_OFFSET);

  const int tid = threadIdx.x;
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&bar[s], 1);
    mbar_init_fence();
#pragma unroll
    for (int k = 0; k < S::NIN; ++k) prefetch_tmap(&a.in[k]);
#pragma unroll
    for (int k = 0; k < S::NOUT; ++k) prefetch_tmap(&a.out[k]);
  }
  __syncthreads();

  // Loads in flight (maintained by thread 0): bit s of `pending` set while
  // stage s has an issued, not yet consumed load, of parity bit s of `pph`.
  uint32_t pending = 0, pph = 0;
  auto issue = [&](int s, int j, int tile) {
    mbar_arrive_expect_tx(&bar[s], S::STAGE_BYTES);
#pragma unroll
    for (int k = 0; k < S::NIN; ++k)
      tma_load_2d(in_stage + s * S::STAGE_BYTES + k * S::IN_BYTES, &a.in[k], &bar[s], 0,
                  tile * TILE);
    pending |= 1u << s;
    pph = (pph & ~(1u << s)) | ((static_cast<uint32_t>(j / NSTAGE) & 1u) << s);
  };
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) {
      const int tile = blockIdx.x + s * gridDim.x;
      if (tile < a.ntiles) issue(s, s, tile);
    }
  }

  bool failed = false;
  int it = 0;
  for (int tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++it) {
    const int s = it % NSTAGE;
    const uint32_t ph = static_cast<uint32_t>(it / NSTAGE) & 1u;
    const bool ok = mbar_wait(&bar[s], ph, kWaitLimitNs);
    if (!__syncthreads_and(ok)) {
      failed = true;
      break;
    }
    Tok in0, in1;
    TileIO<TIn>::load(in_stage + s * S::STAGE_BYTES, tid, in0.v);
    if constexpr (S::NIN == 2) TileIO<TIn>::load(in_stage + s * S::STAGE_BYTES + S::IN_BYTES, tid, in1.v);
    __syncthreads();  // stage s fully read: refill it
    if (tid == 0) {
      pending &= ~(1u << s);
      const int next = tile + NSTAGE * static_cast<int>(gridDim.x);
      if (next < a.ntiles) issue(s, it + NSTAGE, next);
    }

    const int64_t tok = static_cast<int64_t>(tile) * TILE + tid;
    const bool valid = tok < a.T;
    Tok out0, out1;
    token_compute<M, TIn>(a, tok, valid, in0, in1, out0, out1);

    const int os = it % NOSTAGE;
    if (tid == 0) bulk_wait_read<NOSTAGE - 1>();  // the store that used stage os is done
    __syncthreads();
    unsigned char* ob = out_stage + os * S::OSTAGE_BYTES;
    TileIO<TOut>::store(ob, tid, out0.v);
    if constexpr (S::NOUT == 2) TileIO<TOut>::store(ob + S::OUT_BYTES, tid, out1.v);
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < S::NOUT; ++k) tma_store_2d(&a.out[k], ob + k * S::OUT_BYTES, 0, tile * TILE);
      bulk_commit();
    }
  }
  if (tid == 0) {
    bulk_wait_all();
    if (failed) {
      if (a.fault != nullptr) atomicOr(a.fault, 1u);
      // drain the loads this CTA issued before leaving (again time-limited)
      for (int s = 0; s < NSTAGE; ++s)
        if (pending & (1u << s)) (void)mbar_wait(&bar[s], (pph >> s) & 1u, kWaitLimitNs);
    }
  }
}

// Plain-load variant for base addresses without 16-byte alignment.
template <Mode M, class TIn, class TOut>
__global__ void __launch_bounds__(256) plain_kernel(const __grid_constant__ KParams a) {
  constexpr int NIN = ModeTraits<M>::NIN;
  constexpr int NOUT = ModeTraits<M>::NOUT;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * 256; base < a.T;
       base += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t tok = base + threadIdx.x;
    const bool valid = tok < a.T;
    Tok in0, in1, out0, out1;
    if (valid) {
      TileIO<TIn>::gload(a.gin[0], tok, in0.v);
      if constexpr (NIN == 2) TileIO<TIn>::gload(a.gin[1], tok, in1.v);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) in0.v[k] = in1.v[k] = make_float2(0.0f, 0.0f);
    }
    token_compute<M, TIn>(a, tok, valid, in0, in1, out0, out1);
    if (valid) {
      TileIO<TOut>::gstore(a.gout[0], tok, out0.v);
      if constexpr (NOUT == 2) TileIO<TOut>::gstore(a.gout[1], tok, out1.v);
    }
  }
}

}  // namespace b4
