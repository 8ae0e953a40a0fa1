// b4_queue.cuh -- the Newton passes (forward, fused, recompute) with per-warp
// compaction of slow tokens.
//
// "Accelerating the Birkhoff Projection for Manifold-Constrained
// Hyper-Connections", s2.1 (Newton on the reduced dual) and s2.3 (a batched
// per-token kernel).  With one thread per token, a warp runs as long as its
// slowest token: at N(0,10^2) a token needs 7 evaluations on average but the
// slowest of 32 needs 11.4, so a third of the lanes' issue slots go idle.
// Here a warp solves its tokens in rounds:
//   * a fresh round takes the warp's 32 tokens of the next CTA tile (a TMA
//     ring shared by the CTA's warps) and runs at most K1 evaluations (every
//     N(0,1) token is solved within 5);
//   * a token still unsolved after its round parks its state -- the dual
//     beta, the last residual, its index and evaluation count, 24 bytes -- in
//     the warp's queue in shared memory;
//   * whenever 32 tokens are parked, a resume round pops them, re-evaluates
//     each P in the log domain from X (re-read from global memory) and beta,
//     and runs at most K2 more evaluations; unsolved ones are parked again;
//   * after the CTA's last tile the warp drains its queue the same way.
// Lanes of a resume round are all slow tokens, so few of them idle.  The
// re-evaluation on resume replaces the periodic log-domain refresh of the
// single-round kernel (it is not counted as an evaluation); tokens solved in
// their fresh round take exactly the arithmetic of that kernel.
//
// Warps never wait for each other: a stage of the TMA ring is refilled by
// whichever warp reads it last (a counter per stage), and results go straight
// from registers to global memory (each token's row is one 64- or 32-byte
// run).  The fused and recompute passes read dP when a token is solved; its
// rows are prefetched into L2 when the fresh round starts.
#pragma once

#include "b4_device.cuh"
#include "b4_kernels.cuh"
#include "b4_math.cuh"
#include "b4_types.h"

namespace b4 {

template <Mode M, class TIn, class TOut, int WARPS, int NSTAGE, int QC>
struct QueueShape {
  static constexpr int TILE = WARPS * 32;
  static constexpr int STAGE_BYTES = TILE * TileIO<TIn>::ROW_BYTES;  // X only
  static constexpr int BAR_OFFSET = NSTAGE * STAGE_BYTES;
  // full barriers (8 B each), then the consumed and issued counters
  static constexpr int CNT_OFFSET = BAR_OFFSET + 8 * NSTAGE;
  static constexpr int ISSUED_OFFSET = CNT_OFFSET + 4 * NSTAGE;
  static constexpr int FAIL_OFFSET = ISSUED_OFFSET + 4 * NSTAGE;
  // per warp: QC float4 (beta0, beta1, beta2, prev) and QC int2 (token, evals)
  static constexpr int QA_OFFSET = (FAIL_OFFSET + 4 + 15) / 16 * 16;
  static constexpr int QB_OFFSET = QA_OFFSET + WARPS * QC * 16;
  static constexpr int SMEM_BYTES = QB_OFFSET + WARPS * QC * 8 + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-aligned");
  static_assert((QC & (QC - 1)) == 0 && QC >= 64, "queue capacity: a power of two >= 64");
};

// Results of one solved token: written straight to global memory.
template <Mode M, class TIn, class TOut>
__device__ __forceinline__ void queue_finish(const KParams& a, int tok, const Tok& p,
                                             const float beta[3], int evals) {
  if constexpr (M == Mode::Forward) {
    TileIO<TOut>::gstore_vec(a.gout[0], tok, p.v);
    if (a.b != nullptr) {
      const float b0 = beta[0] * LN2, b1 = beta[1] * LN2, b2 = beta[2] * LN2;
      float* bp = a.b + 4 * static_cast<int64_t>(tok);  // 4 tok can pass 2^31
      if (a.b_vec) {
        *reinterpret_cast<float4*>(bp) = make_float4(b0, b1, b2, 0.0f);
      } else {
        bp[0] = b0;
        bp[1] = b1;
        bp[2] = b2;
        bp[3] = 0.0f;
      }
    }
  } else {
    Tok G, dx;
    TileIO<TIn>::gload_vec(a.gin[1], tok, G.v);
    implicit_backward<false>(p, G, dx);  // p is an evaluation: unit row sums
    if constexpr (M == Mode::Fused) {
      TileIO<TOut>::gstore_vec(a.gout[0], tok, p.v);
      TileIO<TOut>::gstore_vec(a.gout[1], tok, dx.v);
    } else {
      TileIO<TOut>::gstore_vec(a.gout[0], tok, dx.v);
    }
  }
  if (a.evals_out != nullptr) a.evals_out[tok] = evals;
}

template <Mode M, class TIn, class TOut, int WARPS, int NSTAGE, int QC, int K1, int K2, int MINB>
__global__ void __launch_bounds__(WARPS * 32, MINB) queue_kernel(const __grid_constant__ KParams a) {
  using S = QueueShape<M, TIn, TOut, WARPS, NSTAGE, QC>;
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* stage = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::BAR_OFFSET);
  unsigned* consumed = reinterpret_cast<unsigned*>(smem + S::CNT_OFFSET);
  unsigned* issued = reinterpret_cast<unsigned*>(smem + S::ISSUED_OFFSET);
  unsigned* any_failed = reinterpret_cast<unsigned*>(smem + S::FAIL_OFFSET);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float4* qa = reinterpret_cast<float4*>(smem + S::QA_OFFSET) + warp * QC;
  int2* qb = reinterpret_cast<int2*>(smem + S::QB_OFFSET) + warp * QC;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      consumed[s] = 0;
      issued[s] = 0;
    }
    *any_failed = 0;
    mbar_init_fence();
    prefetch_tmap(&a.in[0]);
  }
  __syncthreads();

  // a load of tile `t` into stage s (one thread)
  auto issue = [&](int s, int t) {
    mbar_arrive_expect_tx(&full[s], S::STAGE_BYTES);
    tma_load_2d(stage + s * S::STAGE_BYTES, &a.in[0], &full[s], 0, t * S::TILE);
    atomicAdd(&issued[s], 1u);  // read only at the end, after a block barrier
  };
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) {
      const int t = blockIdx.x + s * gridDim.x;
      if (t < a.ntiles) issue(s, t);
    }
  }

  // warp-uniform queue cursors (ring of QC entries).  Resume rounds run while
  // 32 tokens are parked, so a fresh round starts with at most 31 and adds at
  // most 32: QC = 64 entries never overflow.
  unsigned qh = 0, qt = 0;
  unsigned misses = 0;  // lane 0: tokens that stopped above tol
  bool failed = false;
  auto reload = [&](Tok&) {};  // no periodic refresh here: resume re-evaluates
  const int T = static_cast<int>(a.T);  // a launch covers at most 2^30 tokens
  int tile = blockIdx.x, it = 0;

  for (;;) {
    const unsigned size = qt - qh;
    const bool more = tile < a.ntiles;
    if (!more && size == 0u) break;
    const bool resume = !more || size >= 32u;

    Tok p;
    float beta[3] = {0.0f, 0.0f, 0.0f};
    float prev = 3.0e38f;
    int evals = 0, until, tok = 0;
    bool active;  // this lane runs Newton steps in this round
    bool solved;  // finished before any step (non-finite input: P is NaN)
    if (resume) {
      const unsigned n = size < 32u ? size : 32u;
      active = static_cast<unsigned>(lane) < n;
      solved = false;
      if (active) {
        const unsigned e = (qh + lane) & (QC - 1);
        const float4 st = qa[e];
        const int2 ix = qb[e];
        beta[0] = st.x;
        beta[1] = st.y;
        beta[2] = st.z;
        prev = st.w;
        tok = ix.x;
        evals = ix.y;
        Tok x;
        TileIO<TIn>::gload_vec(a.gin[0], tok, x.v);
        eval_log(x, beta, p);
      }
      qh += n;
      until = evals + K2;
    } else {
      const int s = it % NSTAGE;
      const uint32_t ph = static_cast<uint32_t>(it / NSTAGE) & 1u;
      const bool ok = mbar_wait(&full[s], ph, kWaitLimitNs);
      if (!__all_sync(FULL, ok)) {
        failed = true;
        break;
      }
      Tok x;
      TileIO<TIn>::load(stage + s * S::STAGE_BYTES, warp * 32 + lane, x.v);
      __syncwarp();
      if (lane == 0) {
        // the last of the CTA's warps to read stage s refills it (the
        // acquire-release add orders every warp's reads of the stage before
        // the refill)
        unsigned old;
        asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                     : "=r"(old)
                     : "r"(smem_addr(&consumed[s]))
                     : "memory");
        if (old % WARPS == WARPS - 1) {
          const int next = tile + NSTAGE * static_cast<int>(gridDim.x);
          if (next < a.ntiles) issue(s, next);
        }
      }
      const int base = tile * S::TILE + warp * 32;
      if constexpr (M != Mode::Forward) {
        // dP rows of this warp's tokens, needed when each is solved
        if (lane == 0 && base < T) {
          const int rows = T - base < 32 ? T - base : 32;
          prefetch_l2_bulk(static_cast<const unsigned char*>(a.gin[1]) +
                               static_cast<int64_t>(base) * TileIO<TIn>::ROW_BYTES,
                           static_cast<uint32_t>(rows * TileIO<TIn>::ROW_BYTES));
        }
      }
      tok = base + lane;
      const bool valid = tok < T;
      active = valid && newton_start(x, p, beta, evals);
      solved = valid && !active;
      until = K1;
      tile += gridDim.x;
      ++it;
    }

    int st = kPaused;
    if (active) st = newton_run<false>(p, beta, prev, evals, until, a.cfg, reload);
    if (solved || (active && st != kPaused)) queue_finish<M, TIn, TOut>(a, tok, p, beta, evals);
    const unsigned miss = __ballot_sync(FULL, solved || st == kCapped);
    const bool park = active && st == kPaused;
    const unsigned pm = __ballot_sync(FULL, park);
    if (lane == 0) misses += __popc(miss);
    if (pm != 0u) {
      __syncwarp();  // every popped entry has been read
      if (park) {
        const unsigned e = (qt + __popc(pm & ((1u << lane) - 1u))) & (QC - 1);
        qa[e] = make_float4(beta[0], beta[1], beta[2], prev);
        qb[e] = make_int2(tok, evals);
      }
      qt += __popc(pm);
      __syncwarp();
    }
  }

  if (lane == 0 && misses != 0u && a.nonconv != nullptr) atomicAdd(a.nonconv, (unsigned long long)misses);
  if (failed && lane == 0) {
    atomicOr(any_failed, 1u);
    if (a.fault != nullptr) atomicOr(a.fault, 1u);
  }
  __syncthreads();
  if (threadIdx.x == 0 && *any_failed != 0u) {
    // drain the loads still in flight before the CTA's shared memory goes
    // away (every wait time-limited)
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s)
      if (issued[s] > 0u) (void)mbar_wait(&full[s], (issued[s] - 1u) & 1u, kWaitLimitNs);
  }
}

}  // namespace b4
