// b4_lanes4.cuh -- the forward with four lanes per token (one row per lane).
//
// "Accelerating the Birkhoff Projection for Manifold-Constrained
// Hyper-Connections", s2.3: the pages' kernel spreads one matrix over a
// group of lanes and forms column sums with __shfl_xor_sync.  This kernel is
// that mapping at four lanes per token, built to compare with one thread per
// token (B4_SCHED_LANES4): lane r of a group holds row r of its token, so a
// warp loads and stores eight whole tokens with contiguous 16-byte accesses
// and needs no staging.  Column sums and the six Hessian edge weights are
// butterfly sums over the group (xor 1, then xor 2); the 3x3 solve and the
// step are computed redundantly by the four lanes, which therefore take
// identical decisions.  A warp iterates until all eight of its tokens are
// solved (finished groups idle), so it waits for the slowest of 8 tokens
// instead of 32.  The arithmetic is that of the one-thread kernels: the same
// start, evaluations, Laplacian solve, safeguards and stopping rule.
#pragma once

#include "b4_device.cuh"
#include "b4_kernels.cuh"
#include "b4_math.cuh"
#include "b4_types.h"

namespace b4 {

// Sum of v over the four lanes of a group (all 32 lanes take part).
__device__ __forceinline__ float group_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// Row softmax of (x log2e + beta) for this lane's row, shifted by its max.
__device__ __forceinline__ void row_eval_log(const float4& x, const float beta[3], float p[4]) {
  const float z0 = fmaf(x.x, LOG2E, beta[0]), z1 = fmaf(x.y, LOG2E, beta[1]);
  const float z2 = fmaf(x.z, LOG2E, beta[2]), z3 = x.w * LOG2E;
  const float m = fmaxf(max3(z0, z1, z2), z3);
  const float e0 = ex2(z0 - m), e1 = ex2(z1 - m), e2 = ex2(z2 - m), e3 = ex2(z3 - m);
  const float r = rcp((e0 + e1) + (e2 + e3));
  p[0] = e0 * r;
  p[1] = e1 * r;
  p[2] = e2 * r;
  p[3] = e3 * r;
}

template <class TIn, class TOut>
__global__ void __launch_bounds__(256) lanes4_kernel(const __grid_constant__ KParams a) {
  static_assert(sizeof(TIn) == 4 && sizeof(TOut) == 4, "fp32 tokens");
  const int lane = threadIdx.x & 31;
  const int r = lane & 3;  // the row this lane holds
  const int64_t groups_per_cta = blockDim.x / 4;
  const float4* X = static_cast<const float4*>(a.gin[0]);
  float4* P = static_cast<float4*>(a.gout[0]);
  unsigned misses = 0;
  for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * groups_per_cta; t0 < a.T;
       t0 += static_cast<int64_t>(gridDim.x) * groups_per_cta) {
    const int64_t tok = t0 + (threadIdx.x >> 2);
    const bool valid = tok < a.T;
    float4 x = valid ? __ldg(X + 4 * tok + r) : make_float4(0.f, 0.f, 0.f, 0.f);
    // column sums of X: the column-mean start b_j = -(mean_i X_ij - mean_i X_i3)
    const float c0 = group_sum(x.x), c1 = group_sum(x.y), c2 = group_sum(x.z), c3 = group_sum(x.w);
    const bool finite = isfinite((c0 + c1) + (c2 + c3));
    float beta[3], p[4];
    const float q = 0.25f * LOG2E;
    beta[0] = (c3 - c0) * q;
    beta[1] = (c3 - c1) * q;
    beta[2] = (c3 - c2) * q;
    row_eval_log(x, beta, p);
    int evals = 1;
    bool done = !valid || !finite;  // the same in the four lanes of a group
    bool ok = false;
    float prev = 3.0e38f;
    int k = 0;
    while (__any_sync(0xffffffffu, !done)) {
      // gradient: column sums minus one
      const float g0 = group_sum(p[0]) - 1.0f, g1 = group_sum(p[1]) - 1.0f;
      const float g2 = group_sum(p[2]) - 1.0f, g3 = group_sum(p[3]) - 1.0f;
      const float res = fmaxf(max3(fabsf(g0), fabsf(g1), fabsf(g2)), fabsf(g3));
      const bool stop = (res <= a.cfg.tol) || (res <= kStagnation * a.cfg.tol && res > 0.5f * prev);
      if (!done && stop) {
        done = true;
        ok = true;
      } else if (!done && evals >= a.cfg.max_evals) {
        done = true;
      }
      // Laplacian edge weights w_jk = sum_i p_ij p_ik (+ ridge)
      const float w01 = group_sum(p[0] * p[1]) + kRidge, w02 = group_sum(p[0] * p[2]) + kRidge;
      const float w03 = group_sum(p[0] * p[3]) + kRidge, w12 = group_sum(p[1] * p[2]) + kRidge;
      const float w13 = group_sum(p[1] * p[3]) + kRidge, w23 = group_sum(p[2] * p[3]) + kRidge;
      if (done) continue;
      prev = res;
      const float w[6] = {w01, w02, w03, w12, w13, w23};
      const float g[3] = {g0, g1, g2};
      float d[3];
      laplacian_solve(w, g, d);
      float lim = 1.0f;
      if (k >= kDampFrom) {
        const float lam2 = fmaf(g[0], d[0], fmaf(g[1], d[1], g[2] * d[2]));
        if (lam2 > 1.0f) lim = rcp(1.0f + lam2 * rsqrt(lam2));
      }
      const float dmax = max3(fabsf(d[0]), fabsf(d[1]), fabsf(d[2]));
      const float scale = LOG2E * fminf(lim, kClamp * rcp(dmax));
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        d[j] *= scale;
        beta[j] -= d[j];
      }
      if ((k & (kRefreshEvery - 1)) == kRefreshEvery - 1) {
        row_eval_log(x, beta, p);  // x stays in registers: one row per lane
      } else {
        const float q0 = p[0] * ex2(-d[0]), q1 = p[1] * ex2(-d[1]), q2 = p[2] * ex2(-d[2]), q3 = p[3];
        const float rs = rcp((q0 + q1) + (q2 + q3));
        p[0] = q0 * rs;
        p[1] = q1 * rs;
        p[2] = q2 * rs;
        p[3] = q3 * rs;
      }
      ++evals;
      ++k;
    }
    if (valid) {
      P[4 * tok + r] = finite ? make_float4(p[0], p[1], p[2], p[3])
                              : make_float4(__int_as_float(0x7fffffff), __int_as_float(0x7fffffff),
                                            __int_as_float(0x7fffffff), __int_as_float(0x7fffffff));
      if (r == 0) {
        if (a.b != nullptr) {
          const float nan = __int_as_float(0x7fffffff);
          const float4 bv = finite ? make_float4(beta[0] * LN2, beta[1] * LN2, beta[2] * LN2, 0.0f)
                                   : make_float4(nan, nan, nan, nan);
          float* bp = a.b + 4 * tok;
          if (a.b_vec) {
            *reinterpret_cast<float4*>(bp) = bv;
          } else {
            bp[0] = bv.x;
            bp[1] = bv.y;
            bp[2] = bv.z;
            bp[3] = bv.w;
          }
        }
        if (a.evals_out != nullptr) a.evals_out[tok] = finite ? evals : 0;
      }
    }
    const unsigned miss = __ballot_sync(0xffffffffu, valid && r == 0 && !ok);
    if (lane == 0) misses += __popc(miss);
  }
  if (lane == 0 && misses != 0u && a.nonconv != nullptr) atomicAdd(a.nonconv, (unsigned long long)misses);
}

}  // namespace b4
