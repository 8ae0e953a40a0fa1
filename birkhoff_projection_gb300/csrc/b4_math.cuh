// b4_math.cuh -- per-token arithmetic of the 4x4 Birkhoff projection, one
// thread per token, everything in registers, fp32.
//
// Source: "Accelerating the Birkhoff Projection for Manifold-Constrained
// Hyper-Connections" (technical summary of arXiv 2606.07574), s2.1 (Newton on
// the 3-variable reduced dual, closed-form gradient and Hessian, row-max
// shift), s2.2 (implicit-differentiation backward, Hessian reuse), s1
// (fixed-iteration Sinkhorn-Knopp as used in current mHC).
//
// A token lives in registers as eight float2 pairs (row i = pairs 2i, 2i+1:
// (x_i0, x_i1), (x_i2, x_i3)), so that row scalings, row sums and column
// sums run on the packed fp32x2 FMA pipe (FFMA2/FADD2/FMUL2, sm_100+).
// beta is the column dual in base-2 units (beta_j = b_j log2 e), beta_3 = 0.
#pragma once

#include "b4_device.cuh"
#include "b4_types.h"

namespace b4 {

struct Tok {
  float2 v[8];  // v[2i] = (t_i0, t_i1), v[2i+1] = (t_i2, t_i3)
  __device__ __forceinline__ float at(int i, int j) const {
    const float2 q = v[2 * i + (j >> 1)];
    return (j & 1) ? q.y : q.x;
  }
};

__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 splat(float a) { return make_float2(a, a); }

// Newton-step safeguards (values chosen by simulation of this exact fp32
// iteration on N(0,1), N(0,10^2) and large-magnitude (|X| ~ 200) tokens, and
// by the GPU parity runs on 2^26 tokens):
constexpr float kRidge = 1e-7f;      // added to every Hessian edge weight
constexpr float kClamp = 3.0f;       // max-norm of a step, natural-log units
constexpr int kDampFrom = 4;         // Newton-decrement damping from this step on
constexpr float kStagnation = 64.0f; // stop if residual <= 64 tol and not halving
constexpr int kRefreshEvery = 8;     // log-domain re-evaluation period

// Row softmax of (x log2e + beta) in base 2, every row shifted by its
// maximum [s2.1, numerical stability].
__device__ __forceinline__ void eval_log(const Tok& x, const float beta[3], Tok& p) {
  const float2 L = splat(LOG2E);
  const float2 b01 = make_float2(beta[0], beta[1]), b23 = make_float2(beta[2], 0.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 z01 = fma2(x.v[2 * i], L, b01);
    float2 z23 = fma2(x.v[2 * i + 1], L, b23);
    const float m = fmaxf(max3(z01.x, z01.y, z23.x), z23.y);
    z01 = add2(z01, splat(-m));
    z23 = add2(z23, splat(-m));
    const float2 e01 = make_float2(ex2(z01.x), ex2(z01.y));
    const float2 e23 = make_float2(ex2(z23.x), ex2(z23.y));
    const float2 s = add2(e01, e23);
    const float2 r = splat(rcp(s.x + s.y));
    p.v[2 * i] = mul2(e01, r);
    p.v[2 * i + 1] = mul2(e23, r);
  }
}

// The same row softmax after beta_j += e_j, from the previous (row-normalised)
// p: p_ij <- p_ij 2^{e_j} / sum_k p_ik 2^{e_k}.  Mathematically identical to
// eval_log at the new beta; its rounding does not grow with |X|.
__device__ __forceinline__ void eval_mul(Tok& p, const float e[3]) {
  const float2 w01 = make_float2(ex2(e[0]), ex2(e[1]));
  const float2 w23 = make_float2(ex2(e[2]), 1.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q01 = mul2(p.v[2 * i], w01);
    const float2 q23 = mul2(p.v[2 * i + 1], w23);
    const float2 s = add2(q01, q23);
    const float2 r = splat(rcp(s.x + s.y));
    p.v[2 * i] = mul2(q01, r);
    p.v[2 * i + 1] = mul2(q23, r);
  }
}

// Column sums minus one (the gradient of the reduced dual [s2.1]), all four.
__device__ __forceinline__ void colsum_minus_one(const Tok& p, float2& g01, float2& g23) {
  const float2 c01 = add2(add2(p.v[0], p.v[2]), add2(p.v[4], p.v[6]));
  const float2 c23 = add2(add2(p.v[1], p.v[3]), add2(p.v[5], p.v[7]));
  g01 = add2(c01, splat(-1.0f));
  g23 = add2(c23, splat(-1.0f));
}

// Edge weights of the dual Hessian seen as a graph Laplacian over the four
// columns: w_jk = sum_i p_ij p_ik.  Because rows of p sum to one,
//   H_jk = -w_jk (j != k),  H_jj = sum_{l != j} w_jl   [s2.1: Hessian
//   sum_i diag(p_i) - p_i p_i^T, restricted to columns 0..2 by b_3 = 0],
// which keeps the diagonal free of the cancellation in p (1 - p) when a row
// is nearly one-hot.  Order: 01, 02, 03, 12, 13, 23.
__device__ __forceinline__ void laplacian_weights(const Tok& p, float w[6], float base) {
  float2 w0213 = splat(base);  // (w02, w13) accumulate as a pair
  float w01 = base, w03 = base, w12 = base, w23 = base;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 ab = p.v[2 * i], cd = p.v[2 * i + 1];
    w0213 = fma2(ab, cd, w0213);
    w01 = fmaf(ab.x, ab.y, w01);
    w03 = fmaf(ab.x, cd.y, w03);
    w12 = fmaf(ab.y, cd.x, w12);
    w23 = fmaf(cd.x, cd.y, w23);
  }
  w[0] = w01;
  w[1] = w0213.x;
  w[2] = w03;
  w[3] = w12;
  w[4] = w0213.y;
  w[5] = w23;
}

// Solve H x = g (H the Laplacian of weights w with column 3 grounded) by
// Gaussian elimination in Laplacian form: eliminating a column adds
// w_aj w_ak / d_a to the remaining edge weights (a Schur complement of a
// Laplacian is a Laplacian), so every pivot d is a sum of positive terms and
// nothing cancels in the matrix however small the weights.
// GUARD keeps every pivot >= 1e-30; without it the weights must include a
// positive ridge (every pivot is then a sum of positive terms).
template <bool GUARD = true>
__device__ __forceinline__ void laplacian_solve(const float w[6], const float g[3], float x[3]) {
  auto pivot = [](float v) { return GUARD ? fmaxf(v, 1e-30f) : v; };
  // eliminate column 0
  const float d0 = pivot(w[0] + w[1] + w[2]);
  const float i0 = rcp(d0);
  const float t1 = w[0] * i0, t2 = w[1] * i0;
  const float w12 = fmaf(t1, w[1], w[3]);
  const float w13 = fmaf(t1, w[2], w[4]);
  const float w23 = fmaf(t2, w[2], w[5]);
  const float g1 = fmaf(t1, g[0], g[1]);
  const float g2 = fmaf(t2, g[0], g[2]);
  // eliminate column 1
  const float d1 = pivot(w12 + w13);
  const float i1 = rcp(d1);
  const float u2 = w12 * i1;
  const float d2 = pivot(fmaf(u2, w13, w23));
  const float h2 = fmaf(u2, g1, g2);
  // back substitution
  x[2] = h2 * rcp(d2);
  x[1] = fmaf(w12, x[2], g1) * i1;
  x[0] = fmaf(w[0], x[1], fmaf(w[1], x[2], g[0])) * i0;
}

// Start of the forward solve of one token [s2.1]: the column-mean dual and
// the first (log-domain) evaluation.  Returns false for a token with NaN or
// infinite logits (or sums beyond the fp32 range): p and beta are then NaN
// and evals 0.
__device__ __forceinline__ bool newton_start(const Tok& x, Tok& p, float beta[3], int& evals) {
  // Column-mean start: the exact dual when X_ij = u_i + v_j, and a first-order
  // estimate otherwise: b_j = -(mean_i X_ij - mean_i X_i3).
  const float2 cs01 = add2(add2(x.v[0], x.v[2]), add2(x.v[4], x.v[6]));
  const float2 cs23 = add2(add2(x.v[1], x.v[3]), add2(x.v[5], x.v[7]));
  const float all = (cs01.x + cs01.y) + (cs23.x + cs23.y);
  if (!isfinite(all)) {
    const float nan = __int_as_float(0x7fffffff);
#pragma unroll
    for (int k = 0; k < 8; ++k) p.v[k] = splat(nan);
    beta[0] = beta[1] = beta[2] = nan;
    evals = 0;
    return false;
  }
  const float q = 0.25f * LOG2E;
  beta[0] = (cs23.y - cs01.x) * q;
  beta[1] = (cs23.y - cs01.y) * q;
  beta[2] = (cs23.y - cs23.x) * q;
  eval_log(x, beta, p);
  evals = 1;
  return true;
}

// Outcome of newton_run.
enum NewtonStatus : int { kPaused = 0, kConverged = 1, kCapped = 2 };

// Newton iterations of one token from the state (p, beta, prev, evals) [s2.1],
// until the residual reaches tol (or its stagnation floor): kConverged; or
// until cfg.max_evals evaluations: kCapped; or, with the token unfinished,
// until `until` evaluations: kPaused (the state is then complete: calling
// again continues the same iteration, redoing only the residual test).
// prev is the previous residual (3e38 before the first step).  With REFRESH,
// every 8th step re-evaluates P in the log domain from X, which
// reload(Tok&) fetches, so that X does not have to stay live in registers
// through the iteration.
template <bool REFRESH, class Reload>
__device__ __forceinline__ int newton_run(Tok& p, float beta[3], float& prev, int& evals, int until,
                                          const NewtonCfg& cfg, Reload&& reload) {
  const int lim = until < cfg.max_evals ? until : cfg.max_evals;
  for (;;) {
    float2 g01, g23;
    colsum_minus_one(p, g01, g23);
    const float res = fmaxf(max3(fabsf(g01.x), fabsf(g01.y), fabsf(g23.x)), fabsf(g23.y));
    const bool stop = (res <= cfg.tol) || (res <= kStagnation * cfg.tol && res > 0.5f * prev);
    if (stop) return kConverged;
    if (evals >= lim) return evals >= cfg.max_evals ? kCapped : kPaused;
    prev = res;
    const int k = evals - 1;  // Newton steps taken so far
    // Newton step on b_0..b_2 (natural-log units)
    float w[6], d[3];
    const float g[3] = {g01.x, g01.y, g23.x};
    laplacian_weights(p, w, kRidge);
    laplacian_solve<false>(w, g, d);  // the ridge keeps every pivot positive
    // The step is clamped to kClamp in the max norm (rcp(0) = inf leaves a
    // zero step unscaled).  From the kDampFrom-th step on it is also damped by
    // 1/(1 + lambda) when the Newton decrement lambda = sqrt(g^T H^-1 g)
    // exceeds 1: rare tokens (about one in 10^6 at N(0,10^2)) otherwise cycle.
    // Lanes that start together share k, so warps whose tokens all converge
    // earlier (every N(0,1) warp) never run this branch.
    float lim = 1.0f;
    if (k >= kDampFrom) {
      const float lam2 = fmaf(g[0], d[0], fmaf(g[1], d[1], g[2] * d[2]));
      if (lam2 > 1.0f) lim = rcp(1.0f + lam2 * rsqrt(lam2));
    }
    const float dmax = max3(fabsf(d[0]), fabsf(d[1]), fabsf(d[2]));
    // the negated step in base-2 units, beta_j += e_j: -log2(e) min(lim,
    // kClamp / dmax) (rcp(0) = inf leaves a zero step zero)
    const float nscale = fmaxf(-LOG2E * lim, (-LOG2E * kClamp) * rcp(dmax));
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      d[j] *= nscale;
      beta[j] += d[j];
    }
    if (REFRESH && (k & (kRefreshEvery - 1)) == kRefreshEvery - 1) {
      Tok xr;
      reload(xr);
      eval_log(xr, beta, p);
    } else {
      eval_mul(p, d);
    }
    ++evals;
  }
}

// Forward solve of one token [s2.1] to the end.  Returns true if the
// residual reached tol (or its stagnation floor); p is the last evaluation,
// beta the dual.
template <class Reload>
__device__ __forceinline__ bool newton_forward(const Tok& x, Tok& p, float beta[3], int& evals,
                                               const NewtonCfg& cfg, Reload&& reload) {
  if (!newton_start(x, p, beta, evals)) return false;
  float prev = 3.0e38f;
  return newton_run<true>(p, beta, prev, evals, 0x7fffffff, cfg, reload) == kConverged;
}

// Backward of one token [s2.2]: dX = (dP/dX)^T G from P and G.
//   D_kl = G_kl - sum_j p_kj G_kj = sum_j p_kj (G_kl - G_kj)
//   v_l = sum_k p_kl D_kl,  H lambda = v (lambda_3 = 0)
//   dX_kq = p_kq (D_kq - sum_l p_kl (lambda_q - lambda_l))
// The two sums are written in their difference forms (valid for unit row
// sums, enforced first) so that nothing cancels when a row is nearly one-hot;
// H is regularised by 1e-7 * max weight.
// RENORM rescales the rows of P to unit sums first (a stored P, possibly
// rounded to bf16); a P straight from an evaluation has them already.
template <bool RENORM = true>
__device__ __forceinline__ void implicit_backward(const Tok& pin, const Tok& G, Tok& dx) {
  Tok p;
  if constexpr (RENORM) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 s = add2(pin.v[2 * k], pin.v[2 * k + 1]);
      const float2 r = splat(rcp(s.x + s.y));
      p.v[2 * k] = mul2(pin.v[2 * k], r);
      p.v[2 * k + 1] = mul2(pin.v[2 * k + 1], r);
    }
  } else {
    p = pin;
  }
  Tok D;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float g0 = G.at(k, 0), g1 = G.at(k, 1), g2 = G.at(k, 2), g3 = G.at(k, 3);
    const float q0 = p.at(k, 0), q1 = p.at(k, 1), q2 = p.at(k, 2), q3 = p.at(k, 3);
    const float e01 = g0 - g1, e02 = g0 - g2, e03 = g0 - g3;
    const float e12 = g1 - g2, e13 = g1 - g3, e23 = g2 - g3;
    D.v[2 * k] = make_float2(fmaf(q1, e01, fmaf(q2, e02, q3 * e03)),
                             fmaf(q2, e12, fmaf(q3, e13, -q0 * e01)));
    D.v[2 * k + 1] = make_float2(fmaf(q3, e23, -fmaf(q0, e02, q1 * e12)),
                                 -fmaf(q0, e03, fmaf(q1, e13, q2 * e23)));
  }
  // v_l = sum_k p_kl D_kl for l = 0..2 (the column-3 half is unused)
  float2 v01 = mul2(p.v[0], D.v[0]);
  float2 v23 = mul2(p.v[1], D.v[1]);
#pragma unroll
  for (int k = 1; k < 4; ++k) {
    v01 = fma2(p.v[2 * k], D.v[2 * k], v01);
    v23 = fma2(p.v[2 * k + 1], D.v[2 * k + 1], v23);
  }
  float w[6];
  laplacian_weights(p, w, 0.0f);
  const float wmax = fmaxf(max3(w[0], w[1], w[2]), max3(w[3], w[4], w[5]));
  const float ridge = 1e-7f * wmax;
#pragma unroll
  for (int e = 0; e < 6; ++e) w[e] += ridge;
  const float v[3] = {v01.x, v01.y, v23.x};
  float lam[3];
  laplacian_solve(w, v, lam);
  const float l01 = lam[0] - lam[1], l02 = lam[0] - lam[2], l12 = lam[1] - lam[2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float q0 = p.at(k, 0), q1 = p.at(k, 1), q2 = p.at(k, 2), q3 = p.at(k, 3);
    const float c0 = fmaf(q1, l01, fmaf(q2, l02, q3 * lam[0]));
    const float c1 = fmaf(q2, l12, fmaf(q3, lam[1], -q0 * l01));
    const float c2 = fmaf(q3, lam[2], -fmaf(q0, l02, q1 * l12));
    const float c3 = -fmaf(q0, lam[0], fmaf(q1, lam[1], q2 * lam[2]));
    dx.v[2 * k] = mul2(p.v[2 * k], add2(D.v[2 * k], make_float2(-c0, -c1)));
    dx.v[2 * k + 1] = mul2(p.v[2 * k + 1], add2(D.v[2 * k + 1], make_float2(-c2, -c3)));
  }
}

// Fixed-iteration log-domain Sinkhorn-Knopp [s1]: `iters` times a row
// normalisation then a column normalisation, from b = 0; P = exp(X + a + b).
// Base-2 duals; every log-sum-exp is shifted by its maximum.
__device__ __forceinline__ void sinkhorn_fixed(const Tok& x, Tok& p, int iters) {
  float y[16];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) y[4 * i + j] = x.at(i, j) * LOG2E;
  float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float z0 = y[4 * i] + b[0], z1 = y[4 * i + 1] + b[1];
      const float z2 = y[4 * i + 2] + b[2], z3 = y[4 * i + 3] + b[3];
      const float m = fmaxf(max3(z0, z1, z2), z3);
      a[i] = -(m + lg2((ex2(z0 - m) + ex2(z1 - m)) + (ex2(z2 - m) + ex2(z3 - m))));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float z0 = y[j] + a[0], z1 = y[4 + j] + a[1];
      const float z2 = y[8 + j] + a[2], z3 = y[12 + j] + a[3];
      const float m = fmaxf(max3(z0, z1, z2), z3);
      b[j] = -(m + lg2((ex2(z0 - m) + ex2(z1 - m)) + (ex2(z2 - m) + ex2(z3 - m))));
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    p.v[2 * i] = make_float2(ex2((y[4 * i] + a[i]) + b[0]), ex2((y[4 * i + 1] + a[i]) + b[1]));
    p.v[2 * i + 1] = make_float2(ex2((y[4 * i + 2] + a[i]) + b[2]), ex2((y[4 * i + 3] + a[i]) + b[3]));
  }
}

}  // namespace b4
