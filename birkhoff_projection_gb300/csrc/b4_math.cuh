// b4_math.cuh -- per-token arithmetic of the 4x4 Birkhoff projection, one
// thread per token, everything in registers, fp32.
//
// Source: "Accelerating the Birkhoff Projection for Manifold-Constrained
// Hyper-Connections" (technical summary of arXiv 2606.07574), s2.1 (Newton on
// the 3-variable reduced dual, closed-form gradient and Hessian, row-max
// shift), s2.2 (implicit-differentiation backward, Hessian reuse), s1
// (fixed-iteration Sinkhorn-Knopp as used in current mHC).
//
// Notation: x = X (row-major, x[4i+j]), p = P, beta = the column dual in
// base-2 units (beta_j = b_j * log2(e)), beta_3 = 0.
#pragma once

#include "b4_device.cuh"
#include "b4_types.h"

namespace b4 {

// Newton-step safeguards (values chosen by simulation of this exact fp32
// iteration on N(0,1), N(0,10^2) and large-magnitude (|X| ~ 200) tokens):
constexpr float kRidge = 1e-7f;      // added to every Hessian edge weight
constexpr float kDampAbove = 1.0f;   // damp when the Newton decrement exceeds this
constexpr float kClamp = 4.0f;       // max-norm of a step, natural-log units
constexpr float kStagnation = 64.0f; // stop if residual <= 64 tol and not halving
constexpr int kRefreshEvery = 8;     // log-domain re-evaluation period

// Row softmax of (x*log2e + beta) in base 2, every row shifted by its
// maximum [s2.1, numerical stability].
__device__ __forceinline__ void eval_log(const float x[16], const float beta[3], float p[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float z0 = fmaf(x[4 * i + 0], LOG2E, beta[0]);
    const float z1 = fmaf(x[4 * i + 1], LOG2E, beta[1]);
    const float z2 = fmaf(x[4 * i + 2], LOG2E, beta[2]);
    const float z3 = x[4 * i + 3] * LOG2E;
    const float m = fmaxf(max3(z0, z1, z2), z3);
    const float e0 = ex2(z0 - m), e1 = ex2(z1 - m), e2 = ex2(z2 - m), e3 = ex2(z3 - m);
    const float r = rcp((e0 + e1) + (e2 + e3));
    p[4 * i + 0] = e0 * r;
    p[4 * i + 1] = e1 * r;
    p[4 * i + 2] = e2 * r;
    p[4 * i + 3] = e3 * r;
  }
}

// The same row softmax after beta_j -= d_j, from the previous (row-normalised)
// p: p_ij <- p_ij 2^{-d_j} / sum_k p_ik 2^{-d_k}.  Mathematically identical to
// eval_log at the new beta; its rounding does not grow with |X|.
__device__ __forceinline__ void eval_mul(float p[16], const float d[3]) {
  const float w0 = ex2(-d[0]), w1 = ex2(-d[1]), w2 = ex2(-d[2]);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float q0 = p[4 * i + 0] * w0, q1 = p[4 * i + 1] * w1, q2 = p[4 * i + 2] * w2;
    const float q3 = p[4 * i + 3];
    const float r = rcp((q0 + q1) + (q2 + q3));
    p[4 * i + 0] = q0 * r;
    p[4 * i + 1] = q1 * r;
    p[4 * i + 2] = q2 * r;
    p[4 * i + 3] = q3 * r;
  }
}

// Edge weights of the dual Hessian seen as a graph Laplacian over the four
// columns: w_jk = sum_i p_ij p_ik.  Because rows of p sum to one,
//   H_jk = -w_jk (j != k),  H_jj = sum_{l != j} w_jl   [s2.1: Hessian
//   sum_i diag(p_i) - p_i p_i^T, restricted to columns 0..2 by b_3 = 0],
// which keeps the diagonal free of the cancellation in p (1 - p) when a row
// is nearly one-hot.  Order: 01, 02, 03, 12, 13, 23.
__device__ __forceinline__ void laplacian_weights(const float p[16], float w[6], float base) {
  w[0] = w[1] = w[2] = w[3] = w[4] = w[5] = base;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = p[4 * i + 0], b = p[4 * i + 1], c = p[4 * i + 2], d = p[4 * i + 3];
    w[0] = fmaf(a, b, w[0]);
    w[1] = fmaf(a, c, w[1]);
    w[2] = fmaf(a, d, w[2]);
    w[3] = fmaf(b, c, w[3]);
    w[4] = fmaf(b, d, w[4]);
    w[5] = fmaf(c, d, w[5]);
  }
}

// Solve H x = g (H the Laplacian of weights w with column 3 grounded) by
// Gaussian elimination in Laplacian form: eliminating a column adds
// w_aj w_ak / d_a to the remaining edge weights (a Schur complement of a
// Laplacian is a Laplacian), so every pivot d is a sum of positive terms and
// nothing cancels in the matrix however small the weights.
__device__ __forceinline__ void laplacian_solve(const float w[6], const float g[3], float x[3]) {
  // eliminate column 0
  const float d0 = fmaxf(w[0] + w[1] + w[2], 1e-30f);
  const float i0 = rcp(d0);
  const float t1 = w[0] * i0, t2 = w[1] * i0;
  const float w12 = fmaf(t1, w[1], w[3]);
  const float w13 = fmaf(t1, w[2], w[4]);
  const float w23 = fmaf(t2, w[2], w[5]);
  const float g1 = fmaf(t1, g[0], g[1]);
  const float g2 = fmaf(t2, g[0], g[2]);
  // eliminate column 1
  const float d1 = fmaxf(w12 + w13, 1e-30f);
  const float i1 = rcp(d1);
  const float u2 = w12 * i1;
  const float d2 = fmaxf(fmaf(u2, w13, w23), 1e-30f);
  const float h2 = fmaf(u2, g1, g2);
  // back substitution
  x[2] = h2 * rcp(d2);
  x[1] = fmaf(w12, x[2], g1) * i1;
  x[0] = fmaf(w[0], x[1], fmaf(w[1], x[2], g[0])) * i0;
}

// Forward solve of one token [s2.1].  Returns true if the residual reached
// tol (or its stagnation floor); p is the last evaluation, beta the dual.
__device__ __forceinline__ bool newton_forward(const float x[16], float p[16], float beta[3],
                                               int& evals, const NewtonCfg& cfg) {
  // Column-mean start: the exact dual when X_ij = u_i + v_j, and a first-order
  // estimate otherwise: b_j = -(mean_i X_ij - mean_i X_i3).
  float cs[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) cs[j] = (x[j] + x[4 + j]) + (x[8 + j] + x[12 + j]);
  const float all = (cs[0] + cs[1]) + (cs[2] + cs[3]);
  if (!isfinite(all)) {
    // NaN or infinite logits (or sums beyond the fp32 range): no projection
#pragma unroll
    for (int k = 0; k < 16; ++k) p[k] = __int_as_float(0x7fffffff);
    beta[0] = beta[1] = beta[2] = __int_as_float(0x7fffffff);
    evals = 0;
    return false;
  }
#pragma unroll
  for (int j = 0; j < 3; ++j) beta[j] = (cs[3] - cs[j]) * (0.25f * LOG2E);
  eval_log(x, beta, p);
  evals = 1;
  float prev = 3.0e38f;
  for (int k = 0;; ++k) {
    // gradient: column sums of the row softmax minus one [s2.1]
    float g[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) g[j] = ((p[j] + p[4 + j]) + (p[8 + j] + p[12 + j])) - 1.0f;
    const float res = fmaxf(max3(fabsf(g[0]), fabsf(g[1]), fabsf(g[2])), fabsf(g[3]));
    if (res <= cfg.tol) return true;
    if (res <= kStagnation * cfg.tol && res > 0.5f * prev) return true;
    if (evals >= cfg.max_evals) return false;
    prev = res;
    // Newton step on b_0..b_2 (natural-log units)
    float w[6], d[3];
    laplacian_weights(p, w, kRidge);
    laplacian_solve(w, g, d);
    // damped when the Newton decrement lambda = sqrt(g^T H^-1 g) exceeds 1
    const float lam2 = fmaf(g[0], d[0], fmaf(g[1], d[1], g[2] * d[2]));
    float scale = LOG2E;
    if (lam2 > kDampAbove * kDampAbove) scale *= rcp(1.0f + lam2 * rsqrt(lam2));
    // and clamped to kClamp in the max norm
    const float dmax = max3(fabsf(d[0]), fabsf(d[1]), fabsf(d[2])) * scale;
    if (dmax > kClamp * LOG2E) scale *= (kClamp * LOG2E) * rcp(dmax);
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      d[j] *= scale;  // base-2 units
      beta[j] -= d[j];
    }
    if ((k + 1) % kRefreshEvery == 0)
      eval_log(x, beta, p);
    else
      eval_mul(p, d);
    ++evals;
  }
}

// Backward of one token [s2.2]: dX = (dP/dX)^T G from P and G.
//   D_kl = G_kl - sum_j p_kj G_kj = sum_j p_kj (G_kl - G_kj)
//   v_l = sum_k p_kl D_kl,  H lambda = v (lambda_3 = 0)
//   dX_kq = p_kq (D_kq - sum_l p_kl (lambda_q - lambda_l))
// The two sums are written in their difference forms (valid for unit row
// sums, enforced first) so that nothing cancels when a row is nearly one-hot;
// H is regularised by 1e-7 * max weight.
__device__ __forceinline__ void implicit_backward(const float pin[16], const float G[16],
                                                  float dx[16]) {
  float p[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float r = rcp((pin[4 * k] + pin[4 * k + 1]) + (pin[4 * k + 2] + pin[4 * k + 3]));
#pragma unroll
    for (int j = 0; j < 4; ++j) p[4 * k + j] = pin[4 * k + j] * r;
  }
  float D[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float* g = G + 4 * k;
    const float* q = p + 4 * k;
    const float e01 = g[0] - g[1], e02 = g[0] - g[2], e03 = g[0] - g[3];
    const float e12 = g[1] - g[2], e13 = g[1] - g[3], e23 = g[2] - g[3];
    D[4 * k + 0] = fmaf(q[1], e01, fmaf(q[2], e02, q[3] * e03));
    D[4 * k + 1] = fmaf(q[2], e12, fmaf(q[3], e13, -q[0] * e01));
    D[4 * k + 2] = fmaf(q[3], e23, -fmaf(q[0], e02, q[1] * e12));
    D[4 * k + 3] = -fmaf(q[0], e03, fmaf(q[1], e13, q[2] * e23));
  }
  float v[3];
#pragma unroll
  for (int l = 0; l < 3; ++l)
    v[l] = fmaf(p[l], D[l], fmaf(p[4 + l], D[4 + l], fmaf(p[8 + l], D[8 + l], p[12 + l] * D[12 + l])));
  float w[6];
  laplacian_weights(p, w, 0.0f);
  const float wmax = fmaxf(max3(w[0], w[1], w[2]), max3(w[3], w[4], w[5]));
  const float ridge = 1e-7f * wmax;
#pragma unroll
  for (int e = 0; e < 6; ++e) w[e] += ridge;
  float lam[3];
  laplacian_solve(w, v, lam);
  const float l01 = lam[0] - lam[1], l02 = lam[0] - lam[2], l12 = lam[1] - lam[2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float* q = p + 4 * k;
    const float c0 = fmaf(q[1], l01, fmaf(q[2], l02, q[3] * lam[0]));
    const float c1 = fmaf(q[2], l12, fmaf(q[3], lam[1], -q[0] * l01));
    const float c2 = fmaf(q[3], lam[2], -fmaf(q[0], l02, q[1] * l12));
    const float c3 = -fmaf(q[0], lam[0], fmaf(q[1], lam[1], q[2] * lam[2]));
    dx[4 * k + 0] = q[0] * (D[4 * k + 0] - c0);
    dx[4 * k + 1] = q[1] * (D[4 * k + 1] - c1);
    dx[4 * k + 2] = q[2] * (D[4 * k + 2] - c2);
    dx[4 * k + 3] = q[3] * (D[4 * k + 3] - c3);
  }
}

// Fixed-iteration log-domain Sinkhorn-Knopp [s1]: `iters` times a row
// normalisation then a column normalisation, from b = 0; P = exp(X + a + b).
// Base-2 duals; every log-sum-exp is shifted by its maximum.
__device__ __forceinline__ void sinkhorn_fixed(const float x[16], float p[16], int iters) {
  float y[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) y[k] = x[k] * LOG2E;
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
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) p[4 * i + j] = ex2((y[4 * i + j] + a[i]) + b[j]);
}

}  // namespace b4
