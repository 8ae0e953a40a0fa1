// b4_nxn.cuh -- the projection for n x n tokens (2 <= n <= 8), one thread per
// token: Newton on the dual reduced to n-1 free variables and the
// implicit-differentiation backward ("Accelerating the Birkhoff Projection
// for Manifold-Constrained Hyper-Connections", s2.1: m-1 free variables for
// m columns; s2.2).  The same iteration as the 4 x 4 kernels (column-mean
// start, row-max-shifted first evaluation, multiplicative re-evaluation with
// a log-domain refresh every 8 steps, Laplacian-form Hessian and elimination,
// step clamp 3 with Newton-decrement damping from the fifth step), written
// for any n; for n = 2 the single free dual variable has a closed form,
// which the forward uses instead.  Tokens are staged through shared memory
// with plain coalesced loads (float4 where the tile allows, see
// nxn_tile_in): n x n rows of n^2 * 4 bytes are not all multiples of 16
// bytes, which TMA tiles need.
#pragma once

#include "b4_device.cuh"
#include "b4_types.h"

namespace b4 {

template <int N>
struct NxnShape {
  static constexpr int NN = N * N;
  // row stride of a token in shared memory: odd, so that lanes reading the
  // same element of consecutive tokens hit different banks.  For n = 6 and 8
  // it is 38 and 68 instead, so that every row is 8- or 16-byte aligned and
  // moves as 64- or 128-bit accesses (NxnRowVec), free of bank conflicts:
  // for 128-bit accesses the 16-byte slots of eight consecutive tokens,
  // (272 t + 32 r) mod 128, are distinct, and for 64-bit accesses the
  // 8-byte slots of sixteen consecutive tokens, (152 t + 24 r) / 8 mod 16 =
  // (3 t + 3 r) mod 16, are.  (At n = 4 a stride of 20 sped the forward up
  // by 4% but slowed the bandwidth-bound backward by 5-8%: the float4 tile
  // stores of neighbouring tokens collide two ways there.)
  static constexpr int STRIDE = (N == 8) ? 68 : (N == 6) ? 38 : (NN % 2 == 0) ? NN + 1 : NN;
};

// Width (floats) of the shared-memory accesses that move one row of a token.
template <int N>
struct NxnRowVec {
  static constexpr int value = (N == 8) ? 4 : (N == 6) ? 2 : 1;
};

// One row of a token in shared memory, loaded or stored in order (each
// row is fetched where it is used), NxnRowVec<N> floats per access.
template <int N>
__device__ __forceinline__ void nxn_row_ld(const float* r, float v[N]) {
  constexpr int W = NxnRowVec<N>::value;
  if constexpr (W == 4) {  // rows 16-byte aligned
#pragma unroll
    for (int j = 0; j < N; j += 4)
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(v[j]), "=f"(v[j + 1]), "=f"(v[j + 2]), "=f"(v[j + 3])
                   : "r"(smem_addr(r + j)));
  } else if constexpr (W == 2) {  // rows 8-byte aligned
#pragma unroll
    for (int j = 0; j < N; j += 2)
      asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v[j]), "=f"(v[j + 1]) : "r"(smem_addr(r + j)));
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v[j]) : "r"(smem_addr(r + j)));
  }
}
template <int N>
__device__ __forceinline__ void nxn_row_st(float* r, const float v[N]) {
  constexpr int W = NxnRowVec<N>::value;
  if constexpr (W == 4) {
#pragma unroll
    for (int j = 0; j < N; j += 4)
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(smem_addr(r + j)), "f"(v[j]),
                   "f"(v[j + 1]), "f"(v[j + 2]), "f"(v[j + 3])
                   : "memory");
  } else if constexpr (W == 2) {
#pragma unroll
    for (int j = 0; j < N; j += 2)
      asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(smem_addr(r + j)), "f"(v[j]), "f"(v[j + 1])
                   : "memory");
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) asm volatile("st.shared.f32 [%0], %1;" ::"r"(smem_addr(r + j)), "f"(v[j]) : "memory");
  }
}

constexpr float kNxnRidge = 1e-7f;
constexpr float kNxnClamp = 3.0f;
constexpr int kNxnDampFrom = 4;
// From this n on the forward keeps P in shared memory (nxn_newton_smem).
#ifndef B4_NXN_SMEM_FROM
#define B4_NXN_SMEM_FROM 7
#endif
constexpr int kNxnSmemFrom = B4_NXN_SMEM_FROM;
// The backward keeps P in shared memory (nxn_backward_smem) for odd n and
// from n = 7 on.  Measured on GB300 (1 GiB of X per n): n = 3 went 0.594 ->
// 0.532 ms and n = 5 0.623 -> 0.588 ms that way, while n = 4 and 6 are
// faster with P in registers (0.568 against 0.584 ms, 0.647 against 0.657).
template <int N>
struct NxnBwdSmem {
  static constexpr bool value = (N % 2 == 1) || N >= 7;
};

// Row softmax of (x log2e + beta), rows shifted by their maximum; x is the
// token's row in shared memory.
template <int N>
__device__ __forceinline__ void nxn_eval_log(const float* xs, const float beta[N], float p[N * N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float z[N], x[N];
    nxn_row_ld<N>(xs + N * i, x);
    float m = -3.0e38f;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      z[j] = fmaf(x[j], LOG2E, beta[j]);
      m = fmaxf(m, z[j]);
    }
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      z[j] = ex2(z[j] - m);
      s += z[j];
    }
    const float r = rcp(s);
#pragma unroll
    for (int j = 0; j < N; ++j) p[N * i + j] = z[j] * r;
  }
}

// The row softmax after beta_j -= d_j, from the previous row-normalised p.
template <int N>
__device__ __forceinline__ void nxn_eval_mul(float p[N * N], const float d[N - 1]) {
  float w[N];
#pragma unroll
  for (int j = 0; j < N - 1; ++j) w[j] = ex2(-d[j]);
  w[N - 1] = 1.0f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      p[N * i + j] *= w[j];
      s += p[N * i + j];
    }
    const float r = rcp(s);
#pragma unroll
    for (int j = 0; j < N; ++j) p[N * i + j] *= r;
  }
}

// Laplacian edge weights w[j][k] = sum_i p_ij p_ik (+ base) for j < k.
template <int N>
__device__ __forceinline__ void nxn_weights(const float p[N * N], float w[N][N], float base) {
#pragma unroll
  for (int j = 0; j < N; ++j)
#pragma unroll
    for (int k = j + 1; k < N; ++k) {
      float s = base;
#pragma unroll
      for (int i = 0; i < N; ++i) s = fmaf(p[N * i + j], p[N * i + k], s);
      w[j][k] = s;
    }
}

// Solve H x = g for the Laplacian of w with column N-1 grounded (N-1
// unknowns), by elimination in Laplacian form: eliminating column a adds
// w_aj w_ak / d_a to the remaining weights, so every pivot is a sum of
// positive terms.  w is overwritten.
template <int N>
__device__ __forceinline__ void nxn_solve(float w[N][N], const float g[N - 1], float x[N - 1]) {
  if constexpr (N == 3) {
    // the same elimination written out for two unknowns (the general loops
    // left w in a 40-byte local-memory frame at n = 3); same operations,
    // same order
    const float i0 = rcp(fmaxf(w[0][1] + w[0][2], 1e-30f));
    const float t = w[0][1] * i0;
    const float w12 = fmaf(t, w[0][2], w[1][2]);
    const float g1 = fmaf(t, g[0], g[1]);
    x[1] = g1 * rcp(fmaxf(w12, 1e-30f));
    x[0] = fmaf(w[0][1], x[1], g[0]) * i0;
  } else {
    float gg[N - 1], inv[N - 1];
#pragma unroll
    for (int j = 0; j < N - 1; ++j) gg[j] = g[j];
#pragma unroll
    for (int a = 0; a < N - 1; ++a) {
      float d = 0.0f;
#pragma unroll
      for (int k = a + 1; k < N; ++k) d += w[a][k];
      inv[a] = rcp(fmaxf(d, 1e-30f));
#pragma unroll
      for (int j = a + 1; j < N; ++j) {
        const float t = w[a][j] * inv[a];
        if (j < N - 1) gg[j] = fmaf(t, gg[a], gg[j]);
#pragma unroll
        for (int k = j + 1; k < N; ++k) w[j][k] = fmaf(t, w[a][k], w[j][k]);
      }
    }
#pragma unroll
    for (int a = N - 2; a >= 0; --a) {
      float s = gg[a];
#pragma unroll
      for (int j = a + 1; j < N - 1; ++j) s = fmaf(w[a][j], x[j], s);
      x[a] = s * inv[a];
    }
  }
}

// Forward solve of one n x n token; xs is its row in shared memory (read at
// the start and by the periodic refresh).  beta[N-1] = 0 (base 2).
template <int N>
__device__ __forceinline__ bool nxn_newton(const float* xs, float p[N * N], float beta[N],
                                           int& evals, const NewtonCfg& cfg) {
  if constexpr (N == 2) {
    // closed form: P = [[q, 1 - q], [1 - q, q]], q = sigma(u) with
    // u = (x00 + x11 - x01 - x10) / 2 (the one free dual variable solves a
    // scalar equation); b0 = (x01 + x11 - x00 - x10) / 2, b1 = 0
    const float x00 = xs[0], x01 = xs[1], x10 = xs[2], x11 = xs[3];
    if (!isfinite(x00 + x01 + x10 + x11)) {
      const float nan = __int_as_float(0x7fffffff);
      p[0] = p[1] = p[2] = p[3] = nan;
      beta[0] = beta[1] = nan;
      evals = 0;
      return false;
    }
    const float u = 0.5f * ((x00 + x11) - (x01 + x10));
    const float e = ex2(-fabsf(u) * LOG2E);  // exp(-|u|)
    const float big = rcp(1.0f + e);        // sigma(|u|)
    const float small = e * big;            // 1 - sigma(|u|), without cancellation
    const float q = u >= 0.0f ? big : small;
    const float qc = u >= 0.0f ? small : big;
    p[0] = q;
    p[1] = qc;
    p[2] = qc;
    p[3] = q;
    beta[0] = 0.5f * ((x01 + x11) - (x00 + x10)) * LOG2E;
    beta[1] = 0.0f;
    evals = 1;
    return true;
  }
  float cs[N];
  float all = 0.0f;
#pragma unroll
  for (int j = 0; j < N; ++j) cs[j] = 0.0f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float x[N];
    nxn_row_ld<N>(xs + N * i, x);
#pragma unroll
    for (int j = 0; j < N; ++j) cs[j] += x[j];
  }
#pragma unroll
  for (int j = 0; j < N; ++j) all += cs[j];
  if (!isfinite(all)) {
    const float nan = __int_as_float(0x7fffffff);
#pragma unroll
    for (int k = 0; k < N * N; ++k) p[k] = nan;
#pragma unroll
    for (int j = 0; j < N; ++j) beta[j] = nan;
    evals = 0;
    return false;
  }
  // column-mean start b_j = -(mean_i X_ij - mean_i X_i,N-1)
#pragma unroll
  for (int j = 0; j < N; ++j) beta[j] = (cs[N - 1] - cs[j]) * (LOG2E / N);
  nxn_eval_log<N>(xs, beta, p);
  evals = 1;
  float prev = 3.0e38f;
  for (int k = 0;; ++k) {
    float g[N];
    float res = 0.0f;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < N; ++i) s += p[N * i + j];
      g[j] = s - 1.0f;
      res = fmaxf(res, fabsf(g[j]));
    }
    const bool stop = (res <= cfg.tol) || (res <= 64.0f * cfg.tol && res > 0.5f * prev);
    if (stop) return true;
    if (evals >= cfg.max_evals) return false;
    prev = res;
    float w[N][N], d[N - 1];
    nxn_weights<N>(p, w, kNxnRidge);
    nxn_solve<N>(w, g, d);
    float lim = 1.0f;
    if (k >= kNxnDampFrom) {
      float lam2 = 0.0f;
#pragma unroll
      for (int j = 0; j < N - 1; ++j) lam2 = fmaf(g[j], d[j], lam2);
      if (lam2 > 1.0f) lim = rcp(1.0f + lam2 * rsqrt(lam2));
    }
    float dmax = 0.0f;
#pragma unroll
    for (int j = 0; j < N - 1; ++j) dmax = fmaxf(dmax, fabsf(d[j]));
    const float scale = LOG2E * fminf(lim, kNxnClamp * rcp(dmax));
#pragma unroll
    for (int j = 0; j < N - 1; ++j) {
      d[j] *= scale;
      beta[j] -= d[j];
    }
    if ((k & 7) == 7)
      nxn_eval_log<N>(xs, beta, p);
    else
      nxn_eval_mul<N>(p, d);
    ++evals;
  }
}

// The same forward with P kept in the token's own row of shared memory
// instead of registers (for large n, where P, the Hessian and the solve do
// not fit the register budget of several resident CTAs).  `row` holds X on
// entry and P on return; xg is the token's X in global memory, read again by
// the periodic log-domain refresh.  Every evaluation streams the rows --
// load, scale, normalise, store -- and accumulates the column sums and the
// Hessian edge weights of the new P on the way, so only those, the dual and
// one row are live.  The operations and their order are those of nxn_newton:
// the results are the same bit for bit.
// Column sums and edge weights (+ base) accumulated over rows.
template <int N>
struct NxnAccum {
  float c[N];
  float w[N][N];
  __device__ __forceinline__ void reset(float base) {
#pragma unroll
    for (int j = 0; j < N; ++j) {
      c[j] = 0.0f;
#pragma unroll
      for (int k = j + 1; k < N; ++k) w[j][k] = base;
    }
  }
  __device__ __forceinline__ void add(const float p[N]) {
#pragma unroll
    for (int j = 0; j < N; ++j) {
      c[j] += p[j];
#pragma unroll
      for (int k = j + 1; k < N; ++k) w[j][k] = fmaf(p[j], p[k], w[j][k]);
    }
  }
};

template <int N>
__device__ __forceinline__ bool nxn_newton_smem(float* row, const float* xg, float beta[N], int& evals,
                                                const NewtonCfg& cfg) {
  static_assert(N >= 3, "n >= 3");
  float cs[N];
  float all = 0.0f;
#pragma unroll
  for (int j = 0; j < N; ++j) cs[j] = 0.0f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float x[N];
    nxn_row_ld<N>(row + N * i, x);
#pragma unroll
    for (int j = 0; j < N; ++j) cs[j] += x[j];
  }
#pragma unroll
  for (int j = 0; j < N; ++j) all += cs[j];
  if (!isfinite(all)) {
    const float nan = __int_as_float(0x7fffffff);
    float v[N];
#pragma unroll
    for (int j = 0; j < N; ++j) v[j] = nan;
#pragma unroll
    for (int i = 0; i < N; ++i) nxn_row_st<N>(row + N * i, v);
#pragma unroll
    for (int j = 0; j < N; ++j) beta[j] = nan;
    evals = 0;
    return false;
  }
#pragma unroll
  for (int j = 0; j < N; ++j) beta[j] = (cs[N - 1] - cs[j]) * (LOG2E / N);
  NxnAccum<N> acc;
  // log-domain evaluation of row i from x (row-max shift), stored and accumulated
  auto eval_log_row = [&](int i, const float x[N]) {
    float z[N];
    float m = -3.0e38f;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      z[j] = fmaf(x[j], LOG2E, beta[j]);
      m = fmaxf(m, z[j]);
    }
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      z[j] = ex2(z[j] - m);
      sum += z[j];
    }
    const float r = rcp(sum);
#pragma unroll
    for (int j = 0; j < N; ++j) z[j] *= r;
    nxn_row_st<N>(row + N * i, z);
    acc.add(z);
  };
  acc.reset(kNxnRidge);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float x[N];
    nxn_row_ld<N>(row + N * i, x);
    eval_log_row(i, x);
  }
  evals = 1;
  float prev = 3.0e38f;
  for (int k = 0;; ++k) {
    float g[N];
    float res = 0.0f;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      g[j] = acc.c[j] - 1.0f;
      res = fmaxf(res, fabsf(g[j]));
    }
    const bool stop = (res <= cfg.tol) || (res <= 64.0f * cfg.tol && res > 0.5f * prev);
    if (stop) return true;
    if (evals >= cfg.max_evals) return false;
    prev = res;
    float d[N - 1];
    nxn_solve<N>(acc.w, g, d);
    float lim = 1.0f;
    if (k >= kNxnDampFrom) {
      float lam2 = 0.0f;
#pragma unroll
      for (int j = 0; j < N - 1; ++j) lam2 = fmaf(g[j], d[j], lam2);
      if (lam2 > 1.0f) lim = rcp(1.0f + lam2 * rsqrt(lam2));
    }
    float dmax = 0.0f;
#pragma unroll
    for (int j = 0; j < N - 1; ++j) dmax = fmaxf(dmax, fabsf(d[j]));
    const float scale = LOG2E * fminf(lim, kNxnClamp * rcp(dmax));
#pragma unroll
    for (int j = 0; j < N - 1; ++j) {
      d[j] *= scale;
      beta[j] -= d[j];
    }
    acc.reset(kNxnRidge);
    if ((k & 7) == 7) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        float x[N];
#pragma unroll
        for (int j = 0; j < N; ++j) x[j] = __ldg(xg + N * i + j);
        eval_log_row(i, x);
      }
    } else {
      float wv[N];
#pragma unroll
      for (int j = 0; j < N - 1; ++j) wv[j] = ex2(-d[j]);
      wv[N - 1] = 1.0f;
#pragma unroll
      for (int i = 0; i < N; ++i) {
        float q[N];
        nxn_row_ld<N>(row + N * i, q);
        float sum = 0.0f;
#pragma unroll
        for (int j = 0; j < N; ++j) {
          q[j] *= wv[j];
          sum += q[j];
        }
        const float r = rcp(sum);
#pragma unroll
        for (int j = 0; j < N; ++j) q[j] *= r;
        nxn_row_st<N>(row + N * i, q);
        acc.add(q);
      }
    }
    ++evals;
  }
}

// Backward of one n x n token [s2.2], the difference forms of the 4 x 4
// kernel: D_kl = sum_j p_kj (G_kl - G_kj), v_l = sum_k p_kl D_kl,
// H lambda = v (lambda_{N-1} = 0, ridge 1e-7 max w),
// dX_kq = p_kq (D_kq - sum_l p_kl (lambda_q - lambda_l)); the sums over the
// other columns of a row are formed in O(n) by nxn_excl_diff.  G is the token's
// row in shared memory; P is read from its row Ps into registers first, so
// dX may be written to `out` == Ps.  Both passes over D go row by
// row -- a row of G is loaded, its row of D formed and used -- so that only
// p, the Hessian and one row are live (holding D or G whole spills at n = 8).
template <int N>
__device__ __forceinline__ void nxn_load_row(const float* g, float G[N]) {
  nxn_row_ld<N>(g, G);  // ordered shared loads: each row is fetched where it is used
}

// out_c = sum_{j != c} q_j (h_c - h_j) for every c of one row.  From n = 5
// on in O(N) instead of O(N^2): with R_c and S_c the sums of q_j and of
// q_j h_j over j != c, each a prefix sum (j < c) plus a suffix sum (j > c),
// out_c = h_c R_c - S_c.  R_c is a sum of the other entries of the row,
// never 1 - q_c, so nothing cancels when the row is nearly one-hot.
// Measured on GB300 (1 GiB of X per n), the n = 7 and 8 backwards went
// 0.796 -> 0.647 ms and 1.032 -> 0.780 ms; for n <= 4 the direct sums are
// cheaper and stay.
template <int N>
__device__ __forceinline__ void nxn_excl_diff(const float* q, const float h[N], float out[N]) {
  if constexpr (N <= 4) {
#pragma unroll
    for (int c = 0; c < N; ++c) {
      float s = 0.0f;
#pragma unroll
      for (int j = 0; j < N; ++j)
        if (j != c) s = fmaf(q[j], h[c] - h[j], s);
      out[c] = s;
    }
  } else {
    float pr[N], ps[N];
    float a = 0.0f, b = 0.0f;
#pragma unroll
    for (int c = 0; c < N; ++c) {
      pr[c] = a;
      ps[c] = b;
      a += q[c];
      b = fmaf(q[c], h[c], b);
    }
    a = 0.0f;
    b = 0.0f;
#pragma unroll
    for (int c = N - 1; c >= 0; --c) {
      out[c] = fmaf(h[c], pr[c] + a, -(ps[c] + b));
      a += q[c];
      b = fmaf(q[c], h[c], b);
    }
  }
}

template <int N>
__device__ __forceinline__ void nxn_D_row(const float p[N * N], const float G[N], int k, float D[N]) {
  nxn_excl_diff<N>(p + N * k, G, D);
}

template <int N>
__device__ __forceinline__ void nxn_backward(const float* Ps, const float* Gs, float* out) {
  // P from its shared-memory row, rescaled to unit row sums
  float p[N * N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    float row[N];
    nxn_load_row<N>(Ps + N * k, row);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < N; ++j) s += row[j];
    const float r = rcp(s);
#pragma unroll
    for (int j = 0; j < N; ++j) p[N * k + j] = row[j] * r;
  }
  float v[N - 1];
#pragma unroll
  for (int l = 0; l < N - 1; ++l) v[l] = 0.0f;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    float G[N], D[N];
    nxn_load_row<N>(Gs + N * k, G);
    nxn_D_row<N>(p, G, k, D);
#pragma unroll
    for (int l = 0; l < N - 1; ++l) v[l] = fmaf(p[N * k + l], D[l], v[l]);
  }
  float w[N][N];
  nxn_weights<N>(p, w, 0.0f);
  float wmax = 0.0f;
#pragma unroll
  for (int j = 0; j < N; ++j)
#pragma unroll
    for (int k = j + 1; k < N; ++k) wmax = fmaxf(wmax, w[j][k]);
#pragma unroll
  for (int j = 0; j < N; ++j)
#pragma unroll
    for (int k = j + 1; k < N; ++k) w[j][k] = fmaf(1e-7f, wmax, w[j][k]);
  float lam[N];
  nxn_solve<N>(w, v, lam);
  lam[N - 1] = 0.0f;
  // dX_kq = p_kq sum_{l != q} p_kl ((G_kq - lam_q) - (G_kl - lam_l))
#pragma unroll
  for (int k = 0; k < N; ++k) {
    float H[N], E[N];
    nxn_load_row<N>(Gs + N * k, H);
#pragma unroll
    for (int q = 0; q < N; ++q) H[q] -= lam[q];
    nxn_excl_diff<N>(p + N * k, H, E);
#pragma unroll
    for (int q = 0; q < N; ++q) E[q] *= p[N * k + q];
    nxn_row_st<N>(out + N * k, E);
  }
}

// The same backward with P kept in its shared-memory row (for large n, where
// holding P and the Hessian in registers puts them in local memory):
// pass 1 rescales each row of P to unit sum in place and accumulates the
// edge weights, pass 2 forms v from rows of P and dP, pass 3 forms dX row by
// row into the same row of shared memory.  `row` holds P on entry and dX on
// return.
template <int N>
__device__ __forceinline__ void nxn_backward_smem(float* row, const float* Gs) {
  NxnAccum<N> acc;
  acc.reset(0.0f);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    float q[N];
    nxn_row_ld<N>(row + N * k, q);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < N; ++j) s += q[j];
    const float r = rcp(s);
#pragma unroll
    for (int j = 0; j < N; ++j) q[j] *= r;
    nxn_row_st<N>(row + N * k, q);
    acc.add(q);
  }
  float v[N - 1];
#pragma unroll
  for (int l = 0; l < N - 1; ++l) v[l] = 0.0f;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    float q[N], G[N], D[N];
    nxn_row_ld<N>(row + N * k, q);
    nxn_row_ld<N>(Gs + N * k, G);
    nxn_excl_diff<N>(q, G, D);
#pragma unroll
    for (int l = 0; l < N - 1; ++l) v[l] = fmaf(q[l], D[l], v[l]);
  }
  float wmax = 0.0f;
#pragma unroll
  for (int j = 0; j < N; ++j)
#pragma unroll
    for (int k = j + 1; k < N; ++k) wmax = fmaxf(wmax, acc.w[j][k]);
#pragma unroll
  for (int j = 0; j < N; ++j)
#pragma unroll
    for (int k = j + 1; k < N; ++k) acc.w[j][k] = fmaf(1e-7f, wmax, acc.w[j][k]);
  float lam[N];
  nxn_solve<N>(acc.w, v, lam);
  lam[N - 1] = 0.0f;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    float q[N], H[N], o[N];
    nxn_row_ld<N>(row + N * k, q);
    nxn_row_ld<N>(Gs + N * k, H);
#pragma unroll
    for (int c = 0; c < N; ++c) H[c] -= lam[c];
    nxn_excl_diff<N>(q, H, o);
#pragma unroll
    for (int c = 0; c < N; ++c) o[c] *= q[c];
    nxn_row_st<N>(row + N * k, o);
  }
}

// Copy a tile of `nel` floats between global memory and the padded token
// layout in shared memory (token t at t * STRIDE).  With a 16-byte aligned
// global tile the copy moves float4s: for odd n the layouts coincide
// (STRIDE = n^2) and the float4 goes straight across; for even n (n^2 a
// multiple of 4) each float4 lies inside one token and goes into its row
// as one float4 or two float2s where the stride aligns the row (n = 8, 6),
// else as four floats.  The last nel % 4 floats, or all of them when the
// tile is not aligned, go one by one.  Measured on GB300 (1 GiB of X per
// n): the float4 copy lifts the n = 3 ... 8 forward and the n = 3, 5 ... 8
// backward by 2-22 points of HBM bandwidth, but the four-float scatter's
// bank conflicts cost the bandwidth-bound n = 2 and n = 4 backward 6-8
// points, so those keep the one-by-one copy (as does the n = 2 forward,
// where it made no difference).
template <int N, bool FWD>
struct NxnVecCopy {
  static constexpr bool value = FWD ? N >= 3 : ((N % 2 == 1) || N >= 6);
};

template <int N, int TILE, bool FWD>
__device__ __forceinline__ void nxn_tile_in(float* s, const float* g, int nel) {
  using S = NxnShape<N>;
  int done = 0;
  if (NxnVecCopy<N, FWD>::value && (reinterpret_cast<uintptr_t>(g) & 15u) == 0u) {
    const int n4 = nel >> 2;
    const float4* g4 = reinterpret_cast<const float4*>(g);
    for (int i = threadIdx.x; i < n4; i += TILE) {
      const float4 v = __ldg(g4 + i);
      if constexpr (S::STRIDE == S::NN) {
        *reinterpret_cast<float4*>(s + 4 * i) = v;
      } else {
        static_assert(S::NN % 4 == 0, "a float4 stays inside one token");
        const int t = (4 * i) / S::NN;
        float* d = s + t * S::STRIDE + (4 * i - t * S::NN);
        if constexpr (S::STRIDE % 4 == 0) {
          *reinterpret_cast<float4*>(d) = v;
        } else if constexpr (S::STRIDE % 2 == 0) {
          reinterpret_cast<float2*>(d)[0] = make_float2(v.x, v.y);
          reinterpret_cast<float2*>(d)[1] = make_float2(v.z, v.w);
        } else {
          d[0] = v.x;
          d[1] = v.y;
          d[2] = v.z;
          d[3] = v.w;
        }
      }
    }
    done = n4 << 2;
  }
  for (int i = done + threadIdx.x; i < nel; i += TILE) s[(i / S::NN) * S::STRIDE + i % S::NN] = __ldg(g + i);
}

template <int N, int TILE, bool FWD>
__device__ __forceinline__ void nxn_tile_out(float* g, const float* s, int nel) {
  using S = NxnShape<N>;
  int done = 0;
  if (NxnVecCopy<N, FWD>::value && (reinterpret_cast<uintptr_t>(g) & 15u) == 0u) {
    const int n4 = nel >> 2;
    float4* g4 = reinterpret_cast<float4*>(g);
    for (int i = threadIdx.x; i < n4; i += TILE) {
      float4 v;
      if constexpr (S::STRIDE == S::NN) {
        v = *reinterpret_cast<const float4*>(s + 4 * i);
      } else {
        const int t = (4 * i) / S::NN;
        const float* d = s + t * S::STRIDE + (4 * i - t * S::NN);
        if constexpr (S::STRIDE % 4 == 0) {
          v = *reinterpret_cast<const float4*>(d);
        } else if constexpr (S::STRIDE % 2 == 0) {
          const float2 lo = reinterpret_cast<const float2*>(d)[0], hi = reinterpret_cast<const float2*>(d)[1];
          v = make_float4(lo.x, lo.y, hi.x, hi.y);
        } else {
          v = make_float4(d[0], d[1], d[2], d[3]);
        }
      }
      g4[i] = v;
    }
    done = n4 << 2;
  }
  for (int i = done + threadIdx.x; i < nel; i += TILE) g[i] = s[(i / S::NN) * S::STRIDE + i % S::NN];
}

struct NxnParams {
  const float* in0;  // X (forward) or P (backward)
  const float* in1;  // dP (backward)
  float* out;        // P (forward) or dX (backward)
  float* b;          // forward: optional [T, N] dual
  int64_t T;
  NewtonCfg cfg;
};

// Persistent kernel over tiles of TILE tokens: coalesced copy into shared
// memory, per-token compute, coalesced copy out.
// Resident CTAs per SM the register allocation aims at (launch-bounds
// minimum), swept on GB300.  Forward (128-thread CTAs): 3 / 4 for n = 5 / 6,
// where P, the Hessian and the solve live in registers (128-255 of them
// uncapped; n = 7 went 1.63 -> 1.00 ms with a cap); 7 / 5 for n = 7 / 8,
// where P lives in shared memory (nxn_newton_smem: 72 / 96 registers, no
// spill; n = 8 went 0.72 -> 0.36 ms at 512 MiB; with its 128-bit row
// accesses a cap of 6 spilled 32 bytes and took 0.599 against 0.579 ms at
// 1 GiB).  Backward (64-thread CTAs,
// P and dP tiles in shared memory): the most CTAs that both the shared
// memory and a spill-free register allocation allow, 11 / 10 / 9 / 6 (the
// backward forms D row by row, so it needs far fewer registers than it
// once did).
#ifndef B4_NXN_F5
#define B4_NXN_F5 3
#endif
#ifndef B4_NXN_F6
#define B4_NXN_F6 4
#endif
#ifndef B4_NXN_F7
#define B4_NXN_F7 7
#endif
#ifndef B4_NXN_F8
#define B4_NXN_F8 5
#endif
template <int N, bool FWD>
constexpr int nxn_minb() {
  return N == 5 ? (FWD ? B4_NXN_F5 : 11) : N == 6 ? (FWD ? B4_NXN_F6 : 10)
       : N == 7 ? (FWD ? B4_NXN_F7 : 9) : N == 8 ? (FWD ? B4_NXN_F8 : 6) : 1;
}

template <int N, int TILE, bool FWD>
__global__ void __launch_bounds__(TILE, (nxn_minb<N, FWD>())) nxn_kernel(const NxnParams a) {
  using S = NxnShape<N>;
  extern __shared__ __align__(16) float sm[];
  float* s0 = sm;                     // X or P tile, reused for the output
  float* s1 = sm + TILE * S::STRIDE;  // dP tile (backward)
  const int tid = threadIdx.x;
  const int64_t step = static_cast<int64_t>(gridDim.x) * TILE;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * TILE; base < a.T; base += step) {
    const int64_t left = a.T - base;
    const int ntok = left < TILE ? static_cast<int>(left) : TILE;
    const int nel = ntok * S::NN;
    if (tid == 0 && base + step < a.T) {
      // this CTA's next tile into L2 while the current one is computed (a
      // whole tile is TILE * n^2 * 4 bytes from a 16-byte aligned start
      // when the arrays are; the last one is rounded down to 16 bytes)
      const int64_t nl = a.T - (base + step) < TILE ? a.T - (base + step) : TILE;
      const uint32_t bytes = static_cast<uint32_t>(nl * S::NN * 4) & ~15u;
      const float* n0 = a.in0 + (base + step) * S::NN;
      if (bytes != 0u && (reinterpret_cast<uintptr_t>(n0) & 15u) == 0u) prefetch_l2_bulk(n0, bytes);
      if constexpr (!FWD) {
        const float* n1 = a.in1 + (base + step) * S::NN;
        if (bytes != 0u && (reinterpret_cast<uintptr_t>(n1) & 15u) == 0u) prefetch_l2_bulk(n1, bytes);
      }
    }
    nxn_tile_in<N, TILE, FWD>(s0, a.in0 + base * S::NN, nel);
    if constexpr (!FWD) nxn_tile_in<N, TILE, FWD>(s1, a.in1 + base * S::NN, nel);
    __syncthreads();
    float out[(FWD && N < kNxnSmemFrom) ? S::NN : 1];
    const bool valid = tid < ntok;
    if (valid) {
      if constexpr (FWD) {
        float beta[N];
        int evals = 0;
        if constexpr (N >= kNxnSmemFrom)
          nxn_newton_smem<N>(s0 + tid * S::STRIDE, a.in0 + (base + tid) * S::NN, beta, evals, a.cfg);
        else
          nxn_newton<N>(s0 + tid * S::STRIDE, out, beta, evals, a.cfg);
        if (a.b != nullptr) {
          float* bp = a.b + (base + tid) * N;
#pragma unroll
          for (int j = 0; j < N - 1; ++j) bp[j] = beta[j] * LN2;
          bp[N - 1] = 0.0f;
        }
      } else {
        // P is read from the token's own row of s0 and dX written back
        // there (each thread touches only its own rows)
        if constexpr (NxnBwdSmem<N>::value)
          nxn_backward_smem<N>(s0 + tid * S::STRIDE, s1 + tid * S::STRIDE);
        else
          nxn_backward<N>(s0 + tid * S::STRIDE, s1 + tid * S::STRIDE, s0 + tid * S::STRIDE);
      }
    }
    if constexpr (FWD && N < kNxnSmemFrom) {
      __syncthreads();  // every token's inputs have been read
      if (valid) {
#pragma unroll
        for (int i = 0; i < N; ++i) nxn_row_st<N>(s0 + tid * S::STRIDE + N * i, out + N * i);
      }
    }
    __syncthreads();
    nxn_tile_out<N, TILE, FWD>(a.out + base * S::NN, s0, nel);
    __syncthreads();  // the tile is free for the next load
  }
}

}  // namespace b4
