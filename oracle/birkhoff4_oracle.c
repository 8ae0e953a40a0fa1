/*
 * birkhoff4_oracle.c -- float64 CPU oracle for the per-token 4x4 Birkhoff
 * projection.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain checker that the
 * CUDA path is compared against.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load it.  It shares no code,
 * header, table or constant with the CUDA library, and nothing in the product
 * path may call it.
 *
 * Sources (page titles and sections):
 *   [mHC] "Accelerating the Birkhoff Projection for Manifold-Constrained
 *         Hyper-Connections" (technical summary, arXiv 2606.07574), in its
 *         Spanish and French renderings.
 *     s1   : the projection maps each residual mixing matrix onto the Birkhoff
 *            polytope (doubly stochastic matrices); current mHC runs
 *            Sinkhorn-Knopp for it, often with a small fixed iteration count.
 *     s2   : the projection is entropic optimal transport.
 *     s2.1 : the dual is reduced to m-1 = 3 free variables (the duals are only
 *            defined up to a common scalar shift); closed-form gradient and
 *            Hessian; Newton's method; rows shifted by their maximum before the
 *            softmax.
 *     s2.2 : the backward pass uses the implicit function theorem on that
 *            dual; the last Newton Hessian is the matrix of the linear system.
 *
 * Every token is one X in R^{4x4}, row-major: element (t,i,j) sits at offset
 * 16*t + 4*i + j.  The projection is P = diag(e^a) exp(X) diag(e^b) with unit
 * row and column sums (entropic OT with epsilon = 1 and uniform unit
 * marginals); P is unique by Sinkhorn's theorem.  The gauge is b[3] = 0.
 *
 * Functions (all batched over T tokens, OpenMP over tokens):
 *   oracle_sinkhorn64   : log-domain Sinkhorn-Knopp.  With tol > 0 it runs to
 *                         max(row, column residual) < tol or max_iters; with
 *                         tol <= 0 it runs exactly max_iters iterations (the
 *                         fixed-iteration scheme of [mHC s1]).
 *   oracle_newton64     : Newton's method on the reduced 3-variable dual
 *                         [mHC s2.1] with an Armijo backtracking line search.
 *   oracle_backward64   : vector-Jacobian product dX = (dP/dX)^T G through the
 *                         implicit function theorem on the reduced dual
 *                         [mHC s2.2].
 *
 * Build: gcc -O2 -fopenmp -fPIC -shared (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_VERSION 1

int oracle_version(void) { return ORACLE_VERSION; }

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads used by later calls (the CPU baseline times one core and all). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* log(sum_k exp(v[k])) for four values, shifted by the maximum. */
static double lse4(double v0, double v1, double v2, double v3)
{
    double m = v0;
    if (v1 > m) m = v1;
    if (v2 > m) m = v2;
    if (v3 > m) m = v3;
    if (isinf(m) && m < 0) return m;
    return m + log(exp(v0 - m) + exp(v1 - m) + exp(v2 - m) + exp(v3 - m));
}

/* max over rows of |row sum - 1| and over columns of |column sum - 1|. */
static double marginal_residual(const double p[16])
{
    double res = 0.0;
    for (int i = 0; i < 4; ++i) {
        double s = p[4 * i] + p[4 * i + 1] + p[4 * i + 2] + p[4 * i + 3];
        double d = fabs(s - 1.0);
        if (d > res || isnan(d)) res = d;
    }
    for (int j = 0; j < 4; ++j) {
        double s = p[j] + p[4 + j] + p[8 + j] + p[12 + j];
        double d = fabs(s - 1.0);
        if (d > res || isnan(d)) res = d;
    }
    return res;
}

/* A token with a NaN or infinite logit has no projection (exp(X) is not a
 * strictly positive finite matrix); its outputs are all NaN. */
static int nonfinite_token(const double x[16], double p[16], double *b)
{
    for (int k = 0; k < 16; ++k) {
        if (!isfinite(x[k])) {
            for (int q = 0; q < 16; ++q) p[q] = NAN;
            if (b)
                for (int q = 0; q < 4; ++q) b[q] = NAN;
            return 1;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Sinkhorn-Knopp in the log domain [mHC s1, s2].                            */
/* One iteration: a_i = -LSE_j(X_ij + b_j) (rows), then                      */
/*                b_j = -LSE_i(X_ij + a_i) (columns).                        */
/* The output is P = exp(X_ij + a_i + b_j) after the last column step.       */
/* ------------------------------------------------------------------------ */
static int sinkhorn_token(const double x[16], double p[16], double bout[4],
                          double tol, int32_t max_iters, int32_t *iters)
{
    double a[4] = {0, 0, 0, 0}, b[4] = {0, 0, 0, 0};
    int converged = 0;
    if (nonfinite_token(x, p, bout)) {
        if (iters) *iters = 0;
        return 0;
    }
    int32_t it = 0;
    while (it < max_iters) {
        for (int i = 0; i < 4; ++i)
            a[i] = -lse4(x[4 * i] + b[0], x[4 * i + 1] + b[1], x[4 * i + 2] + b[2],
                         x[4 * i + 3] + b[3]);
        for (int j = 0; j < 4; ++j)
            b[j] = -lse4(x[j] + a[0], x[4 + j] + a[1], x[8 + j] + a[2], x[12 + j] + a[3]);
        ++it;
        if (tol > 0.0) {
            double q[16];
            for (int i = 0; i < 4; ++i)
                for (int j = 0; j < 4; ++j) q[4 * i + j] = exp(x[4 * i + j] + a[i] + b[j]);
            if (marginal_residual(q) < tol) {
                converged = 1;
                break;
            }
        }
    }
    for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 4; ++j) p[4 * i + j] = exp(x[4 * i + j] + a[i] + b[j]);
    if (bout) {
        /* gauge b[3] = 0; a absorbs the shift (P is unchanged) */
        double s = b[3];
        for (int j = 0; j < 4; ++j) bout[j] = b[j] - s;
    }
    if (iters) *iters = it;
    if (tol <= 0.0) converged = 1;
    return converged;
}

/* Returns the number of tokens that did not reach tol (0 when tol <= 0). */
int64_t oracle_sinkhorn64(const double *X, double *P, double *b, int64_t T, double tol,
                          int32_t max_iters, int32_t *iters_out)
{
    int64_t nonconv = 0;
    if (T <= 0) return 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : nonconv)
    for (int64_t t = 0; t < T; ++t) {
        int32_t it = 0;
        int ok = sinkhorn_token(X + 16 * t, P + 16 * t, b ? b + 4 * t : NULL, tol, max_iters, &it);
        if (!ok) ++nonconv;
        if (iters_out) iters_out[t] = it;
    }
    return nonconv;
}

/* ------------------------------------------------------------------------ */
/* Newton's method on the reduced dual [mHC s2.1].                           */
/*                                                                           */
/*   phi(b) = sum_i LSE_j(X_ij + b_j) - sum_j b_j,   b_3 = 0                 */
/*   p_ij(b) = softmax_j(X_ij + b_j)        (row softmax, rows shifted by     */
/*                                           their maximum)                  */
/*   grad_j  = sum_i p_ij - 1                                   (j = 0..2)   */
/*   Hess_jk = sum_i p_ij (delta_jk - p_ik)                     (j,k = 0..2) */
/*                                                                           */
/* The diagonal term p_ij (1 - p_ij) is evaluated as p_ij * sum_{l!=j} p_il  */
/* (equal because every row of p sums to one) so that it does not cancel     */
/* when p_ij is close to 1.  The 3x3 system is solved in closed form by the */
/* matrix-tree theorem (hessian_solve).  A Newton step longer than 32 in     */
/* the max norm is scaled down to 32 (far from the solution the dual is      */
/* nearly flat along some directions and the raw step is unbounded); the     */
/* step length then comes from Armijo backtracking on phi (on the marginal  */
/* residual once the predicted decrease of phi is below its rounding error). */
/* The iteration stops at residual <= tol, after                             */
/* max_iters steps, or when the residual is below 1e-10 and has not improved */
/* for 8 steps (rounding regime); the                                        */
/* best iterate seen is returned.                                            */
/* ------------------------------------------------------------------------ */

/* Evaluate the row softmax p(b), phi(b) and the gradient (all four columns). */
static double dual_eval(const double x[16], const double b[4], double p[16], double g[4])
{
    double phi = -(b[0] + b[1] + b[2] + b[3]);
    for (int i = 0; i < 4; ++i) {
        double z[4];
        double m = -INFINITY;
        for (int j = 0; j < 4; ++j) {
            z[j] = x[4 * i + j] + b[j];
            if (z[j] > m) m = z[j];
        }
        double e[4], s = 0.0;
        for (int j = 0; j < 4; ++j) {
            e[j] = exp(z[j] - m);
            s += e[j];
        }
        for (int j = 0; j < 4; ++j) p[4 * i + j] = e[j] / s;
        phi += m + log(s);
    }
    for (int j = 0; j < 4; ++j) g[j] = p[j] + p[4 + j] + p[8 + j] + p[12 + j] - 1.0;
    return phi;
}

/* The reduced Hessian as a graph Laplacian.  Because every row of p sums to
 * one, p_ij (1 - p_ij) = p_ij sum_{l!=j} p_il, so
 *   Hess_jk = -w_jk (j != k),   Hess_jj = sum_{l != j} w_jl,
 *   w_jk = sum_i p_ij p_ik      (j, k = 0..3, j != k),
 * i.e. Hess is the Laplacian of the complete graph on the four columns with
 * edge weights w, restricted to columns 0..2 (column 3 is grounded by the
 * gauge b_3 = 0).  Edge e joins columns EDGE[e][0] and EDGE[e][1]. */
static const int EDGE[6][2] = {{0, 1}, {0, 2}, {0, 3}, {1, 2}, {1, 3}, {2, 3}};

static void hessian_weights(const double p[16], double w[6])
{
    for (int e = 0; e < 6; ++e) {
        int j = EDGE[e][0], k = EDGE[e][1];
        double s = 0.0;
        for (int i = 0; i < 4; ++i) s += p[4 * i + j] * p[4 * i + k];
        w[e] = s;
    }
}

/* Connected components of the graph on columns 0..3 with the edges in mask;
 * comp[v] is a representative of v's component.  Returns the count. */
static int edge_components(unsigned mask, int comp[4])
{
    int par[4] = {0, 1, 2, 3};
    for (int e = 0; e < 6; ++e) {
        if (!(mask & (1u << e))) continue;
        int a = EDGE[e][0], b = EDGE[e][1];
        while (par[a] != a) a = par[a];
        while (par[b] != b) b = par[b];
        if (a != b) par[a] = b;
    }
    int n = 0;
    for (int v = 0; v < 4; ++v) {
        int a = v;
        while (par[a] != a) a = par[a];
        comp[v] = a;
        if (a == v) ++n;
    }
    return n;
}

/* Solve Hess x = r through the matrix-tree theorem (the inverse of a grounded
 * Laplacian in closed form):
 *   det Hess       = sum over spanning trees T of the four columns of w(T),
 *   (Hess^-1)_jk   = sum over spanning forests F with two trees, column 3 in
 *                    one and columns j and k in the other, of w(F), / det,
 * where w(.) is the product of the edge weights.  Every term is positive, so
 * nothing cancels however small the weights are; the sums run in long double
 * to keep products of tiny weights off the underflow threshold.  The four
 * columns have 16 spanning trees and 15 two-tree forests (every pair of
 * edges); which edge subsets they are, and which (j,k) each forest serves, is
 * enumerated once by brute force over the 2^6 edge subsets.
 * Returns -1 if the determinant is not positive (a zero weight pattern that
 * disconnects the graph). */
static struct {
    int ntree, nforest;
    unsigned tree[16];
    unsigned forest[15];
    unsigned char serves[15][3][3]; /* forest f contributes to (j,k) */
} MT;

static void matrix_tree_tables(void)
{
    int nt = 0, nf = 0;
    for (unsigned mask = 0; mask < 64; ++mask) {
        int ne = __builtin_popcount(mask);
        if (ne != 2 && ne != 3) continue;
        int comp[4];
        int nc = edge_components(mask, comp);
        if (ne == 3 && nc == 1) MT.tree[nt++] = mask;
        if (ne == 2 && nc == 2) {
            for (int j = 0; j < 3; ++j)
                for (int k = 0; k < 3; ++k)
                    MT.serves[nf][j][k] = (comp[j] == comp[k] && comp[j] != comp[3]);
            MT.forest[nf++] = mask;
        }
    }
    MT.ntree = nt;
    MT.nforest = nf;
}

static long double edge_product(const double w[6], unsigned mask)
{
    long double prod = 1.0L;
    for (int e = 0; e < 6; ++e)
        if (mask & (1u << e)) prod *= (long double)w[e];
    return prod;
}

static int hessian_solve(const double w[6], const double r[3], double x[3])
{
    long double det = 0.0L, F[3][3] = {{0.0L}};
    for (int t = 0; t < MT.ntree; ++t) det += edge_product(w, MT.tree[t]);
    for (int f = 0; f < MT.nforest; ++f) {
        long double prod = edge_product(w, MT.forest[f]);
        for (int j = 0; j < 3; ++j)
            for (int k = 0; k < 3; ++k)
                if (MT.serves[f][j][k]) F[j][k] += prod;
    }
    if (!(det > 0.0L)) return -1;
    for (int j = 0; j < 3; ++j)
        x[j] = (double)((F[j][0] * r[0] + F[j][1] * r[1] + F[j][2] * r[2]) / det);
    return 0;
}

/* Batched form of hessian_solve for the tests: w [n,6] (edge order
 * (0,1),(0,2),(0,3),(1,2),(1,3),(2,3)), r and x [n,3].  Returns the number of
 * systems with a non-positive determinant (their x is NaN). */
int64_t oracle_laplacian_solve64(const double *w, const double *r, double *x, int64_t n)
{
    int64_t bad = 0;
    matrix_tree_tables();
    for (int64_t t = 0; t < n; ++t) {
        if (hessian_solve(w + 6 * t, r + 3 * t, x + 3 * t) != 0) {
            x[3 * t] = x[3 * t + 1] = x[3 * t + 2] = NAN;
            ++bad;
        }
    }
    return bad;
}

static int newton_token(const double x[16], double pout[16], double bout[4], double tol,
                        int32_t max_iters, int32_t *iters, double *trace, int32_t trace_len)
{
    double b[4] = {0, 0, 0, 0};
    double p[16], g[4];
    if (nonfinite_token(x, pout, bout)) {
        if (iters) *iters = 0;
        if (trace)
            for (int32_t q = 0; q < trace_len; ++q) trace[q] = NAN;
        return 0;
    }
    double best_p[16], best_b[4], best_res = INFINITY;
    int32_t best_k = 0, since_best = 0;
    double phi = dual_eval(x, b, p, g);
    int32_t k = 0;
    if (trace)
        for (int32_t q = 0; q < trace_len; ++q) trace[q] = NAN;
    for (;;) {
        double res = marginal_residual(p);
        if (trace && k < trace_len) trace[k] = res;
        if (k == 0 || res < best_res) { /* k == 0: a NaN token keeps its NaN P */
            best_res = res;
            memcpy(best_p, p, sizeof best_p);
            memcpy(best_b, b, sizeof best_b);
            best_k = k;
            since_best = 0;
        } else {
            ++since_best;
        }
        if (res <= tol || k >= max_iters || isnan(res)) break;
        /* stalled in the rounding regime: more steps cannot help */
        if (since_best >= 8 && best_res < 1e-10) break;

        double w[6], step[3];
        hessian_weights(p, w);
        if (hessian_solve(w, g, step) != 0) {
            /* not numerically positive definite: fall back to a gradient step */
            for (int j = 0; j < 3; ++j) step[j] = g[j];
        }
        double smax = fmax(fabs(step[0]), fmax(fabs(step[1]), fabs(step[2])));
        if (smax > 32.0)
            for (int j = 0; j < 3; ++j) step[j] *= 32.0 / smax;
        double slope = g[0] * step[0] + g[1] * step[1] + g[2] * step[2];
        double t = 1.0;
        double bn[4], pn[16], gn[4], phin = phi;
        int accepted = 0;
        for (int ls = 0; ls < 60; ++ls) {
            bn[0] = b[0] - t * step[0];
            bn[1] = b[1] - t * step[1];
            bn[2] = b[2] - t * step[2];
            bn[3] = 0.0;
            phin = dual_eval(x, bn, pn, gn);
            /* Armijo sufficient decrease on phi */
            if (phin <= phi - 1e-4 * t * slope) {
                accepted = 1;
                break;
            }
            /* Near the solution the predicted decrease t*slope falls below the
             * rounding error of phi itself and the Armijo test is noise; there
             * the step is judged by the marginal residual instead. */
            if (t * slope <= 1e-12 * (fabs(phi) + 1.0) && marginal_residual(pn) < res) {
                accepted = 1;
                break;
            }
            t *= 0.5;
        }
        ++k;
        if (!accepted) {
            /* no decrease possible in floating point: stop at the best iterate */
            break;
        }
        memcpy(b, bn, sizeof b);
        memcpy(p, pn, sizeof p);
        memcpy(g, gn, sizeof g);
        phi = phin;
    }
    memcpy(pout, best_p, sizeof best_p);
    if (bout) memcpy(bout, best_b, sizeof best_b);
    if (iters) *iters = best_k;
    return best_res <= tol;
}

/* Returns the number of tokens whose best residual stayed above tol.
 * trace (optional) is [T, trace_len]: residual after each Newton step
 * (index 0 = at b = 0), NaN past the end. */
int64_t oracle_newton64(const double *X, double *P, double *b, int64_t T, double tol,
                        int32_t max_iters, int32_t *iters_out, double *trace, int32_t trace_len)
{
    int64_t nonconv = 0;
    if (T <= 0) return 0;
    matrix_tree_tables();
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : nonconv)
    for (int64_t t = 0; t < T; ++t) {
        int32_t it = 0;
        int ok = newton_token(X + 16 * t, P + 16 * t, b ? b + 4 * t : NULL, tol, max_iters, &it,
                              trace ? trace + (int64_t)trace_len * t : NULL, trace_len);
        if (!ok) ++nonconv;
        if (iters_out) iters_out[t] = it;
    }
    return nonconv;
}

/* ------------------------------------------------------------------------ */
/* Backward pass by the implicit function theorem [mHC s2.2].                */
/*                                                                           */
/* P(X) = p(X, b*(X)) with p the row softmax of X + b and b* defined by      */
/* F(X, b) = grad_b phi = colsum(p) - 1 = 0 (components 0..2, b_3 = 0).      */
/* For a loss L with G = dL/dP:                                              */
/*   dL/dX = dL/dX|_b  -  lambda^T dF/dX,   Hess lambda = dL/db|_X            */
/* where, with r_k = sum_j G_kj p_kj and D_kl = G_kl - r_k,                  */
/*   dL/dX_kl |_b = p_kl D_kl                                                 */
/*   dL/db_l  |_X = v_l = sum_k p_kl D_kl                       (l = 0..2)   */
/*   dF_l/dX_kq   = p_kl (delta_lq - p_kq)                                    */
/* so that  dX_kq = p_kq (D_kq - sum_l p_kl (lambda_q - lambda_l)),           */
/* lambda_3 = 0.  Hess is the dual Hessian at P (the matrix of the last      */
/* Newton step), solved in closed form by hessian_solve.                     */
/*                                                                           */
/* P is first rescaled to unit row sums (P from the forward pass has them up */
/* to rounding; storing P in a narrower type perturbs them).  With unit row  */
/* sums two identities hold exactly and are used to avoid cancellation when  */
/* a row of P is close to one-hot:                                           */
/*   D_kl = sum_j p_kj (G_kl - G_kj),                                         */
/*   lambda_q - sum_l p_kl lambda_l = sum_l p_kl (lambda_q - lambda_l).       */
/* ------------------------------------------------------------------------ */
static void backward_token(const double pin[16], const double G[16], double dX[16])
{
    double p[16], D[16];
    for (int k = 0; k < 4; ++k) {
        double s = pin[4 * k] + pin[4 * k + 1] + pin[4 * k + 2] + pin[4 * k + 3];
        for (int j = 0; j < 4; ++j) p[4 * k + j] = pin[4 * k + j] / s;
    }
    for (int k = 0; k < 4; ++k)
        for (int l = 0; l < 4; ++l) {
            double d = 0.0;
            for (int j = 0; j < 4; ++j)
                if (j != l) d += p[4 * k + j] * (G[4 * k + l] - G[4 * k + j]);
            D[4 * k + l] = d;
        }
    double v[3];
    for (int l = 0; l < 3; ++l)
        v[l] = p[l] * D[l] + p[4 + l] * D[4 + l] + p[8 + l] * D[8 + l] + p[12 + l] * D[12 + l];
    double w[6], lam[4] = {0, 0, 0, 0};
    hessian_weights(p, w);
    if (hessian_solve(w, v, lam) != 0) lam[0] = lam[1] = lam[2] = NAN;
    for (int k = 0; k < 4; ++k)
        for (int q = 0; q < 4; ++q) {
            double c = 0.0;
            for (int l = 0; l < 4; ++l)
                if (l != q) c += p[4 * k + l] * (lam[q] - lam[l]);
            dX[4 * k + q] = p[4 * k + q] * (D[4 * k + q] - c);
        }
}

void oracle_backward64(const double *P, const double *G, double *dX, int64_t T)
{
    if (T <= 0) return;
    matrix_tree_tables();
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) backward_token(P + 16 * t, G + 16 * t, dX + 16 * t);
}

/* ======================================================================== */
/* General n x n (2 <= n <= 16): the same projection for an n x n logit     */
/* matrix, the dual reduced to n-1 free variables (b_{n-1} = 0) [mHC s2.1: */
/* m-1 free variables for m columns].  Written separately from the 4 x 4    */
/* code above (which it is checked against at n = 4); the Newton system is  */
/* solved by Cholesky after symmetric diagonal scaling, in long double.     */
/* ======================================================================== */
#define NMAX 16

static double lse_n(const double *v, int n, int stride)
{
    double m = -INFINITY;
    for (int k = 0; k < n; ++k)
        if (v[k * stride] > m) m = v[k * stride];
    if (isinf(m) && m < 0) return m;
    double s = 0.0;
    for (int k = 0; k < n; ++k) s += exp(v[k * stride] - m);
    return m + log(s);
}

static double marginal_residual_n(const double *p, int n)
{
    double res = 0.0;
    for (int i = 0; i < n; ++i) {
        double s = 0.0, c = 0.0;
        for (int j = 0; j < n; ++j) {
            s += p[n * i + j];
            c += p[n * j + i];
        }
        double d = fmax(fabs(s - 1.0), fabs(c - 1.0));
        if (d > res || isnan(d)) res = d;
    }
    return res;
}

static int nonfinite_n(const double *x, double *p, double *b, int n)
{
    for (int k = 0; k < n * n; ++k) {
        if (!isfinite(x[k])) {
            for (int q = 0; q < n * n; ++q) p[q] = NAN;
            if (b)
                for (int q = 0; q < n; ++q) b[q] = NAN;
            return 1;
        }
    }
    return 0;
}

/* Log-domain Sinkhorn-Knopp for one n x n token (as sinkhorn_token). */
static int sinkhorn_token_n(const double *x, double *p, double *bout, int n, double tol,
                            int32_t max_iters, int32_t *iters)
{
    double a[NMAX] = {0}, b[NMAX] = {0}, z[NMAX];
    if (nonfinite_n(x, p, bout, n)) {
        if (iters) *iters = 0;
        return 0;
    }
    int converged = 0;
    int32_t it = 0;
    while (it < max_iters) {
        for (int i = 0; i < n; ++i) {
            for (int j = 0; j < n; ++j) z[j] = x[n * i + j] + b[j];
            a[i] = -lse_n(z, n, 1);
        }
        for (int j = 0; j < n; ++j) {
            for (int i = 0; i < n; ++i) z[i] = x[n * i + j] + a[i];
            b[j] = -lse_n(z, n, 1);
        }
        ++it;
        if (tol > 0.0) {
            double q[NMAX * NMAX];
            for (int i = 0; i < n; ++i)
                for (int j = 0; j < n; ++j) q[n * i + j] = exp(x[n * i + j] + a[i] + b[j]);
            if (marginal_residual_n(q, n) < tol) {
                converged = 1;
                break;
            }
        }
    }
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) p[n * i + j] = exp(x[n * i + j] + a[i] + b[j]);
    if (bout)
        for (int j = 0; j < n; ++j) bout[j] = b[j] - b[n - 1];
    if (iters) *iters = it;
    return tol <= 0.0 ? 1 : converged;
}

int64_t oracle_sinkhorn64_n(const double *X, double *P, double *b, int32_t n, int64_t T,
                            double tol, int32_t max_iters, int32_t *iters_out)
{
    int64_t nonconv = 0;
    if (T <= 0 || n < 2 || n > NMAX) return 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : nonconv)
    for (int64_t t = 0; t < T; ++t) {
        int32_t it = 0;
        int ok = sinkhorn_token_n(X + (int64_t)n * n * t, P + (int64_t)n * n * t,
                                  b ? b + (int64_t)n * t : NULL, n, tol, max_iters, &it);
        if (!ok) ++nonconv;
        if (iters_out) iters_out[t] = it;
    }
    return nonconv;
}

/* phi(b), the row softmax p(b) and the gradient colsum(p) - 1, for n x n. */
static double dual_eval_n(const double *x, const double *b, double *p, double *g, int n)
{
    double phi = 0.0;
    for (int j = 0; j < n; ++j) phi -= b[j];
    for (int i = 0; i < n; ++i) {
        double m = -INFINITY;
        for (int j = 0; j < n; ++j) {
            double z = x[n * i + j] + b[j];
            if (z > m) m = z;
        }
        double s = 0.0;
        for (int j = 0; j < n; ++j) {
            p[n * i + j] = exp(x[n * i + j] + b[j] - m);
            s += p[n * i + j];
        }
        for (int j = 0; j < n; ++j) p[n * i + j] /= s;
        phi += m + log(s);
    }
    for (int j = 0; j < n; ++j) {
        double c = 0.0;
        for (int i = 0; i < n; ++i) c += p[n * i + j];
        g[j] = c - 1.0;
    }
    return phi;
}

/* Hessian of phi on b_0..b_{n-2}: H_jk = sum_i p_ij (delta_jk - p_ik), the
 * diagonal as p_ij sum_{l != j} p_il (rows of p sum to one). */
static void dual_hessian_n(const double *p, int n, long double H[NMAX][NMAX])
{
    for (int j = 0; j < n - 1; ++j)
        for (int k = 0; k < n - 1; ++k) {
            long double h = 0.0L;
            for (int i = 0; i < n; ++i) {
                const double *pi = p + n * i;
                if (j == k) {
                    long double rest = 0.0L;
                    for (int l = 0; l < n; ++l)
                        if (l != j) rest += pi[l];
                    h += (long double)pi[j] * rest;
                } else {
                    h -= (long double)pi[j] * pi[k];
                }
            }
            H[j][k] = h;
        }
}

/* Solve H x = r (m = n-1 unknowns) by Cholesky after symmetric diagonal
 * scaling, in long double.  Returns -1 if H is not numerically positive
 * definite. */
static int spd_solve_n(long double H[NMAX][NMAX], const double *r, double *x, int m)
{
    long double d[NMAX], L[NMAX][NMAX], y[NMAX], z[NMAX];
    for (int j = 0; j < m; ++j) {
        if (!(H[j][j] > 0.0L)) return -1;
        d[j] = 1.0L / sqrtl(H[j][j]);
    }
    for (int j = 0; j < m; ++j) {
        long double s = d[j] * H[j][j] * d[j];
        for (int k = 0; k < j; ++k) s -= L[j][k] * L[j][k];
        if (!(s > 0.0L)) return -1;
        L[j][j] = sqrtl(s);
        for (int i = j + 1; i < m; ++i) {
            long double t = d[i] * H[i][j] * d[j];
            for (int k = 0; k < j; ++k) t -= L[i][k] * L[j][k];
            L[i][j] = t / L[j][j];
        }
    }
    for (int j = 0; j < m; ++j) {
        long double s = d[j] * r[j];
        for (int k = 0; k < j; ++k) s -= L[j][k] * y[k];
        y[j] = s / L[j][j];
    }
    for (int j = m - 1; j >= 0; --j) {
        long double s = y[j];
        for (int k = j + 1; k < m; ++k) s -= L[k][j] * z[k];
        z[j] = s / L[j][j];
    }
    for (int j = 0; j < m; ++j) x[j] = (double)(d[j] * z[j]);
    return 0;
}

/* Newton with Armijo backtracking for one n x n token (as newton_token). */
static int newton_token_n(const double *x, double *pout, double *bout, int n, double tol,
                          int32_t max_iters, int32_t *iters)
{
    double b[NMAX] = {0}, p[NMAX * NMAX], g[NMAX];
    double best_p[NMAX * NMAX], best_b[NMAX], best_res = INFINITY;
    int32_t best_k = 0, since_best = 0;
    if (nonfinite_n(x, pout, bout, n)) {
        if (iters) *iters = 0;
        return 0;
    }
    double phi = dual_eval_n(x, b, p, g, n);
    int32_t k = 0;
    for (;;) {
        double res = marginal_residual_n(p, n);
        if (k == 0 || res < best_res) {
            best_res = res;
            memcpy(best_p, p, sizeof(double) * n * n);
            memcpy(best_b, b, sizeof(double) * n);
            best_k = k;
            since_best = 0;
        } else {
            ++since_best;
        }
        if (res <= tol || k >= max_iters || isnan(res)) break;
        if (since_best >= 8 && best_res < 1e-10) break;
        long double H[NMAX][NMAX];
        double step[NMAX];
        dual_hessian_n(p, n, H);
        if (spd_solve_n(H, g, step, n - 1) != 0)
            for (int j = 0; j < n - 1; ++j) step[j] = g[j];
        double smax = 0.0;
        for (int j = 0; j < n - 1; ++j) smax = fmax(smax, fabs(step[j]));
        if (smax > 32.0)
            for (int j = 0; j < n - 1; ++j) step[j] *= 32.0 / smax;
        double slope = 0.0;
        for (int j = 0; j < n - 1; ++j) slope += g[j] * step[j];
        double t = 1.0, bn[NMAX], pn[NMAX * NMAX], gn[NMAX], phin = phi;
        int accepted = 0;
        for (int ls = 0; ls < 60; ++ls) {
            for (int j = 0; j < n - 1; ++j) bn[j] = b[j] - t * step[j];
            bn[n - 1] = 0.0;
            phin = dual_eval_n(x, bn, pn, gn, n);
            if (phin <= phi - 1e-4 * t * slope) {
                accepted = 1;
                break;
            }
            if (t * slope <= 1e-12 * (fabs(phi) + 1.0) && marginal_residual_n(pn, n) < res) {
                accepted = 1;
                break;
            }
            t *= 0.5;
        }
        ++k;
        if (!accepted) break;
        memcpy(b, bn, sizeof(double) * n);
        memcpy(p, pn, sizeof(double) * n * n);
        memcpy(g, gn, sizeof(double) * n);
        phi = phin;
    }
    memcpy(pout, best_p, sizeof(double) * n * n);
    if (bout) memcpy(bout, best_b, sizeof(double) * n);
    if (iters) *iters = best_k;
    return best_res <= tol;
}

int64_t oracle_newton64_n(const double *X, double *P, double *b, int32_t n, int64_t T, double tol,
                          int32_t max_iters, int32_t *iters_out)
{
    int64_t nonconv = 0;
    if (T <= 0 || n < 2 || n > NMAX) return 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : nonconv)
    for (int64_t t = 0; t < T; ++t) {
        int32_t it = 0;
        int ok = newton_token_n(X + (int64_t)n * n * t, P + (int64_t)n * n * t,
                                b ? b + (int64_t)n * t : NULL, n, tol, max_iters, &it);
        if (!ok) ++nonconv;
        if (iters_out) iters_out[t] = it;
    }
    return nonconv;
}

/* Implicit-function-theorem backward for one n x n token (as backward_token,
 * same difference forms, Cholesky solve). */
static void backward_token_n(const double *pin, const double *G, double *dX, int n)
{
    double p[NMAX * NMAX], D[NMAX * NMAX], v[NMAX], lam[NMAX];
    for (int k = 0; k < n; ++k) {
        double s = 0.0;
        for (int j = 0; j < n; ++j) s += pin[n * k + j];
        for (int j = 0; j < n; ++j) p[n * k + j] = pin[n * k + j] / s;
    }
    for (int k = 0; k < n; ++k)
        for (int l = 0; l < n; ++l) {
            double d = 0.0;
            for (int j = 0; j < n; ++j)
                if (j != l) d += p[n * k + j] * (G[n * k + l] - G[n * k + j]);
            D[n * k + l] = d;
        }
    for (int l = 0; l < n - 1; ++l) {
        double s = 0.0;
        for (int k = 0; k < n; ++k) s += p[n * k + l] * D[n * k + l];
        v[l] = s;
    }
    long double H[NMAX][NMAX];
    dual_hessian_n(p, n, H);
    if (spd_solve_n(H, v, lam, n - 1) != 0)
        for (int l = 0; l < n - 1; ++l) lam[l] = NAN;
    lam[n - 1] = 0.0;
    for (int k = 0; k < n; ++k)
        for (int q = 0; q < n; ++q) {
            double c = 0.0;
            for (int l = 0; l < n; ++l)
                if (l != q) c += p[n * k + l] * (lam[q] - lam[l]);
            dX[n * k + q] = p[n * k + q] * (D[n * k + q] - c);
        }
}

void oracle_backward64_n(const double *P, const double *G, double *dX, int32_t n, int64_t T)
{
    if (T <= 0 || n < 2 || n > NMAX) return;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        backward_token_n(P + (int64_t)n * n * t, G + (int64_t)n * n * t, dX + (int64_t)n * n * t, n);
}
