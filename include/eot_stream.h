/* eot_stream.h -- streaming entropic optimal transport between point clouds
 * on one GB300 (part of libbirkhoff4.so).
 *
 * Follows "FlashSinkhorn: IO-Aware Entropic OT on GPU", Methodik s1-s2:
 * the log-domain Sinkhorn update for the quadratic Euclidean cost
 *
 *     f_i <- -eps LSE_j[ (g_j - ||x_i - y_j||^2) / eps + log b_j ]
 *
 * computed in the pages' attention form (s1, Proposition 1): with
 * ||x - y||^2 = ||x||^2 + ||y||^2 - 2 x.y the update is
 *     f_i = ||x_i||^2 - eps LSE_j[ (2 x_i.y_j + g_j - ||y_j||^2) / eps + log b_j ],
 * a row-wise log-sum-exp of a biased dot-product score matrix.  The n x m
 * cost matrix is never stored (s2): a CTA keeps 128 query rows and streams
 * every key tile through shared memory (TMA), the dot products run on the
 * tensor cores (tcgen05, accumulators in tensor memory), and a running
 * maximum and sum of exponentials per row stay in registers (online LSE,
 * row-stationary traversal).
 *
 * Arithmetic: point coordinates are rounded to TF32 for the products and
 * accumulated in fp32 (EOT_TF32), or split x = hi + lo into two TF32 parts
 * with the products hi.hi + hi.lo + lo.hi (EOT_TF32X3, near-fp32 accuracy,
 * three MMAs per step).  Norms, biases and the log-sum-exp are fp32.
 *
 * Layout: X [n, d], Y [m, d] row-major fp32 (point i at X + i*d); log_a [n],
 * log_b [m], f [n], g [m] fp32.  All pointers are device memory owned by the
 * caller; the library allocates nothing.  Work is asynchronous on `stream`.
 *
 * Workspace: the clouds are repacked once per call into the workspace (rows
 * padded to a multiple of 256, coordinates padded with zeros to a multiple of
 * 32, rounded to TF32), with their squared norms and one bias vector;
 * eot_workspace_bytes gives the size.  It must be 256-byte aligned.
 *
 * Errors (return values, from birkhoff4.h): B4_EINVAL for a NULL pointer with
 * work to do, n < 0, m < 0, m == 0 < n, d < 1 or d > 16384, eps not a positive
 * finite number, iters < 0, passes not 1 or 3, more than 2^31 - 512 points,
 * or a workspace that is too small or misaligned; B4_ECUDA for a launch
 * error (birkhoff4_last_cuda_error has the code).  n == 0 does nothing.  A
 * tensor-pipeline wait that runs out (2 s) sets bit 2 of the fault latch
 * (birkhoff4_device_status) and the kernel returns; it never traps.
 */
#ifndef EOT_STREAM_H
#define EOT_STREAM_H

#include <stddef.h>
#include <stdint.h>

#include "birkhoff4.h"

#ifdef __cplusplus
extern "C" {
#endif

#define EOT_TF32 1   /* one TF32 product per coordinate pair */
#define EOT_TF32X3 3 /* split hi + lo, three TF32 products (near fp32) */

/* Bytes of workspace that eot_sinkhorn / eot_update need for n points
 * against m points in d dimensions (0 for invalid sizes or passes). */
size_t eot_workspace_bytes(int64_t n, int64_t m, int32_t d, int32_t passes);

/* One potential update [FlashSinkhorn, Methodik s1]:
 *     out_i = -eps LSE_j[ (h_j - ||xq_i - xk_j||^2) / eps + log_w_j ],
 * i < nq, j < nk.  Xq [nq, d] are the query points (the side whose potential
 * is written), Xk [nk, d] the key points, h [nk] the key-side potential,
 * log_w [nk] the key-side log weights.  The f update is (X, Y, g, log_b);
 * the g update is (Y, X, f, log_a).  out may not alias the other inputs. */
int eot_update(const float *Xq, const float *Xk, const float *h, const float *log_w, float *out,
               int64_t nq, int64_t nk, int32_t d, float eps, int32_t passes, void *workspace,
               size_t workspace_bytes, birkhoff4_stream_t stream);

/* `iters` alternating Sinkhorn iterations [FlashSinkhorn, Methodik s1]:
 * each iteration updates f from g (keys Y, weights b), then g from the new f
 * (keys X, weights a).  f [n] and g [m] hold the starting potentials on
 * entry (zeros for a cold start) and the result on return.  The clouds are
 * repacked once per call, not per iteration. */
int eot_sinkhorn(const float *X, const float *Y, const float *log_a, const float *log_b, float *f,
                 float *g, int64_t n, int64_t m, int32_t d, float eps, int32_t iters,
                 int32_t passes, void *workspace, size_t workspace_bytes,
                 birkhoff4_stream_t stream);

/* Transport application [FlashSinkhorn, Methodik s3]: with the plan of
 * the potentials f [n] and g [m],
 *     pi_ij = a_i b_j exp((f_i + g_j - ||x_i - y_j||^2) / eps),
 * computes PY [n, d] = pi Y (PY_i = sum_j pi_ij y_j) and mass [n] = pi 1
 * without storing pi.  If grad is not NULL it also writes grad [n, d] =
 * 2 (mass_i x_i - PY_i): at Sinkhorn-converged potentials this is the
 * gradient of the entropic OT cost <f, a> + <g, b> with respect to X
 * (envelope theorem); PY_i / mass_i is the barycentric map.  For f the exact
 * update of g (eot_update), pi's rows are normalised softmax weights, so no
 * running maximum is needed.  Otherwise pi is evaluated as given, and
 * potentials far from consistent can overflow.
 * Arithmetic: TF32 products with fp32 accumulation for both chained
 * products (S = X Y^T, then pi Y, with pi held in tensor memory);
 * exponentials and masses in fp32.  The value coordinates are processed 256
 * at a time, one launch each.
 * Workspace: eot_transport_workspace_bytes(n, m, d), 256-byte aligned.
 * Errors as for eot_update; PY, mass must not alias the inputs or each
 * other, grad may be NULL. */
size_t eot_transport_workspace_bytes(int64_t n, int64_t m, int32_t d);

/* The plan of f and g applied to any values V [m, dv] (row-major fp32) at
 * the key points [FlashSinkhorn, Methodik s3: the transport matrix applied
 * without materialising it]: out [n, dv] = pi V, mass [n] = pi 1, with pi
 * as for eot_transport (which is the case V = Y).  Same arithmetic, errors
 * and conditions; the workspace is eot_apply_plan_workspace_bytes(n, m, d,
 * dv) bytes. */
size_t eot_apply_plan_workspace_bytes(int64_t n, int64_t m, int32_t d, int32_t dv);
int eot_apply_plan(const float *X, const float *Y, const float *f, const float *g,
                   const float *log_a, const float *log_b, const float *V, int32_t dv, float *out,
                   float *mass, int64_t n, int64_t m, int32_t d, float eps, void *workspace,
                   size_t workspace_bytes, birkhoff4_stream_t stream);
int eot_transport(const float *X, const float *Y, const float *f, const float *g,
                  const float *log_a, const float *log_b, float *PY, float *mass, float *grad,
                  int64_t n, int64_t m, int32_t d, float eps, void *workspace,
                  size_t workspace_bytes, birkhoff4_stream_t stream);

/* Hessian-vector product of the entropic OT cost with respect to the points
 * X [FlashSinkhorn, Methodik s3: the HVP as a sequence of transport-vector
 * and transport-matrix products, the n d x n d Hessian never formed]: out
 * [n, d] = H V for a direction V [n, d], at potentials (f, g) that
 * Sinkhorn has converged.  With pi the plan, dC_ij = 2 (x_i - y_j).v_i and
 * the row marginals fixed:
 *     (H V)_i = 2 a_i v_i - 2 sum_j dpi_ij y_j,
 *     dpi_ij = pi_ij (df_i + dg_j - dC_ij) / eps,
 * where (df, dg) solve the linearised marginal conditions
 *     [[diag(a), pi], [pi^T, diag(b)]] [df; dg] = [pi dC 1; pi^T dC 1]
 * by at most cg_iters steps of conjugate gradients with the diagonal as
 * preconditioner.  The two plan products of a step carry their own score
 * rounding, so the operator is symmetric only to about 1e-3 and the
 * residual levels off: the iteration stops, on the device, once
 * r^T diag^-1 r is 1e-8 of its first value or has risen 1e4-fold above its
 * smallest value, and the iterate with the smallest value is used.  Its
 * component along (1, -1), which leaves H V unchanged, is removed.
 * cg_iters is a maximum: the plan products of the steps after the stop are
 * skipped on the device.  Each step applies pi and pi^T once
 * to one column (two streaming passes over the n x m scores); the
 * remaining terms are plan applications (pi Y, pi^T [x.v, V],
 * pi [dg, dg y]) and one second-moment pass sum_j pi_ij (v_i . y_j) y_j.
 * The scores are one TF32 pass; the CG runs in fp32 with fp64 dot
 * products, with no host synchronisation.
 * Workspace: eot_hvp_workspace_bytes(n, m, d), 256-byte aligned.  Errors as
 * for eot_update, and B4_EINVAL for cg_iters outside 0..100000. */
/* Diagnostic (host only, no GPU needed): the transport kernel's work split
 * of n_rb row blocks of n_kt key tiles over `ctas` CTAs, as used by
 * eot_transport, eot_apply_plan and eot_hvp.  CTA b first takes whole row
 * blocks b, b + ctas, ..., then an equal contiguous run of the remaining
 * tiles.  The split is played on the host with the kernel's own tile walk
 * and partial-slot rule and checked against the fix-up's slot rule:
 *   - every tile is visited once;
 *   - each row block is either one CTA's whole segment, or is split among
 *     CTAs whose partial slots are the ones the fix-up sums;
 *   - no slot holds two row blocks.
 * owner [n_rb * n_kt] (row block major), or NULL, receives the CTA of each
 * tile.  Returns B4_OK; B4_EINVAL unless n_rb >= 1, n_kt >= 1,
 * 1 <= ctas <= min(256, n_rb n_kt) and n_rb n_kt <= 2^28; or minus the
 * number of inconsistencies found. */
int eot_transport_schedule(int64_t n_rb, int32_t n_kt, int32_t ctas, int64_t *owner);

size_t eot_hvp_workspace_bytes(int64_t n, int64_t m, int32_t d);
int eot_hvp(const float *X, const float *Y, const float *f, const float *g, const float *log_a,
            const float *log_b, const float *V, float *out, int64_t n, int64_t m, int32_t d,
            float eps, int32_t cg_iters, void *workspace, size_t workspace_bytes,
            birkhoff4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EOT_STREAM_H */
