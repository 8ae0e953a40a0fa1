"""Float64 CPU oracle for entropic optimal transport between point clouds
(test infrastructure only: the product path never imports this module).

Follows "FlashSinkhorn: IO-Aware Entropic OT on GPU", Methodik, s1: the
log-domain Sinkhorn update for the quadratic Euclidean cost,

    f_i <- -eps * LSE_j[ (g_j - C_ij) / eps + log b_j ],   C_ij = ||x_i - y_j||^2,

and, by the symmetry of the problem in (x, a, f) <-> (y, b, g), the update of
g from f.  One Sinkhorn iteration is the f update followed by the g update
with the new f (the standard alternating scheme; the pages do not spell out
the order).  The cost is formed here directly from the differences x_i - y_j,
not in the expanded dot-product ("attention") form of the pages' Proposition
1, so this module shares no arithmetic with a kernel that uses that form.

The transport application of s3 (the plan applied to the key points, and
from it the gradient of the cost and the barycentric map) is the plan
pi_ij = a_i b_j exp((f_i + g_j - C_ij)/eps) formed densely and multiplied.

Everything is dense numpy float64 over the full n x m cost matrix, processed
in row blocks to bound memory; it is meant for n, m up to a few thousand.
"""
from __future__ import annotations

import numpy as np

_BLOCK_ELEMS = 1 << 22  # cost-matrix entries per row block


def _as64(A, name, ndim):
    A = np.asarray(A, dtype=np.float64)
    if A.ndim != ndim:
        raise ValueError("%s must have %d dimensions" % (name, ndim))
    return A


def sqeuclid_cost64(X, Y) -> np.ndarray:
    """C_ij = sum_k (x_ik - y_jk)^2, from the differences (float64)."""
    X = _as64(X, "X", 2)
    Y = _as64(Y, "Y", 2)
    if X.shape[1] != Y.shape[1]:
        raise ValueError("X and Y must have the same number of columns")
    C = np.empty((X.shape[0], Y.shape[0]))
    rows = max(1, _BLOCK_ELEMS // max(1, Y.shape[0] * max(1, X.shape[1])))
    for r0 in range(0, X.shape[0], rows):
        D = X[r0:r0 + rows, None, :] - Y[None, :, :]
        C[r0:r0 + rows] = np.einsum("ijk,ijk->ij", D, D)
    return C


def lse64(M, axis) -> np.ndarray:
    """log sum exp along `axis`, shifted by the maximum (float64)."""
    M = np.asarray(M, dtype=np.float64)
    mx = M.max(axis=axis, keepdims=True)
    mx = np.where(np.isfinite(mx), mx, 0.0)
    return np.squeeze(mx, axis=axis) + np.log(np.exp(M - mx).sum(axis=axis))


def f_update64(X, Y, g, log_b, eps) -> np.ndarray:
    """f_i = -eps LSE_j[(g_j - C_ij)/eps + log b_j]  (Methodik, s1)."""
    g = _as64(g, "g", 1)
    log_b = _as64(log_b, "log_b", 1)
    if eps <= 0:
        raise ValueError("eps must be positive")
    C = sqeuclid_cost64(X, Y)
    return -eps * lse64((g[None, :] - C) / eps + log_b[None, :], axis=1)


def g_update64(X, Y, f, log_a, eps) -> np.ndarray:
    """g_j = -eps LSE_i[(f_i - C_ij)/eps + log a_i]: the f update with the
    roles of the two clouds exchanged."""
    return f_update64(Y, X, f, log_a, eps)


def sinkhorn64(X, Y, log_a, log_b, eps, iters, f0=None, g0=None):
    """`iters` alternating iterations (f update, then g update with the new
    f) from (f0, g0) (default zeros).  Returns (f, g)."""
    n, m = np.shape(X)[0], np.shape(Y)[0]
    g = np.zeros(m) if g0 is None else _as64(g0, "g0", 1).copy()
    f = np.zeros(n) if f0 is None else _as64(f0, "f0", 1).copy()
    C = sqeuclid_cost64(X, Y)
    la = _as64(log_a, "log_a", 1)
    lb = _as64(log_b, "log_b", 1)
    for _ in range(int(iters)):
        f = -eps * lse64((g[None, :] - C) / eps + lb[None, :], axis=1)
        g = -eps * lse64((f[:, None] - C) / eps + la[:, None], axis=0)
    return f, g


def plan64(X, Y, f, g, log_a, log_b, eps) -> np.ndarray:
    """P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps), the transport plan of the
    dual potentials."""
    C = sqeuclid_cost64(X, Y)
    f = _as64(f, "f", 1)
    g = _as64(g, "g", 1)
    return np.exp((f[:, None] + g[None, :] - C) / eps + _as64(log_a, "log_a", 1)[:, None]
                  + _as64(log_b, "log_b", 1)[None, :])


def primal_cost64(X, Y, P, log_a, log_b, eps) -> float:
    """<C, P> + eps KL(P | a b^T), the entropic OT objective of a plan."""
    C = sqeuclid_cost64(X, Y)
    P = np.asarray(P, dtype=np.float64)
    la = _as64(log_a, "log_a", 1)
    lb = _as64(log_b, "log_b", 1)
    with np.errstate(divide="ignore"):
        logP = np.log(P)
    kl = np.sum(np.where(P > 0, P * (logP - la[:, None] - lb[None, :]) - P, 0.0)) \
        + np.exp(la).sum() * np.exp(lb).sum()
    return float(np.sum(C * P) + eps * kl)


def transport64(X, Y, f, g, log_a, log_b, eps):
    """Transport application ("FlashSinkhorn", Methodik s3): with
    pi_ij = a_i b_j exp((f_i + g_j - C_ij)/eps), returns (pi Y [n, d],
    pi 1 [n]), the weighted sums of the key points and the row masses."""
    P = plan64(X, Y, f, g, log_a, log_b, eps)
    return P @ np.asarray(Y, dtype=np.float64), P.sum(1)


def grad_x64(X, Y, f, g, log_a, log_b, eps):
    """Gradient of the entropic OT cost with respect to the points X at
    optimal potentials (envelope theorem on the dual):
    d/dx_i = sum_j pi_ij d C_ij / d x_i = 2 (r_i x_i - (pi Y)_i)."""
    PY, r = transport64(X, Y, f, g, log_a, log_b, eps)
    return 2.0 * (r[:, None] * np.asarray(X, dtype=np.float64) - PY)


def eot_cost64(X, Y, log_a, log_b, eps, iters):
    """The entropic OT cost <f, a> + <g, b> after `iters` alternating
    iterations from zero potentials (the dual value at convergence)."""
    f, g = sinkhorn64(X, Y, log_a, log_b, eps, iters)
    return float(f @ np.exp(_as64(log_a, "log_a", 1)) + g @ np.exp(_as64(log_b, "log_b", 1)))


def apply_plan64(X, Y, f, g, log_a, log_b, eps, V):
    """The plan of (f, g) applied to values V [m, dv]: (pi V, pi 1)."""
    P = plan64(X, Y, f, g, log_a, log_b, eps)
    return P @ np.asarray(V, dtype=np.float64), P.sum(1)


def hvp64(X, Y, f, g, log_a, log_b, eps, V):
    """Hessian-vector product of the entropic OT cost with respect to X at
    converged potentials ("FlashSinkhorn", Methodik s3: the HVP as transport
    products), written out densely.

    With pi the plan, the row marginals fixed (sum_j dpi_ij = 0) and
    dC_ij = 2 (x_i - y_j).v_i:
        (H v)_i = 2 a_i v_i - 2 sum_j dpi_ij y_j,
        dpi_ij = pi_ij (df_i + dg_j - dC_ij) / eps,
    where (df, dg) solve the linearised marginal conditions
        a_i df_i + (pi dg)_i = sum_j pi_ij dC_ij,
        (pi^T df)_j + b_j dg_j = sum_i pi_ij dC_ij
    (a singular symmetric system with null vector (1, -1), solved here by
    least squares).  Returns H v [n, d]."""
    X = _as64(X, "X", 2)
    Y = _as64(Y, "Y", 2)
    V = _as64(V, "V", 2)
    n = X.shape[0]
    a = np.exp(_as64(log_a, "log_a", 1))
    b = np.exp(_as64(log_b, "log_b", 1))
    P = plan64(X, Y, f, g, log_a, log_b, eps)
    dC = 2.0 * ((X * V).sum(1)[:, None] - V @ Y.T)
    r = (P * dC).sum(1)
    c = (P * dC).sum(0)
    A = np.block([[np.diag(a), P], [P.T, np.diag(b)]])
    sol = np.linalg.lstsq(A, np.r_[r, c], rcond=None)[0]
    df, dg = sol[:n], sol[n:]
    dP = P * (df[:, None] + dg[None, :] - dC) / eps
    return 2.0 * a[:, None] * V - 2.0 * dP @ Y
