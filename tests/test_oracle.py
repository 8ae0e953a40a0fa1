"""Pins for the float64 oracle (CPU only).

The oracle is checked against facts that do not come from the oracle itself:
  * closed forms (tests/golden/closed_forms.json, derived by hand from the
    definition of the projection and of its backward pass);
  * the fixed-point family X = log Q + u 1^T + 1 v^T, whose projection is Q;
  * invariants the definition fixes: unit marginals, positivity, the
    diag(e^a) exp(X) diag(e^b) form (double-centred log P - X vanishes),
    equivariance under row/column permutations and transposition, invariance
    under row/column offsets;
  * two independent solvers (Sinkhorn-Knopp and Newton) agreeing;
  * quadratic convergence of Newton's method ("Accelerating the Birkhoff
    Projection for Manifold-Constrained Hyper-Connections", s2.1);
  * the implicit-differentiation backward (s2.2) against central finite
    differences, against autodiff through a long unrolled Sinkhorn-Knopp, and
    against the symmetry of the Jacobian (P is the gradient of a convex
    function of X);
  * the pages' qualitative accuracy claim (s4): fixed 20-iteration
    Sinkhorn-Knopp is accurate at N(0,1) but far off at N(0,10^2).
Planted mistakes (a transposed operand, a dropped term, a wrong sign) are
shown to fail these pins at the end of the file.
"""
import json
import os

import numpy as np
import pytest

import oracle
from birkhoff_projection_gb300 import workloads

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "closed_forms.json")))


def rng(seed):
    return np.random.default_rng(seed)


def large_mag(T, seed):
    x, _ = workloads.large_magnitude(T)
    return x.double().numpy()


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
@pytest.mark.parametrize("case", GOLDEN["forward"], ids=lambda c: c["name"])
def test_closed_form_forward(case):
    X = np.array(case["X"])[None]
    P = np.array(case["P"])[None]
    Pn = oracle.newton64(X)[0]
    Ps = oracle.sinkhorn64(X)[0]
    assert np.abs(Pn - P).max() <= 1e-13
    assert np.abs(Ps - P).max() <= 1e-13


@pytest.mark.parametrize("case", GOLDEN["backward"], ids=lambda c: c["name"])
def test_closed_form_backward(case):
    X = np.array(case["X"])[None]
    G = np.array(case["G"])[None]
    dX = np.array(case["dX"])[None]
    P = oracle.newton64(X)[0]
    assert np.abs(oracle.backward64(P, G) - dX).max() <= 1e-13


@pytest.mark.parametrize("c", [-30.0, -3.0, 0.7, 5.0, 40.0])
def test_scaled_identity(c):
    """X = cI: P_ii = e^c/(e^c+3), P_ij = 1/(e^c+3) for any c."""
    X = (c * np.eye(4))[None]
    P = oracle.newton64(X)[0][0]
    # written stably for large |c|
    diag = 1.0 / (1.0 + 3.0 * np.exp(-c))
    off = 1.0 / (np.exp(c) + 3.0)
    want = np.where(np.eye(4) > 0, diag, off)
    assert np.allclose(P, want, rtol=1e-12, atol=0)


def test_circulant_is_row_softmax():
    r = rng(3)
    x = r.standard_normal((200, 4)) * 3.0
    idx = (np.arange(4)[None, :] - np.arange(4)[:, None]) % 4
    X = x[:, idx]
    P = oracle.newton64(X)[0]
    e = np.exp(X - X.max(axis=2, keepdims=True))
    soft = e / e.sum(axis=2, keepdims=True)
    assert np.abs(P - soft).max() <= 1e-13


@pytest.mark.parametrize("spread,floor", [(5.0, 1e-3), (60.0, 1e-3), (20.0, 1e-12), (5.0, 1e-30)])
def test_fixed_point_family(spread, floor):
    X, Q = workloads.fixed_point_family(2000, seed=11, spread=spread, floor=floor)
    P = oracle.newton64(X.numpy())[0]
    Q = Q.numpy()
    assert np.abs(P - Q).max() <= 1e-12
    # relative accuracy on the small entries as well
    assert (np.abs(P - Q) / Q).max() <= 1e-8


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def families():
    r = rng(5)
    return {
        "n01": r.standard_normal((3000, 4, 4)),
        "sigma10": 10.0 * r.standard_normal((3000, 4, 4)),
        "large_magnitude": large_mag(3000, 2),
    }


@pytest.mark.parametrize("name", ["n01", "sigma10", "large_magnitude"])
def test_marginals_positivity_and_form(name):
    X = families()[name]
    P, b, it, nonconv = oracle.newton64(X)
    assert nonconv == 0
    assert oracle.marginal_residual(P).max() <= 1e-13
    assert (P > 0).all()
    # log P - X = a_i + b_j: its double-centred part vanishes
    D = np.log(P) - X
    Dc = D - D.mean(axis=2, keepdims=True) - D.mean(axis=1, keepdims=True) \
        + D.mean(axis=(1, 2), keepdims=True)
    assert np.abs(Dc).max() <= 1e-9 * max(1.0, np.abs(X).max() / 10)
    # gauge of the returned dual and consistency P = rowsoftmax(X + b)
    assert (b[:, 3] == 0).all()
    z = X + b[:, None, :]
    e = np.exp(z - z.max(axis=2, keepdims=True))
    assert np.abs(e / e.sum(axis=2, keepdims=True) - P).max() <= 1e-12


@pytest.mark.parametrize("name", ["n01", "sigma10", "large_magnitude"])
def test_permutation_and_transpose_equivariance(name):
    X = families()[name][:500]
    r = rng(7)
    P = oracle.newton64(X)[0]
    rows = np.array([r.permutation(4) for _ in range(len(X))])
    cols = np.array([r.permutation(4) for _ in range(len(X))])
    t = np.arange(len(X))[:, None, None]
    Xp = X[t, rows[:, :, None], cols[:, None, :]]
    Pp = oracle.newton64(Xp)[0]
    assert np.abs(Pp - P[t, rows[:, :, None], cols[:, None, :]]).max() <= 1e-12
    PT = oracle.newton64(np.swapaxes(X, 1, 2))[0]
    assert np.abs(PT - np.swapaxes(P, 1, 2)).max() <= 1e-12


def test_offset_invariance():
    r = rng(8)
    X = r.standard_normal((1000, 4, 4)) * 3
    u = r.uniform(-40, 40, (1000, 4, 1))
    v = r.uniform(-40, 40, (1000, 1, 4))
    P = oracle.newton64(X)[0]
    P2 = oracle.newton64(X + u + v)[0]
    assert np.abs(P - P2).max() <= 1e-12


# --------------------------------------------------------------------------
# two solvers
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["n01", "sigma10", "large_magnitude"])
def test_sinkhorn_and_newton_agree(name):
    X = families()[name][:400]
    Pn = oracle.newton64(X)[0]
    Ps, bs, its, nonconv = oracle.sinkhorn64(X, tol=1e-13, max_iters=20000)
    conv = its < 20000
    assert conv.sum() >= 100  # enough converged tokens to compare
    assert np.abs(Ps[conv] - Pn[conv]).max() <= 1e-12
    # where Sinkhorn-Knopp is capped it is still on its way to the same P
    if (~conv).any():
        assert oracle.marginal_residual(Ps[~conv]).max() < 1e-3


def test_newton_converges_quadratically():
    X = rng(9).standard_normal((300, 4, 4))
    P, b, it, nonconv, tr = oracle.newton64(X, tol=1e-15, trace_len=30)
    checked = 0
    for t in range(len(X)):
        r = tr[t][~np.isnan(tr[t])]
        for k in range(len(r) - 1):
            if 1e-12 < r[k + 1] and r[k] < 1e-2:
                # e_{k+1} <= C e_k^2 in the local regime
                assert r[k + 1] <= 50.0 * r[k] ** 2
                checked += 1
    assert checked > 100
    assert it.max() <= 10  # "very few iterations" at N(0,1)


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------
def test_backward_matches_finite_differences():
    r = rng(10)
    X = np.concatenate([r.standard_normal((40, 4, 4)), 4.0 * r.standard_normal((20, 4, 4))])
    G = r.standard_normal(X.shape)
    P = oracle.newton64(X)[0]
    dX = oracle.backward64(P, G)
    fd = oracle.fd_backward64(X, G, h=1e-3)
    scale = np.abs(G).max()
    assert np.abs(dX - fd).max() <= 1e-9 * scale


def test_backward_matches_unrolled_sinkhorn_autodiff():
    r = rng(12)
    X = r.standard_normal((64, 4, 4))
    G = r.standard_normal(X.shape)
    P = oracle.newton64(X)[0]
    dX = oracle.backward64(P, G)
    Pu, dXu = oracle.unrolled_sinkhorn_backward64(X, G, iters=400)
    assert np.abs(Pu - P).max() <= 1e-13
    assert np.abs(dXu - dX).max() <= 1e-11


@pytest.mark.parametrize("name,tol", [("n01", 1e-12), ("large_magnitude", 1e-7)])
def test_backward_structure(name, tol):
    """tol: float64 rounding amplified by the conditioning of the dual Hessian.
    On nearly one-hot tokens of the large-magnitude family the dual potentials
    reach ~1e8, so solving for them in float64 leaves residuals ~1e-8 (the
    60-digit comparison below bounds the same effect)."""
    r = rng(13)
    X = r.standard_normal((1000, 4, 4)) if name == "n01" else large_mag(1000, 2)
    G = r.standard_normal(X.shape)
    P = oracle.newton64(X)[0]
    dX = oracle.backward64(P, G)
    g = np.abs(G).max()
    # the projection is invariant to row/column offsets of X: dX has zero
    # row and column sums
    assert np.abs(dX.sum(axis=1)).max() <= tol * g
    assert np.abs(dX.sum(axis=2)).max() <= tol * g
    # and an upstream gradient of the form u_i + v_j changes nothing (the
    # marginals are fixed), so dX = 0
    U = r.standard_normal((len(X), 4, 1)) + r.standard_normal((len(X), 1, 4))
    assert np.abs(oracle.backward64(P, U)).max() <= tol * 100
    # the Jacobian is positive semidefinite (Hessian of a convex function)
    assert (np.einsum("tij,tij->t", G, dX) >= -tol).all()


def test_backward_against_60_digit_arithmetic():
    """The float64 backward against the same formula evaluated with 60
    significant digits (mpmath), on the same P rescaled to unit row sums."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60

    def exact(P, G):
        p = [[mpmath.mpf(float(v)) for v in row] for row in P]
        p = [[v / sum(row) for v in row] for row in p]
        g = [[mpmath.mpf(float(v)) for v in row] for row in G]
        r = [sum(p[k][j] * g[k][j] for j in range(4)) for k in range(4)]
        v = [sum(p[k][l] * (g[k][l] - r[k]) for k in range(4)) for l in range(3)]
        H = mpmath.matrix(3, 3)
        for j in range(3):
            for k in range(3):
                H[j, k] = (sum(p[i][j] * (1 - p[i][j]) for i in range(4)) if j == k
                           else -sum(p[i][j] * p[i][k] for i in range(4)))
        lam = list(mpmath.lu_solve(H, mpmath.matrix(v))) + [mpmath.mpf(0)]
        out = np.zeros((4, 4))
        for k in range(4):
            s = sum(lam[l] * p[k][l] for l in range(4))
            for q in range(4):
                out[k, q] = float(p[k][q] * (g[k][q] - r[k] - lam[q] + s))
        return out

    r = rng(19)
    for X, tol in ((r.standard_normal((60, 4, 4)), 1e-14), (large_mag(200, 2), 1e-8)):
        G = r.standard_normal(X.shape)
        P = oracle.newton64(X)[0]
        dX = oracle.backward64(P, G)
        err = max(np.abs(exact(P[t], G[t]) - dX[t]).max() for t in range(len(X)))
        assert err <= tol


def test_backward_is_symmetric_jacobian():
    """P(X) is the gradient of a convex function of X, so the VJP with G equals
    the directional derivative of P along G."""
    r = rng(14)
    X = np.concatenate([r.standard_normal((200, 4, 4)), 5.0 * r.standard_normal((100, 4, 4))])
    G = r.standard_normal(X.shape)
    P = oracle.newton64(X)[0]
    dX = oracle.backward64(P, G)
    h = 1e-4
    jvp1 = (oracle.newton64(X + h * G, tol=1e-15)[0] - oracle.newton64(X - h * G, tol=1e-15)[0]) / (2 * h)
    h2 = h / 2
    jvp2 = (oracle.newton64(X + h2 * G, tol=1e-15)[0] - oracle.newton64(X - h2 * G, tol=1e-15)[0]) / (2 * h2)
    jvp = (4 * jvp2 - jvp1) / 3
    assert np.abs(jvp - dX).max() <= 1e-8


# --------------------------------------------------------------------------
# fixed-iteration Sinkhorn-Knopp
# --------------------------------------------------------------------------
def test_sinkhorn_fixed_one_iteration_definition():
    """One iteration = row normalisation then column normalisation; the output
    is the column-normalised row softmax."""
    X = rng(15).standard_normal((300, 4, 4)) * 2
    P1 = oracle.sinkhorn_fixed64(X, 1)
    e = np.exp(X - X.max(axis=2, keepdims=True))
    rs = e / e.sum(axis=2, keepdims=True)
    want = rs / rs.sum(axis=1, keepdims=True)
    assert np.abs(P1 - want).max() <= 1e-14
    assert np.abs(oracle.sinkhorn_fixed64(X, 0) - np.exp(X)).max() <= 1e-12


def test_sinkhorn20_accuracy_claim():
    """The pages: with N(0,1) inputs every method is reasonable; with
    N(0,10^2) inputs fixed-iteration Sinkhorn has far larger median error."""
    r = rng(16)
    for sigma, lo, hi in ((1.0, 0.0, 1e-6), (10.0, 1e-3, 1.0)):
        X = sigma * r.standard_normal((2000, 4, 4))
        P = oracle.newton64(X)[0]
        P20 = oracle.sinkhorn_fixed64(X, 20)
        err = np.abs(P20 - P).reshape(len(X), -1).max(axis=1)
        assert lo <= np.median(err) <= hi


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------
def test_empty_and_nonfinite():
    P, b, it, n = oracle.newton64(np.zeros((0, 4, 4)))
    assert P.shape == (0, 4, 4) and n == 0
    X = rng(17).standard_normal((3, 4, 4))
    X[1, 2, 3] = np.nan
    P = oracle.newton64(X)[0]
    assert np.isnan(P[1]).all()
    assert np.isfinite(P[[0, 2]]).all()
    X[1, 2, 3] = np.inf
    assert np.isnan(oracle.newton64(X)[0][1]).all()
    assert np.isnan(oracle.sinkhorn64(X)[0][1]).all()


# --------------------------------------------------------------------------
# planted mistakes fail the pins (mutations are applied on the CPU, to the
# oracle's outputs or inputs, never to the GPU path)
# --------------------------------------------------------------------------
def test_planted_mistakes_are_caught():
    r = rng(18)
    X = r.standard_normal((30, 4, 4)) * 2
    G = r.standard_normal(X.shape)
    P = oracle.newton64(X)[0]
    fd = oracle.fd_backward64(X, G, h=1e-3)
    good = oracle.backward64(P, G)
    assert np.abs(good - fd).max() <= 1e-9 * np.abs(G).max()
    # transposed operand: P^T in place of P
    bad = np.swapaxes(oracle.backward64(np.swapaxes(P, 1, 2), G), 1, 2)
    assert np.abs(bad - fd).max() > 1e-3
    bad = oracle.backward64(np.swapaxes(P, 1, 2), G)
    assert np.abs(bad - fd).max() > 1e-3
    # dropped implicit term: only the explicit part p (G - r)
    r_ = (G * P).sum(axis=2, keepdims=True)
    bad = P * (G - r_)
    assert np.abs(bad - fd).max() > 1e-3
    # wrong sign of the implicit term
    bad = 2 * bad - good
    assert np.abs(bad - fd).max() > 1e-3
    # forward: one Sinkhorn step is not the projection (marginal pin)
    assert oracle.marginal_residual(oracle.sinkhorn_fixed64(X, 1)).max() > 1e-3
    # forward: a row softmax with the wrong sign of the dual fails the form pin
    Pn, b, _, _ = oracle.newton64(X)
    z = X - b[:, None, :]
    e = np.exp(z - z.max(axis=2, keepdims=True))
    assert np.abs(e / e.sum(axis=2, keepdims=True) - Pn).max() > 1e-3


# --------------------------------------------------------------------------
# the Hessian solve exported by the oracle ("Accelerating the Birkhoff
# Projection for Manifold-Constrained Hyper-Connections", s2.1: the 3x3 system
# of the reduced dual), against an LU solve of the explicitly assembled matrix
# --------------------------------------------------------------------------
EDGES = [(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)]


def grounded_laplacian(w):
    """3x3 matrix of the Laplacian with edge weights w (node 3 grounded):
    H_jj = sum of the weights of the edges at j, H_jk = -w_jk."""
    H = np.zeros((len(w), 4, 4))
    for e, (a, b) in enumerate(EDGES):
        H[:, a, b] -= w[:, e]
        H[:, b, a] -= w[:, e]
        H[:, a, a] += w[:, e]
        H[:, b, b] += w[:, e]
    return H[:, :3, :3]


def test_laplacian_solve_matches_lu_solve():
    r = rng(19)
    n = 4000
    # weights over many decades (nearly disconnected graphs included)
    w = 10.0 ** r.uniform(-6, 1, (n, 6))
    rhs = r.standard_normal((n, 3))
    x = oracle.laplacian_solve64(w, rhs)
    H = grounded_laplacian(w)
    want = np.linalg.solve(H, rhs[..., None])[..., 0]
    cond = np.linalg.cond(H)
    err = np.abs(x - want).max(1) / np.abs(want).max(1)
    assert np.all(err <= 1e-13 * cond)
    # the residual of the oracle's own solution, in the assembled matrix
    res = np.abs(np.einsum("tjk,tk->tj", H, x) - rhs).max(1)
    assert np.all(res <= 1e-12 * (np.abs(H).max((1, 2)) * np.abs(x).max(1) + np.abs(rhs).max(1)))
    # the Hessian of a token: H = diag(colsum P) - P^T P on columns 0..2,
    # whose edge weights are w_jk = sum_i p_ij p_ik (rows of P sum to one)
    X = r.standard_normal((200, 4, 4))
    P = oracle.newton64(X)[0]
    wp = np.stack([(P[:, :, a] * P[:, :, b]).sum(1) for a, b in EDGES], 1)
    Hp = (np.eye(4)[None] * P.sum(1)[:, None, :] - np.einsum("tij,tik->tjk", P, P))[:, :3, :3]
    g = r.standard_normal((200, 3))
    assert np.abs(oracle.laplacian_solve64(wp, g) - np.linalg.solve(Hp, g[..., None])[..., 0]).max() <= 1e-11
    # a disconnected graph (all weights zero) has no solution: NaN, counted
    z = oracle.laplacian_solve64(np.zeros((1, 6)), np.ones((1, 3)))
    assert np.isnan(z).all()


def test_laplacian_solve_planted_mistake():
    """A transposed edge order (the (0,3) and (1,2) weights exchanged)
    fails the LU pin."""
    r = rng(20)
    w = 10.0 ** r.uniform(-2, 1, (500, 6))
    rhs = r.standard_normal((500, 3))
    want = np.linalg.solve(grounded_laplacian(w), rhs[..., None])[..., 0]
    bad = oracle.laplacian_solve64(w[:, [0, 1, 3, 2, 4, 5]], rhs)
    assert np.abs(bad - want).max() > 1e-3
