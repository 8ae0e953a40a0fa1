"""Pins for the float64 entropic-OT oracle (oracle/eot.py), CPU only.

The streaming EOT update ("FlashSinkhorn: IO-Aware Entropic OT on GPU",
Methodik, s1) is checked against facts that do not come from the oracle's own
formula:
  * n = m with uniform weights: the converged plan times n is the Birkhoff
    projection of -C/eps, computed by the separately written n x n Newton
    oracle (C code);
  * the 2 x 2 uniform case in closed form;
  * strong duality at convergence: <f, a> + <g, b> equals the primal
    objective <C, P> + eps KL(P | a b^T) of the plan built from f and g;
  * the eps -> infinity limit (with g = 0, f_i tends to the b-weighted mean
    cost sum_j b_j C_ij) and the eps -> 0 limit (f_i tends to
    min_j (C_ij - g_j), the c-transform), each within its asymptotic error
    bound;
  * invariances: a common translation of both clouds, the scaling
    (c X, c Y, c^2 eps) -> (c^2 f, c^2 g), permutations;
  * the cost against a brute-force double loop on a tiny case;
  * marginals at convergence with non-uniform weights;
  * planted mistakes (a sign of g, the weights dropped, the cost unsquared,
    eps misplaced) each fail at least one pin.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import eot

R = np.random.default_rng


def clouds(n, m, d, seed, shift=0.5):
    r = R(seed)
    X = r.standard_normal((n, d)) / math.sqrt(d)
    Y = r.standard_normal((m, d)) / math.sqrt(d)
    Y[:, 0] += shift
    return X, Y


def uniform(n):
    return np.full(n, -math.log(n))


def test_cost_matches_double_loop():
    X, Y = clouds(3, 4, 5, seed=0)
    C = eot.sqeuclid_cost64(X, Y)
    for i in range(3):
        for j in range(4):
            s = 0.0
            for k in range(5):
                s += (X[i, k] - Y[j, k]) ** 2
            assert C[i, j] == pytest.approx(s, rel=1e-15, abs=1e-15)


@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_uniform_square_case_is_birkhoff_projection(n):
    X, Y = clouds(n, n, 3, seed=n)
    eps = 1.0
    f, g = eot.sinkhorn64(X, Y, uniform(n), uniform(n), eps, iters=3000)
    P = eot.plan64(X, Y, f, g, uniform(n), uniform(n), eps)
    B = oracle.newton64_n(-eot.sqeuclid_cost64(X, Y)[None] / eps)[0][0]
    assert np.abs(n * P - B).max() <= 1e-11


def test_two_by_two_closed_form():
    X, Y = clouds(2, 2, 4, seed=1)
    eps = 0.2
    f, g = eot.sinkhorn64(X, Y, uniform(2), uniform(2), eps, iters=4000)
    P = eot.plan64(X, Y, f, g, uniform(2), uniform(2), eps)
    C = eot.sqeuclid_cost64(X, Y)
    q = 1.0 / (1.0 + math.exp(-(C[0, 1] + C[1, 0] - C[0, 0] - C[1, 1]) / (2 * eps)))
    want = 0.5 * np.array([[q, 1 - q], [1 - q, q]])
    assert np.abs(P - want).max() <= 1e-13


@pytest.mark.parametrize("n,m,d,eps", [(40, 60, 3, 0.1), (25, 17, 16, 0.5), (30, 30, 2, 0.05)])
def test_strong_duality_and_marginals(n, m, d, eps):
    X, Y = clouds(n, m, d, seed=n + m)
    r = R(7)
    a = r.uniform(0.2, 1.0, n)
    a /= a.sum()
    b = r.uniform(0.2, 1.0, m)
    b /= b.sum()
    la, lb = np.log(a), np.log(b)
    f, g = eot.sinkhorn64(X, Y, la, lb, eps, iters=20000)
    P = eot.plan64(X, Y, f, g, la, lb, eps)
    assert np.abs(P.sum(1) - a).max() <= 1e-12
    assert np.abs(P.sum(0) - b).max() <= 1e-14
    dual = float(f @ a + g @ b)
    assert dual == pytest.approx(eot.primal_cost64(X, Y, P, la, lb, eps), rel=1e-10, abs=1e-12)


def test_large_eps_limit_is_mean_cost():
    X, Y = clouds(20, 30, 4, seed=3)
    r = R(4)
    b = r.uniform(0.5, 1.0, 30)
    b /= b.sum()
    eps = 1e6
    C = eot.sqeuclid_cost64(X, Y)
    f = eot.f_update64(X, Y, np.zeros(30), np.log(b), eps)
    mean = C @ b
    # -eps log E_b exp(-C/eps) = E_b C - Var_b(C)/(2 eps) + O(eps^-2)
    assert np.abs(f - mean).max() <= (C.max() ** 2) / eps
    assert np.abs(f - mean).max() > 0.0


def test_small_eps_limit_is_c_transform():
    X, Y = clouds(25, 35, 3, seed=5)
    g = R(6).standard_normal(35) * 0.1
    lb = uniform(35)
    eps = 1e-4
    f = eot.f_update64(X, Y, g, lb, eps)
    ct = (eot.sqeuclid_cost64(X, Y) - g[None, :]).min(1)
    # with uniform b, f_i = ct_i + eps log m - eps log(sum_j exp(-(C_ij - g_j - ct_i)/eps)),
    # and that sum lies in [1, m], so f_i is in [ct_i, ct_i + eps log m]
    assert np.all(f - ct <= eps * math.log(35) + 1e-12)
    assert np.all(f - ct >= -1e-12)


def test_single_target_point():
    X, Y = clouds(10, 1, 6, seed=8)
    g = np.array([0.37])
    f = eot.f_update64(X, Y, g, np.array([0.0]), 0.25)
    assert np.allclose(f, eot.sqeuclid_cost64(X, Y)[:, 0] - 0.37, rtol=0, atol=1e-15)


def test_translation_scaling_permutation():
    X, Y = clouds(30, 20, 5, seed=9)
    la, lb = uniform(30), uniform(20)
    f, g = eot.sinkhorn64(X, Y, la, lb, 0.2, iters=50)
    t = R(10).standard_normal(5) * 3
    f2, g2 = eot.sinkhorn64(X + t, Y + t, la, lb, 0.2, iters=50)
    assert np.abs(f2 - f).max() <= 1e-11 and np.abs(g2 - g).max() <= 1e-11
    c = 1.7
    f3, g3 = eot.sinkhorn64(c * X, c * Y, la, lb, 0.2 * c * c, iters=50)
    assert np.abs(f3 - c * c * f).max() <= 1e-11 and np.abs(g3 - c * c * g).max() <= 1e-11
    pi, pj = R(11).permutation(30), R(12).permutation(20)
    f4, g4 = eot.sinkhorn64(X[pi], Y[pj], la, lb, 0.2, iters=50)
    assert np.abs(f4 - f[pi]).max() <= 1e-12 and np.abs(g4 - g[pj]).max() <= 1e-12


def _pins_hold(update):
    """The duality / limit pins evaluated with a replacement f update."""
    X, Y = clouds(12, 12, 3, seed=13)
    eps = 1.0
    la = lb = uniform(12)
    g = np.zeros(12)
    C = eot.sqeuclid_cost64(X, Y)
    for _ in range(3000):
        f = update(X, Y, g, lb, eps)
        g = update(Y, X, f, la, eps)
    P = eot.plan64(X, Y, f, g, la, lb, eps)
    B = oracle.newton64_n(-C[None] / eps)[0][0]
    ok_birkhoff = np.abs(12 * P - B).max() <= 1e-9
    gb = R(14).standard_normal(12) * 0.1
    ok_ctransform = np.all(np.abs(update(X, Y, gb, lb, 1e-4) - (C - gb).min(1)) <= 1e-3)
    return ok_birkhoff and ok_ctransform


def test_planted_mistakes_fail():
    assert _pins_hold(eot.f_update64)

    def sign_of_g(X, Y, g, lb, eps):
        C = eot.sqeuclid_cost64(X, Y)
        return -eps * eot.lse64((-g[None, :] - C) / eps + lb[None, :], axis=1)

    def weights_dropped(X, Y, g, lb, eps):
        return eot.f_update64(X, Y, g, np.zeros_like(lb), eps)

    def unsquared(X, Y, g, lb, eps):
        C = np.sqrt(eot.sqeuclid_cost64(X, Y))
        return -eps * eot.lse64((g[None, :] - C) / eps + lb[None, :], axis=1)

    def eps_misplaced(X, Y, g, lb, eps):
        C = eot.sqeuclid_cost64(X, Y)
        return -eot.lse64((g[None, :] - C) / eps + lb[None, :], axis=1)

    for bad in (sign_of_g, weights_dropped, unsquared, eps_misplaced):
        assert not _pins_hold(bad), bad.__name__


def test_gradient_matches_finite_differences_of_the_cost():
    """grad_x64 (a formula in pi) against central differences of the
    converged dual value, which is computed without it."""
    X, Y = clouds(5, 7, 2, seed=21)
    r = R(22)
    la = np.log(r.uniform(0.3, 1.0, 5))
    la -= np.log(np.exp(la).sum())
    lb = uniform(7)
    eps, iters, h = 0.5, 4000, 1e-5
    f, g = eot.sinkhorn64(X, Y, la, lb, eps, iters)
    G = eot.grad_x64(X, Y, f, g, la, lb, eps)
    fd = np.zeros_like(X)
    for i in range(X.shape[0]):
        for k in range(X.shape[1]):
            Xp, Xm = X.copy(), X.copy()
            Xp[i, k] += h
            Xm[i, k] -= h
            fd[i, k] = (eot.eot_cost64(Xp, Y, la, lb, eps, iters)
                        - eot.eot_cost64(Xm, Y, la, lb, eps, iters)) / (2 * h)
    assert np.abs(G - fd).max() <= 1e-8


def test_transport_masses_and_single_target():
    X, Y = clouds(30, 40, 3, seed=23)
    la, lb = uniform(30), uniform(40)
    f, g = eot.sinkhorn64(X, Y, la, lb, 0.3, iters=5000)
    PY, r = eot.transport64(X, Y, f, g, la, lb, 0.3)
    assert np.abs(r - np.exp(la)).max() <= 1e-13
    # the barycentric map of a single target point is that point
    Y1 = Y[:1]
    f1, g1 = eot.sinkhorn64(X, Y1, la, np.zeros(1), 0.3, iters=3)
    PY1, r1 = eot.transport64(X, Y1, f1, g1, la, np.zeros(1), 0.3)
    assert np.abs(PY1 / r1[:, None] - Y1).max() <= 1e-14
    # translating both clouds translates the barycentric map
    t = np.array([0.3, -1.2, 2.0])
    f2, g2 = eot.sinkhorn64(X + t, Y + t, la, lb, 0.3, iters=5000)
    PY2, r2 = eot.transport64(X + t, Y + t, f2, g2, la, lb, 0.3)
    assert np.abs(PY2 / r2[:, None] - (PY / r[:, None] + t)).max() <= 1e-10


def test_planted_transport_mistake_fails():
    """A gradient with the sign of (pi Y) flipped fails the FD pin."""
    X, Y = clouds(4, 5, 2, seed=24)
    la, lb = uniform(4), uniform(5)
    f, g = eot.sinkhorn64(X, Y, la, lb, 0.5, 4000)
    PY, r = eot.transport64(X, Y, f, g, la, lb, 0.5)
    bad = 2.0 * (r[:, None] * X + PY)
    h = 1e-5
    Xp = X.copy()
    Xp[0, 0] += h
    Xm = X.copy()
    Xm[0, 0] -= h
    fd = (eot.eot_cost64(Xp, Y, la, lb, 0.5, 4000) - eot.eot_cost64(Xm, Y, la, lb, 0.5, 4000)) / (2 * h)
    assert abs(bad[0, 0] - fd) > 1e-3
    assert abs(eot.grad_x64(X, Y, f, g, la, lb, 0.5)[0, 0] - fd) <= 1e-8


def test_apply_plan_is_linear_and_matches_transport():
    X, Y = clouds(9, 11, 3, seed=25)
    la, lb = uniform(9), uniform(11)
    f, g = eot.sinkhorn64(X, Y, la, lb, 0.4, iters=200)
    PY, r = eot.transport64(X, Y, f, g, la, lb, 0.4)
    PV, r2 = eot.apply_plan64(X, Y, f, g, la, lb, 0.4, Y)
    assert np.array_equal(PV, PY) and np.array_equal(r, r2)
    ones, _ = eot.apply_plan64(X, Y, f, g, la, lb, 0.4, np.ones((11, 1)))
    assert np.abs(ones[:, 0] - r).max() <= 1e-15


def test_hvp_matches_finite_differences_of_the_gradient():
    """hvp64 (dense implicit differentiation) against central differences of
    the gradient at re-converged potentials, which use no Hessian formula."""
    X, Y = clouds(6, 7, 2, seed=31)
    la, lb = uniform(6), uniform(7)
    eps, iters, h = 0.5, 4000, 1e-5
    V = R(32).standard_normal(X.shape)
    f, g = eot.sinkhorn64(X, Y, la, lb, eps, iters)
    Hv = eot.hvp64(X, Y, f, g, la, lb, eps, V)

    def grad(Xs):
        fs, gs = eot.sinkhorn64(Xs, Y, la, lb, eps, iters)
        return eot.grad_x64(Xs, Y, fs, gs, la, lb, eps)

    fd = (grad(X + h * V) - grad(X - h * V)) / (2 * h)
    assert np.abs(Hv - fd).max() <= 1e-6 * max(1.0, np.abs(fd).max())


def test_hvp_along_a_common_translation_sums_to_2t():
    """Moving every x_i by t changes sum_i grad_i = 2 (sum_i a_i x_i - sum_j b_j y_j)
    by 2 t (total mass 1), so sum_i (H v)_i = 2 t for v_i = t."""
    X, Y = clouds(9, 12, 3, seed=33)
    r = R(34)
    la = np.log(r.uniform(0.3, 1.0, 9))
    la -= np.log(np.exp(la).sum())
    lb = uniform(12)
    f, g = eot.sinkhorn64(X, Y, la, lb, 0.3, 5000)
    t = np.array([0.7, -1.1, 0.25])
    Hv = eot.hvp64(X, Y, f, g, la, lb, 0.3, np.tile(t, (9, 1)))
    assert np.abs(Hv.sum(0) - 2 * t).max() <= 1e-9


def test_planted_hvp_cost_sign_mistake_fails():
    """dC_ij built from (x_i + y_j).v_i instead of (x_i - y_j).v_i, carried
    through the whole implicit solve, breaks the finite-difference pin."""
    X, Y = clouds(5, 6, 2, seed=37)
    la, lb = uniform(5), uniform(6)
    eps, iters, h = 0.5, 4000, 1e-5
    V = R(38).standard_normal(X.shape)
    f, g = eot.sinkhorn64(X, Y, la, lb, eps, iters)
    a, b = np.exp(la), np.exp(lb)
    P = eot.plan64(X, Y, f, g, la, lb, eps)
    dC = 2.0 * ((X * V).sum(1)[:, None] + V @ Y.T)  # the planted sign
    A = np.block([[np.diag(a), P], [P.T, np.diag(b)]])
    sol = np.linalg.lstsq(A, np.r_[(P * dC).sum(1), (P * dC).sum(0)], rcond=None)[0]
    dP = P * (sol[:5][:, None] + sol[5:][None, :] - dC) / eps
    bad = 2.0 * a[:, None] * V - 2.0 * dP @ Y

    def grad(Xs):
        fs, gs = eot.sinkhorn64(Xs, Y, la, lb, eps, iters)
        return eot.grad_x64(Xs, Y, fs, gs, la, lb, eps)

    fd = (grad(X + h * V) - grad(X - h * V)) / (2 * h)
    assert np.abs(bad - fd).max() > 1e-2


def test_planted_hvp_mistake_fails():
    """Dropping the implicit (df, dg) term breaks the finite-difference pin."""
    X, Y = clouds(5, 6, 2, seed=35)
    la, lb = uniform(5), uniform(6)
    eps, iters, h = 0.5, 4000, 1e-5
    V = R(36).standard_normal(X.shape)
    f, g = eot.sinkhorn64(X, Y, la, lb, eps, iters)
    P = eot.plan64(X, Y, f, g, la, lb, eps)
    dC = 2.0 * ((X * V).sum(1)[:, None] - V @ Y.T)
    bad = 2.0 * np.exp(la)[:, None] * V - 2.0 * (P * -dC / eps) @ Y

    def grad(Xs):
        fs, gs = eot.sinkhorn64(Xs, Y, la, lb, eps, iters)
        return eot.grad_x64(Xs, Y, fs, gs, la, lb, eps)

    fd = (grad(X + h * V) - grad(X - h * V)) / (2 * h)
    assert np.abs(bad - fd).max() > 1e-2
