"""Pins for the general n x n oracle functions (CPU only).

The n x n projection reduces the dual to n-1 free variables ("Accelerating
the Birkhoff Projection for Manifold-Constrained Hyper-Connections", s2.1:
m-1 free variables for m columns).  The general-n oracle is checked against
the separately written 4 x 4 oracle at n = 4, against closed forms (X = cI,
X = u 1^T + 1 v^T, circulants, and the whole 2 x 2 case), against the
fixed-point family, against invariants, against Sinkhorn-Knopp, and its
backward against finite differences; a planted mistake fails.
"""
import numpy as np
import pytest

import oracle
from birkhoff_projection_gb300 import workloads

NS = [2, 3, 5, 6, 7, 8]


def rng(seed):
    return np.random.default_rng(seed)


def test_agrees_with_4x4_oracle():
    r = rng(0)
    X = np.concatenate([r.standard_normal((500, 4, 4)), 10 * r.standard_normal((500, 4, 4))])
    G = r.standard_normal(X.shape)
    P4 = oracle.newton64(X)[0]
    Pn = oracle.newton64_n(X)[0]
    assert np.abs(P4 - Pn).max() <= 1e-12
    assert np.abs(oracle.backward64(P4, G) - oracle.backward64_n(P4, G)).max() <= 1e-9


@pytest.mark.parametrize("n", NS)
def test_closed_forms(n):
    for c in (-3.0, 0.5, 4.0):
        P = oracle.newton64_n((c * np.eye(n))[None])[0][0]
        diag = 1.0 / (1.0 + (n - 1) * np.exp(-c))
        off = 1.0 / (np.exp(c) + n - 1)
        assert np.allclose(P, np.where(np.eye(n) > 0, diag, off), rtol=1e-12, atol=0)
    r = rng(n)
    u, v = r.standard_normal((50, n, 1)) * 5, r.standard_normal((50, 1, n)) * 5
    assert np.abs(oracle.newton64_n(u + v)[0] - 1.0 / n).max() <= 1e-13
    x = r.standard_normal((50, n)) * 2
    idx = (np.arange(n)[None, :] - np.arange(n)[:, None]) % n
    X = x[:, idx]
    e = np.exp(X - X.max(2, keepdims=True))
    assert np.abs(oracle.newton64_n(X)[0] - e / e.sum(2, keepdims=True)).max() <= 1e-13


def test_two_by_two_closed_form():
    """n = 2: P = [[q, 1-q], [1-q, q]] with q = sigmoid((x00 + x11 - x01 - x10)/2)
    (the cross ratio P00 P11 / (P01 P10) = exp(x00 + x11 - x01 - x10) is
    invariant under row and column scaling); the backward is
    dX = (G00 + G11 - G01 - G10) q (1 - q) / 2 * [[1, -1], [-1, 1]]."""
    r = rng(2)
    X = r.standard_normal((1000, 2, 2)) * 3
    G = r.standard_normal(X.shape)
    s = (X[:, 0, 0] + X[:, 1, 1] - X[:, 0, 1] - X[:, 1, 0]) / 2
    q = 1.0 / (1.0 + np.exp(-s))
    want = np.stack([np.stack([q, 1 - q], -1), np.stack([1 - q, q], -1)], 1)
    P = oracle.newton64_n(X)[0]
    assert np.abs(P - want).max() <= 1e-13
    gam = G[:, 0, 0] + G[:, 1, 1] - G[:, 0, 1] - G[:, 1, 0]
    k = gam * q * (1 - q) / 2
    dwant = k[:, None, None] * np.array([[1.0, -1.0], [-1.0, 1.0]])[None]
    assert np.abs(oracle.backward64_n(P, G) - dwant).max() <= 1e-12


@pytest.mark.parametrize("n", NS)
def test_fixed_point_family(n):
    X, Q = workloads.fixed_point_family_n(n, 500, seed=n)
    P = oracle.newton64_n(X.numpy())[0]
    assert np.abs(P - Q.numpy()).max() <= 1e-12


@pytest.mark.parametrize("n", NS)
def test_invariants_and_sinkhorn_agreement(n):
    r = rng(10 + n)
    X = r.standard_normal((400, n, n)) * 3
    P, b, it, nonconv = oracle.newton64_n(X)
    assert nonconv == 0
    assert oracle.marginal_residual(P).max() <= 1e-13
    assert (P > 0).all()
    D = np.log(P) - X
    Dc = D - D.mean(2, keepdims=True) - D.mean(1, keepdims=True) + D.mean((1, 2), keepdims=True)
    assert np.abs(Dc).max() <= 1e-9
    rows = np.array([r.permutation(n) for _ in range(len(X))])
    cols = np.array([r.permutation(n) for _ in range(len(X))])
    t = np.arange(len(X))[:, None, None]
    Pp = oracle.newton64_n(X[t, rows[:, :, None], cols[:, None, :]])[0]
    assert np.abs(Pp - P[t, rows[:, :, None], cols[:, None, :]]).max() <= 1e-12
    Ps, _, its, _ = oracle.sinkhorn64_n(X)
    conv = its < 20000
    assert conv.sum() >= 100
    assert np.abs(Ps[conv] - P[conv]).max() <= 1e-12


@pytest.mark.parametrize("n", [2, 3, 6])
def test_backward_matches_finite_differences(n):
    r = rng(20 + n)
    X = r.standard_normal((12, n, n)) * 2
    G = r.standard_normal(X.shape)
    P = oracle.newton64_n(X)[0]
    dX = oracle.backward64_n(P, G)
    fd = oracle.fd_backward64_n(X, G)
    assert np.abs(dX - fd).max() <= 1e-8 * np.abs(G).max()
    # planted mistake: dropping the implicit (dual) term fails the same pin
    # (a transposed P would not: every 2 x 2 doubly stochastic P is symmetric)
    bad = P * (G - (P * G).sum(2, keepdims=True))
    assert np.abs(bad - fd).max() > 1e-4
    # structural: zero row and column sums
    assert np.abs(dX.sum(1)).max() <= 1e-12 and np.abs(dX.sum(2)).max() <= 1e-12
