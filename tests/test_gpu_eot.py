"""GPU parity of the streaming entropic-OT kernels (eot_update, eot_sinkhorn)
against the float64 oracle (oracle/eot.py), through the C ABI.

Tolerance: a per-row bound derived from the kernel's arithmetic.  With
A_i = max_j sum_k |x_ik y_jk|, N_i = ||x_i||^2, B = max_j ||y_j||^2:
  * dot products: each coordinate rounded to TF32 (relative 2^-11, so 2^-10
    per product) for one pass, or represented as hi + lo to 2^-22 with the
    lo.lo product dropped (2^-20 per product) for the split form; fp32
    accumulation over d_pad terms (d_pad 2^-23);
  * squared norms in fp32 (d 2^-23 relative);
  * biases, the running maximum, ex2 / lg2 and the final combination in fp32
    (2^-21 relative to every magnitude involved, plus eps 2^-18);
the log-sum-exp is 1-Lipschitz in the max norm of its arguments, so the
error of f_i is at most the largest error of an argument in row i, and a
sequence of updates adds the bounds of its steps.  The tests assert twice
that bound.
"""
import math

import numpy as np
import pytest
import torch

from birkhoff_projection_gb300 import eot, workloads
from oracle import eot as oeot
from _helpers import rna_tf32

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def row_bound(X, Y, h, log_w, f_ref, eps, passes):
    """Per-row error bound of one update of the X side against keys Y."""
    X = np.asarray(X, np.float64)
    Y = np.asarray(Y, np.float64)
    d = X.shape[1]
    d_pad = -(-d // 32) * 32
    A = (np.abs(X) @ np.abs(Y).T).max(1)
    N = (X * X).sum(1)
    B = (Y * Y).sum(1).max()
    H = np.abs(h).max()
    W = eps * np.abs(log_w).max()
    u = 2.0 ** -10 if passes == 1 else 2.0 ** -20
    t = (2 * (u + d_pad * 2.0 ** -23) * A + d * 2.0 ** -23 * (N + B)
         + 2.0 ** -21 * (2 * A + H + B + W + np.abs(f_ref) + N) + eps * 2.0 ** -18)
    return 2.0 * t


CASES = [
    (1000, 1500, 64),
    (777, 300, 3),
    (300, 1000, 100),
    (1, 1, 1),
    (129, 257, 32),
    (20000, 300, 8),  # more row blocks than SMs
    (64, 3000, 520),  # d past one 512-wide span, ragged
    (1000, 5000, 64),  # few row blocks: the keys split into segments, partials merged
]


@pytest.mark.parametrize("passes", [eot.TF32, eot.TF32X3])
@pytest.mark.parametrize("nq,nk,d", CASES)
def test_update_parity(nq, nk, d, passes):
    X, Y, _, log_b = workloads.eot_clouds(nq, nk, d, seed=nq + nk + d, device=DEV, random_weights=True)
    gen = torch.Generator(device="cpu").manual_seed(d)
    h = (torch.randn(nk, generator=gen) * 0.3).to(DEV)
    eps = workloads.EOT_EPS
    f = eot.update(X, Y, h, log_b, eps, passes=passes)
    ref = oeot.f_update64(np64(X), np64(Y), np64(h), np64(log_b), eps)
    err = np.abs(np64(f) - ref)
    tol = row_bound(np64(X), np64(Y), np64(h), np64(log_b), ref, eps, passes)
    assert np.all(np.isfinite(np64(f)))
    assert np.all(err <= tol), (err.max(), tol[err.argmax()])


@pytest.mark.parametrize("passes", [eot.TF32, eot.TF32X3])
def test_split_form_is_near_fp32(passes):
    """The split form must be far more accurate than one TF32 pass."""
    X, Y, _, log_b = workloads.eot_clouds(1000, 1500, 256, seed=5, device=DEV)
    h = torch.zeros(1500, device=DEV)
    f = eot.update(X, Y, h, log_b, 0.1, passes=passes)
    ref = oeot.f_update64(np64(X), np64(Y), np64(h), np64(log_b), 0.1)
    err = np.abs(np64(f) - ref).max()
    assert err <= (2e-3 if passes == eot.TF32 else 2e-5)


@pytest.mark.parametrize("passes", [eot.TF32, eot.TF32X3])
def test_sinkhorn_parity(passes):
    n, m, d, K = 500, 700, 16, 5
    eps = 0.1
    X, Y, log_a, log_b = workloads.eot_clouds(n, m, d, seed=1, device=DEV, random_weights=True)
    f, g = eot.sinkhorn(X, Y, log_a, log_b, eps, K, passes=passes)
    fr, gr = oeot.sinkhorn64(np64(X), np64(Y), np64(log_a), np64(log_b), eps, K)
    mag = max(np.abs(fr).max(), np.abs(gr).max())
    tf = row_bound(np64(X), np64(Y), np.full(m, mag), np64(log_b), np.full(n, mag), eps, passes)
    tg = row_bound(np64(Y), np64(X), np.full(n, mag), np64(log_a), np.full(m, mag), eps, passes)
    total = 2 * K * max(tf.max(), tg.max())
    assert np.abs(np64(f) - fr).max() <= total
    assert np.abs(np64(g) - gr).max() <= total


def test_sinkhorn_warm_start_and_zero_iters():
    X, Y, log_a, log_b = workloads.eot_clouds(300, 400, 8, seed=2, device=DEV)
    f, g = eot.sinkhorn(X, Y, log_a, log_b, 0.1, 3)
    f2, g2 = eot.sinkhorn(X, Y, log_a, log_b, 0.1, 0, f=f.clone(), g=g.clone())
    assert torch.equal(f2, f) and torch.equal(g2, g)
    # 3 + 2 iterations from a warm start == 5 from cold, up to rounding
    fa, ga = eot.sinkhorn(X, Y, log_a, log_b, 0.1, 2, f=f.clone(), g=g.clone())
    fb, gb = eot.sinkhorn(X, Y, log_a, log_b, 0.1, 5)
    assert torch.allclose(fa, fb, atol=1e-5) and torch.allclose(ga, gb, atol=1e-5)


def test_converged_plan_marginals():
    n, m, d, eps = 600, 800, 4, 0.1
    X, Y, log_a, log_b = workloads.eot_clouds(n, m, d, seed=3, device=DEV, random_weights=True)
    f, g = eot.sinkhorn(X, Y, log_a, log_b, eps, 300, passes=eot.TF32X3)
    P = oeot.plan64(np64(X), np64(Y), np64(f), np64(g), np64(log_a), np64(log_b), eps)
    a, b = np.exp(np64(log_a)), np.exp(np64(log_b))
    # columns are exact after a g update up to the fp32 rounding of g / eps
    assert np.abs(P.sum(0) / b - 1).max() <= 2e-3
    assert np.abs(P.sum(1) / a - 1).max() <= 2e-2


def test_full_size_sampled_rows():
    """The benchmark's size (65536 x 65536 points, d = 512): sampled rows
    of one f update against the oracle evaluated row by row."""
    n = m = 65536
    d = 512
    X, Y, _, log_b = workloads.eot_clouds(n, m, d, seed=0, device=DEV)
    h = torch.zeros(m, device=DEV)
    for passes in (eot.TF32, eot.TF32X3):
        f = eot.update(X, Y, h, log_b, workloads.EOT_EPS, passes=passes)
        rows = np.r_[0, 1, 127, 128, 40000, n - 129, n - 1, np.random.default_rng(0).integers(0, n, 9)]
        Xs = np64(X[torch.as_tensor(rows, device=DEV)])
        Yn = np64(Y)
        ref = oeot.f_update64(Xs, Yn, np.zeros(m), np64(log_b), workloads.EOT_EPS)
        tol = row_bound(Xs, Yn, np.zeros(m), np64(log_b), ref, workloads.EOT_EPS, passes)
        assert np.all(np.abs(np64(f)[rows] - ref) <= tol)
        assert np.all(np.isfinite(np64(f)))


def transport_bounds(X, Y, f, g, log_a, log_b, eps):
    """Element bounds for (pi Y, pi 1) from one TF32 pass: each pi_ij is off
    by at most exp(e_i) - 1 relative, e_i the exponent error of row i (the
    update's per-row bound over eps, plus the ex2 approximation); the second
    product adds TF32 truncation of pi (2^-10) and rounding of y (2^-11) and
    fp32 accumulation over m_pad keys.  The tests assert twice the bound."""
    X = np.asarray(X, np.float64)
    Y = np.asarray(Y, np.float64)
    m_pad = -(-Y.shape[0] // 256) * 256
    fr = np.abs(f) + eps * np.abs(log_a)
    t = row_bound(X, Y, g, log_b, fr, eps, eot.TF32) / 2.0
    rel = np.expm1(t / eps + 2.0 ** -20)
    P = oeot.plan64(X, Y, f, g, log_a, log_b, eps)
    acc = m_pad * 2.0 ** -23
    b_py = (rel + 2.0 ** -10 + 2.0 ** -11 + acc)[:, None] * (P @ np.abs(Y))
    b_mass = (rel + acc) * P.sum(1)
    return 2.0 * b_py, 2.0 * b_mass


TRANSPORT_CASES = [
    (1000, 1500, 64),
    (300, 700, 3),
    (129, 257, 160),   # two value slices, ragged everything
    (1, 1, 1),
    (20000, 300, 8),   # more row blocks than SMs
    (40000, 200, 4),   # CTA runs spanning two or three row blocks: whole and split ones
    (300, 400, 520),   # five value slices
]


@pytest.mark.parametrize("n,m,d", TRANSPORT_CASES)
def test_transport_parity(n, m, d):
    eps = workloads.EOT_EPS
    X, Y, log_a, log_b = workloads.eot_clouds(n, m, d, seed=n + 3 * m + d, device=DEV,
                                              random_weights=True)
    f64, g64 = oeot.sinkhorn64(np64(X), np64(Y), np64(log_a), np64(log_b), eps, 30)
    f = torch.tensor(f64, dtype=torch.float32, device=DEV)
    g = torch.tensor(g64, dtype=torch.float32, device=DEV)
    PY, mass, grad = eot.transport(X, Y, f, g, log_a, log_b, eps, want_grad=True)
    args = (np64(X), np64(Y), np64(f), np64(g), np64(log_a), np64(log_b), eps)
    PYr, mr = oeot.transport64(*args)
    b_py, b_mass = transport_bounds(*args)
    assert np.all(np.isfinite(np64(PY))) and np.all(np.isfinite(np64(mass)))
    assert np.all(np.abs(np64(PY) - PYr) <= b_py)
    assert np.all(np.abs(np64(mass) - mr) <= b_mass)
    Gr = oeot.grad_x64(*args)
    b_g = 2.0 * (b_mass[:, None] * np.abs(np64(X)) + b_py) + 2.0 ** -20 * np.abs(Gr) + 1e-30
    assert np.all(np.abs(np64(grad) - Gr) <= 2.0 * b_g)


def test_transport_row_masses_at_consistent_potentials():
    """With f the (split-form) update of g, every row of pi sums to a_i: the
    GPU masses match the oracle's masses of the same potentials within the
    derived bound, and those are a to the split form's accuracy."""
    n, m, d, eps = 600, 800, 16, 0.1
    X, Y, log_a, log_b = workloads.eot_clouds(n, m, d, seed=11, device=DEV, random_weights=True)
    f, g = eot.sinkhorn(X, Y, log_a, log_b, eps, 50, passes=eot.TF32X3)
    f = eot.update(X, Y, g, log_b, eps, passes=eot.TF32X3)
    PY, mass = eot.transport(X, Y, f, g, log_a, log_b, eps)
    args = (np64(X), np64(Y), np64(f), np64(g), np64(log_a), np64(log_b), eps)
    _, mr = oeot.transport64(*args)
    _, b_mass = transport_bounds(*args)
    assert np.all(np.abs(np64(mass) - mr) <= b_mass)
    a = np.exp(np64(log_a))
    assert np.abs(mr / a - 1).max() <= 1e-3


@pytest.mark.parametrize("d", [64, 512])
def test_transport_full_size_sampled_rows(d):
    """65536 x 65536 points at the bench sizes (d = 64: one value slice of
    192-key f16 tiles; d = 512: two slices of 256-key tiles): sampled rows
    against the oracle's plan rows.  With 512 row blocks on 152 SMs the
    first 456 row blocks go whole to CTAs and the rest in stream-K runs;
    rows on both sides of that line are sampled.  At d = 64 a one-column
    plan product (CUDA cores) is checked on the same rows."""
    n = m = 65536
    eps = workloads.EOT_EPS
    X, Y, log_a, log_b = workloads.eot_clouds(n, m, d, seed=0, device=DEV)
    g = torch.zeros(m, device=DEV)
    f = eot.update(X, Y, g, log_b, eps)
    PY, mass = eot.transport(X, Y, f, g, log_a, log_b, eps)
    rows = np.r_[0, 127, 128, 30000, 58367, 58368, 60000, n - 1,
                 np.random.default_rng(1).integers(0, n, 5)]
    idx = torch.as_tensor(rows, device=DEV)
    args = (np64(X[idx]), np64(Y), np64(f[idx]), np64(g), np64(log_a[idx]), np64(log_b), eps)
    PYr, mr = oeot.transport64(*args)
    b_py, b_mass = transport_bounds(*args)
    assert np.all(np.abs(np64(PY)[rows] - PYr) <= b_py)
    assert np.all(np.abs(np64(mass)[rows] - mr) <= b_mass)
    if d == 64:
        V = torch.randn(m, 1, generator=torch.Generator().manual_seed(9)).to(DEV)
        out, _ = eot.apply_plan(X, Y, f, g, log_a, log_b, V, eps)
        ref, _ = oeot.apply_plan64(*args, np64(V))
        bound = _apply_bound(X[idx], Y, f[idx], g, log_a[idx], log_b, V, eps)
        assert np.all(np.abs(np64(out)[rows] - ref) <= bound)


@pytest.mark.parametrize("n,m,d,dv", [(700, 900, 16, 5), (300, 500, 64, 1), (257, 300, 8, 300)])
def test_apply_plan_parity(n, m, d, dv):
    """pi V for arbitrary values (an odd width, a single column, two
    256-wide slices) against the oracle, within the bound of the transport
    arithmetic with |V| in place of |Y|."""
    eps = workloads.EOT_EPS
    X, Y, log_a, log_b = workloads.eot_clouds(n, m, d, seed=n + m, device=DEV, random_weights=True)
    gen = torch.Generator(device="cpu").manual_seed(dv)
    V = torch.randn(m, dv, generator=gen).to(DEV)
    f64, g64 = oeot.sinkhorn64(np64(X), np64(Y), np64(log_a), np64(log_b), eps, 20)
    f = torch.tensor(f64, dtype=torch.float32, device=DEV)
    g = torch.tensor(g64, dtype=torch.float32, device=DEV)
    out, mass = eot.apply_plan(X, Y, f, g, log_a, log_b, V, eps)
    args = (np64(X), np64(Y), np64(f), np64(g), np64(log_a), np64(log_b), eps)
    ref, mr = oeot.apply_plan64(*args, np64(V))
    fr = np.abs(np64(f)) + eps * np.abs(np64(log_a))
    t = row_bound(np64(X), np64(Y), np64(g), np64(log_b), fr, eps, eot.TF32) / 2.0
    rel = np.expm1(t / eps + 2.0 ** -20)
    P = oeot.plan64(*args)
    m_pad = -(-m // 256) * 256
    bound = 2.0 * (rel + 2.0 ** -10 + 2.0 ** -11 + m_pad * 2.0 ** -23)[:, None] * (P @ np.abs(np64(V)))
    assert np.all(np.abs(np64(out) - ref) <= bound)
    assert np.all(np.abs(np64(mass) - mr) <= 2.0 * (rel + m_pad * 2.0 ** -23) * mr)
    if dv == 1:
        assert out.shape == (n, 1)


def _apply_bound(X, Y, f, g, log_a, log_b, V, eps):
    """Element bound of pi V from one TF32 score pass and 2^-10 + 2^-11
    operand rounding in the second product (what the f16 form also
    satisfies: 2^-11 for P and for the scaled V), fp32 accumulation."""
    args = (np64(X), np64(Y), np64(f), np64(g), np64(log_a), np64(log_b), eps)
    fr = np.abs(np64(f)) + eps * np.abs(np64(log_a))
    t = row_bound(np64(X), np64(Y), np64(g), np64(log_b), fr, eps, eot.TF32) / 2.0
    rel = np.expm1(t / eps + 2.0 ** -20)
    P = oeot.plan64(*args)
    m_pad = -(-Y.shape[0] // 256) * 256
    return 2.0 * (rel + 2.0 ** -10 + 2.0 ** -11 + m_pad * 2.0 ** -23)[:, None] * (P @ np.abs(np64(V)))


@pytest.mark.parametrize("vmag,dv", [(1e6, 40), (1e-6, 40), (1.0, 200)])
def test_apply_plan_f16_overflow_redo_and_value_scale(vmag, dv):
    """The f16 second product scales P by 2^15 / a_i and V by a power of
    two.  Potentials shifted by 4 eps make every row of pi sum to e^4 a_i,
    past that range: the TF32 redo must take over, within the same bound
    (192-key tiles for 40 value columns, 256-key tiles for 200).  Values
    of magnitude 1e6 and 1e-6 exercise the V scale both ways."""
    n, m, d, eps = 400, 500, 8, 0.1
    X, Y, log_a, log_b = workloads.eot_clouds(n, m, d, seed=31, device=DEV, random_weights=True)
    f64, g64 = oeot.sinkhorn64(np64(X), np64(Y), np64(log_a), np64(log_b), eps, 30)
    V = torch.randn(m, dv, generator=torch.Generator().manual_seed(7)).to(DEV) * vmag
    for shift in (0.0, 4.0 * eps):
        f = torch.tensor(f64 + shift, dtype=torch.float32, device=DEV)
        g = torch.tensor(g64, dtype=torch.float32, device=DEV)
        out, mass = eot.apply_plan(X, Y, f, g, log_a, log_b, V, eps)
        ref, mr = oeot.apply_plan64(np64(X), np64(Y), np64(f), np64(g), np64(log_a), np64(log_b),
                                    eps, np64(V))
        assert np.all(np.isfinite(np64(out)))
        assert np.all(np.abs(np64(out) - ref) <= _apply_bound(X, Y, f, g, log_a, log_b, V, eps))
        if shift > 0:
            assert mr.sum() > 50 * np.exp(np64(log_a)).sum()  # rows of pi well past a_i


def test_sinkhorn_iterations_capture_into_a_cuda_graph():
    """After one warm-up call (per-device set-up), eot_sinkhorn enqueues only
    kernels: a CUDA graph of 3 iterations, replayed twice, gives exactly
    the eager result of 6 iterations."""
    n, m, d = 3000, 2000, 32
    X, Y, log_a, log_b = workloads.eot_clouds(n, m, d, seed=12, device=DEV)
    ws = torch.empty(eot.workspace_bytes(n, m, d), dtype=torch.uint8, device=DEV)
    f = torch.zeros(n, device=DEV)
    g = torch.zeros(m, device=DEV)
    eot.sinkhorn(X, Y, log_a, log_b, 0.1, 1, f=f.clone(), g=g.clone(), workspace=ws)  # warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        eot.sinkhorn(X, Y, log_a, log_b, 0.1, 3, f=f, g=g, workspace=ws)
    f.zero_()
    g.zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    fe, ge = eot.sinkhorn(X, Y, log_a, log_b, 0.1, 6, workspace=ws)
    assert torch.equal(f, fe) and torch.equal(g, ge)


def _hvp_case(n, m, d, eps, seed):
    X, Y, log_a, log_b = workloads.eot_clouds(n, m, d, seed=seed, device=DEV, random_weights=True)
    f64, g64 = oeot.sinkhorn64(np64(X), np64(Y), np64(log_a), np64(log_b), eps, 3000)
    f = torch.tensor(f64, dtype=torch.float32, device=DEV)
    g = torch.tensor(g64, dtype=torch.float32, device=DEV)
    return X, Y, log_a, log_b, f, g


def _hvp_bound(X, Y, f, g, log_a, log_b, V, eps):
    """Element bound of H v, entry by entry of the plan.  The kernel forms
        (H v)_i = 2 a_i v_i - (2/eps) [(df_i - 2 xv_i) (pi Y)_i
                                        + sum_j pi_ij dg_j y_j
                                        + 2 sum_j pi_ij (v_i . y_j) y_j]
    (xv_i = x_i . v_i), each sum a plan application.  Plan entry pi_ij
    carries a relative error delta_ij:
      * its score x_i . y_j: the operands are rounded to TF32 exactly as
        the kernel rounds them (cvt.rna), so that part of the error is
        computed here, not bounded; fp32 accumulation adds d_pad 2^-23 of
        sum_k |x_ik y_jk| (rounded operands);
      * norms, biases, ex2 and the exponent's combination as in row_bound,
        but with this entry's own magnitudes;
      * the second product: 2^-10 for pi (TF32 truncation; f16 rounds to
        2^-11) plus 2^-11 for the values, and fp32 accumulation over m_pad
        keys.
    Each term's error is delta_ij times its own magnitude:
    |df_i - 2 xv_i| + |dg_j| + 2 |v_i . y_j|, plus |df_i| + |dg_j| for the
    solve, which is taken to inherit the same relative error (its
    conditioning in the combination df_i + dg_j that enters H v is taken
    as 1).  The moment weights v_i . y_j are a TF32 product of their own
    (rounded the same way, computed here).  2 a_i v_i is rounded once
    (2^-21).  (df, dg) come from the oracle's dense solve."""
    args = (np64(X), np64(Y), np64(f), np64(g), np64(log_a), np64(log_b), eps)
    Xn, Yn, Vn = np64(X), np64(Y), np64(V)
    fn, gn, la, lb = np64(f), np64(g), np64(log_a), np64(log_b)
    n, d = Xn.shape
    m = Yn.shape[0]
    d_pad = -(-d // 32) * 32
    m_pad = -(-m // 256) * 256
    a, b = np.exp(la), np.exp(lb)
    P = oeot.plan64(*args)
    Xt, Yt, Vt = rna_tf32(Xn), rna_tf32(Yn), rna_tf32(Vn)
    xy = Xn @ Yn.T
    score = np.abs(Xt @ Yt.T - xy) + d_pad * 2.0 ** -23 * (np.abs(Xt) @ np.abs(Yt).T)
    N = (Xn * Xn).sum(1)[:, None]
    B = (Yn * Yn).sum(1)[None, :]
    fr = (np.abs(fn) + eps * np.abs(la))[:, None]
    t = (2.0 * score + d * 2.0 ** -23 * (N + B)
         + 2.0 ** -21 * (2.0 * np.abs(xy) + np.abs(gn)[None, :] + B + eps * np.abs(lb)[None, :] + fr + N)
         + eps * 2.0 ** -18)
    delta = np.expm1(t / eps + 2.0 ** -20) + 2.0 ** -10 + 2.0 ** -11 + m_pad * 2.0 ** -23
    xv = (Xn * Vn).sum(1)
    vy = Vn @ Yn.T
    dC = 2.0 * (xv[:, None] - vy)
    A = np.block([[np.diag(a), P], [P.T, np.diag(b)]])
    z = np.linalg.lstsq(A, np.r_[(P * dC).sum(1), (P * dC).sum(0)], rcond=None)[0]
    df, dg = z[:n], z[n:]
    S = (np.abs(df - 2.0 * xv) + np.abs(df))[:, None] + 2.0 * np.abs(dg)[None, :] + 2.0 * np.abs(vy)
    moment = 2.0 * (np.abs(Vt @ Yt.T - vy) + d_pad * 2.0 ** -23 * (np.abs(Vt) @ np.abs(Yt).T))
    return ((2.0 / eps) * ((P * (delta * S + moment)) @ np.abs(Yn))
            + 2.0 ** -21 * 2.0 * a[:, None] * np.abs(Vn))


@pytest.mark.parametrize("n,m,d,eps", [(300, 400, 8, 0.5), (500, 350, 32, 1.0), (200, 600, 3, 0.5)])
def test_hvp_parity(n, m, d, eps):
    """eot_hvp against the dense oracle at the same potentials, every element
    within the bound of _hvp_bound itself (CG runs long enough to converge
    at these sizes)."""
    X, Y, log_a, log_b, f, g = _hvp_case(n, m, d, eps, seed=n + m + d)
    V = torch.randn(n, d, generator=torch.Generator().manual_seed(d)).to(DEV)
    Hv = eot.hvp(X, Y, f, g, log_a, log_b, V, eps, cg_iters=150)
    ref = oeot.hvp64(np64(X), np64(Y), np64(f), np64(g), np64(log_a), np64(log_b), eps, np64(V))
    bound = _hvp_bound(X, Y, f, g, log_a, log_b, V, eps)
    err = np.abs(np64(Hv) - ref)
    assert np.all(np.isfinite(np64(Hv)))
    worst = (err / bound).max()
    assert worst <= 1.0, (worst, np.unravel_index((err / bound).argmax(), err.shape))


def test_hvp_translation_identity_and_zero_direction():
    """Along a common translation v_i = t the cost's gradient sum moves by
    2 t, so sum_i (H v)_i = 2 t; and H 0 = 0 exactly."""
    n, m, d, eps = 400, 300, 4, 0.5
    X, Y, log_a, log_b, f, g = _hvp_case(n, m, d, eps, seed=77)
    t = torch.tensor([0.6, -0.9, 0.3, 1.2], device=DEV)
    Hv = eot.hvp(X, Y, f, g, log_a, log_b, t.expand(n, d).contiguous(), eps, cg_iters=150)
    ref = oeot.hvp64(np64(X), np64(Y), np64(f), np64(g), np64(log_a), np64(log_b), eps,
                     np.tile(np64(t), (n, 1)))
    s = np64(Hv).sum(0)
    assert np.abs(s - 2 * np64(t)).max() <= 2e-2 * np.abs(ref).sum(0).max() / n + 1e-3
    Z = eot.hvp(X, Y, f, g, log_a, log_b, torch.zeros(n, d, device=DEV), eps, cg_iters=10)
    assert torch.count_nonzero(Z) == 0
