"""The token schedules of the Newton passes (birkhoff4_opts.schedule),
through the C ABI.

B4_SCHED_QUEUE (the default) solves each warp's tokens in a fresh round of
at most 7 evaluations (8 in the passes with a backward), parks the unsolved
ones in shared memory and finishes them in resume rounds of 2 evaluations,
re-evaluating P in the log domain on each resume.  B4_SCHED_LANE keeps one token per thread to the end.
  * N(0,1) tokens all finish within their fresh round (at most 5
    evaluations), so both schedules run the same arithmetic: bit-identical
    results for every pass and dtype.
  * At N(0,10^2) and on large-magnitude tokens most tokens are parked at
    least once: every output against the oracle within the large-magnitude
    tolerances, the dual b consistent with P, the fused and recompute passes
    consistent with the forward.
  * Caps inside and beyond the fresh round; non-finite tokens among parked
    ones; ragged token counts.
B4_SCHED_LANES4 (four lanes per token, fp32 forward) against the oracle on
the three magnitude classes and ragged sizes.
"""
import numpy as np
import pytest
import torch

import birkhoff_projection_gb300 as b4
import oracle
from birkhoff_projection_gb300 import workloads
from _helpers import (TOL_DX_REL, TOL_P_LARGE, TOL_P_SMALL, TOL_RES_LARGE, TOL_RES_SMALL,
                      max_abs_err, np64, rel_fro, residual)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_schedules_bit_identical_at_normal(dtype):
    T = 100003
    X = workloads.normal(T, 1.0, seed=40, device=DEV).to(dtype)
    G = workloads.normal(T, 1.0, seed=41, device=DEV).to(dtype)
    Pq, bq, eq, nq = b4.forward(X, return_dual=True, return_stats=True, schedule="queue")
    Pl, bl, el, nl = b4.forward(X, return_dual=True, return_stats=True, schedule="lane")
    assert int(eq.max()) <= 5  # all solved in the fresh round
    assert torch.equal(Pq, Pl) and torch.equal(bq, bl) and torch.equal(eq, el)
    assert int(nq.item()) == int(nl.item()) == 0
    for with_P in (True, False):
        outs = {}
        for sched in ("queue", "lane"):
            P = torch.empty_like(X) if with_P else None
            dX = torch.empty_like(X)
            b4._fused_pass(X, G, P, dX, schedule=sched)
            outs[sched] = (P, dX)
        if with_P:
            assert torch.equal(outs["queue"][0], outs["lane"][0])
            assert torch.equal(outs["queue"][0], Pq)
        assert torch.equal(outs["queue"][1], outs["lane"][1])


def _parked_case(kind, T):
    if kind == "sigma10":
        X = workloads.normal(T, 10.0, seed=42, device=DEV)
        G = workloads.normal(T, 1.0, seed=43, device=DEV)
        return X, G
    return workloads.large_magnitude(T, device=DEV)


@pytest.mark.parametrize("kind,T", [("sigma10", 50017), ("large", 30001)])
def test_queue_parks_and_resumes(kind, T):
    X, G = _parked_case(kind, T)
    P, b, ev, nc = b4.forward(X, return_dual=True, return_stats=True, schedule="queue")
    _, evl, _ = b4.forward(X, return_stats=True, schedule="lane")
    e = ev.cpu().numpy()
    # many tokens needed more than the forward's fresh round of 7 evaluations
    assert (e > 7).mean() > (0.25 if kind == "sigma10" else 0.5)
    assert e.max() <= 48 and int(nc.item()) == 0
    # the same iteration: evaluation counts within a step or two of the
    # single-round schedule's on average (resumes re-evaluate P in the log domain)
    assert abs(float(ev.float().mean()) - float(evl.float().mean())) <= 0.5
    Pst = oracle.project64(np64(X))
    Pg = np64(P)
    assert max_abs_err(Pg, Pst) <= TOL_P_LARGE
    assert residual(Pg).max() <= TOL_RES_LARGE
    bb = b.double().cpu().numpy()
    assert (bb[:, 3] == 0).all()
    if kind == "sigma10":
        z = np64(X) + bb[:, None, :]
        s = np.exp(z - z.max(axis=2, keepdims=True))
        assert max_abs_err(s / s.sum(axis=2, keepdims=True), Pg) <= 1e-4
    # fused: P and dX against the oracle (its fresh round is 8 evaluations
    # against the forward's 7, so a token parked by one is re-evaluated in
    # the log domain at another step than in the other: P agrees within the
    # tolerance, not bit for bit); recompute: the same dX as the fused pass
    Pf, dXf = b4.forward_backward(X, G)
    assert max_abs_err(np64(Pf), Pst) <= TOL_P_LARGE
    assert max_abs_err(np64(Pf), Pg) <= TOL_P_LARGE
    assert rel_fro(np64(dXf), oracle.backward64(Pst, np64(G))) <= TOL_DX_REL
    _, dXr = b4.forward_backward(X, G, want_P=False)
    assert torch.equal(dXr, dXf)
    # bf16 in and out, parked tokens included: the forward, and the fused
    # pass (its own, longer fresh round, parking and resuming with a
    # backward): P within bf16 rounding of the oracle, dX within bf16
    # rounding in the relative Frobenius norm
    Xb = X.bfloat16()
    Gb = G.bfloat16()
    Pb = b4.forward(Xb)
    Pbst = oracle.project64(np64(Xb))
    assert np.abs(np64(Pb) - Pbst).max() <= 2.0 ** -8 + TOL_P_LARGE
    Pbf, dXbf = b4.forward_backward(Xb, Gb)
    assert np.abs(np64(Pbf) - Pbst).max() <= 2.0 ** -8 + TOL_P_LARGE
    assert rel_fro(np64(dXbf), oracle.backward64(Pbst, np64(Gb))) <= 2.0 ** -8 + TOL_DX_REL


@pytest.mark.parametrize("cap", [3, 7, 10])
def test_queue_caps(cap):
    """max_evals within every fresh round of the forward (3, 7: no token is
    parked, so the schedules agree bit for bit) and beyond it (10: the cap
    falls in a resume round)."""
    X = workloads.normal(20000, 10.0, seed=44, device=DEV)
    Pq, eq, nq = b4.forward(X, max_evals=cap, return_stats=True, schedule="queue")
    Pl, el, nl = b4.forward(X, max_evals=cap, return_stats=True, schedule="lane")
    e = eq.cpu().numpy()
    assert e.max() == cap and e.min() >= 1
    if cap <= 7:
        assert torch.equal(Pq, Pl) and torch.equal(eq, el)
        assert int(nq.item()) == int(nl.item())
    res = residual(np64(Pq))
    # tokens stopped below the cap converged (tolerance or its stagnation floor)
    # (the kernel tests its fp32 residual; 7e-5 allows for recomputing it in float64)
    assert res[e < cap].max() <= 7e-5
    # tokens counted as not converged are the ones stopped by the cap above tol
    assert int(nq.item()) <= int((e == cap).sum())
    assert int(nq.item()) >= int(((e == cap) & (res > 7e-5)).sum())


def test_nonfinite_tokens_among_parked():
    T = 10000
    X = workloads.normal(T, 10.0, seed=45, device=DEV)
    bad = [3, 4, 1000, 5555, T - 1]
    X[3, 0, 0] = float("nan")
    X[4, 1, 1] = float("inf")
    X[1000, 2, 3] = -float("inf")
    X[5555, 3, 0] = float("nan")
    X[T - 1, 0, 2] = float("inf")
    P, ev, nc = b4.forward(X, return_stats=True)
    mask = torch.zeros(T, dtype=torch.bool)
    mask[bad] = True
    Pc = P.cpu()
    assert torch.isnan(Pc[mask]).all()
    assert torch.isfinite(Pc[~mask]).all()
    assert (ev.cpu()[mask] == 0).all()
    assert int(nc.item()) == len(bad)
    good = np64(X)[~mask.numpy()]
    assert max_abs_err(Pc[~mask].double().numpy(), oracle.project64(good)) <= TOL_P_LARGE


@pytest.mark.parametrize("T", [1, 31, 33, 127, 129, 4095])
def test_queue_ragged_small(T):
    X = workloads.normal(T, 10.0, seed=46 + T, device=DEV)
    P = b4.forward(X)
    Pst = oracle.project64(np64(X))
    assert max_abs_err(np64(P), Pst) <= TOL_P_LARGE
    assert residual(np64(P)).max() <= TOL_RES_LARGE


@pytest.mark.parametrize("kind,T", [("normal", 40009), ("sigma10", 30011), ("large", 20001)])
def test_lanes4_forward(kind, T):
    """Four lanes per token (B4_SCHED_LANES4, fp32 forward): the same
    iteration with sums taken across lanes.  Parity with the oracle in the
    workload's tolerance class, b consistent with P, evaluation counts as in
    the one-thread kernel up to rounding-order effects."""
    if kind == "normal":
        X = workloads.normal(T, 1.0, seed=47, device=DEV)
    elif kind == "sigma10":
        X = workloads.normal(T, 10.0, seed=48, device=DEV)
    else:
        X = workloads.large_magnitude(T, device=DEV)[0]
    X[T // 2, 1, 1] = float("nan")
    P, b, ev, nc = b4.forward(X, return_dual=True, return_stats=True, schedule="lanes4")
    _, evl, _ = b4.forward(X, return_stats=True, schedule="lane")
    ok = torch.ones(T, dtype=torch.bool)
    ok[T // 2] = False
    Pc = P.cpu()
    assert torch.isnan(Pc[T // 2]).all() and int(ev[T // 2]) == 0
    assert int(nc.item()) == 1
    Pg = Pc[ok].double().numpy()
    Pst = oracle.project64(np64(X)[ok.numpy()])
    tol_p, tol_r = ((TOL_P_SMALL, TOL_RES_SMALL) if kind == "normal" else (TOL_P_LARGE, TOL_RES_LARGE))
    assert max_abs_err(Pg, Pst) <= tol_p
    assert residual(Pg).max() <= tol_r
    bb = b.double().cpu().numpy()[ok.numpy()]
    assert (bb[:, 3] == 0).all()
    assert abs(float(ev[ok].float().mean()) - float(evl[ok].float().mean())) <= 0.05
    if kind != "large":
        z = np64(X)[ok.numpy()] + bb[:, None, :]
        s = np.exp(z - z.max(axis=2, keepdims=True))
        assert max_abs_err(s / s.sum(axis=2, keepdims=True), Pg) <= 10 * tol_p


@pytest.mark.parametrize("T", [1, 7, 8, 9, 63, 65, 1001])
def test_lanes4_ragged(T):
    X = workloads.normal(T, 1.0, seed=49 + T, device=DEV)
    P = b4.forward(X, schedule="lanes4")
    assert max_abs_err(np64(P), oracle.project64(np64(X))) <= TOL_P_SMALL
