"""GPU parity on small cases, through the C ABI (libbirkhoff4.so).

Sizes span several 128-token tiles and ragged tails; closed forms and the
fixed-point family give known answers independent of the oracle; edge cases:
empty input, unaligned pointers (plain-load kernel), in-place use, untouched
guard regions around outputs, non-finite tokens, option statistics, the
device fault latch.
"""
import ctypes
import json
import os

import numpy as np
import pytest
import torch

import birkhoff_projection_gb300 as b4
import oracle
from birkhoff_projection_gb300 import _lib, workloads
from _helpers import (TOL_DX_REL, TOL_P_LARGE, TOL_P_SMALL, TOL_RES_LARGE, TOL_RES_SMALL,
                      max_abs_err, np64, rel_fro, residual)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HERE = os.path.dirname(os.path.abspath(__file__))


def normal(T, sigma=1.0, seed=7):
    return workloads.normal(T, sigma, seed=seed).to(DEV)


@pytest.mark.parametrize("T", [1, 2, 31, 32, 33, 127, 128, 129, 255, 257, 1000, 4097])
def test_forward_small_sizes(T):
    X = normal(T)
    P = b4.forward(X)
    Pst = oracle.project64(np64(X))
    Pg = np64(P)
    assert max_abs_err(Pg, Pst) <= TOL_P_SMALL
    assert residual(Pg).max() <= TOL_RES_SMALL


@pytest.mark.parametrize("T", [1, 33, 129, 4097])
def test_backward_small_sizes(T):
    X = normal(T, seed=8)
    G = normal(T, seed=9)
    P = b4.forward(X)
    dX = b4.backward(G, P=P)
    Pst = oracle.project64(np64(X))
    dXst = oracle.backward64(Pst, np64(G))
    assert rel_fro(np64(dX), dXst) <= TOL_DX_REL
    assert max_abs_err(np64(dX), dXst) <= 1e-5


def test_closed_forms():
    cases = json.load(open(os.path.join(HERE, "golden", "closed_forms.json")))
    X = torch.tensor([c["X"] for c in cases["forward"]], dtype=torch.float32, device=DEV)
    want = np.array([c["P"] for c in cases["forward"]])
    P = np64(b4.forward(X))
    # fp32 rounding of the logits moves P by ~1e-7
    assert max_abs_err(P, want) <= 2e-6
    bw = cases["backward"][0]
    Xb = torch.tensor([bw["X"]], dtype=torch.float32, device=DEV)
    Gb = torch.tensor([bw["G"]], dtype=torch.float32, device=DEV)
    dX = np64(b4.backward(Gb, P=b4.forward(Xb)))
    assert max_abs_err(dX, np.array([bw["dX"]])) <= 2e-6


@pytest.mark.parametrize("spread,floor,tol", [(5.0, 1e-3, TOL_P_SMALL), (40.0, 1e-6, TOL_P_LARGE)])
def test_fixed_point_family(spread, floor, tol):
    """X = log Q + u 1^T + 1 v^T projects to Q exactly (Q doubly stochastic)."""
    X64, Q = workloads.fixed_point_family(4096, seed=21, spread=spread, floor=floor)
    X = X64.float().to(DEV)
    P = np64(b4.forward(X))
    # the known answer for the fp32-rounded logits, and Q itself
    assert max_abs_err(P, oracle.project64(np64(X))) <= tol
    assert max_abs_err(P, Q.numpy()) <= tol


def test_fused_and_recompute_match_separate_passes():
    X = normal(3000, seed=10)
    G = normal(3000, seed=11)
    P = b4.forward(X)
    dX = b4.backward(G, P=P)
    Pf, dXf = b4.forward_backward(X, G)
    assert torch.equal(Pf, P)
    assert max_abs_err(np64(dXf), np64(dX)) <= 1e-6
    _, dXr = b4.forward_backward(X, G, want_P=False)
    dXr2 = b4.backward(G, X=X)
    assert max_abs_err(np64(dXr), np64(dX)) <= 1e-6
    assert max_abs_err(np64(dXr2), np64(dX)) <= 1e-6


def test_autograd_projection():
    X = normal(777, seed=12).requires_grad_(True)
    G = normal(777, seed=13)
    P = b4.project(X)
    (P * G).sum().backward()
    Pst = oracle.project64(np64(X))
    assert max_abs_err(np64(P), Pst) <= TOL_P_SMALL
    assert rel_fro(np64(X.grad), oracle.backward64(Pst, np64(G))) <= TOL_DX_REL


def test_dual_output():
    X = normal(5000, seed=14)
    P, b = b4.forward(X, return_dual=True)
    b = b.cpu().double().numpy()
    assert (b[:, 3] == 0).all()
    z = np64(X) + b[:, None, :]
    e = np.exp(z - z.max(axis=2, keepdims=True))
    assert max_abs_err(e / e.sum(axis=2, keepdims=True), np64(P)) <= TOL_P_SMALL
    bst = oracle.newton64(np64(X))[1]
    assert max_abs_err(b, bst) <= 1e-4


def test_sinkhorn_reference_matches_oracle():
    X = normal(2000, seed=15)
    for iters in (0, 1, 5, 20):
        P = np64(b4.sinkhorn(X, iters=iters))
        want = oracle.sinkhorn_fixed64(np64(X), iters)
        # relative: iters = 0 gives exp(X), up to ~e^4 here
        assert (np.abs(P - want) / np.maximum(want, 1.0)).max() <= 2e-6 * max(1, iters)


def test_empty_input():
    X = torch.empty(0, 4, 4, device=DEV)
    assert b4.forward(X).shape == (0, 4, 4)
    assert b4.backward(X, P=X).shape == (0, 4, 4)
    assert b4.sinkhorn(X).shape == (0, 4, 4)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_unaligned_pointers_use_plain_kernel(dtype):
    T = 1000
    X = normal(T, seed=16).to(dtype)
    G = normal(T, seed=17).to(dtype)
    P = b4.forward(X)
    dX = b4.backward(G, P=P)
    # the same tokens at an address offset by one element
    L = _lib.lib()
    es = X.element_size()
    bufX = torch.zeros(T * 16 + 1, dtype=dtype, device=DEV)
    bufX[1:] = X.reshape(-1)
    bufP = torch.zeros_like(bufX)
    fwd = L.birkhoff4_forward if dtype == torch.float32 else L.birkhoff4_forward_bf16
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert fwd(ctypes.c_void_p(bufX.data_ptr() + es), ctypes.c_void_p(bufP.data_ptr() + es), None, T, s) == 0
    assert torch.equal(bufP[1:].reshape(T, 4, 4), P)
    bufG = torch.zeros_like(bufX)
    bufG[1:] = G.reshape(-1)
    bufD = torch.zeros_like(bufX)
    bwd = L.birkhoff4_backward if dtype == torch.float32 else L.birkhoff4_backward_bf16
    assert bwd(None, ctypes.c_void_p(bufP.data_ptr() + es), ctypes.c_void_p(bufG.data_ptr() + es),
               ctypes.c_void_p(bufD.data_ptr() + es), T, s) == 0
    assert torch.equal(bufD[1:].reshape(T, 4, 4), dX)


def test_in_place():
    X = normal(4097, seed=18)
    G = normal(4097, seed=19)
    P = b4.forward(X)
    dX = b4.backward(G, P=P)
    Y = X.clone()
    b4.forward(Y, out=Y)
    assert torch.equal(Y, P)
    H = G.clone()
    L = _lib.lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.birkhoff4_backward(None, ctypes.c_void_p(P.data_ptr()), ctypes.c_void_p(H.data_ptr()),
                                ctypes.c_void_p(H.data_ptr()), 4097, s) == 0
    assert torch.equal(H, dX)


def test_guard_regions_untouched():
    """Outputs are written exactly where the tokens are: guard regions of 1 KiB
    on both sides keep their bit pattern (ragged T, all passes)."""
    T = 1000 + 37
    guard = 256  # floats
    X = normal(T, seed=20)
    G = normal(T, seed=21)
    canary = torch.full((T * 16 + 2 * guard,), float.fromhex("0x1.deadbep+7"), device=DEV)
    L = _lib.lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = canary.clone()
    optr = ctypes.c_void_p(out.data_ptr() + guard * 4)
    xp, gp = ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(G.data_ptr())
    for call in (lambda: L.birkhoff4_forward(xp, optr, None, T, s),
                 lambda: L.birkhoff4_backward(None, xp, gp, optr, T, s),
                 lambda: L.birkhoff4_sinkhorn(xp, optr, 3, T, s)):
        out.copy_(canary)
        assert call() == 0
        torch.cuda.synchronize()
        assert torch.equal(out[:guard], canary[:guard])
        assert torch.equal(out[-guard:], canary[-guard:])
        assert not torch.equal(out[guard:-guard], canary[guard:-guard])


def test_nonfinite_tokens_are_isolated():
    X = normal(300, seed=22)
    X[5, 1, 2] = float("nan")
    X[77, 0, 0] = float("inf")
    X[78, 3, 3] = -float("inf")
    P = b4.forward(X)
    bad = torch.zeros(300, dtype=torch.bool)
    bad[[5, 77, 78]] = True
    Pc = P.cpu()
    assert torch.isnan(Pc[bad]).all()
    assert torch.isfinite(Pc[~bad]).all()
    good = np64(X)[~bad.numpy()]
    assert max_abs_err(Pc[~bad].double().numpy(), oracle.project64(good)) <= TOL_P_SMALL


def test_statistics_and_options():
    X = normal(4096, seed=23)
    P, evals, nonconv = b4.forward(X, return_stats=True)
    ev = evals.cpu().numpy()
    assert ev.min() >= 1 and ev.max() <= 48
    assert int(nonconv.item()) == 0
    # a cap of one evaluation: tokens above tol are counted, P is the first
    # evaluation (the row softmax at the column-mean start)
    P1, ev1, nc1 = b4.forward(X, max_evals=1, return_stats=True)
    assert (ev1.cpu().numpy() == 1).all()
    res = residual(np64(P1))
    assert int(nc1.item()) == int((res > 1e-6).sum())
    # a looser tolerance stops earlier
    P3, ev3, _ = b4.forward(X, tol=1e-3, return_stats=True)
    assert ev3.float().mean() < evals.float().mean()
    assert residual(np64(P3)).max() <= 64e-3
    # bf16 in -> fp32 out
    Pb = b4.forward(X.bfloat16(), out_dtype=torch.float32)
    assert Pb.dtype == torch.float32
    assert residual(np64(Pb)).max() <= TOL_RES_SMALL


def test_fault_latch_selftest():
    L = _lib.lib()
    v = ctypes.c_uint(0)
    assert L.birkhoff4_device_status(ctypes.byref(v), 1) == 0
    assert v.value & 1 == 0  # no TMA wait has ever run out
    assert L.birkhoff4_selftest_wait_timeout(1_000_000) == 0  # 1 ms
    assert L.birkhoff4_device_status(ctypes.byref(v), 1) == 0
    assert v.value == 2
    assert L.birkhoff4_device_status(ctypes.byref(v), 0) == 0
    assert v.value == 0


def test_large_magnitude_small():
    X, G = workloads.large_magnitude(3000)
    X, G = X.to(DEV), G.to(DEV)
    P = b4.forward(X)
    dX = b4.backward(G, P=P)
    Pst = oracle.project64(np64(X))
    assert max_abs_err(np64(P), Pst) <= TOL_P_LARGE
    assert residual(np64(P)).max() <= TOL_RES_LARGE
    assert rel_fro(np64(dX), oracle.backward64(Pst, np64(G))) <= TOL_DX_REL


@pytest.mark.parametrize("dtype,nstreams,chunk,with_P", [
    (torch.float32, 3, 1024, True), (torch.float32, 1, 777, False), (torch.bfloat16, 2, 1500, True)])
def test_host_streaming_api(dtype, nstreams, chunk, with_P):
    """birkhoff4_forward_backward_host: host tokens through chunked copies on
    caller streams give the device results (ragged last chunk, P optional)."""
    T = 5000
    X = normal(T, seed=24).to(dtype)
    G = normal(T, seed=25).to(dtype)
    P, dX = b4.forward_backward(X, G)
    Xh, Gh = X.cpu().pin_memory(), G.cpu().pin_memory()
    Ph = torch.empty_like(Xh).pin_memory() if with_P else None
    dXh = torch.empty_like(Xh).pin_memory()
    ws = b4.host_workspace(DEV, dtype, chunk_tokens=chunk, nstreams=nstreams)
    b4.forward_backward_host(Xh, Gh, Ph, dXh, device=DEV, workspace=ws, nstreams=nstreams)
    torch.cuda.synchronize()
    if with_P:
        assert torch.equal(Ph, P.cpu())
    assert torch.equal(dXh, dX.cpu())


def test_cuda_graph_capture_and_replay():
    """The passes capture into a CUDA graph (no host synchronisation or
    allocation on the launch path) and replay on new inputs."""
    T = 10000
    X, G = normal(T, seed=30), normal(T, seed=31)
    P, dX = torch.empty_like(X), torch.empty_like(X)
    b4.forward(X, out=P)  # one-time per-device set-up happens outside the capture
    b4.backward(G, P=P, out=dX)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        b4.forward(X, out=P)
        b4.backward(G, P=P, out=dX)
    for seed in (32, 34):
        X.copy_(normal(T, seed=seed))
        G.copy_(normal(T, seed=seed + 1))
        g.replay()
        torch.cuda.synchronize()
        Pe = b4.forward(X)
        assert torch.equal(P, Pe)
        assert torch.equal(dX, b4.backward(G, P=Pe))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [1, 129, 5000])
@pytest.mark.parametrize("with_P", [True, False])
def test_mapped_host_api(dtype, T, with_P):
    """birkhoff4_forward_backward_mapped: the kernel reads and writes pinned
    host tokens in place and gives exactly the device pass's results."""
    X = normal(T, seed=26).to(dtype)
    G = normal(T, seed=27).to(dtype)
    P, dX = b4.forward_backward(X, G)
    Xh, Gh = X.cpu().pin_memory(), G.cpu().pin_memory()
    Ph = torch.empty_like(Xh).pin_memory() if with_P else None
    dXh = torch.empty_like(Xh).pin_memory()
    b4.forward_backward_mapped(Xh, Gh, Ph, dXh, device=DEV)
    torch.cuda.synchronize()
    if with_P:
        assert torch.equal(Ph, P.cpu())
    assert torch.equal(dXh, dX.cpu())


def test_mapped_host_in_place_and_pageable_memory():
    T = 3000
    X, G = normal(T, seed=28), normal(T, seed=29)
    P, dX = b4.forward_backward(X, G)
    Xh, Gh = X.cpu().pin_memory(), G.cpu().pin_memory()
    b4.forward_backward_mapped(Xh, Gh, Xh, Gh, device=DEV)  # P over X, dX over dP
    torch.cuda.synchronize()
    assert torch.equal(Xh, P.cpu()) and torch.equal(Gh, dX.cpu())
    # pageable host memory: refused before anything runs where the device
    # cannot address it, or processed in place where it can (Grace-based
    # systems address all host memory)
    Xp, Gp, Dp = X.cpu(), G.cpu(), torch.empty(T, 4, 4)
    L = _lib.lib()
    st = L.birkhoff4_forward_backward_mapped(ctypes.c_void_p(Xp.data_ptr()), ctypes.c_void_p(Gp.data_ptr()),
                                             None, ctypes.c_void_p(Dp.data_ptr()), T, _lib.B4_F32, None)
    assert st in (_lib.B4_OK, _lib.B4_EINVAL)
    if st == _lib.B4_OK:
        torch.cuda.synchronize()
        assert torch.equal(Dp, dX.cpu())
    assert float(b4.forward(X[:4]).sum()) > 0  # the context is still usable
