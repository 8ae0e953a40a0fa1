"""GPU parity of the n x n kernels (2 <= n <= 8) against the general-n
float64 oracle, through the C ABI (birkhoff4_forward_nxn /
birkhoff4_backward_nxn): several tile counts with ragged tails, N(0,1) and
N(0,5^2) logits, closed forms, the fixed-point family, the n = 4 kernels of
the main path, autograd, in-place use."""
import numpy as np
import pytest
import torch

import birkhoff_projection_gb300 as b4
import oracle
from birkhoff_projection_gb300 import workloads
from _helpers import TOL_DX_REL, max_abs_err, rel_fro, residual

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
NS = [2, 3, 4, 5, 6, 7, 8]


def tokens(n, T, sigma, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(T, n, n, generator=g) * sigma).to(DEV)


@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("T,sigma", [(1, 1.0), (129, 1.0), (5000, 1.0), (3001, 5.0)])
def test_forward_backward_parity(n, T, sigma):
    X = tokens(n, T, sigma, seed=100 * n + T)
    G = tokens(n, T, 1.0, seed=7 * n + T)
    P, b = b4.forward_nxn(X, return_dual=True)
    dX = b4.backward_nxn(G, P=P)
    Pst = oracle.newton64_n(X.double().cpu().numpy())[0]
    dXst = oracle.backward64_n(Pst, G.double().cpu().numpy())
    Pg = P.double().cpu().numpy()
    tolp, tolr = (1e-5, 2e-6) if sigma == 1.0 else (1e-4, 1e-4)
    assert max_abs_err(Pg, Pst) <= tolp
    assert residual(Pg).max() <= tolr
    assert rel_fro(dX.double().cpu().numpy(), dXst) <= TOL_DX_REL
    bb = b.double().cpu().numpy()
    assert (bb[:, n - 1] == 0).all()
    z = X.double().cpu().numpy() + bb[:, None, :]
    e = np.exp(z - z.max(2, keepdims=True))
    assert max_abs_err(e / e.sum(2, keepdims=True), Pg) <= 10 * tolp


@pytest.mark.parametrize("n", NS)
def test_closed_forms_and_fixed_points(n):
    c = torch.tensor([-2.0, 0.0, 1.5, 3.0])
    X = (c[:, None, None] * torch.eye(n)).to(DEV)
    P = b4.forward_nxn(X).double().cpu().numpy()
    cc = c.double().numpy()[:, None, None]
    want = np.where(np.eye(n) > 0, 1 / (1 + (n - 1) * np.exp(-cc)), 1 / (np.exp(cc) + n - 1))
    assert max_abs_err(P, want) <= 2e-6
    Xf, Q = workloads.fixed_point_family_n(n, 2000, seed=n)
    P = b4.forward_nxn(Xf.float().to(DEV)).double().cpu().numpy()
    assert max_abs_err(P, Q.numpy()) <= 1e-5


def test_two_by_two_closed_form():
    X = tokens(2, 4000, 3.0, seed=5)
    G = tokens(2, 4000, 1.0, seed=6)
    P = b4.forward_nxn(X)
    dX = b4.backward_nxn(G, P=P)
    x = X.double().cpu().numpy()
    g = G.double().cpu().numpy()
    q = 1 / (1 + np.exp(-(x[:, 0, 0] + x[:, 1, 1] - x[:, 0, 1] - x[:, 1, 0]) / 2))
    Pw = np.stack([np.stack([q, 1 - q], -1), np.stack([1 - q, q], -1)], 1)
    assert max_abs_err(P.double().cpu().numpy(), Pw) <= 2e-6
    k = (g[:, 0, 0] + g[:, 1, 1] - g[:, 0, 1] - g[:, 1, 0]) * q * (1 - q) / 2
    dw = k[:, None, None] * np.array([[1.0, -1.0], [-1.0, 1.0]])
    assert max_abs_err(dX.double().cpu().numpy(), dw) <= 2e-6


def test_n4_matches_main_path():
    X = tokens(4, 20000, 1.0, seed=8)
    G = tokens(4, 20000, 1.0, seed=9)
    Pa, Pb = b4.forward(X), b4.forward_nxn(X)
    assert max_abs_err(Pa.cpu().numpy(), Pb.cpu().numpy()) <= 2e-6
    da, db = b4.backward(G, P=Pa), b4.backward_nxn(G, P=Pa)
    assert max_abs_err(da.cpu().numpy(), db.cpu().numpy()) <= 2e-6


def test_autograd_and_in_place():
    X = tokens(6, 1000, 1.0, seed=10).requires_grad_(True)
    G = tokens(6, 1000, 1.0, seed=11)
    P = b4.project(X)
    (P * G).sum().backward()
    Pst = oracle.newton64_n(X.detach().double().cpu().numpy())[0]
    assert rel_fro(X.grad.double().cpu().numpy(), oracle.backward64_n(Pst, G.double().cpu().numpy())) <= TOL_DX_REL
    Y = X.detach().clone()
    b4.forward_nxn(Y, out=Y)
    assert torch.equal(Y, P.detach())



def _oracle_rows(X, G, idx):
    x = X[idx].double().cpu().numpy()
    g = G[idx].double().cpu().numpy()
    Pst = oracle.newton64_n(x)[0]
    return Pst, oracle.backward64_n(Pst, g)


@pytest.mark.parametrize("n", [3, 5, 8])
def test_many_tiles_per_cta(n):
    """2^20 + 77 tokens: the persistent grid is at most 152 SMs x 16 CTAs of
    128 tokens (forward) or 152 x 32 CTAs of 64 tokens (backward), so every
    CTA strides over at least three tiles and the last tile is ragged.
    Device residual on every token; the oracle on a 2^17-token random
    sample plus the last 4096 tokens."""
    T = (1 << 20) + 77
    X = tokens(n, T, 1.0, seed=300 + n)
    G = tokens(n, T, 1.0, seed=400 + n)
    P = b4.forward_nxn(X)
    dX = b4.backward_nxn(G, P=P)
    p = P.double()
    res = torch.maximum((p.sum(2) - 1).abs().amax(1), (p.sum(1) - 1).abs().amax(1))
    assert float(res.max()) <= 2e-6
    gsel = torch.Generator(device="cpu").manual_seed(n)
    idx = torch.cat([torch.randperm(T - 4096, generator=gsel)[: 1 << 17],
                     torch.arange(T - 4096, T)]).to(DEV)
    Pst, dXst = _oracle_rows(X, G, idx)
    assert max_abs_err(P[idx].double().cpu().numpy(), Pst) <= 1e-5
    assert rel_fro(dX[idx].double().cpu().numpy(), dXst) <= TOL_DX_REL


@pytest.mark.parametrize("n", [3, 5, 8])
def test_large_magnitude_nxn(n):
    """X_ij = 20 Z_ij + r_i + c_j with offsets U[-50, 50] (|X| up to about
    200): the large-magnitude tolerance class (1e-4 on P and on the
    marginals), every token against the oracle."""
    X, G = workloads.large_magnitude_n(n, 20000, seed=500 + n, device=DEV)
    P = b4.forward_nxn(X)
    dX = b4.backward_nxn(G, P=P)
    Pst = oracle.newton64_n(X.double().cpu().numpy())[0]
    dXst = oracle.backward64_n(Pst, G.double().cpu().numpy())
    Pg = P.double().cpu().numpy()
    assert max_abs_err(Pg, Pst) <= 1e-4
    assert residual(Pg).max() <= 1e-4
    assert rel_fro(dX.double().cpu().numpy(), dXst) <= TOL_DX_REL


@pytest.mark.parametrize("n", [3, 4, 6, 8])
def test_unaligned_arrays_match_aligned(n):
    """Arrays whose base is 4 bytes past a 16-byte boundary take the
    one-float-at-a-time tile copies; the arithmetic is the same as with the
    float4 copies, so P and dX must be equal bit for bit.  1000 tokens:
    several tiles and a ragged last one."""
    T = 1000
    X = tokens(n, T, 1.0, seed=500 + n)
    G = tokens(n, T, 1.0, seed=600 + n)
    P = b4.forward_nxn(X)
    dX = b4.backward_nxn(G, P=P)

    def shifted(t):
        buf = torch.empty(t.numel() + 1, device=DEV)
        v = buf[1:].view(t.shape)
        v.copy_(t)
        return v

    Xu, Gu = shifted(X), shifted(G)
    Pu = shifted(torch.zeros_like(X))
    dXu = shifted(torch.zeros_like(X))
    assert Xu.data_ptr() % 16 == 4
    b4.forward_nxn(Xu, out=Pu)
    b4.backward_nxn(Gu, P=Pu, out=dXu)
    assert torch.equal(Pu, P)
    assert torch.equal(dXu, dX)
