"""The largest token counts: past one kernel launch, and n x n arrays past
2^31 elements.

The launcher splits a pass into launches of at most 2^30 tokens (TMA row
coordinates and the kernels' token indices stay within 32 bits), and inside
a launch the output address of a token's dual is 4 x its index, which
passes 2^31 from index 2^29 on.  One forward over 2^30 + 2^20 + 33 tokens
(in place, with the dual b; about 86 GB of device memory) covers both:
tokens around index 2^29, around the launch boundary at 2^30 and at the
ragged end are checked against the oracle, and b against P.
"""
import numpy as np
import pytest
import torch

import birkhoff_projection_gb300 as b4
import oracle
from _helpers import TOL_DX_REL, TOL_P_SMALL, TOL_RES_SMALL, max_abs_err, np64, rel_fro, residual

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_forward_past_one_launch():
    T = (1 << 30) + (1 << 20) + 33
    torch.cuda.empty_cache()
    need = T * 64 + T * 16 + (4 << 30)
    if torch.cuda.mem_get_info()[0] < need:
        pytest.skip("needs %.0f GB of free device memory" % (need / 1e9))
    g = torch.Generator(device=DEV).manual_seed(77)
    X = torch.empty(T, 4, 4, device=DEV)
    step = 1 << 26
    for s in range(0, T, step):
        X[s:s + step].normal_(generator=g)
    idx = torch.cat([torch.arange(0, 64), torch.arange((1 << 29) - 64, (1 << 29) + 64),
                     torch.arange((1 << 30) - 64, (1 << 30) + 64), torch.arange(T - 64, T)]).to(DEV)
    Xs = np64(X[idx])
    P, b = b4.forward(X, out=X, return_dual=True)  # in place: P over X
    Ps = np64(P[idx])
    bs = np64(b[idx])
    del X, P, b
    torch.cuda.empty_cache()
    Pst = oracle.project64(Xs)
    assert max_abs_err(Ps, Pst) <= TOL_P_SMALL
    assert residual(Ps).max() <= TOL_RES_SMALL
    assert (bs[:, 3] == 0).all()
    z = Xs + bs[:, None, :]
    e = np.exp(z - z.max(axis=2, keepdims=True))
    assert max_abs_err(e / e.sum(axis=2, keepdims=True), Ps) <= 10 * TOL_P_SMALL


def test_nxn_past_2_31_elements():
    """n = 8 with 2^25 + 77 tokens: 2^31 + 4928 floats per array, so element
    offsets pass 2^31 from token 2^25 on.  Forward and backward; tokens
    around that boundary, the first ones and the ragged end against the
    oracle (about 26 GB of device memory)."""
    n = 8
    T = (1 << 25) + 77
    torch.cuda.empty_cache()
    need = 3 * T * n * n * 4 + (4 << 30)
    if torch.cuda.mem_get_info()[0] < need:
        pytest.skip("needs %.0f GB of free device memory" % (need / 1e9))
    g = torch.Generator(device=DEV).manual_seed(78)
    X = torch.randn(T, n, n, device=DEV, generator=g)
    G = torch.randn(T, n, n, device=DEV, generator=g)
    idx = torch.cat([torch.arange(0, 64), torch.arange((1 << 25) - 64, (1 << 25) + 64),
                     torch.arange(T - 64, T)]).to(DEV)
    Xs, Gs = np64(X[idx]), np64(G[idx])
    P = b4.forward_nxn(X)
    del X
    dX = b4.backward_nxn(G, P=P, out=G)  # in place over dP
    Ps, dXs = np64(P[idx]), np64(dX[idx])
    del P, dX, G
    torch.cuda.empty_cache()
    Pst = oracle.newton64_n(Xs)[0]
    assert max_abs_err(Ps, Pst) <= TOL_P_SMALL
    assert residual(Ps).max() <= TOL_RES_SMALL
    assert rel_fro(dXs, oracle.backward64_n(Pst, Gs)) <= TOL_DX_REL
