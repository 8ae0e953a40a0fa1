"""Seeded synthetic inputs for the 4x4 Birkhoff projection.

Shared by the tests, the benchmark and the oracle checks.  This module only
draws random numbers in the shapes and distributions of the workloads; it
holds none of the projection's arithmetic and imports neither the CUDA
library nor the oracle.

Workloads (all tokens are [4,4] row-major; T = number of tokens):
  small_normal     T = 4096, X fp32 iid N(0,1), seed 0 (forward only)
  normal_1m        T = 2^20, X and upstream dP fp32 iid N(0,1), seed 1
  large_magnitude  T = 2^20, X_ij = 20 Z_ij + r_i + c_j, Z ~ N(0,1),
                   r_i, c_j ~ U[-50,50] per token, fp32, seed 2
  mhc_batch        X bf16 [64, 32, 8192, 4, 4] (2^24 tokens),
                   X = Z + 0.5 s I with Z ~ N(0,1) per entry and one
                   s ~ N(0,1) per token (diagonal bias); dP bf16 N(0,1), seed 3
  sweep            T = 2^12 ... 2^26, X fp32 iid N(0, sigma^2),
                   sigma in {1, 10}, seed 4

Point clouds for streaming entropic OT (n x d and m x d, fp32):
  eot_clouds       X rows iid N(0, I_d / d); Y rows iid N(0, I_d / d) shifted
                   by 0.5 along the first axis (so ||x - y||^2 is about 2.25
                   for any d); weights uniform, or with random=True drawn
                   U[0.2, 1] and normalised; seed 100 + seed
"""
from __future__ import annotations

import torch

SWEEP_LOG2_T = list(range(12, 27))
SWEEP_SIGMAS = (1.0, 10.0)


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=torch.device(device)).manual_seed(seed)


def normal(T: int, sigma: float = 1.0, seed: int = 0, device="cpu",
           dtype=torch.float32) -> torch.Tensor:
    """X [T,4,4] iid N(0, sigma^2), drawn in fp32 then cast to ``dtype``."""
    g = _gen(seed, device)
    x = torch.randn(T, 4, 4, generator=g, device=device, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(dtype)


def small_normal(device="cpu") -> torch.Tensor:
    return normal(4096, 1.0, seed=0, device=device)


def normal_1m(T: int = 1 << 20, device="cpu"):
    """(X, dP), both [T,4,4] fp32 iid N(0,1) from one stream, seed 1."""
    g = _gen(1, device)
    x = torch.randn(T, 4, 4, generator=g, device=device, dtype=torch.float32)
    dp = torch.randn(T, 4, 4, generator=g, device=device, dtype=torch.float32)
    return x, dp


def large_magnitude(T: int = 1 << 20, device="cpu"):
    """(X, dP): X_ij = 20 Z_ij + r_i + c_j with r, c ~ U[-50, 50] per token
    (|X| up to about 200); dP iid N(0,1).  Seed 2."""
    g = _gen(2, device)
    z = torch.randn(T, 4, 4, generator=g, device=device, dtype=torch.float32)
    r = torch.rand(T, 4, 1, generator=g, device=device, dtype=torch.float32) * 100.0 - 50.0
    c = torch.rand(T, 1, 4, generator=g, device=device, dtype=torch.float32) * 100.0 - 50.0
    x = 20.0 * z + r + c
    dp = torch.randn(T, 4, 4, generator=g, device=device, dtype=torch.float32)
    return x, dp


def large_magnitude_n(n: int, T: int, seed: int, device="cpu"):
    """(X, dP) for n x n tokens with the large-magnitude recipe:
    X_ij = 20 Z_ij + r_i + c_j, r, c ~ U[-50, 50] per token; dP iid N(0,1)."""
    g = _gen(seed, device)
    z = torch.randn(T, n, n, generator=g, device=device, dtype=torch.float32)
    r = torch.rand(T, n, 1, generator=g, device=device, dtype=torch.float32) * 100.0 - 50.0
    c = torch.rand(T, 1, n, generator=g, device=device, dtype=torch.float32) * 100.0 - 50.0
    x = 20.0 * z + r + c
    dp = torch.randn(T, n, n, generator=g, device=device, dtype=torch.float32)
    return x, dp


MHC_SHAPE = (64, 32, 8192)


def mhc_batch(shape=MHC_SHAPE, device="cpu"):
    """(X, dP) bf16 [*shape, 4, 4]: X = Z + 0.5 s I (one s per token), seed 3."""
    g = _gen(3, device)
    z = torch.randn(*shape, 4, 4, generator=g, device=device, dtype=torch.float32)
    s = torch.randn(*shape, 1, 1, generator=g, device=device, dtype=torch.float32)
    eye = torch.eye(4, device=device, dtype=torch.float32)
    x = (z + 0.5 * s * eye).to(torch.bfloat16)
    dp = torch.randn(*shape, 4, 4, generator=g, device=device,
                     dtype=torch.float32).to(torch.bfloat16)
    return x, dp


def sweep(log2_T: int, sigma: float, device="cpu", shard: int = 0):
    """(X, dP) for the throughput sweep: X fp32 iid N(0, sigma^2), dP N(0,1).
    shard k > 0 draws another 2^log2_T tokens of the same distribution (the
    k-th rank's share of a multi-GPU job)."""
    T = 1 << log2_T
    g = _gen(4 + 1000 * shard, device)
    x = torch.randn(T, 4, 4, generator=g, device=device, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    dp = torch.randn(T, 4, 4, generator=g, device=device, dtype=torch.float32)
    return x, dp


def fixed_point_family(T: int, seed: int, spread: float = 5.0, floor: float = 1e-3,
                       device="cpu", dtype=torch.float64):
    """(X, Q) with Q strictly positive and doubly stochastic and
    X = log Q + u 1^T + 1 v^T (u, v ~ U[-spread, spread] per token).

    Q mixes the 24 permutation matrices with Dirichlet(1) weights plus
    ``floor`` times the uniform matrix, renormalised; the projection of X is Q
    exactly, whatever the offsets.  Built in float64."""
    import itertools

    g = _gen(seed, device)
    perms = torch.tensor(list(itertools.permutations(range(4))), device=device)
    pm = torch.zeros(24, 4, 4, dtype=torch.float64, device=device)
    pm[torch.arange(24).repeat_interleave(4), torch.arange(4).repeat(24), perms.reshape(-1)] = 1.0
    w = -torch.log(torch.rand(T, 24, generator=g, device=device, dtype=torch.float64))
    w = w / w.sum(dim=1, keepdim=True)
    q = torch.einsum("tk,kij->tij", w, pm)
    q = (q + floor / 4.0) / (1.0 + floor)
    u = (torch.rand(T, 4, 1, generator=g, device=device, dtype=torch.float64) * 2 - 1) * spread
    v = (torch.rand(T, 1, 4, generator=g, device=device, dtype=torch.float64) * 2 - 1) * spread
    x = torch.log(q) + u + v
    return x.to(dtype), q


def fixed_point_family_n(n: int, T: int, seed: int, spread: float = 5.0, floor: float = 1e-3,
                         nperm: int = 8, device="cpu", dtype=torch.float64):
    """(X, Q) for n x n tokens: Q = a random mixture of `nperm` random
    permutation matrices plus ``floor`` times the uniform matrix
    (renormalised; strictly positive, doubly stochastic) and
    X = log Q + u 1^T + 1 v^T, whose projection is Q.  Float64."""
    g = _gen(seed, device)
    perms = torch.argsort(torch.rand(T, nperm, n, generator=g, device=device), dim=-1)
    w = -torch.log(torch.rand(T, nperm, generator=g, device=device, dtype=torch.float64))
    w = w / w.sum(dim=1, keepdim=True)
    q = torch.zeros(T, n, n, dtype=torch.float64, device=device)
    rows = torch.arange(n, device=device)
    for k in range(nperm):
        q[torch.arange(T, device=device)[:, None], rows[None, :], perms[:, k, :]] += w[:, k:k + 1]
    q = (q + floor / n) / (1.0 + floor)
    u = (torch.rand(T, n, 1, generator=g, device=device, dtype=torch.float64) * 2 - 1) * spread
    v = (torch.rand(T, 1, n, generator=g, device=device, dtype=torch.float64) * 2 - 1) * spread
    x = torch.log(q) + u + v
    return x.to(dtype), q


EOT_SIZES = {"small": (1000, 1500), "bench": (65536, 65536)}
EOT_DIMS = (64, 512)
EOT_EPS = 0.1


def eot_clouds(n: int, m: int, d: int, seed: int = 0, device="cpu", random_weights: bool = False):
    """(X [n,d], Y [m,d], log_a [n], log_b [m]) fp32 point clouds and log
    weights (see the module docstring)."""
    g = _gen(100 + seed, device)
    X = torch.randn(n, d, generator=g, device=device) * (1.0 / d ** 0.5)
    Y = torch.randn(m, d, generator=g, device=device) * (1.0 / d ** 0.5)
    Y[:, 0] += 0.5
    if random_weights:
        a = torch.rand(n, generator=g, device=device) * 0.8 + 0.2
        b = torch.rand(m, generator=g, device=device) * 0.8 + 0.2
        log_a = torch.log(a / a.sum())
        log_b = torch.log(b / b.sum())
    else:
        log_a = torch.full((n,), -float(torch.log(torch.tensor(float(n)))), device=device)
        log_b = torch.full((m,), -float(torch.log(torch.tensor(float(m)))), device=device)
    return X.contiguous(), Y.contiguous(), log_a, log_b
