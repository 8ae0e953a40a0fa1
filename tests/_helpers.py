"""Host-side metrics and tolerances shared by the GPU parity tests.

Tolerances (fp32 arithmetic on the GPU against the float64 oracle):
  * logits with |X| <= 10 (N(0,1) workloads): max |P - P*| <= 1e-5 and
    marginal residual <= 2e-6;
  * large-magnitude logits (the |X| ~ 200 workload, N(0, 10^2)): both <= 1e-4;
  * backward: global ||dX - dX*||_F / ||dX*||_F <= 1e-4;
  * bf16 outputs: P equal to the round-to-nearest-even bf16 of P*, one bf16
    ulp allowed where P* lies within 4e-6 (the fp32 accuracy of the solve) of
    a rounding midpoint; dX within one bf16 ulp of dX* plus 1e-4 ||dX*||_inf
    per token.
"""
import numpy as np
import torch

TOL_P_SMALL, TOL_RES_SMALL = 1e-5, 2e-6
TOL_P_LARGE, TOL_RES_LARGE = 1e-4, 1e-4
TOL_DX_REL = 1e-4


def np64(t) -> np.ndarray:
    """Tensor (any device/dtype) -> float64 numpy copy of the same shape."""
    return t.detach().to("cpu", torch.float64).numpy()


def residual(P) -> np.ndarray:
    """Per-token max(|P 1 - 1|_inf, |P^T 1 - 1|_inf) of [..., n, n] tokens,
    float64."""
    p = np.asarray(P, dtype=np.float64)
    p = p.reshape(-1, p.shape[-1], p.shape[-1])
    return np.maximum(np.abs(p.sum(2) - 1).max(1), np.abs(p.sum(1) - 1).max(1))


def residual_gpu(P: torch.Tensor) -> torch.Tensor:
    """The same residual computed on the device in float64 (for arrays too
    large to copy back)."""
    p = P.reshape(-1, P.shape[-1], P.shape[-1]).double()
    return torch.maximum((p.sum(2) - 1).abs().amax(1), (p.sum(1) - 1).abs().amax(1))


def max_abs_err(A, B) -> float:
    return float(np.abs(np.asarray(A, np.float64) - np.asarray(B, np.float64)).max())


def rel_fro(A, B) -> float:
    """||A - B||_F / ||B||_F."""
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    return float(np.linalg.norm((A - B).ravel()) / max(np.linalg.norm(B.ravel()), 1e-300))


def rne_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), directly
    from float64 (no intermediate fp32 rounding); returns float64."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m 2^e, 0.5 <= |m| < 1
    r = np.round(m * 256.0)  # 8 significant bits; numpy rounds half to even
    return np.ldexp(r, e - 8)


def rna_tf32(x) -> np.ndarray:
    """Round fp32 values to TF32 as cvt.rna.tf32.f32 does (nearest, ties
    away from zero): add half of the 13 dropped mantissa bits to the
    magnitude field, then clear them.  Returns float64."""
    bits = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    bits = (bits + 0x1000) & ~np.uint64(0x1FFF)
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (normal range)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 1e-38)))
    return np.ldexp(1.0, (e - 7).astype(int))


def near_bf16_midpoint(x, slack) -> np.ndarray:
    """True where x is within `slack` of a point halfway between two bf16
    numbers (where fp32 rounding error can flip the bf16 rounding)."""
    x = np.asarray(x, dtype=np.float64)
    u = bf16_ulp(x)
    lo = np.floor(x / u) * u
    mid = lo + u / 2
    return np.abs(x - mid) <= slack


def to_bf16_values(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its exact values as float64 numpy."""
    return t.detach().to("cpu").float().double().numpy()
