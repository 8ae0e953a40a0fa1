"""Streaming entropic OT between point clouds on the GPU: Python binding of
eot_update / eot_sinkhorn (include/eot_stream.h).  Argument marshalling
only; every step runs in the library's kernels.

"FlashSinkhorn: IO-Aware Entropic OT on GPU", Methodik s1-s2: log-domain
Sinkhorn for the quadratic Euclidean cost, each potential update a row-wise
log-sum-exp of a biased dot-product score matrix that is never stored.

    f, g = sinkhorn(X, Y, log_a, log_b, eps=0.1, iters=10)
"""
from __future__ import annotations

import torch

from . import _ptr, _stream, _on_device
from ._lib import check, lib

TF32 = 1     # one TF32 product per coordinate pair
TF32X3 = 3   # hi + lo split, three TF32 products (near fp32)


def _points(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise ValueError("%s must be a float32 CUDA tensor" % name)
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError("%s must be a contiguous [points, d] tensor" % name)
    return t.shape[0]


def _vector(t: torch.Tensor, name: str, n: int, device) -> None:
    if (not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.device != device
            or t.dim() != 1 or t.shape[0] != n or not t.is_contiguous()):
        raise ValueError("%s must be a contiguous float32 [%d] tensor on %s" % (name, n, device))


def workspace_bytes(n: int, m: int, d: int, passes: int = TF32) -> int:
    b = lib().eot_workspace_bytes(n, m, d, passes)
    if b == 0:
        raise ValueError("invalid sizes or passes")
    return b


def _workspace(ws, n, m, d, passes, device):
    need = workspace_bytes(n, m, d, passes)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
    if ws.numel() < need or ws.device != device:
        raise ValueError("workspace needs %d bytes on %s" % (need, device))
    return ws


def update(Xq: torch.Tensor, Xk: torch.Tensor, h: torch.Tensor, log_w: torch.Tensor, eps: float,
           passes: int = TF32, out: torch.Tensor = None, workspace: torch.Tensor = None):
    """out_i = -eps LSE_j[(h_j - ||xq_i - xk_j||^2)/eps + log_w_j]."""
    nq = _points(Xq, "Xq")
    nk = _points(Xk, "Xk")
    if Xk.device != Xq.device or Xk.shape[1] != Xq.shape[1]:
        raise ValueError("Xq and Xk must share the device and the dimension")
    _vector(h, "h", nk, Xq.device)
    _vector(log_w, "log_w", nk, Xq.device)
    d = Xq.shape[1]
    if out is None:
        out = torch.empty(nq, dtype=torch.float32, device=Xq.device)
    _vector(out, "out", nq, Xq.device)
    ws = _workspace(workspace, nq, nk, d, passes, Xq.device)
    with _on_device(Xq):
        check(lib().eot_update(_ptr(Xq), _ptr(Xk), _ptr(h), _ptr(log_w), _ptr(out), nq, nk, d,
                               float(eps), passes, _ptr(ws), ws.numel(), _stream(Xq)),
              "eot_update")
    return out


def sinkhorn(X: torch.Tensor, Y: torch.Tensor, log_a: torch.Tensor, log_b: torch.Tensor,
             eps: float, iters: int, passes: int = TF32, f: torch.Tensor = None,
             g: torch.Tensor = None, workspace: torch.Tensor = None):
    """`iters` alternating log-domain Sinkhorn iterations (f from g, then g
    from f), starting from f and g (zeros if not given, updated in place).
    Returns (f, g)."""
    n = _points(X, "X")
    m = _points(Y, "Y")
    if Y.device != X.device or Y.shape[1] != X.shape[1]:
        raise ValueError("X and Y must share the device and the dimension")
    _vector(log_a, "log_a", n, X.device)
    _vector(log_b, "log_b", m, X.device)
    if f is None:
        f = torch.zeros(n, dtype=torch.float32, device=X.device)
    if g is None:
        g = torch.zeros(m, dtype=torch.float32, device=X.device)
    _vector(f, "f", n, X.device)
    _vector(g, "g", m, X.device)
    d = X.shape[1]
    ws = _workspace(workspace, n, m, d, passes, X.device)
    with _on_device(X):
        check(lib().eot_sinkhorn(_ptr(X), _ptr(Y), _ptr(log_a), _ptr(log_b), _ptr(f), _ptr(g), n,
                                 m, d, float(eps), int(iters), passes, _ptr(ws), ws.numel(),
                                 _stream(X)),
              "eot_sinkhorn")
    return f, g


def transport(X: torch.Tensor, Y: torch.Tensor, f: torch.Tensor, g: torch.Tensor,
              log_a: torch.Tensor, log_b: torch.Tensor, eps: float, want_grad: bool = False,
              workspace: torch.Tensor = None):
    """Transport application of the plan pi_ij = a_i b_j exp((f_i + g_j -
    ||x_i - y_j||^2)/eps): returns (pi Y [n, d], pi 1 [n]) and, with
    want_grad, also 2 (r_i x_i - (pi Y)_i), the gradient of the entropic OT
    cost with respect to X at converged potentials.  The barycentric map is
    (pi Y) / (pi 1)[:, None]."""
    n = _points(X, "X")
    m = _points(Y, "Y")
    if Y.device != X.device or Y.shape[1] != X.shape[1]:
        raise ValueError("X and Y must share the device and the dimension")
    for t, name, k in ((f, "f", n), (g, "g", m), (log_a, "log_a", n), (log_b, "log_b", m)):
        _vector(t, name, k, X.device)
    d = X.shape[1]
    need = lib().eot_transport_workspace_bytes(n, m, d)
    if need == 0:
        raise ValueError("invalid sizes")
    ws = workspace if workspace is not None else torch.empty(need, dtype=torch.uint8,
                                                             device=X.device)
    if ws.numel() < need or ws.device != X.device:
        raise ValueError("workspace needs %d bytes on %s" % (need, X.device))
    PY = torch.empty(n, d, dtype=torch.float32, device=X.device)
    mass = torch.empty(n, dtype=torch.float32, device=X.device)
    grad = torch.empty(n, d, dtype=torch.float32, device=X.device) if want_grad else None
    with _on_device(X):
        check(lib().eot_transport(_ptr(X), _ptr(Y), _ptr(f), _ptr(g), _ptr(log_a), _ptr(log_b),
                                  _ptr(PY), _ptr(mass), _ptr(grad), n, m, d, float(eps), _ptr(ws),
                                  ws.numel(), _stream(X)),
              "eot_transport")
    return (PY, mass, grad) if want_grad else (PY, mass)


def apply_plan(X: torch.Tensor, Y: torch.Tensor, f: torch.Tensor, g: torch.Tensor,
               log_a: torch.Tensor, log_b: torch.Tensor, V: torch.Tensor, eps: float,
               workspace: torch.Tensor = None):
    """The plan of (f, g) applied to values V [m, dv] at the key points,
    without forming it: returns (pi V [n, dv], pi 1 [n])."""
    n = _points(X, "X")
    m = _points(Y, "Y")
    if Y.device != X.device or Y.shape[1] != X.shape[1]:
        raise ValueError("X and Y must share the device and the dimension")
    if _points(V, "V") != m or V.device != X.device:
        raise ValueError("V must be [m, dv] on the device of X")
    for t, name, k in ((f, "f", n), (g, "g", m), (log_a, "log_a", n), (log_b, "log_b", m)):
        _vector(t, name, k, X.device)
    d, dv = X.shape[1], V.shape[1]
    need = lib().eot_apply_plan_workspace_bytes(n, m, d, dv)
    if need == 0:
        raise ValueError("invalid sizes")
    ws = workspace if workspace is not None else torch.empty(need, dtype=torch.uint8,
                                                             device=X.device)
    if ws.numel() < need or ws.device != X.device:
        raise ValueError("workspace needs %d bytes on %s" % (need, X.device))
    out = torch.empty(n, dv, dtype=torch.float32, device=X.device)
    mass = torch.empty(n, dtype=torch.float32, device=X.device)
    with _on_device(X):
        check(lib().eot_apply_plan(_ptr(X), _ptr(Y), _ptr(f), _ptr(g), _ptr(log_a), _ptr(log_b),
                                   _ptr(V), dv, _ptr(out), _ptr(mass), n, m, d, float(eps),
                                   _ptr(ws), ws.numel(), _stream(X)),
              "eot_apply_plan")
    return out, mass


def hvp(X: torch.Tensor, Y: torch.Tensor, f: torch.Tensor, g: torch.Tensor,
        log_a: torch.Tensor, log_b: torch.Tensor, V: torch.Tensor, eps: float,
        cg_iters: int = 50, workspace: torch.Tensor = None) -> torch.Tensor:
    """Hessian-vector product H V [n, d] of the entropic OT cost with respect
    to X, at Sinkhorn-converged potentials (f, g)."""
    n = _points(X, "X")
    m = _points(Y, "Y")
    if Y.device != X.device or Y.shape[1] != X.shape[1]:
        raise ValueError("X and Y must share the device and the dimension")
    if V.shape != X.shape or V.dtype != torch.float32 or V.device != X.device or not V.is_contiguous():
        raise ValueError("V must be a contiguous float32 tensor shaped like X")
    for t, name, k in ((f, "f", n), (g, "g", m), (log_a, "log_a", n), (log_b, "log_b", m)):
        _vector(t, name, k, X.device)
    d = X.shape[1]
    need = lib().eot_hvp_workspace_bytes(n, m, d)
    if need == 0:
        raise ValueError("invalid sizes")
    ws = workspace if workspace is not None else torch.empty(need, dtype=torch.uint8,
                                                             device=X.device)
    if ws.numel() < need or ws.device != X.device:
        raise ValueError("workspace needs %d bytes on %s" % (need, X.device))
    out = torch.empty_like(X)
    with _on_device(X):
        check(lib().eot_hvp(_ptr(X), _ptr(Y), _ptr(f), _ptr(g), _ptr(log_a), _ptr(log_b), _ptr(V),
                            _ptr(out), n, m, d, float(eps), int(cg_iters), _ptr(ws), ws.numel(),
                            _stream(X)),
              "eot_hvp")
    return out
