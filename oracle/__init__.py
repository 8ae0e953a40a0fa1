"""Float64 CPU oracle for the per-token 4x4 Birkhoff projection.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  It
shares no code with the CUDA library in ``birkhoff_projection_gb300`` and never
imports it.

Sources (page title, section):
  [mHC] "Accelerating the Birkhoff Projection for Manifold-Constrained
        Hyper-Connections" (technical summary of arXiv 2606.07574):
        s1 fixed-iteration Sinkhorn-Knopp in current mHC; s2 projection ==
        entropic OT; s2.1 Newton on the 3-variable reduced dual with a row-max
        shift; s2.2 implicit-function-theorem backward with Hessian reuse.

What each function follows:
  sinkhorn64 / sinkhorn_fixed64  log-domain Sinkhorn-Knopp        [mHC s1, s2]
  newton64                       Newton on the reduced dual       [mHC s2.1]
  backward64                     implicit-function-theorem VJP    [mHC s2.2]
  fd_backward64                  central differences of newton64 (validator)
  unrolled_sinkhorn_backward64   autograd through a long unrolled log-domain
                                 Sinkhorn (validator; the "unrolled" backward
                                 that [mHC s1] names as the memory-heavy
                                 baseline)

Pins: every function is checked in tests/test_oracle.py against closed forms,
invariants and independent validators (see the header of that file).

The C part (birkhoff4_oracle.c) is compiled with gcc on first use (or by
``__graft_entry__.build()``) into ``oracle/liboracle64.so``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "birkhoff4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle64.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        i64 = ctypes.c_int64
        lib.oracle_sinkhorn64.argtypes = [dp, dp, dp, i64, ctypes.c_double, ctypes.c_int32, ip]
        lib.oracle_sinkhorn64.restype = i64
        lib.oracle_newton64.argtypes = [dp, dp, dp, i64, ctypes.c_double, ctypes.c_int32, ip,
                                        dp, ctypes.c_int32]
        lib.oracle_newton64.restype = i64
        lib.oracle_backward64.argtypes = [dp, dp, dp, i64]
        lib.oracle_backward64.restype = None
        lib.oracle_laplacian_solve64.argtypes = [dp, dp, dp, i64]
        lib.oracle_laplacian_solve64.restype = i64
        i32 = ctypes.c_int32
        lib.oracle_sinkhorn64_n.argtypes = [dp, dp, dp, i32, i64, ctypes.c_double, i32, ip]
        lib.oracle_sinkhorn64_n.restype = i64
        lib.oracle_newton64_n.argtypes = [dp, dp, dp, i32, i64, ctypes.c_double, i32, ip]
        lib.oracle_newton64_n.restype = i64
        lib.oracle_backward64_n.argtypes = [dp, dp, dp, i32, i64]
        lib.oracle_backward64_n.restype = None
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        lib.oracle_version.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double if a.dtype == np.float64
                                           else ctypes.c_int32))


def _tokens(X) -> np.ndarray:
    """Any array-like of shape [..., 4, 4] -> C-contiguous float64 [T, 16]."""
    if hasattr(X, "detach"):  # torch tensor (CPU); bf16 is widened exactly
        X = X.detach().to("cpu").double().numpy()
    a = np.ascontiguousarray(np.asarray(X, dtype=np.float64))
    if a.shape[-2:] != (4, 4):
        raise ValueError("expected [..., 4, 4], got %s" % (a.shape,))
    return a.reshape(-1, 16)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> int:
    """Use n threads in later calls; returns the previous count."""
    lib = _load()
    prev = int(lib.oracle_num_threads())
    lib.oracle_set_num_threads(int(n))
    return prev


def sinkhorn64(X, tol: float = 1e-13, max_iters: int = 20000):
    """Log-domain Sinkhorn-Knopp to max marginal residual < tol [mHC s1, s2].

    Returns (P [T,4,4], b [T,4] with b[:,3] = 0, iters [T] int32, nonconverged)."""
    lib = _load()
    x = _tokens(X)
    T = x.shape[0]
    P = np.empty_like(x)
    b = np.empty((T, 4))
    it = np.empty(T, dtype=np.int32)
    n = lib.oracle_sinkhorn64(_ptr(x), _ptr(P), _ptr(b), T, float(tol), int(max_iters), _ptr(it))
    return P.reshape(-1, 4, 4), b, it, int(n)


def sinkhorn_fixed64(X, iters: int):
    """Exactly ``iters`` log-domain Sinkhorn-Knopp iterations (row step then
    column step), output exp(X + a + b) after the last column step [mHC s1]."""
    if iters < 0:
        raise ValueError("iters must be >= 0")
    lib = _load()
    x = _tokens(X)
    T = x.shape[0]
    P = np.empty_like(x)
    lib.oracle_sinkhorn64(_ptr(x), _ptr(P), None, T, 0.0, int(iters), None)
    return P.reshape(-1, 4, 4)


def newton64(X, tol: float = 1e-14, max_iters: int = 200, trace_len: int = 0):
    """Newton's method on the reduced dual with Armijo backtracking [mHC s2.1].

    Returns (P [T,4,4], b [T,4], iters [T], nonconverged[, trace [T,trace_len]])."""
    lib = _load()
    x = _tokens(X)
    T = x.shape[0]
    P = np.empty_like(x)
    b = np.empty((T, 4))
    it = np.empty(T, dtype=np.int32)
    tr = np.empty((T, trace_len)) if trace_len > 0 else None
    n = lib.oracle_newton64(_ptr(x), _ptr(P), _ptr(b), T, float(tol), int(max_iters), _ptr(it),
                            _ptr(tr), int(trace_len))
    out = (P.reshape(-1, 4, 4), b, it, int(n))
    return out + (tr,) if trace_len > 0 else out


def project64(X):
    """The oracle projection P*: newton64 at its default tolerance."""
    return newton64(X)[0]


def backward64(P, G):
    """dX = (dP/dX)^T G by the implicit function theorem [mHC s2.2]."""
    lib = _load()
    p = _tokens(P)
    g = _tokens(G)
    if p.shape != g.shape:
        raise ValueError("P and G shapes differ")
    dX = np.empty_like(p)
    lib.oracle_backward64(_ptr(p), _ptr(g), _ptr(dX), p.shape[0])
    return dX.reshape(-1, 4, 4)


def fd_backward64(X, G, h: float = 1e-4):
    """Validator: dX_kl = sum_ij G_ij dP_ij/dX_kl by central differences of
    newton64 with one Richardson step (steps h and h/2); O(h^4) error."""
    x = _tokens(X).reshape(-1, 4, 4)
    g = _tokens(G).reshape(-1, 4, 4)
    T = x.shape[0]
    eye = np.eye(16).reshape(16, 4, 4)

    def central(step):
        plus = (x[:, None] + step * eye[None]).reshape(-1, 4, 4)
        minus = (x[:, None] - step * eye[None]).reshape(-1, 4, 4)
        Pp = newton64(plus, tol=1e-15)[0].reshape(T, 16, 4, 4)
        Pm = newton64(minus, tol=1e-15)[0].reshape(T, 16, 4, 4)
        return np.einsum("tij,tkij->tk", g, Pp - Pm) / (2.0 * step)

    d1 = central(h)
    d2 = central(h / 2.0)
    return ((4.0 * d2 - d1) / 3.0).reshape(T, 4, 4)


def unrolled_sinkhorn_backward64(X, G, iters: int = 2000):
    """Validator: reverse-mode autodiff (torch, float64, CPU) through ``iters``
    unrolled log-domain Sinkhorn-Knopp iterations; returns (P, dX)."""
    import torch

    x = torch.tensor(_tokens(X).reshape(-1, 4, 4), dtype=torch.float64, requires_grad=True)
    g = torch.tensor(_tokens(G).reshape(-1, 4, 4), dtype=torch.float64)
    b = torch.zeros(x.shape[0], 1, 4, dtype=torch.float64)
    a = torch.zeros(x.shape[0], 4, 1, dtype=torch.float64)
    for _ in range(iters):
        a = -torch.logsumexp(x + b, dim=2, keepdim=True)
        b = -torch.logsumexp(x + a, dim=1, keepdim=True)
    P = torch.exp(x + a + b)
    (P * g).sum().backward()
    return P.detach().numpy(), x.grad.detach().numpy()


def laplacian_solve64(w, r):
    """Solve H x = r where H is the Laplacian of the complete graph on four
    nodes with edge weights w [n,6] (edges (0,1),(0,2),(0,3),(1,2),(1,3),(2,3)),
    restricted to nodes 0..2; closed form by the matrix-tree theorem."""
    lib = _load()
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float64).reshape(-1, 6))
    r = np.ascontiguousarray(np.asarray(r, dtype=np.float64).reshape(-1, 3))
    x = np.empty_like(r)
    lib.oracle_laplacian_solve64(_ptr(w), _ptr(r), _ptr(x), w.shape[0])
    return x


# ---------------------------------------------------------------------------
# General n x n (2 <= n <= 16): the dual reduced to n-1 free variables
# [mHC s2.1]; same methods as the 4 x 4 functions, written for any n.
# ---------------------------------------------------------------------------
def _tokens_n(X):
    if hasattr(X, "detach"):
        X = X.detach().to("cpu").double().numpy()
    a = np.ascontiguousarray(np.asarray(X, dtype=np.float64))
    n = a.shape[-1]
    if a.ndim < 2 or a.shape[-2] != n or not (2 <= n <= 16):
        raise ValueError("expected [..., n, n] with 2 <= n <= 16, got %s" % (a.shape,))
    return a.reshape(-1, n * n), n


def sinkhorn64_n(X, tol: float = 1e-13, max_iters: int = 20000):
    """Log-domain Sinkhorn-Knopp for n x n tokens: (P, b, iters, nonconverged)."""
    lib = _load()
    x, n = _tokens_n(X)
    T = x.shape[0]
    P = np.empty_like(x)
    b = np.empty((T, n))
    it = np.empty(T, dtype=np.int32)
    k = lib.oracle_sinkhorn64_n(_ptr(x), _ptr(P), _ptr(b), n, T, float(tol), int(max_iters), _ptr(it))
    return P.reshape(-1, n, n), b, it, int(k)


def newton64_n(X, tol: float = 1e-14, max_iters: int = 200):
    """Newton on the (n-1)-variable reduced dual: (P, b, iters, nonconverged)."""
    lib = _load()
    x, n = _tokens_n(X)
    T = x.shape[0]
    P = np.empty_like(x)
    b = np.empty((T, n))
    it = np.empty(T, dtype=np.int32)
    k = lib.oracle_newton64_n(_ptr(x), _ptr(P), _ptr(b), n, T, float(tol), int(max_iters), _ptr(it))
    return P.reshape(-1, n, n), b, it, int(k)


def backward64_n(P, G):
    """Implicit-function-theorem VJP for n x n tokens."""
    lib = _load()
    p, n = _tokens_n(P)
    g, n2 = _tokens_n(G)
    if p.shape != g.shape:
        raise ValueError("P and G shapes differ")
    dX = np.empty_like(p)
    lib.oracle_backward64_n(_ptr(p), _ptr(g), _ptr(dX), n, p.shape[0])
    return dX.reshape(-1, n, n)


def fd_backward64_n(X, G, h: float = 1e-3):
    """Validator: central differences of newton64_n with one Richardson step."""
    x, n = _tokens_n(X)
    g, _ = _tokens_n(G)
    T = x.shape[0]
    x = x.reshape(T, n, n)
    g = g.reshape(T, n, n)
    eye = np.eye(n * n).reshape(n * n, n, n)

    def central(step):
        plus = (x[:, None] + step * eye[None]).reshape(-1, n, n)
        minus = (x[:, None] - step * eye[None]).reshape(-1, n, n)
        Pp = newton64_n(plus, tol=1e-15)[0].reshape(T, n * n, n, n)
        Pm = newton64_n(minus, tol=1e-15)[0].reshape(T, n * n, n, n)
        return np.einsum("tij,tkij->tk", g, Pp - Pm) / (2.0 * step)

    return ((4.0 * central(h / 2) - central(h)) / 3.0).reshape(T, n, n)


def marginal_residual(P) -> np.ndarray:
    """Per token max(|P 1 - 1|_inf, |P^T 1 - 1|_inf) (any n x n)."""
    P = np.asarray(P, dtype=np.float64)
    n = P.shape[-1]
    p = P.reshape(-1, n, n)
    r = np.abs(p.sum(axis=2) - 1.0).max(axis=1)
    c = np.abs(p.sum(axis=1) - 1.0).max(axis=1)
    return np.maximum(r, c)
