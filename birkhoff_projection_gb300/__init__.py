"""GB300-native per-token 4x4 Birkhoff projection (mHC, expansion rate n = 4).

Each token's logit matrix X is mapped to the doubly stochastic
P = diag(e^a) exp(X) diag(e^b) by Newton's method on the 3-variable reduced
dual, and the backward pass maps dP to dX by implicit differentiation
("Accelerating the Birkhoff Projection for Manifold-Constrained
Hyper-Connections", s2.1-s2.3).  Every step runs in the sm_103a kernels of
libbirkhoff4.so (C ABI: include/birkhoff4.h); this module only marshals
torch CUDA tensors and the current stream into those calls.

    P = project(X)              # autograd: backward uses the implicit formula
    P, b = forward(X, return_dual=True)
    dX = backward(dP, P=P)      # or backward(dP, X=X): P recomputed, not stored
    P, dX = forward_backward(X, dP)
    P20 = sinkhorn(X, iters=20) # fixed-iteration Sinkhorn-Knopp reference
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import B4_BF16, B4_F32, Birkhoff4Error, Opts, check, lib

__all__ = ["project", "forward", "backward", "forward_backward", "forward_backward_host",
           "forward_nxn", "backward_nxn", "forward_backward_mapped", "sinkhorn", "Birkhoff4Error", "lib", "Projection"]

_DT = {torch.float32: B4_F32, torch.bfloat16: B4_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_tokens(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in _DT:
        raise TypeError("%s must be float32 or bfloat16, got %s" % (name, t.dtype))
    if t.dim() < 2 or tuple(t.shape[-2:]) != (4, 4):
        raise ValueError("%s must have shape [..., 4, 4], got %s" % (name, tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.numel() // 16


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


class _on_device:
    """Make t's device current for the call (a no-op when it already is)."""

    __slots__ = ("ctx",)

    def __init__(self, t: torch.Tensor):
        idx = t.device.index
        self.ctx = None if idx is None or idx == torch.cuda.current_device() else torch.cuda.device(idx)

    def __enter__(self):
        if self.ctx is not None:
            self.ctx.__enter__()

    def __exit__(self, *exc):
        if self.ctx is not None:
            self.ctx.__exit__(*exc)


_SCHED = {"default": _lib.B4_SCHED_DEFAULT, "queue": _lib.B4_SCHED_QUEUE, "lane": _lib.B4_SCHED_LANE,
          "lanes4": _lib.B4_SCHED_LANES4}


def forward(X: torch.Tensor, *, out: torch.Tensor = None, out_dtype=None, return_dual: bool = False,
            tol: float = 0.0, max_evals: int = 0, return_stats: bool = False,
            schedule: str = "default"):
    """Projection of every token of X ([..., 4, 4], fp32 or bf16).

    Returns P (dtype out_dtype, default X.dtype), plus b ([..., 4] fp32,
    natural-log column dual, b[..., 3] = 0) if return_dual, plus
    (evals [...] int32, nonconverged count) if return_stats.  schedule:
    "default", "queue", "lane" or "lanes4" (birkhoff4_schedule; "lanes4"
    for fp32 only)."""
    T = _check_tokens(X, "X")
    odt = out_dtype or X.dtype
    if out is None:
        out = torch.empty(X.shape, dtype=odt, device=X.device)
    else:
        _check_tokens(out, "out")
        if out.shape != X.shape or out.dtype != odt or out.device != X.device:
            raise ValueError("out does not match X")
    b = torch.empty(X.shape[:-1], dtype=torch.float32, device=X.device) if return_dual else None
    opts = Opts(in_dtype=_DT[X.dtype], out_dtype=_DT[odt], max_evals=int(max_evals), tol=float(tol),
                schedule=_SCHED[schedule])
    evals = nonconv = None
    if return_stats:
        evals = torch.empty(X.shape[:-2], dtype=torch.int32, device=X.device)
        nonconv = torch.zeros(1, dtype=torch.int64, device=X.device)
        opts.evals_out = evals.data_ptr()
        opts.nonconv_count = nonconv.data_ptr()
    with _on_device(X):
        check(lib().birkhoff4_forward_ex(_ptr(X), _ptr(out), _ptr(b), T, ctypes.byref(opts),
                                         _stream(X)), "birkhoff4_forward_ex")
    res = (out,)
    if return_dual:
        res += (b,)
    if return_stats:
        res += (evals, nonconv)
    return res[0] if len(res) == 1 else res


def backward(dP: torch.Tensor, *, P: torch.Tensor = None, X: torch.Tensor = None,
             out: torch.Tensor = None) -> torch.Tensor:
    """dX = (dP/dX)^T dP by implicit differentiation, from the stored P or,
    if P is None, from X (P recomputed inside the kernel)."""
    T = _check_tokens(dP, "dP")
    src = P if P is not None else X
    if src is None:
        raise ValueError("backward needs P or X")
    _check_tokens(src, "P" if P is not None else "X")
    if src.shape != dP.shape or src.dtype != dP.dtype or src.device != dP.device:
        raise ValueError("P/X and dP must match in shape, dtype and device")
    if out is None:
        out = torch.empty_like(dP)
    fn = lib().birkhoff4_backward if dP.dtype == torch.float32 else lib().birkhoff4_backward_bf16
    with _on_device(dP):
        check(fn(_ptr(X), _ptr(P), _ptr(dP), _ptr(out), T, _stream(dP)), "birkhoff4_backward")
    return out


def forward_backward(X: torch.Tensor, dP: torch.Tensor, *, want_P: bool = True,
                     schedule: str = "default"):
    """One fused pass: (P, dX) (P is None if not wanted).  schedule:
    "default", "queue" or "lane" (birkhoff4_schedule)."""
    _check_tokens(X, "X")
    _check_tokens(dP, "dP")
    if X.shape != dP.shape or X.dtype != dP.dtype or X.device != dP.device:
        raise ValueError("X and dP must match in shape, dtype and device")
    P = torch.empty_like(X) if want_P else None
    dX = torch.empty_like(dP)
    _fused_pass(X, dP, P, dX, schedule=schedule)
    return P, dX


def _fused_pass(X, dP, P, dX, schedule: str = "default"):
    """The fused pass into preallocated outputs (P may be None)."""
    T = _check_tokens(X, "X")
    opts = Opts(in_dtype=_DT[X.dtype], out_dtype=_DT[X.dtype], schedule=_SCHED[schedule])
    with _on_device(X):
        check(lib().birkhoff4_forward_backward_ex(_ptr(X), _ptr(dP), _ptr(P), _ptr(dX), T,
                                                  ctypes.byref(opts), _stream(X)),
              "birkhoff4_forward_backward_ex")


def sinkhorn(X: torch.Tensor, iters: int = 20, *, out: torch.Tensor = None) -> torch.Tensor:
    """Fixed-iteration log-domain Sinkhorn-Knopp (the reference scheme)."""
    T = _check_tokens(X, "X")
    if out is None:
        out = torch.empty_like(X)
    fn = lib().birkhoff4_sinkhorn if X.dtype == torch.float32 else lib().birkhoff4_sinkhorn_bf16
    with _on_device(X):
        check(fn(_ptr(X), _ptr(out), int(iters), T, _stream(X)), "birkhoff4_sinkhorn")
    return out


def forward_backward_host(X: torch.Tensor, dP: torch.Tensor, P_out, dX_out: torch.Tensor, *,
                          device=None, workspace: torch.Tensor = None, streams=None,
                          chunk_tokens: int = 1 << 22, nstreams: int = 3):
    """Forward + backward of host-resident tokens (birkhoff4_forward_backward_host).

    X, dP (inputs), P_out (or None) and dX_out are contiguous CPU tensors
    [..., 4, 4] of one dtype, pinned for the copies to overlap the kernels.
    The tokens are streamed through the GPU in chunks, round-robin over
    `streams` (created here if not given): copy in, fused forward+backward,
    copy out.  workspace: a device uint8 tensor (allocated here for
    chunk_tokens per stream if not given).  Returns once the work is
    enqueued; the current stream waits for it, so synchronize before
    reading the outputs."""
    T = X.numel() // 16
    for name, t in (("X", X), ("dP", dP), ("dX_out", dX_out)) + ((("P_out", P_out),) if P_out is not None else ()):
        if t.is_cuda or t.dtype != X.dtype or t.numel() != X.numel() or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CPU tensor like X" % name)
    if X.dtype not in _DT:
        raise TypeError("X must be float32 or bfloat16")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if streams is None:
        streams = [torch.cuda.Stream(device=dev) for _ in range(nstreams)]
    rb = 16 * X.element_size()
    if workspace is None:
        workspace = torch.empty(len(streams) * 4 * chunk_tokens * rb, dtype=torch.uint8, device=dev)
    handles = (ctypes.c_void_p * len(streams))(*[s.cuda_stream for s in streams])
    cur = torch.cuda.current_stream(dev)
    start = torch.cuda.Event()
    start.record(cur)
    for s in streams:
        s.wait_event(start)
    with torch.cuda.device(dev):
        check(lib().birkhoff4_forward_backward_host(
            _ptr(X), _ptr(dP), _ptr(P_out), _ptr(dX_out), T, _DT[X.dtype], _ptr(workspace),
            workspace.numel(), ctypes.cast(handles, ctypes.c_void_p), len(streams)),
            "birkhoff4_forward_backward_host")
    for s in streams:
        done = torch.cuda.Event()
        done.record(s)
        cur.wait_event(done)
        workspace.record_stream(s)


def forward_backward_mapped(X: torch.Tensor, dP: torch.Tensor, P_out, dX_out: torch.Tensor, *,
                            device=None):
    """Forward + backward of host-resident tokens without copies
    (birkhoff4_forward_backward_mapped): the kernel on `device` reads X and
    dP and writes P_out (or None) and dX_out in place in pinned host memory.
    Enqueued on the device's current stream; synchronize before reading the
    outputs."""
    T = X.numel() // 16
    for name, t in (("X", X), ("dP", dP), ("dX_out", dX_out)) + ((("P_out", P_out),) if P_out is not None else ()):
        if t.is_cuda or t.dtype != X.dtype or t.numel() != X.numel() or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CPU tensor like X" % name)
        if not t.is_pinned():
            raise ValueError("%s must be in pinned host memory" % name)
    if X.dtype not in _DT:
        raise TypeError("X must be float32 or bfloat16")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        check(lib().birkhoff4_forward_backward_mapped(
            _ptr(X), _ptr(dP), _ptr(P_out), _ptr(dX_out), T, _DT[X.dtype],
            ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)),
            "birkhoff4_forward_backward_mapped")


def host_workspace(device, dtype, chunk_tokens: int = 1 << 22, nstreams: int = 3) -> torch.Tensor:
    """Device staging buffer for forward_backward_host (allocate once, reuse)."""
    rb = 16 * torch.empty((), dtype=dtype).element_size()
    return torch.empty(nstreams * 4 * chunk_tokens * rb, dtype=torch.uint8, device=device)


def _check_nxn(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != torch.float32:
        raise TypeError("%s must be float32 for n x n tokens" % name)
    if t.dim() < 2 or t.shape[-1] != t.shape[-2] or not (2 <= t.shape[-1] <= 8):
        raise ValueError("%s must have shape [..., n, n] with 2 <= n <= 8" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    n = t.shape[-1]
    return n, t.numel() // (n * n)


def forward_nxn(X: torch.Tensor, *, out: torch.Tensor = None, return_dual: bool = False):
    """Projection of n x n tokens X [..., n, n] (fp32, 2 <= n <= 8)."""
    n, T = _check_nxn(X, "X")
    if out is None:
        out = torch.empty_like(X)
    b = torch.empty(X.shape[:-1], dtype=torch.float32, device=X.device) if return_dual else None
    with _on_device(X):
        check(lib().birkhoff4_forward_nxn(_ptr(X), _ptr(out), _ptr(b), n, T, _stream(X)),
              "birkhoff4_forward_nxn")
    return (out, b) if return_dual else out


def backward_nxn(dP: torch.Tensor, *, P: torch.Tensor, out: torch.Tensor = None) -> torch.Tensor:
    """Implicit-differentiation backward for n x n tokens."""
    n, T = _check_nxn(dP, "dP")
    _check_nxn(P, "P")
    if P.shape != dP.shape:
        raise ValueError("P and dP must match")
    if out is None:
        out = torch.empty_like(dP)
    with _on_device(dP):
        check(lib().birkhoff4_backward_nxn(_ptr(P), _ptr(dP), _ptr(out), n, T, _stream(dP)),
              "birkhoff4_backward_nxn")
    return out


class Projection(torch.autograd.Function):
    """P = project(X); the backward is the implicit-differentiation kernel
    applied to the saved P (nothing of the forward iteration is stored)."""

    @staticmethod
    def forward(ctx, X):
        Xc = X.contiguous()
        P = forward(Xc) if X.shape[-1] == 4 else forward_nxn(Xc)
        ctx.save_for_backward(P)
        return P

    @staticmethod
    def backward(ctx, dP):
        (P,) = ctx.saved_tensors
        dP = dP.contiguous().to(P.dtype)
        return backward(dP, P=P) if P.shape[-1] == 4 else backward_nxn(dP, P=P)


def project(X: torch.Tensor) -> torch.Tensor:
    """Differentiable per-token Birkhoff projection of X [..., n, n]
    (n = 4: fp32 or bf16 through the 4 x 4 kernels; 2 <= n <= 8 fp32 through
    the n x n kernels)."""
    return Projection.apply(X)
