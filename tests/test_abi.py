"""The C ABI boundary on the host (no GPU needed).

libbirkhoff4.so must load, export every function include/birkhoff4.h and
include/eot_stream.h declare, and reject invalid arguments on the host before any CUDA call
(these checks never touch a device, so they run on a CPU-only machine).
"""
import ctypes
import os
import re

import pytest

from birkhoff_projection_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("birkhoff4.h", "eot_stream.h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:birkhoff4|eot)_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    return _lib.lib()


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    # and the binding covers exactly the header
    assert set(names) == set(_lib.SIGNATURES)


def test_version_and_strerror(L):
    assert L.birkhoff4_version() == 2
    for code in (0, 1, 2, 3, 99):
        s = L.birkhoff4_strerror(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert b"invalid" in L.birkhoff4_strerror(_lib.B4_EINVAL)


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: rejected before use


def test_negative_T_is_einval(L):
    assert L.birkhoff4_forward(FAKE, FAKE, None, -1, None) == _lib.B4_EINVAL
    assert L.birkhoff4_forward_bf16(FAKE, FAKE, None, -5, None) == _lib.B4_EINVAL
    assert L.birkhoff4_backward(None, FAKE, FAKE, FAKE, -1, None) == _lib.B4_EINVAL
    assert L.birkhoff4_forward_backward(FAKE, FAKE, FAKE, FAKE, -1, None) == _lib.B4_EINVAL
    assert L.birkhoff4_sinkhorn(FAKE, FAKE, 20, -1, None) == _lib.B4_EINVAL


def test_null_pointers_are_einval(L):
    assert L.birkhoff4_forward(None, FAKE, None, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_forward(FAKE, None, None, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_backward(None, None, FAKE, FAKE, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_backward(None, FAKE, None, FAKE, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_backward(None, FAKE, FAKE, None, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_backward_bf16(None, None, FAKE, FAKE, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_forward_backward(None, FAKE, FAKE, FAKE, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_forward_backward(FAKE, None, FAKE, FAKE, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_forward_backward_bf16(FAKE, FAKE, FAKE, None, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_sinkhorn(None, FAKE, 20, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_sinkhorn_bf16(FAKE, None, 20, 4, None) == _lib.B4_EINVAL


def test_nxn_arguments_are_checked(L):
    for n in (1, 9, 0, -3):
        assert L.birkhoff4_forward_nxn(FAKE, FAKE, None, n, 4, None) == _lib.B4_EINVAL
        assert L.birkhoff4_backward_nxn(FAKE, FAKE, FAKE, n, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_forward_nxn(FAKE, FAKE, None, 5, -1, None) == _lib.B4_EINVAL
    assert L.birkhoff4_forward_nxn(None, FAKE, None, 5, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_forward_nxn(FAKE, None, None, 5, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_backward_nxn(None, FAKE, FAKE, 5, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_backward_nxn(FAKE, None, FAKE, 5, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_backward_nxn(FAKE, FAKE, None, 5, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_forward_nxn(None, None, None, 5, 0, None) == _lib.B4_OK
    assert L.birkhoff4_backward_nxn(None, None, None, 8, 0, None) == _lib.B4_OK


def test_eot_arguments_are_checked(L):
    f32 = ctypes.c_float
    ws = ctypes.c_void_p(0x100000)
    need = L.eot_workspace_bytes(100, 200, 64, 1)
    assert need > 0 and L.eot_workspace_bytes(100, 200, 64, 3) > need
    assert L.eot_workspace_bytes(100, 200, 0, 1) == 0
    assert L.eot_workspace_bytes(100, 200, 64, 2) == 0
    assert L.eot_workspace_bytes(-1, 200, 64, 1) == 0

    def upd(nq=100, nk=200, d=64, eps=0.1, passes=1, w=ws, wb=need, ptr=FAKE):
        return L.eot_update(ptr, FAKE, FAKE, FAKE, FAKE, nq, nk, d, f32(eps), passes, w, wb, None)

    assert upd(eps=0.0) == _lib.B4_EINVAL
    assert upd(eps=-1.0) == _lib.B4_EINVAL
    assert upd(eps=float("nan")) == _lib.B4_EINVAL
    assert upd(eps=float("inf")) == _lib.B4_EINVAL
    assert upd(passes=2) == _lib.B4_EINVAL
    assert upd(d=0) == _lib.B4_EINVAL
    assert upd(nk=0) == _lib.B4_EINVAL
    assert upd(ptr=None) == _lib.B4_EINVAL
    assert upd(w=None) == _lib.B4_EINVAL
    assert upd(w=ctypes.c_void_p(0x100001)) == _lib.B4_EINVAL
    assert upd(wb=need - 1) == _lib.B4_EINVAL
    assert upd(nq=0, ptr=None, w=None) == _lib.B4_OK

    def sk(n=100, m=200, iters=3, w=ws, wb=need):
        return L.eot_sinkhorn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, n, m, 64, f32(0.1), iters, 1,
                              w, wb, None)

    assert sk(iters=-1) == _lib.B4_EINVAL
    assert sk(m=0) == _lib.B4_EINVAL
    assert sk(wb=0) == _lib.B4_EINVAL
    assert sk(iters=0) == _lib.B4_OK
    assert sk(n=0, m=0) == _lib.B4_OK


def test_mapped_arguments_are_checked(L):
    f = L.birkhoff4_forward_backward_mapped
    assert f(FAKE, FAKE, FAKE, FAKE, -1, 0, None) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 2, None) == _lib.B4_EINVAL
    assert f(None, FAKE, FAKE, FAKE, 4, 0, None) == _lib.B4_EINVAL
    assert f(FAKE, None, FAKE, FAKE, 4, 0, None) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, FAKE, None, 4, 0, None) == _lib.B4_EINVAL
    assert f(None, None, None, None, 0, 0, None) == _lib.B4_OK


def test_eot_transport_arguments_are_checked(L):
    f32 = ctypes.c_float
    need = L.eot_transport_workspace_bytes(100, 200, 64)
    assert need > 0 and L.eot_transport_workspace_bytes(100, 200, 0) == 0
    ws = ctypes.c_void_p(0x100000)

    def tr(n=100, m=200, d=64, eps=0.1, w=ws, wb=need, py=FAKE, mass=FAKE):
        return L.eot_transport(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, py, mass, None, n, m, d,
                               f32(eps), w, wb, None)

    assert tr(eps=0.0) == _lib.B4_EINVAL
    assert tr(eps=float("nan")) == _lib.B4_EINVAL
    assert tr(d=0) == _lib.B4_EINVAL
    assert tr(m=0) == _lib.B4_EINVAL
    assert tr(py=None) == _lib.B4_EINVAL
    assert tr(mass=None) == _lib.B4_EINVAL
    assert tr(w=ctypes.c_void_p(0x100080)) == _lib.B4_EINVAL
    assert tr(wb=need - 1) == _lib.B4_EINVAL
    assert tr(n=0, w=None, py=None, mass=None) == _lib.B4_OK
    assert L.eot_apply_plan_workspace_bytes(100, 200, 64, 0) == 0
    assert L.eot_apply_plan_workspace_bytes(100, 200, 64, 64) == need
    ap = L.eot_apply_plan
    assert ap(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 3, FAKE, FAKE, 100, 200, 64, f32(0.1),
              ws, need, None) == _lib.B4_EINVAL
    assert ap(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, 100, 200, 64, f32(0.1),
              ws, need, None) == _lib.B4_EINVAL


def test_eot_hvp_arguments_are_checked(L):
    """Every check runs on the host before any CUDA call."""
    f32 = ctypes.c_float
    need = L.eot_hvp_workspace_bytes(100, 200, 16)
    assert need > 0 and L.eot_hvp_workspace_bytes(100, 200, 0) == 0
    ws = ctypes.c_void_p(0x100000)

    def hvp(n=100, m=200, d=16, eps=0.1, it=10, w=ws, wb=need, v=FAKE, out=FAKE):
        return L.eot_hvp(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, v, out, n, m, d, f32(eps), it, w, wb,
                         None)

    E = _lib.B4_EINVAL
    assert hvp(eps=0.0) == E
    assert hvp(eps=float("inf")) == E
    assert hvp(it=-1) == E
    assert hvp(it=100001) == E
    assert hvp(d=0) == E
    assert hvp(m=0) == E
    assert hvp(v=None) == E
    assert hvp(out=None) == E
    assert hvp(w=ctypes.c_void_p(0x100040)) == E   # not 256-byte aligned
    assert hvp(wb=need - 1) == E
    assert hvp(n=0, w=None, out=None) == _lib.B4_OK  # nothing to do


def test_bad_options_are_einval(L):
    def opts(**kw):
        o = _lib.Opts(in_dtype=0, out_dtype=0, max_evals=0, tol=0.0)
        for k, v in kw.items():
            setattr(o, k, v)
        return ctypes.byref(o)

    f = L.birkhoff4_forward_ex
    assert f(FAKE, FAKE, None, 4, None, None) == _lib.B4_EINVAL  # NULL options
    assert f(FAKE, FAKE, None, 4, opts(in_dtype=2), None) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, None, 4, opts(out_dtype=-1), None) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, None, 4, opts(max_evals=-1), None) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, None, 4, opts(max_evals=1025), None) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, None, 4, opts(tol=-1.0), None) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, None, 4, opts(tol=float("nan")), None) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, None, 4, opts(tol=float("inf")), None) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, None, 4, opts(schedule=4), None) == _lib.B4_EINVAL
    # four lanes per token: the fp32 forward only
    assert f(FAKE, FAKE, None, 4, opts(schedule=3, in_dtype=1, out_dtype=1), None) == _lib.B4_ENOTIMPL
    assert f(FAKE, FAKE, None, 4, opts(schedule=-1), None) == _lib.B4_EINVAL
    # the fused pass with options: same checks, one dtype for everything
    g = L.birkhoff4_forward_backward_ex
    assert g(FAKE, FAKE, FAKE, FAKE, 4, None, None) == _lib.B4_EINVAL
    assert g(FAKE, FAKE, FAKE, FAKE, 4, opts(out_dtype=1), None) == _lib.B4_EINVAL
    assert g(FAKE, FAKE, FAKE, FAKE, 4, opts(schedule=7), None) == _lib.B4_EINVAL
    assert g(FAKE, FAKE, FAKE, FAKE, 4, opts(schedule=3), None) == _lib.B4_ENOTIMPL
    assert g(FAKE, FAKE, FAKE, FAKE, 4, opts(max_evals=2000), None) == _lib.B4_EINVAL
    assert g(FAKE, FAKE, FAKE, FAKE, -1, opts(), None) == _lib.B4_EINVAL
    assert g(None, None, None, None, 0, opts(), None) == _lib.B4_OK
    assert g(None, FAKE, FAKE, FAKE, 4, opts(), None) == _lib.B4_EINVAL


def test_host_streaming_argument_checks(L):
    f = L.birkhoff4_forward_backward_host
    streams = (ctypes.c_void_p * 2)(None, None)
    ws = FAKE
    assert f(FAKE, FAKE, FAKE, FAKE, -1, 0, ws, 1 << 20, streams, 2) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 7, ws, 1 << 20, streams, 2) == _lib.B4_EINVAL  # dtype
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 0, ws, 1 << 20, streams, 0) == _lib.B4_EINVAL  # nstreams
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 0, ws, 1 << 20, streams, 17) == _lib.B4_EINVAL
    assert f(None, FAKE, FAKE, FAKE, 4, 0, ws, 1 << 20, streams, 2) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, FAKE, None, 4, 0, ws, 1 << 20, streams, 2) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 0, None, 1 << 20, streams, 2) == _lib.B4_EINVAL
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 0, ws, 1 << 20, None, 2) == _lib.B4_EINVAL
    # a workspace too small for one token per slot (2 slots x 4 x 64 B)
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 0, ws, 511, streams, 2) == _lib.B4_EINVAL
    assert f(None, None, None, None, 0, 0, None, 0, streams, 2) == _lib.B4_OK


def test_negative_iters_is_einval(L):
    assert L.birkhoff4_sinkhorn(FAKE, FAKE, -1, 4, None) == _lib.B4_EINVAL
    assert L.birkhoff4_sinkhorn_bf16(FAKE, FAKE, -3, 4, None) == _lib.B4_EINVAL


def test_empty_batch_is_a_no_op(L):
    # T = 0 returns before any CUDA call, even with NULL pointers
    assert L.birkhoff4_forward(None, None, None, 0, None) == _lib.B4_OK
    assert L.birkhoff4_forward_bf16(None, None, None, 0, None) == _lib.B4_OK
    assert L.birkhoff4_backward(None, None, None, None, 0, None) == _lib.B4_OK
    assert L.birkhoff4_backward_bf16(None, None, None, None, 0, None) == _lib.B4_OK
    assert L.birkhoff4_forward_backward(None, None, None, None, 0, None) == _lib.B4_OK
    assert L.birkhoff4_sinkhorn(None, None, 20, 0, None) == _lib.B4_OK
    o = _lib.Opts(in_dtype=1, out_dtype=0, max_evals=0, tol=0.0)
    assert L.birkhoff4_forward_ex(None, None, None, 0, ctypes.byref(o), None) == _lib.B4_OK


def test_diagnostic_argument_checks(L):
    assert L.birkhoff4_device_status(None, 0) == _lib.B4_EINVAL
    assert L.birkhoff4_selftest_wait_timeout(0) == _lib.B4_EINVAL
    assert L.birkhoff4_selftest_wait_timeout(2_000_000_000) == _lib.B4_EINVAL
    out = (ctypes.c_float * 2)()
    assert L.birkhoff4_mufu_probe(None, 1, 1, None) == _lib.B4_EINVAL
    assert L.birkhoff4_mufu_probe(out, 0, 1, None) == _lib.B4_EINVAL
    assert L.birkhoff4_mufu_probe(out, 1, 0, None) == _lib.B4_EINVAL
    assert L.birkhoff4_last_cuda_error() == 0


def test_python_binding_refuses_cpu_tensors():
    import torch

    import birkhoff_projection_gb300 as b4

    x = torch.zeros(3, 4, 4)
    with pytest.raises(ValueError):
        b4.forward(x)
    with pytest.raises(ValueError):
        b4.backward(x, P=x)
    with pytest.raises(ValueError):
        b4.sinkhorn(x)


def test_missing_library_raises(monkeypatch):
    """With no built library the binding raises instead of computing
    anything another way: there is no fallback path."""
    from birkhoff_projection_gb300 import _build

    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_build, "build", lambda *a, **k: "/nonexistent/libbirkhoff4.so")
    with pytest.raises(_lib.Birkhoff4Error):
        _lib.lib()
