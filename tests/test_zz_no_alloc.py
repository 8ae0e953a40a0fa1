"""The allocation-free entry point birkhoff4_forward_backward_host_static.

Some callers cannot allocate device memory: cudaMalloc synchronises the
device, their device memory may belong to another framework's allocator, or
their host forbids device allocations.  This entry point streams host tokens
through the GPU using a static staging array inside the library instead of a
caller-provided workspace.  The test calls it through the C ABI and checks
its results against the workspace-based entry point
(birkhoff4_forward_backward_host) on two calls in a row, the second with
other tokens, so stale contents of the shared array would show; it also
checks that a chunk larger than the array is refused.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

from birkhoff_projection_gb300 import _lib, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CODES = {torch.float32: _lib.B4_F32, torch.bfloat16: _lib.B4_BF16}


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _handles(streams):
    arr = (ctypes.c_void_p * len(streams))(*[s.cuda_stream for s in streams])
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def _host(T, seed, dtype):
    x = workloads.normal(T, 1.0, seed=seed).to(dtype).pin_memory()
    g = workloads.normal(T, 1.0, seed=seed + 1).to(dtype).pin_memory()
    return x, g


@pytest.mark.parametrize("chunk_tokens", [0, 4097])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_static_scratch_entry_matches_workspace_entry(dtype, chunk_tokens):
    """chunk_tokens 0 takes the largest chunk that fits the array; 4097
    gives many small chunks with a ragged last one."""
    L = _lib.lib()
    torch.cuda.init()
    T = 300001  # several chunks and a ragged tail
    streams = [torch.cuda.Stream(device=DEV) for _ in range(2)]
    arr, hp = _handles(streams)
    ws = torch.empty(2 * 4 * 65536 * 16 * torch.empty((), dtype=dtype).element_size(),
                     dtype=torch.uint8, device=DEV)
    for call in range(2):
        X, G = _host(T, 100 + 10 * call, dtype)
        P1, dX1 = torch.empty_like(X).pin_memory(), torch.empty_like(X).pin_memory()
        P2, dX2 = torch.empty_like(X).pin_memory(), torch.empty_like(X).pin_memory()
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        st = L.birkhoff4_forward_backward_host_static(_p(X), _p(G), _p(P1), _p(dX1), T,
                                                      CODES[dtype], chunk_tokens, hp, len(streams))
        assert st == _lib.B4_OK, L.birkhoff4_strerror(st)
        torch.cuda.synchronize()
        if call == 1:
            # after the first call (which may load the module and reserve the
            # array) a call takes no device memory
            assert torch.cuda.mem_get_info()[0] == free0
        st = L.birkhoff4_forward_backward_host(_p(X), _p(G), _p(P2), _p(dX2), T, CODES[dtype],
                                               _p(ws), ws.numel(), hp, len(streams))
        assert st == _lib.B4_OK, L.birkhoff4_strerror(st)
        torch.cuda.synchronize()
        # the same kernels on the same tokens: identical to the last bit,
        # whatever the chunking
        assert torch.equal(P1, P2) and torch.equal(dX1, dX2)
        assert torch.isfinite(P1.float()).all() and torch.isfinite(dX1.float()).all()
    del arr


def test_static_scratch_refuses_oversized_chunks():
    L = _lib.lib()
    streams = [torch.cuda.Stream(device=DEV) for _ in range(2)]
    arr, hp = _handles(streams)
    fake = ctypes.c_void_p(0x10000)  # never touched: refused before any copy
    # 32 MiB / (2 streams x 4 arrays x 64 B) = 65536 fp32 tokens per chunk
    st = L.birkhoff4_forward_backward_host_static(fake, fake, fake, fake, 10, _lib.B4_F32,
                                                  65537, hp, 2)
    assert st == _lib.B4_ESCRATCH
    assert b"static scratch" in L.birkhoff4_strerror(st)
    st = L.birkhoff4_forward_backward_host_static(None, None, None, None, 0, _lib.B4_F32, 0, hp, 2)
    assert st == _lib.B4_OK
    del arr
