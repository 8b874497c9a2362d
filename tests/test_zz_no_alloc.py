"""fa_bwd_noalloc, the backward pass that allocates nothing.

Some callers cannot allocate device memory (a framework's memory manager
owns every allocation, or the process must not allocate once it runs), so
they can neither give fa_bwd a workspace nor let it take one.
fa_bwd_noalloc serves them from a fixed array inside the library.  This
file is collected last on purpose, and must pass both alone in a fresh
process and after every other test.
"""
import ctypes
import math

import pytest
import torch

from exact_attention_48_gb300 import build as fa_build
from exact_attention_48_gb300.binding import fa_bwd, fa_bwd_noalloc, fa_fwd, fa_device_status, library
from exact_attention_48_gb300.inputs import draw_shape
from parity import check_grad

FA_ERR_WORKSPACE = 3


def _raw_noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, causal, scale):
    """The C entry point itself, called through ctypes with raw pointers."""
    B, H, N, d = q.shape
    f = lib.fa_bwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
             dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, int(causal), float(scale),
             torch.cuda.current_stream().cuda_stream)


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 300, 128, True), (1, 4, 1000, 64, False)])
def test_noalloc_matches_fa_bwd_twice(B, H, N, d, causal):
    fa_build.build()
    lib = library()
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = draw_shape(B, H, N, d, 77, 1.0, "cuda", torch.bfloat16)
    o, lse = fa_fwd(q, k, v, causal, scale)
    ref = fa_bwd(q, k, v, o, do, lse, causal, scale)
    torch.cuda.synchronize()
    for call in range(2):   # two calls in a row share (and reuse) the fixed array
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = _raw_noalloc(lib, q, k, v, o, do, lse, *got, causal, scale)
        assert rc == 0, f"call {call}: status {rc}"
        assert fa_device_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            check_grad(g, r, name, f"fa_bwd_noalloc call {call}")
    # the Python binding of the same name gives the same result
    got = fa_bwd_noalloc(q, k, v, o, do, lse, causal, scale)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check_grad(g, r, name, "fa_bwd_noalloc binding")


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_the_array():
    lib = library()
    q = torch.empty(16, device="cuda", dtype=torch.bfloat16)
    # B*H*Np = 64 * 32768 padded rows need 16 MiB > 8 MiB: rejected on the host, nothing launched
    B, H, N, d = 4, 16, 32768, 64
    f = lib.fa_bwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p]
    f.restype = ctypes.c_int
    base = q.data_ptr()
    ptrs = [base + (i << 36) for i in range(9)]   # never dereferenced: the size check comes first
    rc = f(*ptrs, B, H, N, d, 0, 0.125, None)
    assert rc == FA_ERR_WORKSPACE
