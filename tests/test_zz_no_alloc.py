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

FA_ERR_WORKSPACE = 3
FA_ERR_INVALID_ARGUMENT = 1
CU_MEMPOOL_ATTR_USED_MEM_CURRENT = 7
CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8


def _raw_noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, causal, scale):
    """The C entry point itself, called through ctypes with raw pointers."""
    B, H, N, d = q.shape
    f = lib.fa_bwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
             dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, int(causal), float(scale),
             torch.cuda.current_stream().cuda_stream)


class _DefaultPool:
    """The device's default stream-ordered memory pool (the one
    cudaMallocAsync draws from), read through the driver API."""

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def get(self, attr):
        v = ctypes.c_uint64()
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
        return v.value

    def reset_high(self):
        zero = ctypes.c_uint64(0)   # the high watermark can only be reset to zero (i.e. to the current use)
        assert self.cu.cuMemPoolSetAttribute(self.pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(zero)) == 0


@pytest.mark.gpu
def test_noalloc_matches_fa_bwd_over_changing_shapes():
    """Calls in a row with different shapes: a first one, a larger one whose
    N is not a multiple of 128 (more padded rows of the scratch are used),
    then a smaller causal one that runs over the larger call's leftovers,
    and the first shape again.  Each call gives exactly fa_bwd's gradients
    (both are deterministic), and none takes memory from the default pool
    or from torch's allocator."""
    fa_build.build()
    lib = library()
    pool = _DefaultPool()
    shapes = [(2, 3, 300, 128, True), (3, 5, 1000, 64, False), (1, 2, 200, 128, True), (2, 3, 300, 128, True)]
    for call, (B, H, N, d, causal) in enumerate(shapes):
        scale = 1.0 / math.sqrt(d)
        q, k, v, do = draw_shape(B, H, N, d, 77 + call, 1.0, "cuda", torch.bfloat16)
        o, lse = fa_fwd(q, k, v, causal, scale)
        ref = fa_bwd(q, k, v, o, do, lse, causal, scale)
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        torch.cuda.synchronize()
        pool.reset_high()
        used0 = pool.get(CU_MEMPOOL_ATTR_USED_MEM_CURRENT)
        torch_used0 = torch.cuda.memory_allocated()
        rc = _raw_noalloc(lib, q, k, v, o, do, lse, *got, causal, scale)
        assert rc == 0, f"call {call}: status {rc}"
        assert fa_device_status() == 0
        assert pool.get(CU_MEMPOOL_ATTR_USED_MEM_HIGH) <= used0, f"call {call} took memory from the default pool"
        assert torch.cuda.memory_allocated() == torch_used0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(g, r), f"call {call} {(B, H, N, d, causal)}: {name} differs from fa_bwd"
    # the Python binding of the same name gives the same result
    got = fa_bwd_noalloc(q, k, v, o, do, lse, causal, scale)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert torch.equal(g, r), f"binding: {name} differs from fa_bwd"


@pytest.mark.gpu
def test_noalloc_rejects_before_any_device_work():
    lib = library()
    q = torch.empty(16, device="cuda", dtype=torch.bfloat16)
    f = lib.fa_bwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p]
    f.restype = ctypes.c_int
    base = q.data_ptr()
    ptrs = [base + (i << 36) for i in range(9)]   # never dereferenced: the host checks come first
    # B*H*Np = 64 * 32768 padded rows need 16 MiB > 8 MiB
    assert f(*ptrs, 4, 16, 32768, 64, 0, 0.125, None) == FA_ERR_WORKSPACE
    # a bad causal flag or a non-finite scale
    assert f(*ptrs, 1, 1, 128, 64, 2, 0.125, None) == FA_ERR_INVALID_ARGUMENT
    assert f(*ptrs, 1, 1, 128, 64, 0, float("nan"), None) == FA_ERR_INVALID_ARGUMENT
