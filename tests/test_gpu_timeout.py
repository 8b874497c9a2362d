"""The bounded pipeline waits: a kernel that gives up records
FA_ERR_DEVICE_TIMEOUT and the wait site, returns, and leaves the context
usable.

The failure is made without faulting or hanging anything: a test build of
the library (build.py's "stalltest" variant, its own .so under _build/)
shortens every wait to a millisecond and leaves out
the forward's first V load, so the MMA thread's wait for it runs out.  The
kernel then raises its abort flag, drains the copies and products it
issued, frees its TMEM and exits; fa_device_status reports the timeout
once and clears it.  The product library in the same process keeps
working.
"""
import ctypes
import math

import pytest
import torch

import oracle
from exact_attention_48_gb300 import build as fa_build
from exact_attention_48_gb300 import fa_device_status, fa_fwd
from exact_attention_48_gb300.inputs import draw_shape
from parity import check_lse, check_o

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_DEVICE_TIMEOUT = 0, 5


def _stall_lib():
    lib = ctypes.CDLL(fa_build.build_variant("stalltest"))
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.fa_fwd.restype = i
    lib.fa_device_status.argtypes = [vp]
    lib.fa_device_status.restype = i
    lib.fa_debug_last_wait_site.argtypes = []
    lib.fa_debug_last_wait_site.restype = i
    return lib


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 256, 128), (1, 160, 256, 64)])
def test_timeout_is_reported_and_the_context_survives(B, H, N, d):
    """(1, 1, 256, 128): one CTA, two key blocks.  (1, 160, 256, 64): more
    tiles than SMs, so persistent CTAs that would each walk one or two
    tiles; every one gives up in its first tile and takes no other."""
    scale = 1 / math.sqrt(d)
    q, k, v, _ = draw_shape(B, H, N, d, 61, 1.0, "cuda", torch.bfloat16)
    lib = _stall_lib()
    stream = torch.cuda.current_stream().cuda_stream
    for attempt in range(2):          # the path can be taken again
        o = torch.zeros_like(q)
        lse = torch.zeros(B, H, N, device="cuda", dtype=torch.float32)
        rc = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        B, H, N, d, 0, scale, stream)
        assert rc == FA_OK, f"launch status {rc}"
        torch.cuda.synchronize()      # the kernel has returned: no fault, no hang
        site = lib.fa_debug_last_wait_site()
        assert lib.fa_device_status(stream) == FA_ERR_DEVICE_TIMEOUT, f"attempt {attempt}"
        assert site > 0, f"attempt {attempt}: no wait site recorded"
        assert lib.fa_device_status(stream) == FA_OK      # reported once, then cleared
        assert lib.fa_debug_last_wait_site() == 0
        # the stopped kernel wrote no output row
        assert bool((lse == 0).all()) and bool((o == 0).all())
    # the product library, same process and context: a normal call
    o, lse = fa_fwd(q, k, v, False, scale)
    assert fa_device_status() == FA_OK
    o_ref, lse_ref = oracle.fwd(q[0, 0], k[0, 0], v[0, 0], False, scale)
    check_o(o[0, 0], o_ref, "after the timeout")
    check_lse(lse[0, 0], lse_ref, "after the timeout")
