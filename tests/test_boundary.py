"""C-ABI boundary on the CPU: the library builds, loads, exports every symbol
include/fa.h declares, and rejects invalid arguments on the host before any
CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

from exact_attention_48_gb300 import build as fa_build
from exact_attention_48_gb300.binding import library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]

FA_OK, FA_ERR_INVALID_ARGUMENT, FA_ERR_UNSUPPORTED, FA_ERR_WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return library()


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        # every exported declaration starts with FA_API: "FA_API <type> <name>("
        names += re.findall(r"^\s*FA_API\s+[^(;]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_device_status", "fa_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported by libfa.so"


def test_status_strings(lib):
    for code in range(6):
        s = lib.fa_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.fa_status_string(99).decode() == "unknown status"


# A fake, 256-byte-aligned, non-null device address: validation must reject
# each call below before it touches it (or any CUDA API).
FAKE = 1 << 40


def _fwd(lib, *, q=FAKE, k=FAKE + (1 << 30), v=FAKE + (2 << 30), o=FAKE + (3 << 30), lse=FAKE + (4 << 30),
         B=1, H=2, N=128, d=64, causal=0, scale=0.125):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), FA_ERR_INVALID_ARGUMENT),
    (dict(H=-1), FA_ERR_INVALID_ARGUMENT),
    (dict(N=0), FA_ERR_INVALID_ARGUMENT),
    (dict(d=0), FA_ERR_INVALID_ARGUMENT),
    (dict(d=96), FA_ERR_UNSUPPORTED),
    (dict(d=256), FA_ERR_UNSUPPORTED),
    (dict(causal=2), FA_ERR_INVALID_ARGUMENT),
    (dict(scale=float("nan")), FA_ERR_INVALID_ARGUMENT),
    (dict(scale=float("inf")), FA_ERR_INVALID_ARGUMENT),
    (dict(q=0), FA_ERR_INVALID_ARGUMENT),
    (dict(lse=0), FA_ERR_INVALID_ARGUMENT),
    (dict(k=FAKE + 8), FA_ERR_INVALID_ARGUMENT),          # misaligned
    (dict(o=FAKE + 64), FA_ERR_INVALID_ARGUMENT),         # output overlaps q
    (dict(B=1 << 14, H=1 << 10, N=1 << 10), FA_ERR_INVALID_ARGUMENT),  # 2^40 elements: beyond TMA's strides
    (dict(B=1 << 16, H=1 << 16, N=1), FA_ERR_INVALID_ARGUMENT),         # 2^32 heads: beyond a launch grid
    (dict(B=1 << 15, H=1 << 16, N=1), FA_ERR_INVALID_ARGUMENT),         # 2^31 heads: one past a launch grid
])
def test_fwd_rejects(lib, kw, code):
    assert _fwd(lib, **kw) == code


def _bwd(lib, *, ws=None, ws_bytes=0, dq=FAKE + (10 << 30), B=1, H=2, N=128, d=64, causal=0, scale=0.125,
         lse=FAKE + (5 << 30)):
    return lib.fa_bwd(FAKE, FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (3 << 30), FAKE + (4 << 30), lse,
                      dq, FAKE + (11 << 30), FAKE + (12 << 30), B, H, N, d, causal, scale, ws, ws_bytes, None)


def test_bwd_rejects(lib):
    assert _bwd(lib, d=80) == FA_ERR_UNSUPPORTED
    assert _bwd(lib, N=-3) == FA_ERR_INVALID_ARGUMENT
    assert _bwd(lib, scale=float("nan")) == FA_ERR_INVALID_ARGUMENT
    assert _bwd(lib, dq=FAKE + 16) == FA_ERR_INVALID_ARGUMENT        # dq overlaps q
    assert _bwd(lib, lse=0) == FA_ERR_INVALID_ARGUMENT
    need = lib.fa_bwd_workspace_bytes(1, 2, 128, 64)
    assert _bwd(lib, ws=FAKE + (20 << 30), ws_bytes=need - 1) == FA_ERR_WORKSPACE
    assert _bwd(lib, ws=FAKE + (20 << 30) + 16, ws_bytes=need) == FA_ERR_INVALID_ARGUMENT  # not 256-aligned
    assert _bwd(lib, ws=FAKE + (3 << 30), ws_bytes=need) == FA_ERR_INVALID_ARGUMENT        # overlaps o


def test_sizes_beyond_2_31_elements_are_accepted(lib):
    """Tensors of 2^31 elements and more pass the host checks (element
    offsets are 64-bit): the workspace query answers for them.  2^21 heads
    of 1032 rows at d = 128 are 2.8e11 elements per tensor."""
    r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for B, H, N, d in [(1 << 11, 1 << 10, 1032, 128), (1, 1, (1 << 24) + 3, 128), (1 << 16, 1 << 8, 128, 64)]:
        assert B * H * N * d >= 1 << 31
        Np = (N + 127) // 128 * 128
        assert lib.fa_bwd_workspace_bytes(B, H, N, d) == 2 * r256(B * H * Np * 4)
    assert lib.fa_bwd_workspace_bytes(1 << 16, 1 << 16, 1, 64) == 0     # 2^32 heads: rejected


def test_workspace_bytes(lib):
    def r256(x):
        return (x + 255) // 256 * 256
    for B, H, N, d in [(1, 2, 128, 64), (2, 16, 8192, 128), (1, 1, 1, 64), (3, 5, 129, 128)]:
        Np = (N + 127) // 128 * 128
        want = 2 * r256(B * H * Np * 4)
        assert lib.fa_bwd_workspace_bytes(B, H, N, d) == want
    # linear in N (the pages' O(N) memory claim), not quadratic
    a = lib.fa_bwd_workspace_bytes(1, 1, 4096, 128)
    b = lib.fa_bwd_workspace_bytes(1, 1, 8192, 128)
    assert b == 2 * a
    assert lib.fa_bwd_workspace_bytes(1, 1, 128, 96) == 0
    assert lib.fa_bwd_workspace_bytes(0, 1, 128, 64) == 0


def _s(*v):
    return (ctypes.c_int64 * 3)(*v)


def _fwd_strided(lib, *, qs=None, os_=None, o=FAKE + (3 << 30), B=1, H=2, N=128, d=64):
    c = _s(H * N * d, N * d, d)
    return lib.fa_fwd_strided(FAKE, qs or c, FAKE + (1 << 30), c, FAKE + (2 << 30), c, o, os_ or c,
                              FAKE + (4 << 30), B, H, N, d, 0, 0.125, None)


def test_fwd_strided_rejects(lib):
    H, N, d = 2, 128, 64
    assert _fwd_strided(lib, qs=_s(H * N * d, N * d, d + 4)) == FA_ERR_INVALID_ARGUMENT   # not a multiple of 8
    assert _fwd_strided(lib, qs=_s(H * N * d, 0, d)) == FA_ERR_INVALID_ARGUMENT           # zero stride, extent 2
    assert _fwd_strided(lib, os_=_s(H * N * d, N * d, 8)) == FA_ERR_INVALID_ARGUMENT      # rows of o overlap
    assert _fwd_strided(lib, os_=_s(H * N * d, N * d // 2, d)) == FA_ERR_INVALID_ARGUMENT  # heads of o overlap
    assert _fwd_strided(lib, o=FAKE + (1 << 30) + 256) == FA_ERR_INVALID_ARGUMENT        # o inside k
    assert lib.fa_fwd_strided(FAKE, None, FAKE, None, FAKE, None, FAKE, None, FAKE, 1, 2, 128, 64, 0, 0.125,
                              None) == FA_ERR_INVALID_ARGUMENT                             # no strides
    assert _fwd_strided(lib, d=96) == FA_ERR_UNSUPPORTED


def test_bwd_strided_rejects(lib):
    H, N, d = 2, 128, 64
    c = _s(H * N * d, N * d, d)

    def call(dq=FAKE + (10 << 30), dqs=c, dk=FAKE + (11 << 30), dks=c):
        return lib.fa_bwd_strided(FAKE, c, FAKE + (1 << 30), c, FAKE + (2 << 30), c, FAKE + (3 << 30), c,
                                  FAKE + (4 << 30), c, FAKE + (5 << 30), dq, dqs, dk, dks, FAKE + (12 << 30), c,
                                  1, H, N, d, 0, 0.125, None, 0, None)
    assert call(dk=FAKE + (10 << 30) + 4096) == FA_ERR_INVALID_ARGUMENT                  # dk overlaps dq
    assert call(dks=_s(H * N * d, d, d)) == FA_ERR_INVALID_ARGUMENT                      # dk rows collide
    assert call(dq=FAKE + (2 << 30)) == FA_ERR_INVALID_ARGUMENT                          # dq is v
    assert call(dqs=_s(H * N * d, N * d, 12)) == FA_ERR_INVALID_ARGUMENT                 # not a multiple of 8
    # slices of one packed [B, N, 3, H, d] buffer: dk one head (d elements)
    # after dq collides with dq's second head (a gap of H*d would not)
    packed = _s(N * 3 * H * d, d, 3 * H * d)
    assert call(dqs=packed, dk=FAKE + (10 << 30) + 2 * d, dks=packed) == FA_ERR_INVALID_ARGUMENT


def test_varlen_rejects(lib):
    H, T, d = 2, 300, 64
    c = (ctypes.c_int64 * 2)(H * d, d)

    def fwd(cu=FAKE + (6 << 30), qs=c, B=3, maxlen=200, o=FAKE + (3 << 30)):
        return lib.fa_fwd_varlen(FAKE, qs, FAKE + (1 << 30), c, FAKE + (2 << 30), c, o, c, FAKE + (4 << 30), cu,
                                 B, H, T, maxlen, d, 1, 0.125, None)
    assert fwd(cu=None) == FA_ERR_INVALID_ARGUMENT
    assert fwd(cu=FAKE + (6 << 30) + 2) == FA_ERR_INVALID_ARGUMENT                        # misaligned offsets
    assert fwd(B=0) == FA_ERR_INVALID_ARGUMENT
    assert fwd(maxlen=0) == FA_ERR_INVALID_ARGUMENT
    assert fwd(qs=(ctypes.c_int64 * 2)(H * d + 4, d)) == FA_ERR_INVALID_ARGUMENT          # row stride not x8
    assert fwd(o=FAKE + (2 << 30) + 1024) == FA_ERR_INVALID_ARGUMENT                     # o inside v
    assert lib.fa_bwd_varlen(FAKE, c, FAKE, c, FAKE, c, FAKE, c, FAKE, c, FAKE, FAKE, c, FAKE, c, FAKE, c, None,
                             3, H, T, 200, d, 0, 0.125, None, 0, None) == FA_ERR_INVALID_ARGUMENT


def test_decode_workspace_bytes(lib):
    # one 128-key tile per head: a single chunk, nothing to merge
    assert lib.fa_decode_workspace_bytes(8, 32, 1, 128, 64) == 0
    # a long cache over few heads: several chunks, partial O (fp32) + lse per chunk
    need = lib.fa_decode_workspace_bytes(1, 2, 2, 40000, 128)
    assert need > 0 and need % 256 == 0
    assert lib.fa_decode_workspace_bytes(0, 1, 1, 128, 64) == 0       # invalid shape
    assert lib.fa_decode_workspace_bytes(1, 1, 9, 4096, 64) == 0      # Nq above 8
    assert lib.fa_decode_workspace_bytes(1, 1, 1, 4096, 96) == 0      # unsupported d


def test_decode_rejects(lib):
    B, H, Nq, Nk, d = 2, 2, 2, 1000, 64
    cq = _s(H * Nq * d, Nq * d, d)
    ck = _s(H * Nk * d, Nk * d, d)
    need = lib.fa_decode_workspace_bytes(B, H, Nq, Nk, d)

    def call(q=FAKE, qs=cq, k=FAKE + (1 << 30), ks=ck, v=FAKE + (2 << 30), o=FAKE + (3 << 30), os_=cq,
             lse=FAKE + (4 << 30), cl=None, b=B, nq=Nq, nk=Nk, dd=d, causal=0, scale=0.125, ws=None, ws_bytes=0):
        return lib.fa_fwd_decode(q, qs, k, ks, v, ks, o, os_, lse, cl, b, H, nq, nk, dd, causal, scale, ws,
                                 ws_bytes, None)
    assert call(nq=0) == FA_ERR_INVALID_ARGUMENT
    assert call(nq=9) == FA_ERR_INVALID_ARGUMENT
    assert call(nk=0) == FA_ERR_INVALID_ARGUMENT
    assert call(b=0) == FA_ERR_INVALID_ARGUMENT
    assert call(dd=96) == FA_ERR_UNSUPPORTED
    assert call(causal=2) == FA_ERR_INVALID_ARGUMENT
    assert call(scale=float("nan")) == FA_ERR_INVALID_ARGUMENT
    assert call(q=0) == FA_ERR_INVALID_ARGUMENT
    assert call(lse=0) == FA_ERR_INVALID_ARGUMENT
    assert call(cl=FAKE + (6 << 30) + 2) == FA_ERR_INVALID_ARGUMENT                   # misaligned lengths
    assert call(qs=None) == FA_ERR_INVALID_ARGUMENT
    assert call(ks=_s(H * Nk * d, Nk * d, d + 4)) == FA_ERR_INVALID_ARGUMENT           # row stride not x8
    assert call(os_=_s(H * Nq * d, Nq * d, 8)) == FA_ERR_INVALID_ARGUMENT              # rows of o overlap
    assert call(o=FAKE + 64) == FA_ERR_INVALID_ARGUMENT                               # o overlaps q
    assert call(o=FAKE + (1 << 30) + 4096) == FA_ERR_INVALID_ARGUMENT                 # o inside the key cache
    assert call(lse=FAKE + (2 << 30) + 256) == FA_ERR_INVALID_ARGUMENT                # lse inside the value cache
    assert call(lse=FAKE + (3 << 30) + 16) == FA_ERR_INVALID_ARGUMENT                 # lse overlaps o
    assert call(cl=FAKE + (3 << 30)) == FA_ERR_INVALID_ARGUMENT                       # lengths inside o
    if need:
        assert call(ws=FAKE + (20 << 30), ws_bytes=need - 1) == FA_ERR_WORKSPACE
        assert call(ws=FAKE + (20 << 30) + 16, ws_bytes=need) == FA_ERR_INVALID_ARGUMENT
        assert call(ws=FAKE + (1 << 30), ws_bytes=need) == FA_ERR_INVALID_ARGUMENT    # workspace inside k


def test_fp8_rejects(lib):
    def call(q=FAKE, k=FAKE + (1 << 30), v=FAKE + (2 << 30), o=FAKE + (3 << 30), lse=FAKE + (4 << 30),
             sq=0.01, sk=0.01, sv=0.01, B=1, H=2, N=256, d=128, causal=0, scale=0.088):
        return lib.fa_fwd_fp8(q, k, v, sq, sk, sv, o, lse, B, H, N, d, causal, scale, None)
    assert call(d=64) == FA_ERR_UNSUPPORTED
    assert call(d=96) == FA_ERR_UNSUPPORTED
    assert call(N=0) == FA_ERR_INVALID_ARGUMENT
    assert call(causal=3) == FA_ERR_INVALID_ARGUMENT
    assert call(sq=float("inf")) == FA_ERR_INVALID_ARGUMENT
    assert call(sv=float("nan")) == FA_ERR_INVALID_ARGUMENT
    assert call(scale=float("nan")) == FA_ERR_INVALID_ARGUMENT
    assert call(k=0) == FA_ERR_INVALID_ARGUMENT
    assert call(v=FAKE + (2 << 30) + 8) == FA_ERR_INVALID_ARGUMENT          # misaligned
    assert call(o=FAKE + 1024) == FA_ERR_INVALID_ARGUMENT                    # o overlaps q
    assert call(lse=FAKE + (3 << 30) + 4096) == FA_ERR_INVALID_ARGUMENT      # lse inside o
