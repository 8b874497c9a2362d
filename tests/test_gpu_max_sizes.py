"""Large-extent cases: many heads (a grid of tens of thousands of CTAs),
tensors of more than 2^31 elements, and a key/value cache of a million keys
with a ragged last tile for decode, each checked on sampled rows against
the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_48_gb300 import fa_bwd, fa_device_status, fa_fwd, fa_fwd_decode, fa_decode_workspace_bytes
from exact_attention_48_gb300.inputs import draw_shape
from parity import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


def test_many_heads_short_sequences():
    """B*H = 32768 heads of 130 rows (d 64): 32768 forward CTAs, ragged last
    block in every head; sampled heads forward and backward."""
    B, H, N, d = 256, 128, 130, 64
    q, k, v, do = draw_shape(B, H, N, d, 91, 1.0, "cuda", torch.bfloat16)
    o, lse = fa_fwd(q, k, v, True)
    dq, dk, dv = fa_bwd(q, k, v, o, do, lse, True)
    assert fa_device_status() == 0
    scale = 1 / math.sqrt(d)
    for b, h in ((0, 0), (B - 1, H - 1), (137, 61)):
        o_ref, lse_ref = oracle.fwd(q[b, h], k[b, h], v[b, h], True, scale)
        check_o(o[b, h], o_ref, f"head ({b},{h})")
        check_lse(lse[b, h], lse_ref, f"head ({b},{h})")
        refs = oracle.bwd(q[b, h], k[b, h], v[b, h], do[b, h], True, scale)
        for name, g, r in zip(("dq", "dk", "dv"), (dq[b, h], dk[b, h], dv[b, h]), refs):
            check_grad(g, r, name, f"head ({b},{h})")


def test_tensors_beyond_2_31_elements():
    """B*H = 16384 heads of N = 1032 rows at d = 128: 2.16e9 elements per
    tensor (4.3 GB of bf16, more than 2^31 elements), forward and backward.
    The heads checked against the oracle include the first, the one that
    straddles element 2^31, the first one wholly past it and the last; all
    outputs are finite."""
    B, H, N, d = 64, 256, 1032, 128
    assert B * H * N * d > 1 << 31
    scale = 1 / math.sqrt(d)
    q, k, v, do = draw_shape(B, H, N, d, 93, 1.0, "cuda", torch.bfloat16)
    o, lse = fa_fwd(q, k, v, False)
    dq, dk, dv = fa_bwd(q, k, v, o, do, lse, False)
    assert fa_device_status() == 0
    straddle = (1 << 31) // (N * d)           # head whose elements cross index 2^31
    assert straddle * N * d < 1 << 31 < (straddle + 1) * N * d
    for hh in (0, straddle, straddle + 1, B * H - 1):
        b, h = divmod(hh, H)
        o_ref, lse_ref = oracle.fwd(q[b, h], k[b, h], v[b, h], False, scale)
        check_o(o[b, h], o_ref, f"head {hh}")
        check_lse(lse[b, h], lse_ref, f"head {hh}")
        refs = oracle.bwd(q[b, h], k[b, h], v[b, h], do[b, h], False, scale)
        for name, g, r in zip(("dq", "dk", "dv"), (dq[b, h], dk[b, h], dv[b, h]), refs):
            check_grad(g, r, name, f"head {hh}")
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())


def test_decode_million_keys():
    """Two heads against a cache of 2^20 + 37 keys (a ragged last tile): 64
    chunks per head, merged; both query rows of each head against the
    oracle."""
    B, H, Nq, Nk, d = 1, 2, 2, (1 << 20) + 37, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(92)
    k, v = (torch.randn(B, H, Nk, d, generator=g, device="cuda").to(torch.bfloat16) for _ in range(2))
    q = torch.randn(B, H, Nq, d, generator=g, device="cuda").to(torch.bfloat16)
    assert fa_decode_workspace_bytes(B, H, Nq, Nk, d) > 0
    o, lse = fa_fwd_decode(q, k, v, None, True)
    assert fa_device_status() == 0
    scale = 1 / math.sqrt(d)
    for h in range(H):
        for i in range(Nq):
            end = Nk - Nq + i + 1
            o_ref, lse_ref = oracle.fwd(q[0, h, i:i + 1], k[0, h, :end], v[0, h, :end], False, scale)
            err = float(np.max(np.abs(o[0, h, i:i + 1].double().cpu().numpy() - o_ref)))
            assert err <= 1e-2, f"head {h} row {i}: O err {err:.3e}"
            assert abs(float(lse[0, h, i]) - float(lse_ref[0])) <= 1e-3
