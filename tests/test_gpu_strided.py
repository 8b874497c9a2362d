"""Strided layouts through fa_fwd_strided / fa_bwd_strided.

Layouts a framework hands over: [B, N, H, d] tensors ("BNHD", seen as
[B, H, N, d] views with transposed strides) and the q, k, v slices of one
packed [B, N, 3, H, d] projection, with the gradients written back into one
packed buffer.  The kernels do the same arithmetic whatever the strides, so
the results must equal the contiguous entry points' bit for bit; one small
ragged causal case is also checked against the fp64 oracle.
"""
import pytest
import torch

import oracle
from exact_attention_48_gb300 import (fa_bwd, fa_bwd_strided, fa_device_status, fa_fwd, fa_fwd_strided)
from exact_attention_48_gb300.inputs import draw_shape
from parity import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


def _contig(*ts):
    return [t.contiguous() for t in ts]


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 200, 64, False), (1, 4, 384, 128, True), (2, 2, 129, 128, False),
                                             (2, 80, 700, 64, False), (3, 60, 1000, 128, True)])
def test_bnhd_matches_contiguous_bitwise(B, H, N, d, causal):
    """(The last two shapes have more 256-row tiles than SMs: their forward
    runs the persistent grid, with the same strides.)"""
    q, k, v, do = draw_shape(B, H, N, d, 7 + N, 1.0, "cuda", torch.bfloat16)
    # the same values stored as [B, N, H, d]; the views are [B, H, N, d]
    qs, ks, vs, dos = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (q, k, v, do))
    assert qs.stride() == (N * H * d, d, H * d, 1)
    o_ref, lse_ref = fa_fwd(q, k, v, causal)
    o_bnhd = torch.empty(B, N, H, d, device="cuda", dtype=torch.bfloat16).transpose(1, 2)
    o, lse = fa_fwd_strided(qs, ks, vs, causal, o=o_bnhd)
    g_ref = fa_bwd(q, k, v, o_ref, do, lse_ref, causal)
    grads = fa_bwd_strided(qs, ks, vs, o, dos, lse, causal,
                           dq=torch.empty(B, N, H, d, device="cuda", dtype=torch.bfloat16).transpose(1, 2))
    assert fa_device_status() == 0
    assert torch.equal(o.contiguous(), o_ref) and torch.equal(lse, lse_ref)
    for g, r in zip(grads, g_ref):
        assert torch.equal(g.contiguous(), r)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_qkv_projection(causal):
    B, H, N, d = 2, 4, 300, 128
    q, k, v, do = draw_shape(B, H, N, d, 11, 1.0, "cuda", torch.bfloat16)
    qkv = torch.stack([t.transpose(1, 2) for t in (q, k, v)], dim=2).contiguous()  # [B, N, 3, H, d]
    qp, kp, vp = (qkv[:, :, i].transpose(1, 2) for i in range(3))
    assert qp.stride() == (N * 3 * H * d, d, 3 * H * d, 1)
    o_ref, lse_ref = fa_fwd(q, k, v, causal)
    o, lse = fa_fwd_strided(qp, kp, vp, causal)
    gbuf = torch.empty_like(qkv)  # packed gradients, [B, N, 3, H, d]
    dq, dk, dv = (gbuf[:, :, i].transpose(1, 2) for i in range(3))
    fa_bwd_strided(qp, kp, vp, o, do, lse, causal, dq=dq, dk=dk, dv=dv)
    g_ref = fa_bwd(q, k, v, o_ref, do, lse_ref, causal)
    assert fa_device_status() == 0
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    for i, r in enumerate(g_ref):
        assert torch.equal(gbuf[:, :, i].transpose(1, 2).contiguous(), r)


def test_strided_against_oracle():
    B, H, N, d, causal, scale = 1, 2, 200, 64, True, 0.125
    q, k, v, do = draw_shape(B, H, N, d, 21, 1.0, "cuda", torch.bfloat16)
    qs, ks, vs, dos = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (q, k, v, do))
    o, lse = fa_fwd_strided(qs, ks, vs, causal, scale)
    dq, dk, dv = fa_bwd_strided(qs, ks, vs, o, dos, lse, causal, scale)
    assert fa_device_status() == 0
    for h in range(H):
        qh, kh, vh, doh = (t[0, h] for t in (q, k, v, do))
        o_r, lse_r = oracle.fwd(qh, kh, vh, causal, scale)
        check_o(o[0, h], o_r, f"strided head {h}", oracle.fwd_spread(qh, kh, vh, causal, scale))
        check_lse(lse[0, h], lse_r, f"strided head {h}")
        refs = oracle.bwd(qh, kh, vh, doh, causal, scale)
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
            check_grad(g[0, h], r, name, f"strided head {h}")
