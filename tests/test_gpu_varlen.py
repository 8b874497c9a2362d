"""Packed variable-length sequences through fa_fwd_varlen / fa_bwd_varlen.

B sequences of different lengths lie back to back along one row axis of T
rows ([T, H, d] tensors, lse [H, T]); each attends only to itself.  Every
sequence must give exactly what the batched call gives on that sequence
alone (the same tiles and masks, so the same bits), whatever rows of the
neighbouring sequences the tile loads pick up; one case is also checked
against the fp64 oracle.
"""
import pytest
import torch

import oracle
from exact_attention_48_gb300 import fa_bwd, fa_bwd_varlen, fa_device_status, fa_fwd, fa_fwd_varlen
from parity import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


def _pack(lengths, H, d, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    T = sum(lengths)
    q, k, v, do = (torch.randn(T, H, d, generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    cu = torch.tensor([0] + list(torch.tensor(lengths).cumsum(0).tolist()), dtype=torch.int32, device="cuda")
    return q, k, v, do, cu


def _seq(t, cu, b):
    """Sequence b of a packed [T, H, d] tensor as a contiguous [1, H, n, d] tensor."""
    s, e = int(cu[b]), int(cu[b + 1])
    return t[s:e].transpose(0, 1).unsqueeze(0).contiguous()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_per_sequence_calls(d, causal):
    lengths = [200, 1, 333, 0, 128, 257]
    H = 3
    q, k, v, do, cu = _pack(lengths, H, d, 5 + d)
    max_len = max(lengths) + 40  # larger than needed: the extra blocks have no work
    o, lse = fa_fwd_varlen(q, k, v, cu, max_len, causal)
    dq, dk, dv = fa_bwd_varlen(q, k, v, o, do, lse, cu, max_len, causal)
    assert fa_device_status() == 0
    for b, n in enumerate(lengths):
        if n == 0:
            continue
        qs, ks, vs, dos = (_seq(t, cu, b) for t in (q, k, v, do))
        o_r, lse_r = fa_fwd(qs, ks, vs, causal)
        g_r = fa_bwd(qs, ks, vs, o_r, dos, lse_r, causal)
        s, e = int(cu[b]), int(cu[b + 1])
        assert torch.equal(_seq(o, cu, b), o_r), f"o of sequence {b}"
        assert torch.equal(lse[:, s:e].unsqueeze(0), lse_r), f"lse of sequence {b}"
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), g_r):
            assert torch.equal(_seq(g, cu, b), r), f"{name} of sequence {b}"


def test_varlen_against_oracle():
    lengths = [130, 77, 256]
    H, d, causal, scale = 2, 64, True, 0.125
    q, k, v, do, cu = _pack(lengths, H, d, 99)
    o, lse = fa_fwd_varlen(q, k, v, cu, max(lengths), causal, scale)
    dq, dk, dv = fa_bwd_varlen(q, k, v, o, do, lse, cu, max(lengths), causal, scale)
    assert fa_device_status() == 0
    for b in range(len(lengths)):
        s, e = int(cu[b]), int(cu[b + 1])
        for h in range(H):
            qh, kh, vh, doh = (t[s:e, h] for t in (q, k, v, do))
            o_r, lse_r = oracle.fwd(qh, kh, vh, causal, scale)
            what = f"sequence {b} head {h}"
            check_o(o[s:e, h], o_r, what, oracle.fwd_spread(qh, kh, vh, causal, scale))
            check_lse(lse[h, s:e], lse_r, what)
            for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), oracle.bwd(qh, kh, vh, doh, causal, scale)):
                check_grad(g[s:e, h], r, name, what)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_backward_same_bits_with_and_without_block_pairs(d, causal):
    """The backward of short sequences runs two mirror blocks (j and nb-1-j)
    per CTA -- causal: up to 32 blocks per sequence in the dK/dV kernel and
    16 in the dQ kernel; non-causal: up to 16 in both -- and of longer ones
    one block per CTA.  In a pack whose longest sequence is past those limits
    every sequence runs one block per CTA, while each short sequence alone
    runs in pairs: the tiles' arithmetic is the same either way, so the bits
    must be."""
    lengths = [4200, 1000, 2100, 300, 129, 1]  # blocks: 33, 8, 17, 3, 2, 1
    H = 2
    q, k, v, do, cu = _pack(lengths, H, d, 41 + d)
    o, lse = fa_fwd_varlen(q, k, v, cu, max(lengths), causal)
    dq, dk, dv = fa_bwd_varlen(q, k, v, o, do, lse, cu, max(lengths), causal)
    assert fa_device_status() == 0
    for b in range(1, len(lengths)):
        qs, ks, vs, dos = (_seq(t, cu, b) for t in (q, k, v, do))
        o_r, lse_r = fa_fwd(qs, ks, vs, causal)
        g_r = fa_bwd(qs, ks, vs, o_r, dos, lse_r, causal)
        assert torch.equal(_seq(o, cu, b), o_r), f"o of sequence {b}"
        for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), g_r):
            assert torch.equal(_seq(g, cu, b), r), f"{name} of sequence {b} ({lengths[b]} rows)"
