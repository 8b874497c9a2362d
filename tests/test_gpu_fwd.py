"""Forward parity: fa_fwd (CUDA, through the C ABI) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_48_gb300 import fa_device_status, fa_fwd, fa_fwd_varlen
from exact_attention_48_gb300.inputs import draw_shape
from parity import check_lse, check_o

pytestmark = pytest.mark.gpu

SMALL_N = [1, 64, 127, 128, 129, 200, 256, 384]


def _run(B, H, N, d, causal, scale=None, seed=7, mult=1.0):
    q, k, v, _ = draw_shape(B, H, N, d, seed, mult, "cpu", torch.bfloat16, with_dout=False)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qc, float("nan"))
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    fa_fwd(qc, kc, vc, causal, scale, o=o, lse=lse)
    assert fa_device_status() == 0
    o_ref, lse_ref = oracle.fwd(q, k, v, causal, scale)
    return o, lse, o_ref, lse_ref


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", SMALL_N)
def test_fwd_small(N, d, causal):
    o, lse, o_ref, lse_ref = _run(2, 2, N, d, causal, seed=100 + N + d)
    check_o(o, o_ref, f"N={N} d={d} causal={causal}")
    check_lse(lse, lse_ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("scale", [-0.3, 0.0, 0.5])
def test_fwd_scale_values(scale):
    """Negative, zero and a large scale (0.5 at d = 64: logits of std 4, a
    very sharp softmax, checked with the bound derived from bf16 weights)."""
    for causal in (False, True):
        o, lse, o_ref, lse_ref = _run(1, 2, 200, 64, causal, scale=scale, seed=3)
        q, k, v, _ = draw_shape(1, 2, 200, 64, 3, 1.0, "cpu", torch.bfloat16, with_dout=False)
        spread = oracle.fwd_spread(q, k, v, causal, scale)
        check_o(o, o_ref, f"scale={scale}", spread)
        check_lse(lse, lse_ref, f"scale={scale}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_rescale_every_block(d, causal):
    """Scores that climb along the keys by about 8.5 (log2 units) per
    128-key block: every block's maximum beats the running maximum by more
    than the rescale threshold, so O (and at d = 64 the row sums the P V
    product forms beside it) is rescaled at every block."""
    N = 1000
    scale = 1.0 / math.sqrt(d)
    beta = 8.5 / (128 * scale * math.log2(math.e))  # score step per key, in units of q . k
    u = torch.full((d,), 1.0 / math.sqrt(d), dtype=torch.float64)
    q = u.expand(1, 1, N, d).clone()
    k = (torch.arange(N, dtype=torch.float64)[:, None] * beta * u).expand(1, 1, N, d).clone()
    g = torch.Generator().manual_seed(17)
    v = torch.randn(1, 1, N, d, generator=g, dtype=torch.float64)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    o, lse = fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    assert fa_device_status() == 0
    o_ref, lse_ref = oracle.fwd(q, k, v, causal, scale)
    check_o(o, o_ref, f"ramp d={d} causal={causal}", oracle.fwd_spread(q, k, v, causal, scale))
    check_lse(lse, lse_ref, f"ramp d={d} causal={causal}")


def test_fwd_deterministic():
    q, k, v, _ = draw_shape(2, 4, 1000, 128, 11, 1.0, "cuda", torch.bfloat16, with_dout=False)
    o1, l1 = fa_fwd(q, k, v, True)
    for _ in range(3):
        o2, l2 = fa_fwd(q, k, v, True)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("H,d,causal", [(3, 64, False), (160, 64, False), (160, 128, True)])
def test_fwd_guard_bands(H, d, causal):
    """Writes stay inside o and lse: canaries around both survive (160 heads:
    the persistent grid, whose CTAs write several tiles' rows)."""
    B, N = 1, 300
    q, k, v, _ = draw_shape(B, H, N, d, 5, 1.0, "cuda", torch.bfloat16, with_dout=False)
    pad = 4096
    ob = torch.full((B * H * N * d + 2 * pad,), 7.0, device="cuda", dtype=torch.bfloat16)
    lb = torch.full((B * H * N + 2 * pad,), 7.0, device="cuda")
    o = ob[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = lb[pad:pad + B * H * N].view(B, H, N)
    fa_fwd(q, k, v, causal, o=o, lse=lse)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    assert torch.all(ob[:pad] == 7) and torch.all(ob[-pad:] == 7)
    assert torch.all(lb[:pad] == 7) and torch.all(lb[-pad:] == 7)


def test_fwd_constant_v_and_zero_q():
    B, H, N, d = 1, 2, 333, 128
    q, k, v, _ = draw_shape(B, H, N, d, 9, 1.0, "cuda", torch.bfloat16, with_dout=False)
    c = torch.randn(d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    vc = c.expand(B, H, N, d).contiguous()
    for causal in (False, True):
        o, _ = fa_fwd(q, k, vc, causal)
        assert torch.allclose(o.float(), vc.float(), atol=2e-2, rtol=0)
    z = torch.zeros_like(q)
    o, lse = fa_fwd(z, k, v, False)
    mean = v.double().mean(2, keepdim=True).expand_as(o)
    assert torch.allclose(o.double(), mean, atol=1e-2)
    assert torch.allclose(lse.double(), torch.full_like(lse.double(), math.log(N)), atol=1e-3)


@pytest.mark.parametrize("d,causal", [(64, False), (64, True), (128, False), (128, True)])
@pytest.mark.parametrize("B,H,N", [(3, 40, 1000), (1, 200, 1), (1, 160, 300), (2, 100, 129)])
def test_fwd_persistent_same_bits_as_one_cta_per_tile(B, H, N, d, causal):
    """With more 256-row tiles than SMs, the batched forward of short
    sequences runs one persistent CTA per SM that walks several tiles (more
    Q slots, the K/V ring and every barrier's phase carried from tile to
    tile); the packed-sequence call runs one CTA per tile.  A tile's
    arithmetic is the same either way, so the bits must be.  The shapes give
    ragged last tiles, single-key heads and tile counts that are not
    multiples of the SM count (some CTAs take one tile more than others);
    heads of the first and the last turn are also checked against the
    oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert B * H * ((N + 255) // 256) > sms
    q, k, v, _ = draw_shape(B, H, N, d, 500 + N, 1.0, "cuda", torch.bfloat16, with_dout=False)
    o, lse = fa_fwd(q, k, v, causal)
    qp, kp, vp = (t.transpose(1, 2).reshape(B * N, H, d).contiguous() for t in (q, k, v))
    cu = torch.arange(0, B * N + 1, N, dtype=torch.int32, device="cuda")
    o_p, lse_p = fa_fwd_varlen(qp, kp, vp, cu, N, causal)
    assert fa_device_status() == 0
    assert torch.equal(o_p.reshape(B, N, H, d).transpose(1, 2), o)
    assert torch.equal(lse_p.reshape(H, B, N).permute(1, 0, 2), lse)
    scale = 1.0 / math.sqrt(d)
    for b, h in {(0, 0), (B - 1, H - 1), (B // 2, H // 2)}:
        o_ref, lse_ref = oracle.fwd(q[b, h].cpu(), k[b, h].cpu(), v[b, h].cpu(), causal, scale)
        what = f"persistent B={B} H={H} N={N} d={d} causal={causal} head ({b}, {h})"
        check_o(o[b, h], o_ref, what)
        check_lse(lse[b, h], lse_ref, what)


@pytest.mark.parametrize("scale", [-0.3, 0.0])
def test_fwd_persistent_scale_values(scale):
    """The persistent grid with a negative and a zero scale (the running
    minimum path and uniform weights), causal and not: the same bits as the
    packed call's one CTA per tile, and two heads against the oracle."""
    B, H, N, d = 1, 160, 300, 64
    q, k, v, _ = draw_shape(B, H, N, d, 77, 1.0, "cuda", torch.bfloat16, with_dout=False)
    qp, kp, vp = (t.transpose(1, 2).reshape(B * N, H, d).contiguous() for t in (q, k, v))
    cu = torch.tensor([0, N], dtype=torch.int32, device="cuda")
    for causal in (False, True):
        o, lse = fa_fwd(q, k, v, causal, scale)
        o_p, lse_p = fa_fwd_varlen(qp, kp, vp, cu, N, causal, scale)
        assert fa_device_status() == 0
        assert torch.equal(o_p.reshape(B, N, H, d).transpose(1, 2), o)
        assert torch.equal(lse_p.reshape(H, B, N).permute(1, 0, 2), lse)
        for h in (0, H - 1):
            o_ref, lse_ref = oracle.fwd(q[0, h].cpu(), k[0, h].cpu(), v[0, h].cpu(), causal, scale)
            spread = oracle.fwd_spread(q[0, h].cpu(), k[0, h].cpu(), v[0, h].cpu(), causal, scale)
            check_o(o[0, h], o_ref, f"persistent scale={scale} causal={causal} head {h}", spread)
            check_lse(lse[0, h], lse_ref, f"persistent scale={scale} causal={causal} head {h}")
