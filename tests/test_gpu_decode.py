"""Decode forward (fa_fwd_decode): Nq <= 8 query rows against a key/value
cache, split over the keys and merged.

Every output row is checked against the fp64 oracle run on exactly the keys
that row sees (the first len_b cache rows; with causal, keys
j <= len_b - Nq + i), so the mask convention is tested by construction.
Rows that see no key must come back as o = 0, lse = -inf.  Two kernels
serve the call: for one query row (and every d = 64 call) the products run
on CUDA cores with the weights P in fp32, and O must then also meet a much
tighter bound (the bf16 rounding of the output plus fp32 accumulation);
from two rows at d = 128 they run on the tensor core with P rounded to
bf16, and O meets the bound every bf16-P path meets.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_48_gb300 import fa_decode_workspace_bytes, fa_device_status, fa_fwd_decode
from parity import bf16_ulp, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu


def _draw(B, H, Nq, Nk, d, seed, cache_layout="bhnd", mult=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q = (torch.randn(B, H, Nq, d, generator=g, device="cuda") * mult).to(torch.bfloat16)
    if cache_layout == "bnhd":  # a cache stored [B, Nk, H, d]
        kc, vc = ((torch.randn(B, Nk, H, d, generator=g, device="cuda") * mult).to(torch.bfloat16) for _ in range(2))
        return q, kc.transpose(1, 2), vc.transpose(1, 2)
    k, v = ((torch.randn(B, H, Nk, d, generator=g, device="cuda") * mult).to(torch.bfloat16) for _ in range(2))
    return q, k, v


def _check(q, k, v, o, lse, lens, causal, scale, what, rows=None):
    B, H, Nq, d = q.shape
    fp32_weights = d == 64 or Nq == 1
    for b in range(B):
        n = lens[b]
        for h in range(H):
            for i in range(Nq):
                if rows is not None and (b, h, i) not in rows:
                    continue
                end = min(n, n - Nq + i + 1) if causal else n
                tag = f"{what} b{b} h{h} row{i} (len {n})"
                if end <= 0:
                    assert torch.all(o[b, h, i] == 0), f"{tag}: o of a row with no visible key"
                    assert float(lse[b, h, i]) == -math.inf, f"{tag}: lse of a row with no visible key"
                    continue
                qi, kb, vb = q[b, h, i:i + 1], k[b, h, :end], v[b, h, :end]
                o_ref, lse_ref = oracle.fwd(qi, kb, vb, False, scale)
                spread = oracle.fwd_spread(qi, kb, vb, False, scale)
                check_o(o[b, h, i:i + 1], o_ref, tag, spread)
                check_lse(lse[b, h, i:i + 1], lse_ref, tag)
                if fp32_weights:
                    err = np.abs(to_np(o[b, h, i:i + 1]) - o_ref)
                    tight = 0.5 * bf16_ulp(o_ref) + 1e-4
                    assert np.all(err <= tight), f"{tag}: O error {err.max():.3e} above the fp32-weights bound"
                assert abs(float(lse[b, h, i]) - float(lse_ref[0])) <= 1e-4, f"{tag}: lse"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq", [1, 3, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_small(d, Nq, causal):
    B, H, Nk = 3, 2, 1000
    q, k, v = _draw(B, H, Nq, Nk, d, 10 + d + Nq)
    lens = [1000, 1, 517]
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = fa_fwd_decode(q, k, v, cl, causal)
    assert fa_device_status() == 0
    _check(q, k, v, o, lse, lens, causal, 1.0 / math.sqrt(d), f"d{d} Nq{Nq} causal{int(causal)}")


@pytest.mark.parametrize("Nk", [1, 100, 128, 129, 4100])
def test_decode_lengths_without_array(Nk):
    """No cache_seqlens: every one of the Nk rows is valid (ragged last tile)."""
    B, H, Nq, d = 2, 3, 2, 128
    q, k, v = _draw(B, H, Nq, Nk, d, 100 + Nk)
    o, lse = fa_fwd_decode(q, k, v, None, True)
    assert fa_device_status() == 0
    _check(q, k, v, o, lse, [Nk] * B, True, 1.0 / math.sqrt(d), f"Nk{Nk}")


@pytest.mark.parametrize("d", [64, 128])
def test_decode_empty_and_fully_masked_rows(d):
    """len 0 (no key at all) and causal rows before the first key: o = 0, lse = -inf."""
    B, H, Nq, Nk = 4, 2, 8, 300
    q, k, v = _draw(B, H, Nq, Nk, d, 7)
    lens = [0, 3, 300, 8]
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = fa_fwd_decode(q, k, v, cl, True, 1.0 / math.sqrt(d))
    assert fa_device_status() == 0
    _check(q, k, v, o, lse, lens, True, 1.0 / math.sqrt(d), "masked")
    assert bool(torch.all(o[0] == 0)) and bool(torch.all(torch.isneginf(lse[0])))
    assert bool(torch.all(torch.isneginf(lse[1, :, :5])))  # rows 0..4 see no key when len = 3


def test_decode_out_of_range_lengths_are_clamped():
    """Values outside [0, Nk] in cache_seqlens are clamped, never read past the cache."""
    B, H, Nq, Nk, d = 3, 2, 1, 256, 128
    q, k, v = _draw(B, H, Nq, Nk, d, 8)
    cl = torch.tensor([-5, 10 ** 6, 200], dtype=torch.int32, device="cuda")
    o, lse = fa_fwd_decode(q, k, v, cl, False)
    assert fa_device_status() == 0
    _check(q, k, v, o, lse, [0, Nk, 200], False, 1.0 / math.sqrt(d), "clamped")


@pytest.mark.parametrize("d", [64, 128])
def test_decode_bnhd_cache_and_strided_query(d):
    """Cache stored [B, Nk, H, d]; q and o as [B, Nq, H, d] storage."""
    B, H, Nq, Nk = 2, 4, 4, 3000
    _, k, v = _draw(B, H, Nq, Nk, d, 21, cache_layout="bnhd")
    qs = torch.randn(B, Nq, H, d, device="cuda").to(torch.bfloat16)
    q = qs.transpose(1, 2)
    os_ = torch.empty_like(qs)
    lens = [3000, 1234]
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = fa_fwd_decode(q, k, v, cl, True, o=os_.transpose(1, 2))
    assert fa_device_status() == 0
    assert o.data_ptr() == os_.data_ptr()
    _check(q, k, v, o, lse, lens, True, 1.0 / math.sqrt(d), f"bnhd d{d}")
    # the same numbers as contiguous tensors
    o2, lse2 = fa_fwd_decode(q.contiguous(), k.contiguous(), v.contiguous(), cl, True)
    assert torch.equal(o2, o.contiguous()) and torch.equal(lse2, lse)


@pytest.mark.parametrize("Nq", [2, 8])
def test_decode_many_splits_and_workspace(Nq):
    """One head, a long cache: the keys go to many chunks and the merge
    kernel; with a caller workspace the result is the same bits."""
    B, H, Nk, d = 1, 2, 40000, 128
    q, k, v = _draw(B, H, Nq, Nk, d, 33, mult=2.0)
    need = fa_decode_workspace_bytes(B, H, Nq, Nk, d)
    assert need > 0
    o, lse = fa_fwd_decode(q, k, v, None, False)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o2, lse2 = fa_fwd_decode(q, k, v, None, False, workspace=ws)
    assert fa_device_status() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    _check(q, k, v, o, lse, [Nk], False, 1.0 / math.sqrt(d), "long")


@pytest.mark.parametrize("Nq,d", [(1, 64), (4, 128)])
def test_decode_single_chunk_path(Nq, d):
    """Many heads and a short cache: one chunk per head, no merge kernel."""
    B, H, Nk = 8, 32, 128
    assert fa_decode_workspace_bytes(B, H, Nq, Nk, d) == 0
    q, k, v = _draw(B, H, Nq, Nk, d, 44)
    o, lse = fa_fwd_decode(q, k, v, None, False)
    assert fa_device_status() == 0
    rows = {(b, h, i) for b in range(0, B, 3) for h in range(0, H, 7) for i in range(Nq)}
    _check(q, k, v, o, lse, [Nk] * B, False, 1.0 / math.sqrt(d), "single chunk", rows)


@pytest.mark.parametrize("scale", [0.0, -0.3])
@pytest.mark.parametrize("Nq,d", [(1, 128), (2, 64), (5, 128)])
def test_decode_zero_and_negative_scale(scale, Nq, d):
    """scale 0 gives every visible key the same weight (O is the mean of the
    visible V rows); a negative scale favours the keys least like q.  Both
    kernels, with causal masking and ragged cache lengths."""
    B, H, Nk = 2, 3, 700
    q, k, v = _draw(B, H, Nq, Nk, d, 140 + Nq + d)
    lens = [700, 301]
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = fa_fwd_decode(q, k, v, cl, True, scale)
    assert fa_device_status() == 0
    _check(q, k, v, o, lse, lens, True, scale, f"scale{scale} Nq{Nq} d{d}")


@pytest.mark.parametrize("Nq,d", [(1, 128), (4, 128), (2, 64)])
def test_decode_rescale_every_tile(Nq, d):
    """Scores that climb along the cache by about 8.5 (log2 units) per
    128-key tile: each row group's running maximum moves at every tile it
    takes, in both kernels, and the chunks' partial results span a wide
    range of logsumexps for the merge."""
    B, H, Nk = 1, 2, 3000
    scale = 1.0 / math.sqrt(d)
    beta = 8.5 / (128 * scale * math.log2(math.e))
    u = torch.full((d,), 1.0 / math.sqrt(d), device="cuda")
    q = u.expand(B, H, Nq, d).to(torch.bfloat16).contiguous()
    k = (torch.arange(Nk, device="cuda", dtype=torch.float32)[:, None] * beta * u).expand(B, H, Nk, d)
    k = k.to(torch.bfloat16).contiguous()
    g = torch.Generator(device="cuda")
    g.manual_seed(29)
    v = torch.randn(B, H, Nk, d, generator=g, device="cuda").to(torch.bfloat16)
    o, lse = fa_fwd_decode(q, k, v, None, True, scale)
    assert fa_device_status() == 0
    _check(q, k, v, o, lse, [Nk] * B, True, scale, f"ramp Nq{Nq} d{d}")


@pytest.mark.parametrize("Nq", [1, 6])
def test_decode_deterministic(Nq):
    B, H, Nk, d = 2, 8, 20000, 128
    q, k, v = _draw(B, H, Nq, Nk, d, 55 + Nq)
    cl = torch.tensor([20000, 15555], dtype=torch.int32, device="cuda")
    a = fa_fwd_decode(q, k, v, cl, False)
    b = fa_fwd_decode(q, k, v, cl, False)
    assert fa_device_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_full_size_workload():
    """The decode workload bench.py times (B16 H16, 16384 cached keys, d128,
    one query row), in the same launch configuration: sampled heads against
    the oracle, every row finite."""
    import bench
    from exact_attention_48_gb300.inputs import DECODE_B16H16NK16384D128 as w
    pb = bench.Problem(w)
    q, k, v, _ = pb.inputs
    o = pb.outputs[0]
    pb.fwd(q, k, v, o, pb.lse)
    assert fa_device_status() == 0
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(pb.lse).all())
    rows = {(0, 0, 0), (w.B - 1, w.H - 1, 0), (7, 5, 0), (11, 9, 0)}
    _check(q, k, v, o, pb.lse, [w.N] * w.B, False, w.scale, w.name, rows)


@pytest.mark.parametrize("Nq", [2, 3, 5, 8])
def test_decode_tensor_core_many_heads_persistent(Nq):
    """Enough heads that every CTA of the persistent grid takes several
    items of several tiles (the tensor-core path at d = 128), with ragged
    cache lengths and causal masking."""
    B, H, Nk, d = 8, 24, 2000, 128
    q, k, v = _draw(B, H, Nq, Nk, d, 120 + Nq)
    lens = [2000, 1999, 1, 0, 129, 1024, 777, 1500]
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = fa_fwd_decode(q, k, v, cl, True)
    assert fa_device_status() == 0
    rows = {(b, h, i) for b in range(B) for h in (0, H - 1) for i in range(Nq)}
    _check(q, k, v, o, lse, lens, True, 1.0 / math.sqrt(d), f"persistent Nq{Nq}", rows)
