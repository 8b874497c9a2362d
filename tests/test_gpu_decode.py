"""Decode forward (fa_fwd_decode): Nq <= 8 query rows against a key/value
cache, split over the keys and merged.

Every output row is checked against the fp64 oracle run on exactly the keys
that row sees (the first len_b cache rows; with causal, keys
j <= len_b - Nq + i), so the mask convention is tested by construction.
Rows that see no key must come back as o = 0, lse = -inf.  Besides the
tolerances every other test uses, O must also meet a much tighter bound:
this path keeps the weights P in fp32 (no bf16 rounding of P), so its error
is the bf16 rounding of the output plus fp32 accumulation.
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


def test_decode_empty_and_fully_masked_rows():
    """len 0 (no key at all) and causal rows before the first key: o = 0, lse = -inf."""
    B, H, Nq, Nk, d = 4, 2, 8, 300, 64
    q, k, v = _draw(B, H, Nq, Nk, d, 7)
    lens = [0, 3, 300, 8]
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = fa_fwd_decode(q, k, v, cl, True)
    assert fa_device_status() == 0
    _check(q, k, v, o, lse, lens, True, 0.125, "masked")
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


def test_decode_many_splits_and_workspace():
    """One head, a long cache: the keys go to many chunks and the merge
    kernel; with a caller workspace the result is the same bits."""
    B, H, Nq, Nk, d = 1, 2, 2, 40000, 128
    q, k, v = _draw(B, H, Nq, Nk, d, 33, mult=2.0)
    need = fa_decode_workspace_bytes(B, H, Nq, Nk, d)
    assert need > 0
    o, lse = fa_fwd_decode(q, k, v, None, False)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o2, lse2 = fa_fwd_decode(q, k, v, None, False, workspace=ws)
    assert fa_device_status() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    _check(q, k, v, o, lse, [Nk], False, 1.0 / math.sqrt(d), "long")


def test_decode_single_chunk_path():
    """Many heads and a short cache: one chunk per head, no merge kernel."""
    B, H, Nq, Nk, d = 8, 32, 1, 128, 64
    assert fa_decode_workspace_bytes(B, H, Nq, Nk, d) == 0
    q, k, v = _draw(B, H, Nq, Nk, d, 44)
    o, lse = fa_fwd_decode(q, k, v, None, False)
    assert fa_device_status() == 0
    rows = {(b, h, 0) for b in range(0, B, 3) for h in range(0, H, 7)}
    _check(q, k, v, o, lse, [Nk] * B, False, 0.125, "single chunk", rows)


def test_decode_deterministic():
    B, H, Nq, Nk, d = 2, 8, 1, 20000, 128
    q, k, v = _draw(B, H, Nq, Nk, d, 55)
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
