"""Parity at the full workload sizes, in the launch configuration bench.py uses.

For each workload the whole tensors go through fa_fwd / fa_bwd once; the fp64
oracle then recomputes a fixed subset of heads (first, last and two seeded
ones) completely, all rows and all columns.  A secondary check compares every
head against PyTorch fp32 attention on the GPU (a library routine, upcast
from the same bf16 inputs).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_48_gb300 import fa_bwd, fa_device_status, fa_fwd
from exact_attention_48_gb300.inputs import (CAUSAL_B4H32N4096D128, FWD_B8H16N2048D64, LONG_B1H16N16384D128,
                                             TINY, draw, sweep)
from parity import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


def heads_to_check(B, H, n_extra=2, max_heads=4):
    BH = B * H
    r = np.random.default_rng(BH)
    picks = {0, BH - 1}
    while len(picks) < min(BH, 2 + n_extra):
        picks.add(int(r.integers(0, BH)))
    return sorted(picks)[:max_heads]


def _torch_ref_fwd(q, k, v, causal, scale):
    """fp32 GPU reference, one head at a time (O and LSE)."""
    B, H, N, d = q.shape
    o = torch.empty(B, H, N, d, device=q.device, dtype=torch.float32)
    lse = torch.empty(B, H, N, device=q.device, dtype=torch.float32)
    mask = torch.ones(N, N, device=q.device, dtype=torch.bool).triu(1) if causal else None
    for b in range(B):
        for h in range(H):
            s = (q[b, h].float() @ k[b, h].float().T) * scale
            if causal:
                s.masked_fill_(mask, float("-inf"))
            lse[b, h] = torch.logsumexp(s, -1)
            o[b, h] = torch.softmax(s, -1) @ v[b, h].float()
            del s
    return o, lse


def _run(w, heads_max=4, full_torch=True):
    q, k, v, do = draw(w, device="cuda")
    o, lse = fa_fwd(q, k, v, w.causal, w.scale)
    grads = None
    if w.backward:
        grads = fa_bwd(q, k, v, o, do, lse, w.causal, w.scale)
    assert fa_device_status() == 0
    torch.cuda.synchronize()
    heads = heads_to_check(w.B, w.H, max_heads=heads_max)
    qf, kf, vf, dof = (t.view(w.B * w.H, w.N, w.d) for t in (q, k, v, do))
    of, lsef = o.view(w.B * w.H, w.N, w.d), lse.view(w.B * w.H, w.N)
    for hh in heads:
        o_ref, lse_ref = oracle.fwd(qf[hh], kf[hh], vf[hh], w.causal, w.scale)
        spread = oracle.fwd_spread(qf[hh], kf[hh], vf[hh], w.causal, w.scale)
        check_o(of[hh], o_ref, f"{w.name} head {hh}", spread)
        check_lse(lsef[hh], lse_ref, f"{w.name} head {hh}")
        if grads is not None:
            refs = oracle.bwd(qf[hh], kf[hh], vf[hh], dof[hh], w.causal, w.scale)
            for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
                check_grad(g.view(w.B * w.H, w.N, w.d)[hh], r, name, f"{w.name} head {hh}")
    if full_torch:
        # every head against PyTorch fp32 attention on the GPU (flat bound;
        # used on workloads with unit-variance inputs only)
        o_t, lse_t = _torch_ref_fwd(q, k, v, w.causal, w.scale)
        err = (o.float() - o_t).abs()
        bound = torch.clamp(0.5 * torch.exp2(torch.floor(torch.log2(o_t.abs().clamp_min(1e-30)))) / 128 + 2e-3,
                            min=1e-2)
        assert bool((err <= bound + 1e-6).all()), f"{w.name}: O vs torch fp32, max err {float(err.max()):.3e}"
        assert float((lse - lse_t).abs().max()) <= 1e-3
    return q, k, v, o, lse


def test_tiny_workload():
    _run(TINY)


def test_forward_only_b8h16n2048d64():
    _run(FWD_B8H16N2048D64)


def test_causal_b4h32n4096d128():
    _run(CAUSAL_B4H32N4096D128, heads_max=3)


def test_long_context_b1h16n16384d128():
    _run(LONG_B1H16N16384D128, heads_max=2, full_torch=False)


@pytest.mark.parametrize("N", [512, 1024, 2048, 8192, 16384])
@pytest.mark.parametrize("causal", [False, True])
def test_sweep_points_d128(N, causal):
    _run(sweep(N, 128, causal), heads_max=2, full_torch=(N <= 8192))


@pytest.mark.parametrize("N,causal", [(512, True), (1024, False), (2048, False), (4096, True), (16384, False),
                                      (16384, True)])
def test_sweep_points_d64(N, causal):
    _run(sweep(N, 64, causal), heads_max=2, full_torch=(N <= 8192))


def _torch_ref_grads(q, k, v, do, causal, scale, heads_per_batch=8):
    """dQ, dK, dV of PyTorch fp32 attention on the GPU (autograd through
    the materialised softmax), a few heads at a time, from the same bf16
    inputs upcast."""
    B, H, N, d = q.shape
    qf, kf, vf, dof = (t.reshape(B * H, N, d) for t in (q, k, v, do))
    outs = [torch.empty(B * H, N, d, device=q.device, dtype=torch.float32) for _ in range(3)]
    mask = torch.ones(N, N, device=q.device, dtype=torch.bool).triu(1) if causal else None
    for h0 in range(0, B * H, heads_per_batch):
        sl = slice(h0, min(B * H, h0 + heads_per_batch))
        a, b, c = (t[sl].float().requires_grad_(True) for t in (qf, kf, vf))
        s = (a @ b.transpose(1, 2)) * scale
        if causal:
            s = s.masked_fill(mask, float("-inf"))
        o = torch.softmax(s, -1) @ c
        ga, gb, gc = torch.autograd.grad(o, (a, b, c), dof[sl].float())
        for dst, g in zip(outs, (ga, gb, gc)):
            dst[sl] = g
        del a, b, c, s, o, ga, gb, gc
    return [t.view(B, H, N, d) for t in outs]


@pytest.mark.parametrize("N,d,causal", [(2048, 128, False), (4096, 128, True), (2048, 64, False)])
def test_sweep_point_gradients_every_head(N, d, causal):
    """Every head's dQ, dK, dV of a sweep point against PyTorch fp32
    attention on the GPU (the per-head bound: 2e-2 x max|grad| of the
    reference), beside the oracle's sampled heads."""
    w = sweep(N, d, causal)
    q, k, v, do = draw(w, device="cuda")
    o, lse = fa_fwd(q, k, v, w.causal, w.scale)
    grads = fa_bwd(q, k, v, o, do, lse, w.causal, w.scale)
    assert fa_device_status() == 0
    refs = _torch_ref_grads(q, k, v, do, w.causal, w.scale)
    for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
        g, r = g.float().reshape(w.B * w.H, -1), r.reshape(w.B * w.H, -1)
        assert bool(torch.isfinite(g).all()), name
        err = (g - r).abs().amax(dim=1)
        bound = 2e-2 * r.abs().amax(dim=1) + 1e-6
        worst = int(torch.argmax(err / bound))
        assert bool((err <= bound).all()), (f"{w.name} {name}: head {worst} err {float(err[worst]):.3e} "
                                            f"> {float(bound[worst]):.3e}")


def _bench_problem(w):
    import bench
    pb = bench.Problem(w)
    q, k, v, do = pb.inputs
    o, dq, dk, dv = pb.outputs
    pb.fwd(q, k, v, o, pb.lse)
    pb.bwd(q, k, v, o, do, pb.lse, dq, dk, dv)
    assert fa_device_status() == 0
    torch.cuda.synchronize()
    return pb


def test_bnhd_b2h16n8192d128():
    """The headline shape stored [B, N, H, d], through the strided calls as
    bench.py drives them: sampled heads against the oracle, every head of O
    against the contiguous path bit for bit."""
    from exact_attention_48_gb300.inputs import BNHD_B2H16N8192D128 as w
    pb = _bench_problem(w)
    q, k, v, do = (x.transpose(1, 2) for x in pb.inputs)   # [B, H, N, d] views
    o, dq, dk, dv = (x.transpose(1, 2) for x in pb.outputs)
    for hh in heads_to_check(w.B, w.H, max_heads=2):
        b, h = divmod(hh, w.H)
        o_ref, lse_ref = oracle.fwd(q[b, h], k[b, h], v[b, h], w.causal, w.scale)
        spread = oracle.fwd_spread(q[b, h], k[b, h], v[b, h], w.causal, w.scale)
        check_o(o[b, h], o_ref, f"{w.name} head {hh}", spread)
        check_lse(pb.lse[b, h], lse_ref, f"{w.name} head {hh}")
        refs = oracle.bwd(q[b, h], k[b, h], v[b, h], do[b, h], w.causal, w.scale)
        for name, g, r in zip(("dq", "dk", "dv"), (dq[b, h], dk[b, h], dv[b, h]), refs):
            check_grad(g, r, name, f"{w.name} head {hh}")
    oc, lc = fa_fwd(q.contiguous(), k.contiguous(), v.contiguous(), w.causal, w.scale)
    assert torch.equal(oc, o) and torch.equal(lc, pb.lse)


def test_varlen_t16384h16d128_causal():
    """16384 packed tokens of 7 sequences, causal, as bench.py drives them:
    the first, the longest and the last sequence against the oracle (one
    head each), and every output row finite."""
    from exact_attention_48_gb300.inputs import VARLEN_T16384H16D128 as w
    pb = _bench_problem(w)
    q, k, v, do = pb.inputs                                  # [T, H, d]
    o, dq, dk, dv = pb.outputs
    offs = [0]
    for n in w.lengths:
        offs.append(offs[-1] + n)
    longest = max(range(w.B), key=lambda i: w.lengths[i])
    for b, h in ((0, 0), (longest, w.H // 2), (w.B - 1, w.H - 1)):
        r0, r1 = offs[b], offs[b + 1]
        sl = lambda x: x[r0:r1, h]  # noqa: E731
        o_ref, lse_ref = oracle.fwd(sl(q), sl(k), sl(v), w.causal, w.scale)
        spread = oracle.fwd_spread(sl(q), sl(k), sl(v), w.causal, w.scale)
        check_o(sl(o), o_ref, f"{w.name} seq {b} head {h}", spread)
        check_lse(pb.lse[h, r0:r1], lse_ref, f"{w.name} seq {b} head {h}")
        refs = oracle.bwd(sl(q), sl(k), sl(v), sl(do), w.causal, w.scale)
        for name, g, r in zip(("dq", "dk", "dv"), (sl(dq), sl(dk), sl(dv)), refs):
            check_grad(g, r, name, f"{w.name} seq {b} head {h}")
    for t in (o, dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
