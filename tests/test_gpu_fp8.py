"""FP8 forward (fa_fwd_fp8) against the oracle's FP8 definition.

The oracle computes the same weights (e4m3 rounding of 2^(x - M + 8) at
the row's integer maximum) in fp64 and reports, per element, how far the
GPU may differ where a weight's rounding could go either way (a score
within the GPU's fp32 error of a rounding midpoint) or lies below e4m3's
normal range.  On top of that bound the test allows half a bf16 ulp of O
(its rounding) and 2^-12 * max|v| for the fp32 accumulation of the
products.  The result is also checked against exact attention on the
decoded inputs with the error rounding every weight to e4m3 can cause.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_48_gb300 import fa_device_status, fa_fwd_fp8
from exact_attention_48_gb300.inputs import draw_fp8
from parity import bf16_ulp, to_np

pytestmark = pytest.mark.gpu

ACC_REL = 2.0 ** -13  # relative precision assumed for the tensor core's fp32 score sums
STALE = 2             # binades by which the kernel's running maximum may lag a row's maximum


def _dec(x8, s):
    return x8.float().cpu().double().numpy() * s


def _check(q8, k8, v8, scales, o, lse, causal, scale, what, heads=None):
    sq, sk, sv = scales
    B, H, N, d = q8.shape
    qf, kf, vf = (t.reshape(B * H, N, d) for t in (q8, k8, v8))
    of, lf = o.reshape(B * H, N, d), lse.reshape(B * H, N)
    vmax = float(v8.float().abs().max()) * sv
    for hh in (heads if heads is not None else range(B * H)):
        o_ref, lse_ref, bound = oracle.fwd_fp8(qf[hh], kf[hh], vf[hh], sq, sk, sv, causal, scale, acc_rel=ACC_REL,
                                               with_bound=True, stale=STALE)
        og = to_np(of[hh])
        assert np.all(np.isfinite(og)), f"{what} head {hh}: non-finite O"
        err = np.abs(og - o_ref)
        tol = 0.5 * bf16_ulp(o_ref) + bound + 2.0 ** -12 * vmax + 1e-6
        bad = err > tol
        assert not bad.any(), (f"{what} head {hh}: {int(bad.sum())} elements off, worst {err[bad].max():.3e} "
                               f"vs {tol[bad][np.argmax(err[bad])]:.3e}")
        lerr = float(np.max(np.abs(to_np(lf[hh]) - lse_ref)))
        assert lerr <= 1e-3, f"{what} head {hh}: LSE max err {lerr:.3e}"


@pytest.mark.parametrize("N", [1, 128, 129, 200, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_small(N, causal):
    q8, k8, v8, sc = draw_fp8(1, 2, N, 128, 50 + N, device="cuda")
    scale = 1 / math.sqrt(128)
    o, lse = fa_fwd_fp8(q8, k8, v8, *sc, causal, scale)
    assert fa_device_status() == 0
    _check(q8, k8, v8, sc, o, lse, causal, scale, f"N{N} causal{int(causal)}")


@pytest.mark.parametrize("mult", [2.0, 0.25])
def test_fp8_sharp_and_flat_softmax(mult):
    q8, k8, v8, sc = draw_fp8(2, 2, 640, 128, 71, input_mult=mult, device="cuda")
    scale = 1 / math.sqrt(128)
    o, lse = fa_fwd_fp8(q8, k8, v8, *sc, True, scale)
    assert fa_device_status() == 0
    _check(q8, k8, v8, sc, o, lse, True, scale, f"mult{mult}")


def test_fp8_negative_scale_and_uint8_codes():
    q8, k8, v8, sc = draw_fp8(1, 2, 300, 128, 72, device="cuda")
    o, lse = fa_fwd_fp8(q8.view(torch.uint8), k8.view(torch.uint8), v8.view(torch.uint8), *sc, False, -0.05)
    assert fa_device_status() == 0
    _check(q8, k8, v8, sc, o, lse, False, -0.05, "negative scale")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_zero_scale(causal):
    """scale 0: every visible key gets the same weight, so O is the mean of
    the visible rows of V and lse = log(number of visible keys)."""
    q8, k8, v8, sc = draw_fp8(1, 2, 257, 128, 73, device="cuda")
    o, lse = fa_fwd_fp8(q8, k8, v8, *sc, causal, 0.0)
    assert fa_device_status() == 0
    _check(q8, k8, v8, sc, o, lse, causal, 0.0, f"zero scale causal{int(causal)}")
    n_vis = torch.arange(1, 258, device="cuda", dtype=torch.float32) if causal else torch.full((257,), 257.0,
                                                                                              device="cuda")
    assert torch.allclose(lse[0, 0], torch.log(n_vis), atol=1e-5)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_rescale_every_block(causal):
    """Scores that climb along the keys by about 4 (log2 units) per 128-key
    block: the integer running maximum (allowed to lag by 2) moves and O is
    rescaled at nearly every block."""
    from exact_attention_48_gb300.inputs import quantize_e4m3
    N, d = 1000, 128
    scale = 1.0 / math.sqrt(d)
    beta = 4.0 / (128 * scale * math.log2(math.e))
    u = torch.full((d,), 1.0 / math.sqrt(d))
    q8, sq = quantize_e4m3(u.expand(1, 1, N, d).clone())
    k8, sk = quantize_e4m3((torch.arange(N, dtype=torch.float32)[:, None] * beta * u).expand(1, 1, N, d).clone())
    g = torch.Generator().manual_seed(23)
    v8, sv = quantize_e4m3(torch.randn(1, 1, N, d, generator=g))
    q8, k8, v8 = q8.cuda(), k8.cuda(), v8.cuda()
    o, lse = fa_fwd_fp8(q8, k8, v8, sq, sk, sv, causal, scale)
    assert fa_device_status() == 0
    _check(q8, k8, v8, (sq, sk, sv), o, lse, causal, scale, f"ramp causal{int(causal)}")


def test_fp8_close_to_exact_attention():
    """Against exact attention on the decoded inputs: rounding each weight
    to e4m3 (2^-4 relative) and renormalising moves O by at most
    2 * 2^-4/(1 - 2^-4) * spread, plus the terms above."""
    q8, k8, v8, sc = draw_fp8(1, 2, 512, 128, 73, device="cuda")
    sq, sk, sv = sc
    scale = 1 / math.sqrt(128)
    o, lse = fa_fwd_fp8(q8, k8, v8, *sc, False, scale)
    assert fa_device_status() == 0
    for hh in range(2):
        q, k, v = _dec(q8[0, hh], sq), _dec(k8[0, hh], sk), _dec(v8[0, hh], sv)
        o_ex, lse_ex = oracle.fwd(q, k, v, False, scale)
        spread = oracle.fwd_spread(q, k, v, False, scale)
        e = 2.0 ** -4
        tol = 2 * e / (1 - e) * spread + 0.5 * bf16_ulp(o_ex) + 2.0 ** -12 * np.abs(v).max() + 1e-3
        assert np.all(np.abs(to_np(o[0, hh]) - o_ex) <= tol)
        assert np.max(np.abs(to_np(lse[0, hh]) - lse_ex)) <= 1e-3


def test_fp8_deterministic():
    q8, k8, v8, sc = draw_fp8(2, 4, 2048, 128, 74, device="cuda")
    a = fa_fwd_fp8(q8, k8, v8, *sc, True)
    b = fa_fwd_fp8(q8, k8, v8, *sc, True)
    assert fa_device_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_full_size_workload():
    """The FP8 workload bench.py times (B2 H16 N8192 d128, non-causal):
    every output finite, two heads against the oracle."""
    import bench
    from exact_attention_48_gb300.inputs import FP8_B2H16N8192D128 as w
    pb = bench.Problem(w)
    q8, k8, v8, _ = pb.inputs
    o = pb.outputs[0]
    pb.fwd(q8, k8, v8, o, pb.lse)
    assert fa_device_status() == 0
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(pb.lse).all())
    _check(q8, k8, v8, pb.fp8_scales, o, pb.lse, w.causal, w.scale, w.name, heads=[0, w.B * w.H - 1])
