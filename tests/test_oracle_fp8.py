"""Pins of the oracle's FP8 forward (CPU only).

The FP8 forward's definition is in oracle/attn_oracle.c.  What fixes it
independently of that code:
  * the e4m3 format: every code's value and the rounding of real numbers
    against PyTorch's float8_e4m3fn conversion (a library routine);
  * where the rounded weights are exact (integer scores), the FP8 forward
    is exact attention on the decoded values (the plain oracle);
  * the logsumexp is the exact one of the decoded, scaled scores;
  * Q = 0 gives the (prefix) mean of V with LSE = ln(count); constant V
    returns V (the rounded weights are normalised by their own sum);
  * O differs from exact attention by no more than rounding each weight to
    e4m3 can explain (relative 2^-4 per normal weight).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

F8 = torch.float8_e4m3fn


def test_e4m3_values_match_torch(lib=None):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(F8).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(c, lib=lib) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(mine))
    assert set(np.flatnonzero(nan).tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan], mine[~nan])
    assert np.nanmax(mine) == 448.0 and mine[1] == 2.0 ** -9


def test_e4m3_round_matches_torch(lib=None):
    g = torch.Generator().manual_seed(3)
    # magnitudes from far below the subnormals to the top of the range, both signs
    mag = torch.exp2(torch.rand(20000, generator=g, dtype=torch.float64) * 23.0 - 14.0)
    x = (mag * torch.where(torch.rand(20000, generator=g) < 0.5, -1.0, 1.0)).to(torch.float32)
    # every midpoint between neighbouring finite values (ties must go to even)
    vals = np.unique(np.array([oracle.e4m3_value(c) for c in range(0x7F)]))
    mids = torch.tensor((vals[1:] + vals[:-1]) / 2, dtype=torch.float32)
    x = torch.cat([x, mids, -mids, torch.tensor(vals, dtype=torch.float32)])
    x = x[x.abs() <= 448]
    ref = x.to(F8).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_round(float(v), lib=lib) for v in x.tolist()])
    bad = np.flatnonzero(ref != mine)
    assert bad.size == 0, f"{bad.size} mismatches, e.g. x={x[bad[0]].item()!r}: torch {ref[bad[0]]}, oracle {mine[bad[0]]}"
    assert oracle.e4m3_round(500.0) == 448.0 and oracle.e4m3_round(-1e9) == -448.0  # saturation


def _codes(shape, g, lo=-8, hi=8):
    """e4m3 codes of small integers (exact in the format)."""
    ints = torch.randint(lo, hi + 1, shape, generator=g).to(torch.float32)
    return ints.to(F8)


def _dec(x8):
    return x8.to(torch.float64).numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_equals_exact_attention_when_weights_are_exact(causal, lib=None):
    """scale = ln 2 and integer q, k make every score an integer: each weight
    2^(x - M + 8) is then a power of two >= 2^-6 (scores kept within 14 of
    the max), exact in e4m3, so the FP8 forward is exact attention."""
    g = torch.Generator().manual_seed(11)
    N, d = 40, 16
    q8 = _codes((2, N, d), g, -1, 1)
    k8 = _codes((2, N, d), g, -1, 1)
    v8 = (torch.randn(2, N, d, generator=g) * 3).to(F8)
    q, k, v = _dec(q8), _dec(k8), _dec(v8)
    x = np.einsum("hid,hjd->hij", q, k)
    assert np.all(np.abs(x) <= 14)  # keeps every weight normal
    o8, lse8 = oracle.fwd_fp8(q8, k8, v8, 1.0, 1.0, 1.0, causal, math.log(2.0), lib=lib)
    o, lse = oracle.fwd(q, k, v, causal, math.log(2.0))
    np.testing.assert_allclose(o8, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse8, lse, rtol=0, atol=1e-12)


def test_fp8_tensor_scales(lib=None):
    """sq, sk scale the scores and sv scales O: the same exact case with
    scales 2, 1/2, 3 and the softmax scale unchanged in effect."""
    g = torch.Generator().manual_seed(12)
    N, d = 24, 8
    q8, k8 = _codes((1, N, d), g, -1, 1), _codes((1, N, d), g, -1, 1)
    v8 = (torch.randn(1, N, d, generator=g) * 2).to(F8)
    o8, lse8 = oracle.fwd_fp8(q8, k8, v8, 2.0, 0.5, 3.0, False, math.log(2.0), lib=lib)
    o, lse = oracle.fwd(_dec(q8), _dec(k8), 3.0 * _dec(v8), False, math.log(2.0))
    np.testing.assert_allclose(o8, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse8, lse, rtol=0, atol=1e-12)
    o8b, lse8b = oracle.fwd_fp8(q8, k8, v8, 4.0, 1.0, 1.0, False, math.log(2.0), lib=lib)
    ob, lseb = oracle.fwd(4.0 * _dec(q8), _dec(k8), _dec(v8), False, math.log(2.0))
    np.testing.assert_allclose(lse8b, lseb, rtol=0, atol=1e-12)


def _random_case(seed, H=2, N=64, d=32, mult=1.0):
    g = torch.Generator().manual_seed(seed)
    q8, k8, v8 = ((torch.randn(H, N, d, generator=g) * mult * 16).to(F8) for _ in range(3))
    return q8, k8, v8


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_lse_is_exact(causal, lib=None):
    q8, k8, v8 = _random_case(21)
    sq, sk, scale = 1 / 16, 1 / 16, 1 / math.sqrt(32)
    _, lse8 = oracle.fwd_fp8(q8, k8, v8, sq, sk, 1.0, causal, scale, lib=lib)
    _, lse = oracle.fwd(sq * _dec(q8), sk * _dec(k8), _dec(v8), causal, scale)
    np.testing.assert_allclose(lse8, lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_zero_queries_and_constant_values(causal, lib=None):
    _, k8, v8 = _random_case(22)
    H, N, d = k8.shape
    q8 = torch.zeros(H, N, d).to(F8)
    o8, lse8 = oracle.fwd_fp8(q8, k8, v8, 1.0, 1.0, 0.5, causal, 0.3, lib=lib)
    v = 0.5 * _dec(v8)
    cnt = np.arange(1, N + 1)[:, None] if causal else N
    mean = np.cumsum(v, axis=1) / cnt if causal else np.repeat(v.mean(axis=1, keepdims=True), N, axis=1)
    np.testing.assert_allclose(o8, mean, rtol=0, atol=1e-12)
    want = np.broadcast_to(np.arange(1, N + 1), lse8.shape) if causal else np.full(lse8.shape, float(N))
    np.testing.assert_allclose(lse8, np.log(want), rtol=0, atol=1e-12)
    # constant V: the normalised rounded weights return it exactly, whatever the scores
    q8r, _, _ = _random_case(23)
    vc = torch.full((H, N, d), 2.5).to(F8)
    o8c, _ = oracle.fwd_fp8(q8r, k8, vc, 1 / 16, 1 / 16, 1.0, causal, 1 / math.sqrt(d), lib=lib)
    np.testing.assert_allclose(o8c, np.full(o8c.shape, 2.5), rtol=0, atol=1e-12)


@pytest.mark.parametrize("mult", [1.0, 2.0])
def test_fp8_close_to_exact_within_rounding(mult, lib=None):
    """Rounding each weight to e4m3 moves it by at most 2^-4 of itself
    (normal range) or 2^-10 absolute (in the weights' 2^8 scale), and the
    weights are renormalised: |O8 - O| <= 2^-4/(1-2^-4) * 2 * spread + the
    subnormal part."""
    q8, k8, v8 = _random_case(31, N=96, mult=mult)
    sq = sk = 1 / 16
    scale = 1 / math.sqrt(32)
    o8, _ = oracle.fwd_fp8(q8, k8, v8, sq, sk, 1.0, False, scale, lib=lib)
    q, k, v = sq * _dec(q8), sk * _dec(k8), _dec(v8)
    o, _ = oracle.fwd(q, k, v, False, scale)
    spread = oracle.fwd_spread(q, k, v, False, scale)
    e = 2.0 ** -4
    bound = 2 * e / (1 - e) * spread + 96 * 2.0 ** -10 / 128 * np.abs(v).max() + 1e-12
    assert np.all(np.abs(o8 - o) <= bound)
    # and the rounding is visible: the FP8 result is not the exact one
    assert np.abs(o8 - o).max() > 1e-4


def test_fp8_bound_flags_nothing_for_exact_weights():
    g = torch.Generator().manual_seed(41)
    q8, k8 = _codes((1, 16, 8), g, -1, 1), _codes((1, 16, 8), g, -1, 1)
    v8 = torch.randn(1, 16, 8, generator=g).to(F8)
    _, _, b = oracle.fwd_fp8(q8, k8, v8, 1.0, 1.0, 1.0, False, math.log(2.0), acc_rel=0.0, with_bound=True)
    # integer scores: every weight a power of two far from any rounding midpoint
    assert np.all(b == 0.0)


# Plausible mistakes in the FP8 part of the oracle source; each must be
# caught by one of the pins above (run against a mutated copy).
FP8_PINS = [
    lambda lib: test_e4m3_values_match_torch(lib),
    lambda lib: test_e4m3_round_matches_torch(lib),
    lambda lib: [test_fp8_equals_exact_attention_when_weights_are_exact(c, lib) for c in (False, True)],
    lambda lib: test_fp8_tensor_scales(lib),
    lambda lib: [test_fp8_lse_is_exact(c, lib) for c in (False, True)],
    lambda lib: [test_fp8_zero_queries_and_constant_values(c, lib) for c in (False, True)],
    lambda lib: [test_fp8_close_to_exact_within_rounding(m, lib) for m in (1.0, 2.0)],
]
FP8_MUTATIONS = [
    ("normalise_by_unrounded_sum", "oi[cc] = J->sv * acc / W;", "oi[cc] = J->sv * acc / Z;"),
    ("drop_value_scale", "oi[cc] = J->sv * acc / W;", "oi[cc] = acc / W;"),
    ("lse_from_rounded_weights", "log(2.0) * (M - 8.0 + log2(Z));", "log(2.0) * (M - 8.0 + log2(W));"),
    ("drop_query_key_scales", "J->scale * J->sq * J->sk / log(2.0);", "J->scale / log(2.0);"),
    ("natural_exp_for_weights", "double y = exp2(x[j] - M + 8.0);", "double y = exp(x[j] - M + 8.0);"),
    ("weights_unrounded", "w[j] = e4m3_round(y);", "w[j] = y;"),
    ("causal_off_by_one_fp8", "long end = J->causal ? (i + 1 < J->Nk ? i + 1 : J->Nk) : J->Nk;",
     "long end = J->causal ? (i < J->Nk ? i : J->Nk) : J->Nk;"),
    ("mantissa_two_bits", "double ulp = ldexp(1.0, e - 3);", "double ulp = ldexp(1.0, e - 2);"),
    ("exponent_bias_8", "else v = ldexp(1.0 + m / 8.0, e - 7);", "else v = ldexp(1.0 + m / 8.0, e - 8);"),
]


@pytest.mark.parametrize("name,old,new", FP8_MUTATIONS, ids=[m[0] for m in FP8_MUTATIONS])
def test_fp8_pins_catch_mutation(name, old, new, tmp_path):
    import subprocess
    src_path = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")
    text = open(src_path).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not unique"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-shared",
                    "-fPIC", "-pthread", str(src), "-o", str(so), "-lm"], check=True)
    lib = oracle.bind(str(so))
    caught = 0
    for pin in FP8_PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError, FloatingPointError):
            caught += 1
    assert caught, f"no FP8 pin caught mutation {name}"
