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
    e4m3 can explain (relative 2^-4 per normal weight);
  * a hand-worked example (tests/golden/fp8_hand_d4.json) fixes M_i =
    ceil(max) against floor and round: one weight in the subnormal range,
    one maximum whose floor would saturate the largest weight;
  * the per-element bound: it covers the worst change of the flagged
    weights and is tight for it; every weight it leaves unflagged keeps
    its rounding under the score error model; and a tiled pass written
    here, whose integer running maximum lags the row maximum by up to
    STALE binades in random patterns, stays within it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

F8 = torch.float8_e4m3fn
# The tolerance model the GPU tests use: relative precision of the
# hardware's fp32 sums of e4m3 products, and how many binades a tiled pass's
# integer running maximum may lag the row maximum.
ACC_REL = 2.0 ** -13
STALE = 2


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


def _golden_fp8():
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "fp8_hand_d4.json")) as f:
        return json.load(f)


def test_fp8_hand_worked_example(lib=None):
    """The definition evaluated by hand on two tiny heads (derivation in the
    fixture): M = ceil(max x), e4m3 weights, normalised by their sum."""
    g = _golden_fp8()
    q8, k8, v8 = (torch.tensor(g[n], dtype=torch.float32).to(F8) for n in ("q", "k", "v"))
    for n, t in (("q", q8), ("k", k8), ("v", v8)):   # the inputs are exact e4m3 values
        assert np.array_equal(_dec(t), np.array(g[n], dtype=np.float64))
    o, lse = oracle.fwd_fp8(q8, k8, v8, g["sq"], g["sk"], g["sv"], False, g["scale"], lib=lib)
    np.testing.assert_allclose(o, np.array(g["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(g["lse"]), rtol=0, atol=1e-12)
    r = oracle.fwd_fp8_detail(q8, k8, v8, g["sq"], g["sk"], g["sv"], False, g["scale"], lib=lib)
    for h in range(2):
        assert np.all(r["M"][h] == g["M"][h])
        for i in range(3):
            np.testing.assert_array_equal(r["w"][h, i], np.array(g["weights"][h]))


def _bound_case(seed, causal, mult=2.0, N=48, d=32, acc_rel=ACC_REL, stale=STALE, lib=None):
    q8, k8, v8 = _random_case(seed, H=2, N=N, d=d, mult=mult)
    sq = sk = 1 / 16
    scale = 1 / math.sqrt(d)
    r = oracle.fwd_fp8_detail(q8, k8, v8, sq, sk, 1.0, causal, scale, acc_rel, stale, lib=lib)
    return q8, k8, v8, sq, sk, scale, r


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_bound_covers_and_is_tight_for_worst_weight_changes(causal, lib=None):
    """Move every flagged weight by its allowed change (delta) in the
    direction that pushes each output element furthest, renormalise, and
    recompute O directly: the change stays within the bound, and reaches
    it up to the factor (W - sum delta) / (W + sum delta).  Random sign
    patterns stay within it too."""
    _, _, v8, _, _, _, r = _bound_case(51, causal, lib=lib)
    v = _dec(v8)
    w, dl, o, b = r["w"], r["delta"], r["o"], r["bound"]
    assert (dl > 0).sum() > 20, "the case must exercise the bound"
    rng = np.random.default_rng(5)
    H, Nq, Nk = w.shape
    for h in range(H):
        for i in range(Nq):
            flagged = dl[h, i] > 0
            if not flagged.any():
                assert np.all(b[h, i] == 0.0)
                continue
            diff = v[h] - o[h, i][None, :]                      # [Nk, d]
            patterns = [np.sign(diff), -np.sign(diff)] + [rng.choice([-1.0, 1.0], size=diff.shape) for _ in range(4)]
            W, S = w[h, i].sum(), dl[h, i].sum()
            for k, eps in enumerate(patterns):
                wp = w[h, i][:, None] + eps * dl[h, i][:, None]   # per output column
                op = (wp * v[h]).sum(0) / wp.sum(0)
                change = np.abs(op - o[h, i])
                assert np.all(change <= b[h, i] * (1 + 1e-9) + 1e-15), (h, i, k)
                if k == 0:  # the aligned pattern nearly reaches the bound
                    assert np.all(change >= b[h, i] * (W - S) / (W + S) * (1 - 1e-9) - 1e-15), (h, i)


def test_fp8_unflagged_weights_keep_their_rounding(lib=None):
    """The scores recomputed here (decoded values, fp64) moved by the error
    model -- acc_rel * |c| * sum|q k| + 2^-23 |x| on the score, 2^-21
    relative on exp2 -- and rounded with PyTorch's float8 conversion: every
    weight the oracle leaves unflagged in the normal band keeps its value;
    every weight in the band below 2^(-5 + stale) is flagged with one
    subnormal step at the lagged scale; and the oracle's weights themselves
    are PyTorch's rounding of the exact 2^(x - M + 8)."""
    q8, k8, v8, sq, sk, scale, r = _bound_case(52, False, mult=2.0, N=64, lib=lib)
    q, k = sq * _dec(q8), sk * _dec(k8)
    c = scale / math.log(2.0)
    x = c * np.einsum("hid,hjd->hij", q, k)
    mag = abs(c) * np.einsum("hid,hjd->hij", np.abs(q), np.abs(k))
    M = np.ceil(x.max(-1))
    np.testing.assert_array_equal(M, r["M"])
    y = np.exp2(x - M[..., None] + 8.0)
    rnd = lambda a: torch.from_numpy(np.minimum(a, 448.0)).to(F8).to(torch.float64).numpy()  # noqa: E731
    np.testing.assert_array_equal(rnd(y), r["w"])
    dx = ACC_REL * mag + 2.0 ** -23 * np.abs(x)
    band = y < 2.0 ** (-5 + STALE)
    np.testing.assert_array_equal(r["delta"][band], 2.0 ** (-9 + STALE))
    normal_unflagged = (~band) & (r["delta"] == 0)
    for sx in (-1.0, 1.0):
        for se in (-1.0, 1.0):
            yp = np.exp2(x + sx * dx - M[..., None] + 8.0) * (1.0 + se * 2.0 ** -21)
            same = rnd(yp) == r["w"]
            assert np.all(same[normal_unflagged]), "an unflagged weight can round the other way"
    assert (r["delta"][~band] > 0).any(), "the case must flag some weights near a rounding midpoint"


def _tiled_fp8_pass(x, v, lag, rng, blk=8):
    """An FP8 forward pass over key blocks with an integer running maximum
    m that may lag the row maximum seen so far by up to `lag` binades: the
    weights of a block are e4m3(2^(x - m + 8 - lag)) (never above 2^8), the
    sums of weights and of weighted values are kept in fp64 and rescaled by
    2^(m_old - m_new) when m moves (it must once the maximum seen exceeds
    it by more than `lag`; where it lands in the allowed range is drawn at
    random).  x: [Nk] scores in log2 units (-inf where masked); v: [Nk, d]."""
    to8 = lambda a: torch.from_numpy(a).to(F8).to(torch.float64).numpy()  # noqa: E731
    m, acc, wsum, seen = None, np.zeros(v.shape[1]), 0.0, -np.inf
    for j0 in range(0, x.shape[0], blk):
        xb, vb = x[j0:j0 + blk], v[j0:j0 + blk]
        if not np.isfinite(xb).any():
            continue
        seen = max(seen, float(np.max(xb)))
        r = math.ceil(seen)
        if m is None or r - m > lag:
            m_new = r - int(rng.integers(0, lag + 1))
            if m is not None:
                acc, wsum = acc * 2.0 ** (m - m_new), wsum * 2.0 ** (m - m_new)
            m = m_new
        wb = to8(np.exp2(xb - m + 8 - lag))
        acc = acc + wb @ vb
        wsum += wb.sum()
    return acc / wsum


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_tiled_pass_with_lagging_maximum_stays_within_bound(causal, lib=None):
    """Against a tiled pass written here with random lag patterns up to
    STALE (exact scores, so only the rounding grid differs): every output
    element within the oracle's bound for stale = STALE (acc_rel = 0)."""
    q8, k8, v8, sq, sk, scale, r = _bound_case(53, causal, mult=2.5, N=64, acc_rel=0.0, lib=lib)
    q, k, v = sq * _dec(q8), sk * _dec(k8), _dec(v8)
    x = scale / math.log(2.0) * np.einsum("hid,hjd->hij", q, k)
    if causal:
        x = np.where(np.tril(np.ones(x.shape[-2:], dtype=bool)), x, -np.inf)
    rng = np.random.default_rng(9)
    worst = 0.0
    for h in range(x.shape[0]):
        for i in range(x.shape[1]):
            for _ in range(3):
                o_t = _tiled_fp8_pass(x[h, i], v[h], STALE, rng)
                excess = np.abs(o_t - r["o"][h, i]) - r["bound"][h, i]
                assert np.all(excess <= 1e-13), (h, i, float(excess.max()))
                worst = max(worst, float(np.max(np.abs(o_t - r["o"][h, i]))))
    assert worst > 0.0, "the lag must change some roundings"


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
    lambda lib: test_fp8_hand_worked_example(lib),
    lambda lib: [test_fp8_bound_covers_and_is_tight_for_worst_weight_changes(c, lib) for c in (False, True)],
    lambda lib: test_fp8_unflagged_weights_keep_their_rounding(lib),
    lambda lib: [test_fp8_tiled_pass_with_lagging_maximum_stays_within_bound(c, lib) for c in (False, True)],
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
    ("max_scale_floor", "double M = ceil(mx);", "double M = floor(mx);"),
    ("max_scale_round", "double M = ceil(mx);", "double M = nearbyint(mx);"),
    ("bound_halved", "bi[cc] = (W - dsum > 0.0) ? fabs(J->sv) * b / (W - dsum) : INFINITY;",
     "bi[cc] = (W - dsum > 0.0) ? 0.5 * fabs(J->sv) * b / (W - dsum) : INFINITY;"),
    ("bound_ignores_lag_band", "if (y < ldexp(1.0, -5 + J->stale)) {", "if (y < ldexp(1.0, -5)) {"),
    ("bound_ignores_lag_step", "delta = ldexp(1.0, -9 + J->stale);", "delta = ldexp(1.0, -9);"),
    ("bound_ignores_score_error", "if (fabs(y - mid) <= rel * y) delta = ulp;", "if (fabs(y - mid) <= 0.0 * y) delta = ulp;"),
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
