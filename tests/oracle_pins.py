"""Checks that pin the fp64 oracle to facts other than itself.

Each ``pin_*`` function takes an optional ``lib`` (another build of the
oracle source, used by the mutation checks) and raises AssertionError when
the oracle disagrees with the fact it checks.  The facts are closed forms,
invariants of softmax attention, central finite differences, a hand-worked
example stored under ``tests/golden/`` and a library routine (PyTorch's fp64
CPU scaled-dot-product attention with autograd).  Together they are chosen so
that a dropped term, a wrong sign or index, or a swapped operand anywhere in
the oracle trips at least one of them (``test_oracle_mutations.py`` plants
such mistakes and checks that).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _qkv(seed, BH=2, N=16, d=8, Nk=None):
    r = _rng(seed)
    Nk = N if Nk is None else Nk
    q = r.standard_normal((BH, N, d))
    k = r.standard_normal((BH, Nk, d))
    v = r.standard_normal((BH, Nk, d))
    do = r.standard_normal((BH, N, d))
    return q, k, v, do


def pin_hand_example(lib=None):
    """Two-token example worked by hand (closed form), forward and backward."""
    g = json.load(open(os.path.join(GOLDEN, "hand_n2_d1.json")))
    q, k, v, do = (np.array(g[x])[None] for x in ("q", "k", "v", "dout"))
    for mode, causal in (("noncausal", False), ("causal", True)):
        exp = g[mode]
        o, lse = oracle.fwd(q, k, v, causal, g["scale"], lib=lib)
        dq, dk, dv = oracle.bwd(q, k, v, do, causal, g["scale"], lib=lib)
        for name, got in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
            np.testing.assert_allclose(got[0], np.array(exp[name]), rtol=0, atol=1e-13,
                                       err_msg=f"{mode} {name}")


def pin_rows_sum_to_one(lib=None):
    """Each softmax row sums to 1, entries are non-negative, masked entries are 0."""
    q, k, _, _ = _qkv(1, 1, 37, 5)
    for causal in (False, True):
        p = oracle.probs(q[0], k[0], causal, 0.7, lib=lib)
        assert np.all(p >= 0)
        assert np.max(np.abs(p.sum(1) - 1.0)) <= 1e-14
        if causal:
            assert np.all(np.triu(p, 1) == 0)
            assert np.all(np.diag(p) > 0)
        else:
            assert np.all(p > 0)


def pin_constant_v(lib=None):
    """If every value row is the same vector c, every output row is c."""
    q, k, v, _ = _qkv(2, 2, 24, 6)
    c = _rng(3).standard_normal(6)
    v[:] = c
    for causal in (False, True):
        o, _ = oracle.fwd(q, k, v, causal, 0.9, lib=lib)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-14)


def pin_zero_query(lib=None):
    """Q = 0: uniform weights, so O is the mean of the visible values and LSE = ln(count)."""
    _, k, v, _ = _qkv(4, 2, 20, 7)
    q = np.zeros((2, 20, 7))
    o, lse = oracle.fwd(q, k, v, False, 0.5, lib=lib)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(1, keepdims=True), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, np.full(lse.shape, math.log(20)), atol=1e-14)
    o, lse = oracle.fwd(q, k, v, True, 0.5, lib=lib)
    prefix = np.cumsum(v, axis=1) / np.arange(1, 21)[None, :, None]
    np.testing.assert_allclose(o, prefix, atol=1e-14)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, 21)), lse.shape), atol=1e-14)


def pin_causal_row0(lib=None):
    """Causal row 0 sees only key 0: O_0 = v_0 and LSE_0 = s q_0 . k_0."""
    q, k, v, _ = _qkv(5, 3, 11, 9)
    s = 0.37
    o, lse = oracle.fwd(q, k, v, True, s, lib=lib)
    np.testing.assert_allclose(o[:, 0], v[:, 0], atol=1e-15)
    np.testing.assert_allclose(lse[:, 0], s * np.einsum("bc,bc->b", q[:, 0], k[:, 0]), atol=1e-14)


def pin_single_token(lib=None):
    """N = 1: O = v, LSE = s q . k, dV = dO, dQ = dK = 0."""
    q, k, v, do = _qkv(6, 2, 1, 5)
    s = 1.3
    for causal in (False, True):
        o, lse = oracle.fwd(q, k, v, causal, s, lib=lib)
        np.testing.assert_allclose(o, v, atol=1e-15)
        np.testing.assert_allclose(lse[:, 0], s * np.einsum("bc,bc->b", q[:, 0], k[:, 0]), atol=1e-14)
        dq, dk, dv = oracle.bwd(q, k, v, do, causal, s, lib=lib)
        np.testing.assert_allclose(dv, do, atol=1e-15)
        assert np.max(np.abs(dq)) <= 1e-15 and np.max(np.abs(dk)) <= 1e-15


def pin_key_shift(lib=None):
    """Adding one vector u to every key leaves O unchanged and shifts LSE_i by s q_i . u."""
    q, k, v, _ = _qkv(7, 2, 19, 6)
    u = _rng(8).standard_normal(6)
    s = 0.8
    o1, l1 = oracle.fwd(q, k, v, False, s, lib=lib)
    o2, l2 = oracle.fwd(q, k + u, v, False, s, lib=lib)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, s * q @ u, atol=1e-12)


def pin_key_permutation(lib=None):
    """Permuting keys and values together (no mask) changes neither O nor LSE,
    and permutes dK, dV the same way while leaving dQ unchanged."""
    q, k, v, do = _qkv(9, 2, 23, 5)
    perm = _rng(10).permutation(23)
    s = 0.6
    o1, l1 = oracle.fwd(q, k, v, False, s, lib=lib)
    o2, l2 = oracle.fwd(q, k[:, perm], v[:, perm], False, s, lib=lib)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(l2, l1, atol=1e-13)
    g1 = oracle.bwd(q, k, v, do, False, s, lib=lib)
    g2 = oracle.bwd(q, k[:, perm], v[:, perm], do, False, s, lib=lib)
    np.testing.assert_allclose(g2[0], g1[0], atol=1e-12)
    np.testing.assert_allclose(g2[1], g1[1][:, perm], atol=1e-12)
    np.testing.assert_allclose(g2[2], g1[2][:, perm], atol=1e-12)


def pin_gradient_identities(lib=None):
    """sum_j dK_j = 0 (rows of dS sum to 0) and sum_j dV_j = sum_i dO_i (rows of P sum to 1)."""
    q, k, v, do = _qkv(11, 2, 29, 6)
    for causal in (False, True):
        dq, dk, dv = oracle.bwd(q, k, v, do, causal, 0.45, lib=lib)
        np.testing.assert_allclose(dk.sum(1), 0.0, atol=1e-12)
        np.testing.assert_allclose(dv.sum(1), do.sum(1), atol=1e-12)


def pin_scale_sign(lib=None):
    """softmax(-s q k^T) = softmax(s q (-k)^T); s = 0 gives uniform weights."""
    q, k, v, do = _qkv(12, 2, 17, 4)
    for causal in (False, True):
        o1, l1 = oracle.fwd(q, k, v, causal, -0.7, lib=lib)
        o2, l2 = oracle.fwd(q, -k, v, causal, 0.7, lib=lib)
        np.testing.assert_allclose(o1, o2, atol=1e-14)
        np.testing.assert_allclose(l1, l2, atol=1e-14)
    o, lse = oracle.fwd(q, k, v, False, 0.0, lib=lib)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(1, keepdims=True), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(17), atol=1e-14)


def _loss(q, k, v, do, causal, s, lib):
    o, _ = oracle.fwd(q, k, v, causal, s, nthreads=1, lib=lib)
    return float(np.sum(do * o))


def _fd_check(q, k, v, do, causal, s, lib, idx_by_tensor):
    an = oracle.bwd(q, k, v, do, causal, s, nthreads=1, lib=lib)
    ins = [q, k, v]
    for t, idxs in enumerate(idx_by_tensor):
        scale_an = np.max(np.abs(an[t]))
        for idx in idxs:
            x = ins[t]
            x0 = x[idx]
            h = 1e-5 * max(1.0, abs(x0))
            x[idx] = x0 + h
            lp = _loss(*ins, do, causal, s, lib)
            x[idx] = x0 - h
            lm = _loss(*ins, do, causal, s, lib)
            x[idx] = x0
            fd = (lp - lm) / (2 * h)
            a = an[t][idx]
            rel = abs(fd - a) / max(abs(a), 1e-3 * scale_an)
            assert rel <= 1e-6, f"tensor {'qkv'[t]} idx {idx}: fd {fd} analytic {a} rel {rel}"


def pin_finite_differences_all(lib=None):
    """Central differences of L = sum(dO * O) match the analytic gradients on
    every element of a small case (B = H = 1, N = 8, d = 4), causal and not."""
    q, k, v, do = _qkv(13, 1, 8, 4)
    idx = [list(np.ndindex(q.shape))] * 3
    for causal in (False, True):
        _fd_check(q, k, v, do, causal, 0.5, lib, idx)


def pin_finite_differences_sampled(lib=None, n_samples=256):
    """Central differences on 256 seeded elements per tensor of the tiny
    workload's shape (one head of N = 128, d = 64, scale 1/8), non-causal."""
    q, k, v, do = _qkv(14, 1, 128, 64)
    r = _rng(15)
    idx = []
    for _ in range(3):
        flat = r.choice(128 * 64, size=n_samples, replace=False)
        idx.append([(0, int(f // 64), int(f % 64)) for f in flat])
    _fd_check(q, k, v, do, False, 0.125, lib, idx)


def pin_library_sdpa(lib=None):
    """PyTorch fp64 CPU scaled_dot_product_attention (math path) + autograd."""
    for seed, (BH, N, Nk, d, causal, s) in enumerate(
            [(2, 128, 128, 64, False, 0.125), (3, 45, 45, 16, True, 0.3),
             (2, 33, 70, 8, False, -0.4), (1, 64, 64, 32, True, 1.7)]):
        q, k, v, do = _qkv(100 + seed, BH, N, d, Nk)
        o, lse = oracle.fwd(q, k, v, causal, s, lib=lib)
        dq, dk, dv = oracle.bwd(q, k, v, do, causal, s, lib=lib)
        qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        with torch.nn.attention.sdpa_kernel(torch.nn.attention.SDPBackend.MATH):
            ot = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=s)
        ot.backward(torch.tensor(do))
        z = s * torch.tensor(q) @ torch.tensor(k).transpose(-1, -2)
        if causal:
            z = z.masked_fill(torch.ones(N, Nk, dtype=torch.bool).triu(1), float("-inf"))
        np.testing.assert_allclose(o, ot.detach().numpy(), atol=1e-13)
        np.testing.assert_allclose(lse, torch.logsumexp(z, -1).numpy(), atol=1e-13)
        np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-12)


def pin_spread(lib=None):
    """spread = sum_j P_ij |v_j - O_i|: 0 for constant V; for uniform weights
    over values +-1 (mean 0) it is 1; and it bounds the change of O when the
    weights are perturbed by a relative e and renormalised."""
    q, k, v, _ = _qkv(31, 2, 12, 5)
    v[:] = 0.7
    assert np.max(np.abs(oracle.fwd_spread(q, k, v, False, 0.4, lib=lib))) <= 1e-15
    q0 = np.zeros((1, 8, 3))
    v1 = np.tile(np.array([1.0, -1.0])[:, None], (4, 3))[None]
    np.testing.assert_allclose(oracle.fwd_spread(q0, _qkv(32, 1, 8, 3)[1], v1, False, 1.0, lib=lib), 1.0,
                               atol=1e-14)
    # perturbation bound, checked by brute force on one head
    q, k, v, _ = _qkv(33, 1, 9, 4)
    P = oracle.probs(q[0], k[0], False, 0.9, lib=lib)
    sp = oracle.fwd_spread(q, k, v, False, 0.9, lib=lib)[0]
    e = 1e-3
    r = _rng(34)
    for _ in range(20):
        Pt = P * (1 + e * r.uniform(-1, 1, P.shape))
        Pt /= Pt.sum(1, keepdims=True)
        dO = np.abs(Pt @ v[0] - P @ v[0])
        assert np.all(dO <= 2 * e * sp + 1e-15)


ALL_PINS = [
    pin_hand_example,
    pin_rows_sum_to_one,
    pin_constant_v,
    pin_zero_query,
    pin_causal_row0,
    pin_single_token,
    pin_key_shift,
    pin_key_permutation,
    pin_gradient_identities,
    pin_scale_sign,
    pin_finite_differences_all,
    pin_finite_differences_sampled,
    pin_library_sdpa,
    pin_spread,
]
