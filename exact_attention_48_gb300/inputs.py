"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only names the workloads and
draws i.i.d. Gaussian tensors from a seeded generator.  Both the CUDA path
and the fp64 oracle are fed the very same (bf16-rounded) tensors it returns.

Workloads.  The pages measure on GPT-style training without naming a
dataset, so dense i.i.d. N(0, 1) tensors of the training shapes stand in for
it: no padding, no variable lengths, one square mask convention (key j is
visible to query i iff j <= i when causal).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    backward: bool = True
    input_mult: float = 1.0   # Q/K/V are N(0,1) * input_mult (dO stays N(0,1))
    seed: int = 1000
    note: str = field(default="", compare=False)
    layout: str = "bhnd"      # "bhnd" contiguous, "bnhd" ([B, N, H, d] storage), "varlen" (packed sequences),
                              # "decode" (nq query rows against a cache of N keys), "fp8" (e4m3 inputs)
    lengths: tuple = ()       # varlen: the B sequence lengths (N is the longest)
    nq: int = 0               # decode: query rows per head

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops_fwd(self) -> float:
        if self.layout == "varlen":
            f = sum(4.0 * self.H * n * n * self.d for n in self.lengths)
        elif self.layout == "decode":
            f = 4.0 * self.B * self.H * self.nq * self.N * self.d
        else:
            f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        return 2.5 * self.flops_fwd()


# The five workload families: a tiny oracle check, a forward-only shape, a
# causal training shape, a long-context shape and a sequence-length sweep.
TINY = Workload("tiny_b1h2n128d64", 1, 2, 128, 64, False, True, 1.0, 1000,
                "oracle check; drawn in fp32, GPU sees the bf16 cast")
FWD_B8H16N2048D64 = Workload("fwd_b8h16n2048d64", 8, 16, 2048, 64, False, False, 1.0, 1001,
                             "forward only, non-causal")
CAUSAL_B4H32N4096D128 = Workload("causal_b4h32n4096d128", 4, 32, 4096, 128, True, True, 1.0, 1002,
                                 "causal LM training shape")
LONG_B1H16N16384D128 = Workload("long_b1h16n16384d128x2", 1, 16, 16384, 128, True, True, 2.0, 1003,
                                "long context, inputs x2 (sharper softmax)")


def sweep(N: int, d: int, causal: bool) -> Workload:
    """B*N fixed at 16384 tokens, H = 16."""
    B = 16384 // N
    return Workload(f"sweep_b{B}h16n{N}d{d}{'_causal' if causal else ''}", B, 16, N, d, causal,
                    True, 1.0, 1004 + N * 10 + d)


def varlen_lengths(total: int, lo: int, hi: int, seed: int) -> tuple:
    """Seeded sequence lengths in [lo, hi] adding up to ``total`` (the last
    one takes the remainder, at least 1)."""
    g = torch.Generator()
    g.manual_seed(int(seed))
    out, left = [], total
    while left > hi:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g))
        out.append(n)
        left -= n
    out.append(left)
    return tuple(out)


# The strided and packed paths measured on training-like shapes: the
# headline shape stored [B, N, H, d], and 16384 tokens of sequences of
# 256..4096 tokens packed back to back (causal, as in packed LM training).
BNHD_B2H16N8192D128 = Workload("bnhd_b2h16n8192d128", 2, 16, 8192, 128, False, True, 1.0, 1005,
                               "headline shape, [B, N, H, d] storage", layout="bnhd")
_VL = varlen_lengths(16384, 256, 4096, 1006)
VARLEN_T16384H16D128 = Workload("varlen_t16384h16d128_causal", len(_VL), 16, max(_VL), 128, True, True, 1.0,
                                1006, "packed sequences of 256..4096 tokens", layout="varlen", lengths=_VL)

# The headline shape in FP8 (e4m3 Q, K, V with per-tensor scales), forward.
FP8_B2H16N8192D128 = Workload("fp8_b2h16n8192d128", 2, 16, 8192, 128, False, False, 1.0, 1008,
                              "headline shape, e4m3 inputs", layout="fp8")

# Decoding one token per sequence against a 16384-token key/value cache
# (bf16, contiguous [B, H, N, d] cache): HBM-bound, 2 GiB of cache per step.
DECODE_B16H16NK16384D128 = Workload("decode_b16h16nk16384d128", 16, 16, 16384, 128, False, False, 1.0, 1007,
                                    "one query row per head against a 16384-key cache", layout="decode", nq=1)
# The same cache with eight query rows per head (speculative or grouped
# decoding): the products run on the tensor core.
DECODE_B16H16NQ8NK16384D128 = Workload("decode_b16h16nq8nk16384d128", 16, 16, 16384, 128, False, False, 1.0, 1009,
                                       "eight query rows per head against a 16384-key cache", layout="decode",
                                       nq=8)

SWEEP_N = (512, 1024, 2048, 4096, 8192, 16384)
HEADLINE = sweep(8192, 128, False)   # B=2, H=16, N=8192, d=128, non-causal


def draw(w: Workload, device="cpu", dtype=torch.bfloat16, with_dout: bool = True):
    """Return (q, k, v, dout) for workload ``w`` as contiguous [B, H, N, d] tensors.

    Values are drawn in fp32 (order q, k, v, dout) from ``torch.Generator``
    seeded with ``w.seed`` on ``device`` and then cast to ``dtype``.
    """
    return draw_shape(w.B, w.H, w.N, w.d, w.seed, w.input_mult, device, dtype, with_dout)


def draw_shape(B, H, N, d, seed, input_mult=1.0, device="cpu", dtype=torch.bfloat16,
               with_dout=True):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    out = []
    for i in range(4 if with_dout else 3):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if i < 3 and input_mult != 1.0:
            x = x * input_mult
        out.append(x.to(dtype).contiguous())
    if not with_dout:
        out.append(None)
    return tuple(out)


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor e4m3 quantisation of an fp32 tensor for the FP8 inputs:
    scale = amax / 448 (the format's largest finite value), codes = x /
    scale rounded by PyTorch's float8_e4m3fn conversion.  Returns (codes,
    scale)."""
    amax = float(x.abs().max())
    scale = amax / 448.0 if amax > 0 else 1.0
    return (x / scale).to(torch.float8_e4m3fn), scale


def draw_fp8(B, H, N, d, seed, input_mult=1.0, device="cpu"):
    """(q8, k8, v8, (sq, sk, sv)): N(0,1) * input_mult drawn in the order q,
    k, v from a generator seeded with ``seed``, each quantised per tensor."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out, scales = [], []
    for _ in range(3):
        x = torch.randn((B, H, N, d), generator=g, device=device, dtype=torch.float32) * input_mult
        c, s = quantize_e4m3(x)
        out.append(c)
        scales.append(s)
    return out[0], out[1], out[2], tuple(scales)
