"""Two independent key tilings of the same forward must agree within rounding.

fa_fwd walks all keys of a query row in 128-key tiles in one pass with a
running maximum.  fa_fwd_decode cuts the keys into chunks, normalises each
chunk on its own and merges the partial results by their logsumexps.  It
uses fp32 weights on the CUDA cores for one query row and bf16 weights on
the tensor core for 2..8 rows.  For the last Nq query rows of a square
problem the two calls see the same keys: decode's bottom-right causal
alignment makes query i of Nq see keys j <= N - Nq + i, which is exactly
the square causal mask on rows N - Nq .. N - 1.  Each output lies within
its own rounding bound of the fp64 oracle, so the two agree within the sum
of those bounds.  Their logsumexps are both fp32 sums of fp32 weights and
agree much more closely than the oracle tolerance.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_48_gb300 import fa_device_status, fa_fwd, fa_fwd_decode
from parity import o_bound, to_np

pytestmark = pytest.mark.gpu

LSE_AGREE = 1e-4


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq", [1, 4, 8])
def test_forward_and_decode_agree_on_last_rows(d, causal, Nq):
    B, H, N = 2, 3, 2000  # 15 full key tiles and a ragged one; several decode chunks
    g = torch.Generator(device="cuda")
    g.manual_seed(700 + d + 10 * Nq + int(causal))
    q, k, v = (torch.randn(B, H, N, d, generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    scale = 1.0 / math.sqrt(d)
    o_full, lse_full = fa_fwd(q, k, v, causal, scale)
    q_tail = q[:, :, N - Nq:].contiguous()
    o_dec, lse_dec = fa_fwd_decode(q_tail, k, v, None, causal, scale)
    assert fa_device_status() == 0

    o_a, o_b = to_np(o_full[:, :, N - Nq:]), to_np(o_dec)
    lse_err = float(np.max(np.abs(to_np(lse_full[:, :, N - Nq:]) - to_np(lse_dec))))
    assert lse_err <= LSE_AGREE, f"logsumexps differ by {lse_err:.3e}"
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                row = N - Nq + i
                end = row + 1 if causal else N
                qi, kb, vb = q[b, h, row:row + 1], k[b, h, :end], v[b, h, :end]
                o_ref, _ = oracle.fwd(qi, kb, vb, False, scale)
                bound = 2.0 * o_bound(o_ref, to_np(oracle.fwd_spread(qi, kb, vb, False, scale)))
                err = np.abs(o_a[b, h, i:i + 1] - o_b[b, h, i:i + 1])
                assert np.all(err <= bound), (f"b{b} h{h} row {row}: the two tilings differ by {err.max():.3e}, "
                                              f"bound {bound[np.unravel_index(np.argmax(err), err.shape)]:.3e}")
