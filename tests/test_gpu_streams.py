"""Stream semantics of the backward pass, whose dQ kernel runs on a side
stream of the library's next to the dK/dV kernel.

* Work enqueued on the caller's stream right after fa_bwd (no host
  synchronisation in between) sees the finished gradients.
* Host threads calling fa_bwd at the same time on their own streams get
  the same results as one call alone (each thread has its own side stream).
* fa_fwd + fa_bwd captured into a CUDA graph (after a first call outside
  the capture) replay to the same bits as eager calls.
Every comparison is bitwise: the kernels are deterministic.
"""
import math
import threading

import pytest
import torch

from exact_attention_48_gb300 import fa_bwd, fa_bwd_workspace_bytes, fa_device_status, fa_fwd
from exact_attention_48_gb300.binding import fa_debug_time_next_bwd
from exact_attention_48_gb300.inputs import draw_shape

pytestmark = pytest.mark.gpu


def _inputs(B, H, N, d, seed):
    q, k, v, do = draw_shape(B, H, N, d, seed, 1.0, "cuda", torch.bfloat16)
    return q, k, v, do


def _sequential_reference(q, k, v, o, do, lse, causal, scale):
    """The same backward with its kernels one after the other (the timing
    hook makes the call run them in stream order)."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    fa_debug_time_next_bwd(*ev)
    out = fa_bwd(q, k, v, o, do, lse, causal, scale)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_results_visible_to_the_callers_stream(causal):
    B, H, N, d = 2, 8, 2048, 128
    scale = 1 / math.sqrt(d)
    q, k, v, do = _inputs(B, H, N, d, 201)
    o, lse = fa_fwd(q, k, v, causal, scale)
    ref = _sequential_reference(q, k, v, o, do, lse, causal, scale)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            grads = [torch.full_like(q, float("nan")) for _ in range(3)]
            fa_bwd(q, k, v, o, do, lse, causal, scale, dq=grads[0], dk=grads[1], dv=grads[2])
            copies = [g.clone() for g in grads]  # enqueued on s right after the call
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    for name, c, r in zip(("dq", "dk", "dv"), copies, ref):
        assert torch.equal(c, r), f"{name}: the caller's stream saw unfinished results"


def test_concurrent_host_threads():
    B, H, N, d = 2, 4, 1536, 128
    scale = 1 / math.sqrt(d)
    cases = []
    for t in range(3):
        q, k, v, do = _inputs(B, H, N, d, 210 + t)
        o, lse = fa_fwd(q, k, v, t == 1, scale)
        cases.append((q, k, v, o, do, lse, t == 1))
    refs = [_sequential_reference(*c[:6], c[6], scale) for c in cases]
    results = [None] * len(cases)
    errors = []

    def work(t):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                q, k, v, o, do, lse, causal = cases[t]
                outs = None
                for _ in range(4):
                    outs = fa_bwd(q, k, v, o, do, lse, causal, scale)
                results[t] = [x.clone() for x in outs]
            s.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(t,)) for t in range(len(cases))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    for t, (res, ref) in enumerate(zip(results, refs)):
        for name, x, r in zip(("dq", "dk", "dv"), res, ref):
            assert torch.equal(x, r), f"thread {t}: {name} differs from the call alone"


def test_graph_capture_of_forward_and_backward():
    B, H, N, d, causal = 2, 8, 1024, 128, True
    scale = 1 / math.sqrt(d)
    q, k, v, do = _inputs(B, H, N, d, 220)
    o, lse = torch.empty_like(q), torch.empty(B, H, N, device="cuda", dtype=torch.float32)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa_bwd_workspace_bytes(B, H, N, d), device="cuda", dtype=torch.uint8)

    def step():
        fa_fwd(q, k, v, causal, scale, o=o, lse=lse)
        fa_bwd(q, k, v, o, do, lse, causal, scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    step()  # first calls outside the capture (module load, side stream creation)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert fa_device_status() == 0
        for name, x, r in zip(("o", "lse", "dq", "dk", "dv"), (o, lse, dq, dk, dv), eager):
            assert torch.equal(x, r), f"graph replay: {name} differs from the eager call"
