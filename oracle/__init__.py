"""fp64 CPU oracle for exact softmax attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it and
shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain two-pass softmax, analytic
Jacobian gradients, fp64); this module only compiles it with gcc and
marshals numpy arrays through ctypes.  See that file's header for the
definition it follows and the passages of the pages it cites.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libattn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE fp64, no fast-math) and return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
           "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
    lib.oracle_fwd.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, I, D, I]
    lib.oracle_fwd.restype = I
    lib.oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, L, L, L, L, I, D, I]
    lib.oracle_bwd.restype = I
    lib.oracle_probs.argtypes = [dp, dp, dp, L, L, L, I, D]
    lib.oracle_probs.restype = I
    lib.oracle_fwd_spread.argtypes = [dp, dp, dp, dp, L, L, L, L, I, D, I]
    lib.oracle_fwd_spread.restype = I
    u8 = ctypes.POINTER(ctypes.c_uint8)
    lib.e4m3_value.argtypes = [ctypes.c_uint8]
    lib.e4m3_value.restype = D
    lib.e4m3_round.argtypes = [D]
    lib.e4m3_round.restype = D
    lib.oracle_fwd_fp8.argtypes = [u8, u8, u8, D, D, D, dp, dp, dp, L, L, L, L, I, D, D, I, I]
    lib.oracle_fwd_fp8.restype = I
    lib.oracle_fwd_fp8_detail.argtypes = [u8, u8, u8, D, D, D, dp, dp, dp, L, L, L, L, I, D, D, I, I,
                                          dp, dp, dp, dp]
    lib.oracle_fwd_fp8_detail.restype = I
    return lib


def bind(path: str):
    """Load another build of the oracle source (used by the mutation checks)."""
    return _bind(path)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape(q, k):
    if q.ndim < 2 or k.ndim != q.ndim or q.shape[-1] != k.shape[-1] or q.shape[:-2] != k.shape[:-2]:
        raise ValueError(f"incompatible shapes {q.shape} / {k.shape}")
    lead = q.shape[:-2]
    BH = int(np.prod(lead)) if lead else 1
    return lead, BH, q.shape[-2], k.shape[-2], q.shape[-1]


def fwd(q, k, v, causal: bool, scale: float, nthreads: int | None = None, lib=None):
    """O and LSE of softmax(q k^T * scale) v.

    Arrays are [..., Nq, d] (q) and [..., Nk, d] (k, v), any float dtype;
    they are upcast to fp64.  Returns (o [..., Nq, d], lse [..., Nq]) in fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead, BH, Nq, Nk, d = _shape(q, k)
    if v.shape != k.shape:
        raise ValueError("v must have the shape of k")
    o = np.empty(q.shape, np.float64)
    lse = np.empty(lead + (Nq,), np.float64)
    rc = (lib or _load()).oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), BH, Nq, Nk, d,
                            int(bool(causal)), float(scale), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_fwd failed ({rc})")
    return o, lse


def bwd(q, k, v, dout, causal: bool, scale: float, nthreads: int | None = None, lib=None):
    """(dq, dk, dv) of L = sum(dout * O) through the softmax definition, fp64."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    lead, BH, Nq, Nk, d = _shape(q, k)
    if v.shape != k.shape or dout.shape != q.shape:
        raise ValueError("v must match k and dout must match q")
    dq = np.empty(q.shape, np.float64)
    dk = np.empty(k.shape, np.float64)
    dv = np.empty(k.shape, np.float64)
    rc = (lib or _load()).oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                            BH, Nq, Nk, d, int(bool(causal)), float(scale),
                            nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_bwd failed ({rc})")
    return dq, dk, dv


def probs(q, k, causal: bool, scale: float, lib=None):
    """Normalised P [Nq, Nk] of a single head (small cases only)."""
    q, k = _f64(q), _f64(k)
    if q.ndim != 2 or k.ndim != 2:
        raise ValueError("probs takes one head: q [Nq, d], k [Nk, d]")
    Nq, d = q.shape
    Nk = k.shape[0]
    p = np.empty((Nq, Nk), np.float64)
    rc = (lib or _load()).oracle_probs(_ptr(q), _ptr(k), _ptr(p), Nq, Nk, d, int(bool(causal)), float(scale))
    if rc != 0:
        raise RuntimeError(f"oracle_probs failed ({rc})")
    return p


def fwd_spread(q, k, v, causal: bool, scale: float, nthreads: int | None = None, lib=None):
    """spread[..., i, c] = sum_j P_ij |v_jc - O_ic| (fp64).

    A relative perturbation e of every weight P_ij moves O_ic by at most
    e * spread; used to derive the O tolerance for short-format weights."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead, BH, Nq, Nk, d = _shape(q, k)
    out = np.empty(q.shape, np.float64)
    rc = (lib or _load()).oracle_fwd_spread(_ptr(q), _ptr(k), _ptr(v), _ptr(out), BH, Nq, Nk, d,
                                            int(bool(causal)), float(scale), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_fwd_spread failed ({rc})")
    return out


# ---------------------------------------------------------------- FP8

def e4m3_value(code: int, lib=None) -> float:
    """Value of one e4m3 code (the format's definition, written out in C)."""
    return float((lib or _load()).e4m3_value(int(code) & 0xFF))


def e4m3_round(x: float, lib=None) -> float:
    """Nearest e4m3 value (ties to even, saturated to +-448)."""
    return float((lib or _load()).e4m3_round(float(x)))


def _u8(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (float8_e4m3fn or uint8): its bytes
        import torch
        t = x.detach().to("cpu").contiguous()
        if t.dtype != torch.uint8:
            t = t.view(torch.uint8)
        x = t.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.uint8))


def fwd_fp8(q8, k8, v8, sq: float, sk: float, sv: float, causal: bool, scale: float, acc_rel: float = 0.0,
            with_bound: bool = False, stale: int = 0, nthreads: int | None = None, lib=None):
    """FP8 forward (the definition in attn_oracle.c): e4m3 codes [..., N, d]
    (uint8 arrays or float8_e4m3fn tensors) and tensor scales.  Returns
    (o, lse) in fp64, and the per-element bound when with_bound."""
    q, k, v = _u8(q8), _u8(k8), _u8(v8)
    lead, BH, Nq, Nk, d = _shape(q, k)
    if v.shape != k.shape:
        raise ValueError("v must have the shape of k")
    o = np.empty(q.shape, np.float64)
    lse = np.empty(lead + (Nq,), np.float64)
    bound = np.empty(q.shape, np.float64) if with_bound else None
    u8p = ctypes.POINTER(ctypes.c_uint8)
    rc = (lib or _load()).oracle_fwd_fp8(q.ctypes.data_as(u8p), k.ctypes.data_as(u8p), v.ctypes.data_as(u8p),
                                         float(sq), float(sk), float(sv), _ptr(o), _ptr(lse),
                                         _ptr(bound) if with_bound else None, BH, Nq, Nk, d,
                                         int(bool(causal)), float(scale), float(acc_rel), int(stale),
                                         nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_fwd_fp8 failed ({rc})")
    return (o, lse, bound) if with_bound else (o, lse)


def fwd_fp8_detail(q8, k8, v8, sq: float, sk: float, sv: float, causal: bool, scale: float,
                   acc_rel: float = 0.0, stale: int = 0, lib=None):
    """fwd_fp8 with the bound, plus the per-key detail of the definition:
    returns a dict with o, lse, bound [..., Nq, d], x (scores in log2 units,
    -inf where masked), w (rounded weights), delta (the change of each
    weight the bound allows) [..., Nq, Nk] and M [..., Nq].  Small cases."""
    q, k, v = _u8(q8), _u8(k8), _u8(v8)
    lead, BH, Nq, Nk, d = _shape(q, k)
    if v.shape != k.shape:
        raise ValueError("v must have the shape of k")
    out = {"o": np.empty(q.shape, np.float64), "lse": np.empty(lead + (Nq,), np.float64),
           "bound": np.empty(q.shape, np.float64)}
    for name in ("x", "w", "delta"):
        out[name] = np.empty(lead + (Nq, Nk), np.float64)
    out["M"] = np.empty(lead + (Nq,), np.float64)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    rc = (lib or _load()).oracle_fwd_fp8_detail(
        q.ctypes.data_as(u8p), k.ctypes.data_as(u8p), v.ctypes.data_as(u8p), float(sq), float(sk), float(sv),
        _ptr(out["o"]), _ptr(out["lse"]), _ptr(out["bound"]), BH, Nq, Nk, d, int(bool(causal)), float(scale),
        float(acc_rel), int(stale), 1, _ptr(out["x"]), _ptr(out["w"]), _ptr(out["delta"]), _ptr(out["M"]))
    if rc != 0:
        raise RuntimeError(f"oracle_fwd_fp8_detail failed ({rc})")
    return out
