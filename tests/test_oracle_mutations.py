"""Plant plausible mistakes in a copy of the oracle source and check that the
pins catch every one of them (CPU only; the mutated copies live in a temp dir)."""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, original text, replacement): each a mistake someone could make
MUTATIONS = [
    ("drop_scale_in_scores", "p[j] = J->scale * acc;", "p[j] = acc;"),
    ("wrong_sign_in_exp", "p[j] = exp(p[j] - M);", "p[j] = exp(M - p[j]);"),
    ("no_normalisation", "for (long j = 0; j < end; ++j) p[j] /= Z;", ""),
    ("lse_without_max", "J->lse[h * J->Nq + i] = M + log(Z);", "J->lse[h * J->Nq + i] = log(Z);"),
    ("causal_off_by_one", "long e = i + 1;", "long e = i + 2;"),
    ("pv_uses_keys", "oi[c] += p[j] * vj[c];", "oi[c] += p[j] * (kh + j * d)[c];"),
    ("drop_jacobian_row_term", "double ds = p[j] * (dp[j] - rowdot);", "double ds = p[j] * dp[j];"),
    ("dq_uses_queries", "dqi[c] += J->scale * ds * kj[c];", "dqi[c] += J->scale * ds * qi[c];"),
    ("dk_without_scale", "dkj[c] += J->scale * ds * qi[c];", "dkj[c] += ds * qi[c];"),
    ("dv_uses_queries", "dvj[c] += p[j] * doi[c];", "dvj[c] += p[j] * qi[c];"),
    ("dp_uses_keys", "acc += doi[c] * vj[c];", "acc += doi[c] * (kh + j * d)[c];"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(name, old, new, tmp_path):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not unique"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-shared",
                    "-fPIC", "-pthread", str(src), "-o", str(so), "-lm"], check=True)
    lib = oracle.bind(str(so))
    caught = []
    for pin in ALL_PINS:
        if pin.__name__ == "pin_finite_differences_sampled":
            continue  # slow; the full small-case differences cover the same code
        try:
            pin(lib=lib)
        except (AssertionError, RuntimeError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {name}"
