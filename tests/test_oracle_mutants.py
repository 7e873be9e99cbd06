"""Plant plausible mistakes in copies of the oracle (on the CPU) and require
that every one of them trips at least one pin.  This is how the pins are shown
to be strong enough: a dropped term, a wrong sign or index, or a transposed
operand anywhere in the oracle must not go unnoticed."""
import os

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "xfa_oracle.c")

MUTANTS = {
    "key index i instead of j": ("acc += q[i * hd + d] * k[j * hd + d];", "acc += q[i * hd + d] * k[i * hd + d];"),
    "scale dropped in scores": ("s[i * S + j] = scale * acc;", "s[i * S + j] = acc;"),
    "mask off by one (diagonal excluded for rows > 0)": ("if (causal && j > i)", "if (causal && j >= i && i > 0)"),
    "mask removed": ("if (causal && j > i)", "if (causal && j > i + S)"),
    "running max dropped from lse": ("lse[i] = m + log(z);", "lse[i] = log(z);"),
    "softmax not normalised": ("for (long j = 0; j < S; ++j) row[j] /= z;", "for (long j = 0; j < S; ++j) row[j] /= 1.0;"),
    "jacobian row term dropped": ("drow[j] = scale * (prow[j] * (drow[j] - dot));", "drow[j] = scale * (prow[j] * drow[j]);"),
    "jacobian row term sign": ("drow[j] = scale * (prow[j] * (drow[j] - dot));", "drow[j] = scale * (prow[j] * (drow[j] + dot));"),
    "scale dropped in backward": ("drow[j] = scale * (prow[j] * (drow[j] - dot));", "drow[j] = (prow[j] * (drow[j] - dot));"),
    "dQ uses Q instead of K": ("matmul_nn(dP, k, S, hd, dq);", "matmul_nn(dP, q, S, hd, dq);"),
    "dK not transposed": ("matmul_tn(dP, q, S, hd, dk);", "matmul_nn(dP, q, S, hd, dk);"),
    "dV not transposed": ("matmul_tn(P, dout, S, hd, dv);", "matmul_nn(P, dout, S, hd, dv);"),
    "dP operands swapped": ("matmul_nt(dout, v, S, hd, dP);", "matmul_nt(v, dout, S, hd, dP);"),
    "O uses K instead of V": ("matmul_nn(P, v, S, hd, out);", "matmul_nn(P, k, S, hd, out);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    with open(SRC) as f:
        src = f.read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    lib = oracle.compile_source(src.replace(old, new), str(tmp_path / "mutant.so"))
    head = oracle.Oracle(lib).head
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(head)
        except (AssertionError, FloatingPointError, RuntimeError) as e:
            failures.append(f"{pin.__name__}: {e}")
    assert failures, f"mutant '{name}' passed every pin"
