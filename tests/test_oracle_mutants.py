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
    "dV not transposed": ("matmul_tn(C ? Pd : P, dout, S, hd, dv);", "matmul_nn(C ? Pd : P, dout, S, hd, dv);"),
    "dP operands swapped": ("matmul_nt(dout, v, S, hd, dP);", "matmul_nt(v, dout, S, hd, dP);"),
    "O uses K instead of V": ("matmul_nn(C ? Pd : P, v, S, hd, out);", "matmul_nn(C ? Pd : P, k, S, hd, out);"),
    # dropout on the attention probabilities
    "dropout mask missing in the backward": ("dP[e] *= C[e];", "dP[e] *= 1.0;"),
    "dropout not inverted": ("? inv_keep : 0.0;", "? 1.0 : 0.0;"),
    "dV from the undropped P": ("matmul_tn(C ? Pd : P, dout, S, hd, dv);", "matmul_tn(P, dout, S, hd, dv);"),
    "dropout index transposed": ("index_base + (uint64_t)(i * S + j)", "index_base + (uint64_t)(j * S + i)"),
    "keep test reversed": ("return u >= p;", "return u < p;"),
    "keep from the low bits": ("(float)(h >> 40)", "(float)(h & 0xFFFFFF)"),
    "bit-mix constant": ("z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;", "z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B8ull;"),
    "second bit-mix constant": ("* 0x94D049BB133111EBull;", "* 0x94D049BB133111EAull;"),
    "second shift 27 -> 26": ("z = (z ^ (z >> 27))", "z = (z ^ (z >> 26))"),
    "golden increment dropped": ("uint64_t z = x + 0x9E3779B97F4A7C15ull;", "uint64_t z = x;"),
    "final xor-shift dropped": ("return z ^ (z >> 31);", "return z;"),
    "seed added, not xored": ("seed ^ (index * 0x9E3779B97F4A7C15ull)", "seed + (index * 0x9E3779B97F4A7C15ull)"),
    "index not scrambled": ("seed ^ (index * 0x9E3779B97F4A7C15ull)", "seed ^ index"),
    "keep test strict": ("return u >= p;", "return u > p;"),
    "u over 2^23": ("/ 16777216.0f", "/ 8388608.0f"),
    "index base ignored": ("index_base + (uint64_t)(i * S + j)", "(uint64_t)(i * S + j)"),
    "inverted scale 1 - p": ("1.0 / (1.0 - (double)p)", "(1.0 - (double)p)"),
    "softmax row term from the dropped P": ("const double *prow = P + i * S;", "const double *prow = (C ? Pd : P) + i * S;"),
    # plain path
    "L in log2": ("lse[i] = m + log(z);", "lse[i] = m + log2(z);"),
    "running max not subtracted": ("row[j] = exp(row[j] - m);", "row[j] = exp(row[j]);"),
    "row term without P": ("dot += drow[j] * prow[j];", "dot += drow[j];"),
    "dP uses K instead of V": ("matmul_nt(dout, v, S, hd, dP);", "matmul_nt(dout, k, S, hd, dP);"),
    "dK uses K instead of Q": ("matmul_tn(dP, q, S, hd, dk);", "matmul_tn(dP, k, S, hd, dk);"),
    "dS transposed in dQ": ("matmul_nn(dP, k, S, hd, dq);", "matmul_tn(dP, k, S, hd, dq);"),
    "scale applied twice": ("s[i * S + j] = scale * acc;", "s[i * S + j] = scale * scale * acc;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    with open(SRC) as f:
        src = f.read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    lib = oracle.compile_source(src.replace(old, new), str(tmp_path / "mutant.so"))
    orc = oracle.Oracle(lib)
    failures = []
    for pin, arg in [(p, orc.head) for p in oracle_pins.ALL_PINS] + [(p, orc) for p in oracle_pins.DROPOUT_PINS]:
        try:
            pin(arg)
        except (AssertionError, FloatingPointError, RuntimeError) as e:
            failures.append(f"{pin.__name__}: {e}")
    assert failures, f"mutant '{name}' passed every pin"
