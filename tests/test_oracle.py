"""The CPU oracle against its pins (no GPU)."""
import numpy as np
import pytest

import oracle
from bwd_xfa_fwd_gb300 import inputs
from tests import oracle_pins


@pytest.fixture(scope="module")
def head():
    return oracle.default().head


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin, head):
    pin(head)


@pytest.mark.parametrize("pin", oracle_pins.DROPOUT_PINS, ids=lambda p: p.__name__)
def test_oracle_dropout_pin(pin):
    pin(oracle.default())


def test_batched_matches_per_head():
    w = inputs.WORKLOADS[1]
    x = inputs.workload_inputs(w)
    r = oracle.attention(x["q"].exact, x["k"].exact, x["v"].exact, x["dout"].exact, w.scale, heads=[1])
    one = oracle.attention_head(x["q"].exact[1], x["k"].exact[1], x["v"].exact[1], x["dout"].exact[1], w.scale)
    assert np.isnan(r["out"][0]).all()
    for n in ("out", "lse", "dq", "dk", "dv"):
        assert np.array_equal(r[n][1], one[n])


def test_bf16_rounding_is_rne():
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties go to the even mantissa (1.0);
    # 1 + 3*2^-8 ties between 1 + 2^-7 (odd) and 1 + 2^-6 (even): rounds up.
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -8 + 2 ** -20], np.float32)
    got = inputs.bf16_bits_to_f64(inputs.f32_to_bf16_bits(x))
    assert got.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0 + 2 ** -7]


def test_generator_is_seeded_and_ordered():
    w = inputs.WORKLOADS[2]
    a = inputs.workload_inputs(w, bh=2, S=8)
    b = inputs.workload_inputs(w, bh=2, S=8)
    for n in ("q", "k", "v", "dout"):
        assert np.array_equal(a[n].stored, b[n].stored)
    rng = np.random.default_rng(w.seed)
    q = rng.standard_normal((2, 8, w.hd)).astype(np.float32)
    assert np.array_equal(a["q"].stored, q)
    assert abs(float(np.std(a["dout"].exact)) - 0.1) < 0.02
