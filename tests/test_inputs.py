"""The seeded input generators (no GPU): determinism, bf16 rounding, and the score
shapes the structured patterns promise."""
import math

import numpy as np
import pytest

from bwd_xfa_fwd_gb300 import inputs


def test_draw_is_deterministic_and_exact():
    a = inputs.draw((2, 9, 8), "bf16", seed=3)
    b = inputs.draw((2, 9, 8), "bf16", seed=3)
    for n in ("q", "k", "v", "dout"):
        assert np.array_equal(a[n].stored, b[n].stored)
        assert np.array_equal(inputs.bf16_bits_to_f64(a[n].stored), a[n].exact)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 0.0], dtype=np.float32)
    got = inputs.bf16_bits_to_f64(inputs.f32_to_bf16_bits(x))
    assert list(got) == [1.0, 1.0, 1.0 + 2 * 2.0 ** -7, -2.5, 0.0]


@pytest.mark.parametrize("pattern", inputs.PATTERNS)
def test_patterned_scores(pattern):
    S, hd = 600, 64
    x = inputs.patterned((1, S, hd), "f32", pattern, seed=11)
    y = inputs.patterned((1, S, hd), "f32", pattern, seed=11)
    assert all(np.array_equal(x[n].stored, y[n].stored) for n in x)
    s = x["q"].exact[0] @ x["k"].exact[0].T / math.sqrt(hd)
    rows = range(100, S, 50)
    if pattern == "flat":
        assert np.all(x["q"].exact == 0.0)
    elif pattern == "rising":
        # the largest causal score of a row sits close to its diagonal
        assert all(i - int(np.argmax(s[i, : i + 1])) < 40 for i in rows)
    else:
        # the largest causal score of a row is one of its first keys
        assert all(int(np.argmax(s[i, : i + 1])) < 40 for i in rows)
