"""Seeded synthetic inputs for the causal-attention workloads.

This module holds no attention arithmetic: it draws Gaussian Q, K, V, dO and
rounds them to the storage dtype.  It is the one piece of code that both the
CUDA path's tests/benchmark and the CPU oracle consume, so that both see the
same bytes.

Recipe (the same for every workload): ``numpy.random.default_rng(seed)``
draws, in the order Q, K, V, dO, one ``standard_normal((bh, S, hd))`` array
each in fp64; each is multiplied by its standard deviation, rounded to fp32
(round to nearest even) and, for bf16 workloads, further rounded from fp32 to
bf16 (round to nearest even).  The fp64 view handed to the oracle holds exactly
the rounded values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    hd: int
    dtype: str          # "f32" or "bf16"
    scale: float
    seed: int
    qk_std: float = 1.0
    v_std: float = 1.0
    do_std: float = 1.0

    @property
    def bh(self) -> int:
        return self.B * self.H

    def fwd_flops(self) -> float:
        """Causal forward FLOPs: half of the dense 4*bh*S^2*hd (QK^T and PV)."""
        return 2.0 * self.bh * self.S * self.S * self.hd

    def bwd_flops(self) -> float:
        """Backward FLOPs: 2.5x the forward (five S^2*hd contractions against two)."""
        return 2.5 * self.fwd_flops()


# The five causal-attention workloads, smallest first.  Layout [bh, S, hd].
WORKLOADS = {
    1: Workload("causal_f32_bh2_s64_hd32", 1, 2, 64, 32, "f32", 1.0 / math.sqrt(32), seed=0),
    2: Workload("causal_f32_bh16_s256_hd64", 4, 4, 256, 64, "f32", 1.0 / 8.0, seed=2, do_std=0.1),
    3: Workload("causal_bf16_bh96_s1024_hd64", 8, 12, 1024, 64, "bf16", 1.0 / 8.0, seed=3),
    4: Workload("causal_bf16_bh64_s4096_hd128_peaked", 4, 16, 4096, 128, "bf16", 1.0 / math.sqrt(128), seed=4,
                qk_std=2.0),
    5: Workload("causal_bf16_bh32_s8192_hd128", 1, 32, 8192, 128, "bf16", 1.0 / math.sqrt(128), seed=5),
}


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact fp64 value of bf16 bit patterns."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclass
class Tensors:
    """One drawn tensor: ``stored`` is what the GPU receives (float32 array, or
    uint16 bf16 bit patterns), ``exact`` its exact fp64 value for the oracle."""
    stored: np.ndarray
    exact: np.ndarray


def _stored(x32: np.ndarray, dtype: str) -> Tensors:
    if dtype == "f32":
        return Tensors(x32, x32.astype(np.float64))
    bits = f32_to_bf16_bits(x32)
    return Tensors(bits, bf16_bits_to_f64(bits))


def draw(shape, dtype: str, seed: int, stds=(1.0, 1.0, 1.0, 1.0), names=("q", "k", "v", "dout")):
    """Draw the named tensors in order from one generator seeded with ``seed``."""
    if dtype not in ("f32", "bf16"):
        raise ValueError(f"unknown dtype {dtype!r}")
    rng = np.random.default_rng(seed)
    out = {}
    for name, std in zip(names, stds):
        x32 = (rng.standard_normal(shape) * std).astype(np.float32)
        out[name] = _stored(x32, dtype)
        del x32
    return out


PATTERNS = ("rising", "falling", "flat")


def patterned(shape, dtype: str, pattern: str, seed: int, magnitude: float = 16.0, k_noise: float = 2.0):
    """Structured Q and K (V and dO standard normal) for the score shapes that steer the
    online softmax.  Q and K rows have norm ``magnitude`` in the plane of coordinates 0
    and 1, at angle theta_j = pi * j / S for position j:
      "rising":  q_i at theta_i and k_j at theta_j, so s_ij ~ cos(pi (i - j) / S): along a
                 row the scores climb towards the diagonal and the running row maximum
                 keeps moving;
      "falling": q_i fixed at angle 0 and k_j at theta_j, so the scores fall along the row
                 and its maximum is the first key;
      "flat":    Q = 0, all scores equal.
    The norms stay constant along the sequence.  The other coordinates of K carry
    independent N(0, k_noise^2) values, as keys do, and those of Q N(0, 0.1^2) noise, so
    the scores follow the pattern while the keys that share a row's softmax window are
    not nearly parallel (with parallel keys dQ = sum_j dS_ij (K_j - K_i) is a near
    cancellation that any bf16 rounding of dS exposes)."""
    if pattern not in PATTERNS:
        raise ValueError(f"unknown pattern {pattern!r}")
    bh, S, hd = shape
    rng = np.random.default_rng(seed)
    q = rng.standard_normal(shape) * 0.1
    k = rng.standard_normal(shape) * k_noise
    v = rng.standard_normal(shape)
    do = rng.standard_normal(shape)
    theta = np.pi * np.arange(S, dtype=np.float64) / S
    if pattern == "flat":
        q[:] = 0.0
    else:
        k[..., 0] = magnitude * np.cos(theta)
        k[..., 1] = magnitude * np.sin(theta)
        if pattern == "rising":
            q[..., 0] = magnitude * np.cos(theta)
            q[..., 1] = magnitude * np.sin(theta)
        else:
            q[..., 0] = magnitude
            q[..., 1] = 0.0
    return {n: _stored(a.astype(np.float32), dtype) for n, a in (("q", q), ("k", k), ("v", v), ("dout", do))}


def workload_inputs(w: Workload, bh: int | None = None, S: int | None = None):
    """Inputs of a workload (optionally with a different bh or S, same recipe)."""
    bh = w.bh if bh is None else bh
    S = w.S if S is None else S
    return draw((bh, S, w.hd), w.dtype, w.seed, (w.qk_std, w.qk_std, w.v_std, w.do_std))
