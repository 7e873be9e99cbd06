"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the C ABI binding, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bwd_xfa_fwd_gb300 import inputs

# Tolerances (max |gpu - ref| against max |ref| per tensor):
#   fp32 storage: 1e-4 relative on O, L, dQ, dK, dV
#   bf16 storage with fp32 accumulation: 2e-2 relative on O and the grads,
#   1e-2 absolute on L
TOL = {"f32": {"rel": 1e-4, "lse_abs": None}, "bf16": {"rel": 2e-2, "lse_abs": 1e-2}}


def to_device(t: inputs.Tensors, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(t.stored)).cuda()
    bits = torch.from_numpy(np.ascontiguousarray(t.stored).view(np.int16))
    return bits.view(torch.bfloat16).cuda()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_gpu(x, dtype: str, scale: float, impl: int = 0, backward: bool = True, dropout=None, keep: str = "none"):
    """``dropout = (p, seed)``: dropout on the attention probabilities.  ``keep``: "none" (both
    kernels draw the mask), "store" (the forward stores it as bits, the backward reads them) or
    "fill" (xfa_dropout_keep_fill draws it, both kernels read it)."""
    from bwd_xfa_fwd_gb300 import binding
    p_drop, seed = (0.0, 0) if dropout is None else dropout
    q, k, v, do = (to_device(x[n], dtype) for n in ("q", "k", "v", "dout"))
    bits = None
    if p_drop and keep != "none":
        bh, S = q.shape[0], q.shape[1]
        bits = torch.full((binding.dropout_keep_bytes(bh, S),), 0xCD, device=q.device, dtype=torch.uint8)
        if keep == "fill":
            binding.dropout_keep_fill(bh, S, p_drop, seed, bits)
    out, lse = binding.fwd(q, k, v, scale, impl, dropout_p=p_drop, seed=seed, keep_bits=bits,
                           keep_cached=keep == "fill")
    res = {"out": out, "lse": lse}
    if backward:
        dq, dk, dv = binding.bwd(q, k, v, out, do, lse, scale, impl, dropout_p=p_drop, seed=seed, keep_bits=bits)
        res.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert binding.status() == binding.XFA_OK
    return {n: to_f64(t) for n, t in res.items()}


def compare(got: dict, ref: dict, dtype: str, heads=None, names=("out", "lse", "dq", "dk", "dv")):
    """Raise AssertionError listing every tensor out of tolerance; returns the error table."""
    tol = TOL[dtype]
    sel = slice(None) if heads is None else list(heads)
    report, bad = {}, []
    # A gradient that is identically zero by structure (S = 1 gives dQ = dK = 0 exactly,
    # Q = 0 gives dK = 0) would get a zero bound, which no rounding passes.  Only then,
    # when max|ref| is exactly 0, is the bound taken against 1% of the largest gradient
    # of the same call; every other tensor gets tol * max|ref| of its own.
    gmax = max([float(np.max(np.abs(ref[n][sel]))) for n in ("dq", "dk", "dv") if n in ref and n in got] or [0.0])
    for n in names:
        if n not in got:
            continue
        g, r = got[n][sel], ref[n][sel]
        assert np.all(np.isfinite(g)), f"{n}: non-finite GPU values"
        err = float(np.max(np.abs(g - r)))
        scale = float(np.max(np.abs(r)))
        if n in ("dq", "dk", "dv") and scale == 0.0:
            scale = 1e-2 * gmax
        if n == "lse" and tol["lse_abs"] is not None:
            bound = tol["lse_abs"]
        else:
            bound = tol["rel"] * scale
        report[n] = (err, bound)
        if not err <= bound:
            bad.append(f"{n}: max err {err:.3e} > bound {bound:.3e} (max|ref| {scale:.3e})")
    assert not bad, "; ".join(bad)
    return report


_ORACLE_CACHE = {}


def oracle_result(key, x, scale, heads=None, dropout=None):
    """Oracle on inputs ``x`` (fp64 views), memoised under ``key``; ``dropout = (p, seed)``."""
    k = (key, None if heads is None else tuple(heads), dropout)
    if k not in _ORACLE_CACHE:
        _ORACLE_CACHE[k] = oracle.attention(x["q"].exact, x["k"].exact, x["v"].exact, x["dout"].exact, scale,
                                            heads=heads, dropout=dropout)
    return _ORACLE_CACHE[k]
