"""Plain fp64 CPU oracle for causal attention, forward and backward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The CUDA product path
(``bwd_xfa_fwd_gb300``) never imports it, and this package never imports that
one: the two share no code.  Inputs reach both sides from the seeded generator
module ``bwd_xfa_fwd_gb300.inputs``, which holds no attention arithmetic.

The arithmetic lives in ``xfa_oracle.c`` (see the header there for the
definition and the page passages it transcribes).  This module only compiles
that file with the host C compiler, loads it with ctypes and loops over heads.

Pinning (every function here is checked against something other than itself
by ``tests/test_oracle.py``): a hand-worked 2x2 example, the row-sum and
softmax-backward identities of "xtrain docs/13-flash-attention.md"
(sections "什么是 flash-attention" and design decision ③), central finite
differences in fp64, special cases with closed forms (S=1, Q=0, hd=1) and the
unmasked case against a dense numpy softmax.  The optional dropout on the
attention probabilities ("xtrain docs/17-dropout.md", section "Key Design
Decisions") is pinned by ``DROPOUT_PINS`` in ``tests/oracle_pins.py`` (run by
``tests/test_oracle.py``): known outputs of the SplitMix64 generator, the keep
rate, p = 0 against the plain path, finite differences with the mask fixed, the
D identity and the expectation over seeds.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import sysconfig

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "xfa_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

_default = None


def compile_source(src: str, out_path: str) -> str:
    """Compile C source text ``src`` into the shared library ``out_path``."""
    os.makedirs(os.path.dirname(out_path) or ".", exist_ok=True)
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc") or sysconfig.get_config_var("CC")
    tmp_c = out_path + f".{os.getpid()}.c"
    tmp_so = out_path + f".tmp{os.getpid()}"
    with open(tmp_c, "w") as f:
        f.write(src)
    base = [cc, "-O2", "-fPIC", "-shared", "-std=c11", tmp_c, "-o", tmp_so, "-lm"]
    try:
        try:
            subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base, check=True, capture_output=True)
    finally:
        os.remove(tmp_c)
    os.replace(tmp_so, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile ``xfa_oracle.c`` into ``oracle/_build/liboracle.so`` (OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    with open(_SRC) as f:
        return compile_source(f.read(), _LIB)


class Oracle:
    """ctypes handle on one compiled copy of the oracle."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.xfa_oracle_head.argtypes = [dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                                        ctypes.c_int, dp, dp, dp, dp, dp, dp, dp, dp]
        lib.xfa_oracle_head.restype = ctypes.c_int
        lib.xfa_oracle_head_dropout.argtypes = [dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                                                ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint64,
                                                dp, dp, dp, dp, dp, dp, dp, dp]
        lib.xfa_oracle_head_dropout.restype = ctypes.c_int
        lib.xfa_oracle_splitmix64.argtypes = [ctypes.c_uint64]
        lib.xfa_oracle_splitmix64.restype = ctypes.c_uint64
        lib.xfa_oracle_keep.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float]
        lib.xfa_oracle_keep.restype = ctypes.c_int
        lib.xfa_oracle_threads.argtypes = []
        lib.xfa_oracle_threads.restype = ctypes.c_int
        self.lib = lib

    def threads(self) -> int:
        return int(self.lib.xfa_oracle_threads())

    def splitmix64(self, x: int) -> int:
        return int(self.lib.xfa_oracle_splitmix64(x & (2 ** 64 - 1)))

    def keep(self, seed: int, index: int, p: float) -> bool:
        return bool(self.lib.xfa_oracle_keep(seed & (2 ** 64 - 1), index & (2 ** 64 - 1), p))

    def head(self, q, k, v, dout=None, scale=1.0, causal=True, diagnostics=False, dropout=None):
        """See :func:`attention_head`."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        S, hd = q.shape
        if k.shape != (S, hd) or v.shape != (S, hd):
            raise ValueError("q, k, v must share the shape [S, hd]")
        res = {"out": np.empty((S, hd)), "lse": np.empty(S)}
        if dout is not None:
            dout = _f64(dout)
            if dout.shape != (S, hd):
                raise ValueError("dout must have the shape [S, hd]")
            for n in ("dq", "dk", "dv"):
                res[n] = np.empty((S, hd))
        if diagnostics:
            res["p_rowsum"] = np.empty(S)
            if dout is not None:
                res["pdp_rowsum"] = np.empty(S)
                res["ds_rowsum"] = np.empty(S)
        outs = (_ptr(res["out"]), _ptr(res["lse"]), _ptr(res.get("dq")), _ptr(res.get("dk")), _ptr(res.get("dv")),
                _ptr(res.get("p_rowsum")), _ptr(res.get("pdp_rowsum")), _ptr(res.get("ds_rowsum")))
        if dropout is None:
            rc = self.lib.xfa_oracle_head(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), S, hd, float(scale),
                                          int(bool(causal)), *outs)
        else:
            p, seed, index_base = dropout
            rc = self.lib.xfa_oracle_head_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), S, hd, float(scale),
                                                  int(bool(causal)), float(p), seed & (2 ** 64 - 1),
                                                  index_base & (2 ** 64 - 1), *outs)
        if rc != 0:
            raise RuntimeError(f"oracle failed with code {rc}")
        return res


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return default().threads()


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def attention_head(q, k, v, dout=None, scale=1.0, causal=True, diagnostics=False, dropout=None):
    """One head, ``q,k,v,dout`` of shape [S, hd].  Returns a dict of fp64 arrays:
    ``out`` [S,hd], ``lse`` [S] (natural log) and, with ``dout``, ``dq, dk, dv``.
    With ``diagnostics`` also ``p_rowsum`` (sum_j P_ij), ``pdp_rowsum``
    (sum_j P_ij dP_ij) and ``ds_rowsum`` (sum_j dS_ij), one per query row.
    ``dropout = (p, seed, index_base)`` applies dropout of rate p to the attention
    probabilities, element (i, j) drawn with flat index index_base + i*S + j."""
    return default().head(q, k, v, dout, scale, causal, diagnostics, dropout)


def splitmix64(x: int) -> int:
    """One step of the SplitMix64 generator from state ``x`` (the dropout page's bit mix)."""
    return default().splitmix64(x)


def keep(seed: int, index: int, p: float) -> bool:
    """The dropout page's keep decision for element ``index`` under ``seed`` and rate ``p``."""
    return default().keep(seed, index, p)


def attention(q, k, v, dout=None, scale=1.0, causal=True, heads=None, dropout=None):
    """Batched over the leading ``bh`` axis of [bh, S, hd] arrays.  ``heads``
    restricts the computation to a list of head indices (the others are left
    as NaN), which is how the full-size configurations are sampled.
    ``dropout = (p, seed)``: dropout on the [bh, S, S] attention probabilities
    (head b's elements have flat indices b*S*S + i*S + j)."""
    q = np.asarray(q)
    bh, S, hd = q.shape
    heads = list(range(bh)) if heads is None else list(heads)
    res = {"out": np.full((bh, S, hd), np.nan), "lse": np.full((bh, S), np.nan)}
    if dout is not None:
        for n in ("dq", "dk", "dv"):
            res[n] = np.full((bh, S, hd), np.nan)
    for b in heads:
        dd = None if dropout is None else (dropout[0], dropout[1], b * S * S)
        r = attention_head(q[b], k[b], v[b], None if dout is None else dout[b], scale, causal, dropout=dd)
        for n, a in r.items():
            res[n][b] = a
    return res
