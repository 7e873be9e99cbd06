"""Checks that pin the CPU oracle to facts other than itself.

Each ``pin_*`` takes a ``head`` callable with the signature of
``oracle.Oracle.head`` and raises AssertionError when the oracle disagrees
with a worked example, an identity of the method, a closed form, a library
routine or a finite-difference derivative.  ``test_oracle.py`` runs them on the
real oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle with a
planted mistake and requires that each mistake trips at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import logsumexp, softmax

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _close(a, b, tol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        raise AssertionError(f"{what}: shape {a.shape} != {b.shape}")
    if not np.all(np.isfinite(a)):
        raise AssertionError(f"{what}: non-finite values")
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    if err > tol:
        raise AssertionError(f"{what}: max abs err {err:.3e} > {tol:.3e}")


def _rand(rng, S, hd, std=1.0):
    return rng.standard_normal((S, hd)) * std


def pin_hand_2x2(head):
    """The 2x2 example worked by hand from the page formulas (tests/golden/hand_2x2.json)."""
    with open(os.path.join(GOLDEN, "hand_2x2.json")) as f:
        g = json.load(f)
    r = head(np.array(g["q"], float), np.array(g["k"], float), np.array(g["v"], float),
             np.array(g["dout"], float), g["scale"], g["causal"], diagnostics=True)
    e = g["expect"]
    lse = [1.0, 1.0 + math.log(2.0)]
    _close(r["out"], e["out"], 1e-14, "2x2 out")
    _close(r["lse"], lse, 1e-14, "2x2 lse")
    _close(r["dq"], e["dq"], 1e-14, "2x2 dq")
    _close(r["dk"], e["dk"], 1e-14, "2x2 dk")
    _close(r["dv"], e["dv"], 1e-14, "2x2 dv")
    _close(r["pdp_rowsum"], e["D"], 1e-14, "2x2 D")


def _masked_scores(q, k, scale):
    S = q.shape[0]
    s = scale * (q @ k.T)
    s[np.triu(np.ones((S, S), bool), 1)] = -np.inf
    return s


def pin_row_identities(head, shapes=((1, 4), (7, 3), (33, 8), (70, 16)), seeds=(1, 2)):
    """Identities of the method on random inputs:
    sum_j P_ij = 1; sum_j P_ij dP_ij = dO_i . O_i (the D_i of the flash backward);
    sum_j dS_ij = 0; sum_j dK_j = 0 (O is invariant to K -> K + 1 c^T under the
    causal window); dQ_0 = 0, O_0 = V_0, L_0 = s_00 (row 0 sees one key);
    dV_{S-1} = P_{S-1,S-1} dO_{S-1} (the last key is seen by the last row only);
    L_i = logsumexp of the masked row (scipy)."""
    for seed in seeds:
        rng = np.random.default_rng(seed)
        for S, hd in shapes:
            q, k, v, do = (_rand(rng, S, hd) for _ in range(4))
            scale = 1.0 / math.sqrt(hd)
            r = head(q, k, v, do, scale, True, diagnostics=True)
            tag = f"S={S} hd={hd} seed={seed}"
            _close(r["p_rowsum"], np.ones(S), 1e-12, f"sum_j P {tag}")
            D = np.sum(do * r["out"], axis=1)
            _close(r["pdp_rowsum"], D, 1e-11 * max(1.0, np.max(np.abs(D))), f"sum_j P dP = dO.O {tag}")
            _close(r["ds_rowsum"], np.zeros(S), 1e-12, f"sum_j dS {tag}")
            _close(np.sum(r["dk"], axis=0), np.zeros(hd), 1e-11 * S, f"sum_j dK {tag}")
            _close(r["dq"][0], np.zeros(hd), 1e-14, f"dQ_0 {tag}")
            _close(r["out"][0], v[0], 1e-13, f"O_0 {tag}")
            s = _masked_scores(q, k, scale)
            _close(r["lse"][0], s[0, 0], 1e-13, f"L_0 {tag}")
            p_last = math.exp(s[S - 1, S - 1] - r["lse"][S - 1])
            _close(r["dv"][S - 1], p_last * do[S - 1], 1e-12, f"dV_last {tag}")
            _close(r["lse"], logsumexp(s, axis=1), 1e-12, f"L vs scipy logsumexp {tag}")


def pin_dense_library(head, shapes=((5, 3), (40, 8)), seed=3):
    """Without the mask the forward is dense softmax attention: compare with
    scipy's softmax/logsumexp and numpy matmul."""
    rng = np.random.default_rng(seed)
    for S, hd in shapes:
        q, k, v = (_rand(rng, S, hd) for _ in range(3))
        scale = 0.7
        r = head(q, k, v, None, scale, False)
        s = scale * (q @ k.T)
        _close(r["out"], softmax(s, axis=1) @ v, 1e-12, f"dense out S={S}")
        _close(r["lse"], logsumexp(s, axis=1), 1e-12, f"dense lse S={S}")


def pin_special_cases(head):
    """Closed forms: S=1 gives O=V, L = scale q.k, dQ = dK = 0, dV = dO;
    Q=0 gives causal running means O_i = mean_{j<=i} V_j with L_i = ln(i+1);
    hd=1 against a pure-Python scalar softmax."""
    rng = np.random.default_rng(11)
    q, k, v, do = (_rand(rng, 1, 5) for _ in range(4))
    r = head(q, k, v, do, 0.3, True)
    _close(r["out"], v, 1e-15, "S=1 out")
    _close(r["lse"], [0.3 * float(q[0] @ k[0])], 1e-14, "S=1 lse")
    _close(r["dq"], np.zeros((1, 5)), 0.0, "S=1 dq")
    _close(r["dk"], np.zeros((1, 5)), 0.0, "S=1 dk")
    _close(r["dv"], do, 1e-15, "S=1 dv")

    S, hd = 9, 4
    k, v, do = (_rand(rng, S, hd) for _ in range(3))
    r = head(np.zeros((S, hd)), k, v, do, 0.5, True)
    means = np.cumsum(v, axis=0) / np.arange(1, S + 1)[:, None]
    _close(r["out"], means, 1e-14, "Q=0 out")
    _close(r["lse"], np.log(np.arange(1, S + 1)), 1e-14, "Q=0 lse")

    S = 6
    qv = [0.3, -1.2, 0.8, 2.0, -0.4, 1.1]
    kv = [1.5, 0.2, -0.7, 0.9, 0.4, -1.3]
    vv = [0.5, -2.0, 1.0, 3.0, -0.5, 0.25]
    scale = 0.9
    r = head(np.array(qv)[:, None], np.array(kv)[:, None], np.array(vv)[:, None], None, scale, True)
    for i in range(S):
        logits = [scale * qv[i] * kv[j] for j in range(i + 1)]
        m = max(logits)
        w = [math.exp(x - m) for x in logits]
        z = sum(w)
        o = sum(wj * vv[j] for j, wj in enumerate(w)) / z
        if abs(r["out"][i, 0] - o) > 1e-14 or abs(r["lse"][i] - (m + math.log(z))) > 1e-14:
            raise AssertionError(f"hd=1 row {i}: oracle ({r['out'][i, 0]}, {r['lse'][i]}) vs ({o}, {m + math.log(z)})")


def pin_finite_differences(head, cases=((5, 3, 1, True), (8, 4, 2, True), (6, 2, 3, False), (3, 5, 4, True)),
                           h=1e-6, rtol=2e-7):
    """Central differences in fp64 of f = sum(dO o O) with respect to Q, K, V."""
    for S, hd, seed, causal in cases:
        rng = np.random.default_rng(100 + seed)
        x = {n: _rand(rng, S, hd) for n in ("q", "k", "v")}
        do = _rand(rng, S, hd)
        scale = 1.0 / math.sqrt(hd)
        r = head(x["q"], x["k"], x["v"], do, scale, causal)

        def f(**kw):
            a = dict(x)
            a.update(kw)
            return float(np.sum(do * head(a["q"], a["k"], a["v"], None, scale, causal)["out"]))

        for n, gname in (("q", "dq"), ("k", "dk"), ("v", "dv")):
            g = np.zeros((S, hd))
            for i in range(S):
                for d in range(hd):
                    xp = x[n].copy()
                    xm = x[n].copy()
                    xp[i, d] += h
                    xm[i, d] -= h
                    g[i, d] = (f(**{n: xp}) - f(**{n: xm})) / (2 * h)
            tol = rtol * max(1.0, float(np.max(np.abs(g))))
            _close(r[gname], g, tol, f"FD {gname} S={S} hd={hd} causal={causal}")


ALL_PINS = (pin_hand_2x2, pin_row_identities, pin_dense_library, pin_special_cases, pin_finite_differences)


# ---------------------------------------------------------------- dropout on the probabilities
# These take the oracle object (``oracle.Oracle``): besides ``head`` they use its
# ``splitmix64`` and ``keep``.  The generator is the dropout page's ("xtrain
# docs/17-dropout.md", section "Key Design Decisions"): key = seed ^ (idx * golden),
# h = splitmix64(key), u = (h >> 40) / 2^24, keep = u >= p.

GOLDEN_GAMMA = 0x9E3779B97F4A7C15

# Outputs of the reference SplitMix64 generator (Steele, Lea, Flood 2014) started from
# state 0: each step advances the state by the golden gamma and mixes it, so the n-th
# output is splitmix64((n - 1) * gamma) in the one-step form the oracle exports.
SPLITMIX64_FROM_ZERO = (0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F)


def pin_dropout_generator_outputs(orc):
    """The bit mix reproduces the published SplitMix64 outputs."""
    for n, want in enumerate(SPLITMIX64_FROM_ZERO):
        got = orc.splitmix64((n * GOLDEN_GAMMA) % 2 ** 64)
        if got != want:
            raise AssertionError(f"splitmix64 output {n}: {got:#x} != {want:#x}")


def pin_dropout_keep_known_answers(orc):
    """keep() against the page's definition worked by hand from the published outputs:
    (seed, index) = (0, 0) gives key 0 and h = 0xE220A8397B1DCDAF, so u = 0xE220A8 / 2^24
    = 0.883311...; (0, 1) gives key = gamma, h = 0x6E789E6AA1B965F4, u = 0.431528...;
    (2 gamma, 0) gives key = 2 gamma, h = 0x06C45D188009454F, u = 0.026433...
    (gamma, 1) gives key = gamma XOR gamma = 0, so the same u as (0, 0) (the sum
    gamma + gamma would give the u of (2 gamma, 0) instead).
    Each element is kept for p just below its u and dropped for p just above."""
    gamma2 = (2 * GOLDEN_GAMMA) % 2 ** 64
    for seed, index, u in ((0, 0, 0.8833), (0, 1, 0.43153), (gamma2, 0, 0.026433), (GOLDEN_GAMMA, 1, 0.8833)):
        if not orc.keep(seed, index, u - 1e-4) or orc.keep(seed, index, u + 1e-4):
            raise AssertionError(f"keep({seed:#x}, {index}) does not switch at u = {u}")
    # keep = (u >= p): a rate equal to u itself keeps the element.  Both u below are
    # 24-bit fractions, exact in fp32; the next fp32 rate above drops it.
    for seed, index, top24 in ((0, 0, 0xE220A8), (gamma2, 0, 0x06C45D)):
        u = np.float32(top24) / np.float32(2 ** 24)
        if not orc.keep(seed, index, float(u)):
            raise AssertionError(f"keep({seed:#x}, {index}) drops at p = u = {float(u)!r}")
        if orc.keep(seed, index, float(np.nextafter(u, np.float32(1.0)))):
            raise AssertionError(f"keep({seed:#x}, {index}) keeps just above p = u")


def pin_dropout_keep_rate(orc, n=1 << 15, seed=0xC0FFEE):
    """Each element is kept with probability 1 - p: the kept fraction of n indices lies
    within 6 standard deviations of 1 - p; p = 0 keeps everything."""
    if not all(orc.keep(seed, i, 0.0) for i in range(0, n, 37)):
        raise AssertionError("p = 0 dropped an element")
    for p in (0.1, 0.5, 0.9):
        kept = sum(orc.keep(seed, i, p) for i in range(n))
        sd = math.sqrt(n * p * (1 - p))
        if abs(kept - n * (1 - p)) > 6 * sd:
            raise AssertionError(f"p={p}: kept {kept} of {n}, expected {n * (1 - p):.0f} +- {6 * sd:.0f}")


def pin_dropout_p_zero(orc):
    """Rate 0 is the plain operator, bit for bit."""
    rng = np.random.default_rng(41)
    S, hd = 9, 4
    q, k, v, do = (_rand(rng, S, hd) for _ in range(4))
    a = orc.head(q, k, v, do, 0.5, True)
    b = orc.head(q, k, v, do, 0.5, True, dropout=(0.0, 77, 5 * S * S))
    for n in a:
        if not np.array_equal(a[n], b[n]):
            raise AssertionError(f"p = 0 changed {n}")


def pin_dropout_mask_structure(orc, S=6, p=0.4, seed=123, index_base=2 * 36):
    """With V = I the output is P o C itself: every factor C_ij equals keep(seed,
    index_base + i*S + j, p) / (1 - p) where P_ij > 0, and L is the plain L."""
    rng = np.random.default_rng(5)
    q, k = _rand(rng, S, S), _rand(rng, S, S)   # hd = S so that V can be the identity
    v = np.eye(S)
    plain = orc.head(q, k, v, None, 0.7, True)
    drop = orc.head(q, k, v, None, 0.7, True, dropout=(p, seed, index_base))
    _close(drop["lse"], plain["lse"], 0.0, "dropout changed L")
    inv = 1.0 / (1.0 - np.float64(np.float32(p)))
    for i in range(S):
        for j in range(S):
            c = inv if orc.keep(seed, index_base + i * S + j, p) else 0.0
            _close(drop["out"][i, j], plain["out"][i, j] * c, 1e-15, f"factor ({i},{j})")


def pin_dropout_finite_differences(orc, cases=((5, 3, 1), (7, 2, 2)), p=0.3, h=1e-6, rtol=2e-7):
    """With the mask fixed (it depends on (seed, index) only), the gradients are the
    central differences in fp64 of f = sum(dO o O)."""
    for S, hd, seed in cases:
        rng = np.random.default_rng(300 + seed)
        x = {n: _rand(rng, S, hd) for n in ("q", "k", "v")}
        do = _rand(rng, S, hd)
        scale = 1.0 / math.sqrt(hd)
        dd = (p, 1000 + seed, 3 * S * S)
        r = orc.head(x["q"], x["k"], x["v"], do, scale, True, dropout=dd)

        def f(**kw):
            a = dict(x)
            a.update(kw)
            return float(np.sum(do * orc.head(a["q"], a["k"], a["v"], None, scale, True, dropout=dd)["out"]))

        for n, gname in (("q", "dq"), ("k", "dk"), ("v", "dv")):
            g = np.zeros((S, hd))
            for i in range(S):
                for d in range(hd):
                    xp, xm = x[n].copy(), x[n].copy()
                    xp[i, d] += h
                    xm[i, d] -= h
                    g[i, d] = (f(**{n: xp}) - f(**{n: xm})) / (2 * h)
            tol = rtol * max(1.0, float(np.max(np.abs(g))))
            _close(r[gname], g, tol, f"dropout FD {gname} S={S} hd={hd}")


def pin_dropout_d_identity(orc, S=40, hd=8, p=0.25):
    """The row term of the softmax backward still equals dO_i . O_i with dropout on
    (sum_j P_ij dP_ij = sum_j (P o C)_ij (dO V^T)_ij = dO_i . O_i), which is what lets
    the fused backward keep the D pre-pass unchanged."""
    rng = np.random.default_rng(9)
    q, k, v, do = (_rand(rng, S, hd) for _ in range(4))
    r = orc.head(q, k, v, do, 1.0 / math.sqrt(hd), True, diagnostics=True, dropout=(p, 4, 0))
    _close(r["pdp_rowsum"], np.sum(do * r["out"], axis=1), 1e-12, "sum_j P dP != dO . O with dropout")


def pin_dropout_expectation(orc, S=5, hd=2, p=0.5, seeds=600):
    """Inverted dropout keeps the expectation: over many seeds the mean output is the
    plain output (within 6 standard errors of the sample mean)."""
    rng = np.random.default_rng(17)
    q, k, v = (_rand(rng, S, hd) for _ in range(3))
    plain = orc.head(q, k, v, None, 0.8, True)["out"]
    outs = np.stack([orc.head(q, k, v, None, 0.8, True, dropout=(p, s, 0))["out"] for s in range(seeds)])
    mean, se = outs.mean(0), outs.std(0) / math.sqrt(seeds)
    if np.any(np.abs(mean - plain) > 6 * se + 1e-12):
        raise AssertionError(f"mean over seeds drifts: max |mean - plain| {np.max(np.abs(mean - plain)):.3e}")


DROPOUT_PINS = (pin_dropout_generator_outputs, pin_dropout_keep_known_answers, pin_dropout_keep_rate, pin_dropout_p_zero,
                pin_dropout_mask_structure, pin_dropout_finite_differences, pin_dropout_d_identity,
                pin_dropout_expectation)
