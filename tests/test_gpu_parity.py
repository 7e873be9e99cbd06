"""CUDA path against the CPU oracle on identical seeded inputs (GB300 only).

Every call goes through the C ABI (ctypes binding).  All five workloads are
compared in full, element by element; workloads 4-5 (S=4096 and S=8192) in the
launch configuration the benchmark times, with identities that hold for every
head at any size checked besides."""
import math
import os

import numpy as np
import pytest
import torch

from bwd_xfa_fwd_gb300 import inputs
from tests.gpu_helpers import TOL, compare, oracle_result, run_gpu, to_device, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bwd_xfa_fwd_gb300 import binding, build
    build.build()
    binding.load()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("impl", [0, 1], ids=["auto", "simt"])
@pytest.mark.parametrize("wid", [1, 2, 3])
def test_workload_full(wid, impl):
    w = inputs.WORKLOADS[wid]
    x = inputs.workload_inputs(w)
    got = run_gpu(x, w.dtype, w.scale, impl=impl)
    ref = oracle_result(("w", wid), x, w.scale)
    compare(got, ref, w.dtype)


def _identities(got, x, dtype):
    """Exact identities of the operator, checked on every head:
    sum_j dV_j = sum_i dO_i (rows of P sum to 1);  sum_j dK_j = 0 (rows of dS sum
    to 0);  tr(Q^T dQ) = tr(K^T dK) (s depends on Q, K only through Q K^T)."""
    tol = TOL[dtype]["rel"]
    dout = x["dout"].exact
    sv = got["dv"].sum(axis=1) - dout.sum(axis=1)
    assert np.max(np.abs(sv)) <= tol * np.max(np.abs(got["dv"]).sum(axis=1)), "sum dV != sum dO"
    sk = got["dk"].sum(axis=1)
    assert np.max(np.abs(sk)) <= tol * np.max(np.abs(got["dk"]).sum(axis=1)), "sum dK != 0"
    tq = np.einsum("bsd,bsd->b", x["q"].exact, got["dq"])
    tk = np.einsum("bsd,bsd->b", x["k"].exact, got["dk"])
    mag = np.einsum("bsd,bsd->b", np.abs(x["q"].exact), np.abs(got["dq"]))
    assert np.all(np.abs(tq - tk) <= tol * mag), "tr(Q^T dQ) != tr(K^T dK)"


@pytest.mark.parametrize("impl", [0, 3], ids=["auto", "deterministic"])
@pytest.mark.parametrize("wid", [4, 5])
def test_workload_full_size(wid, impl):
    """Workloads 4 (bh 64, S 4096) and 5 (bh 32, S 8192) in the benchmark's launch
    configuration, every element of every head against the oracle (about 25 s and 45 s of
    oracle time on 16 cores, computed once per session), plus the exact identities."""
    w = inputs.WORKLOADS[wid]
    x = inputs.workload_inputs(w)
    got = run_gpu(x, w.dtype, w.scale, impl=impl)
    for n in ("out", "lse", "dq", "dk", "dv"):
        assert np.all(np.isfinite(got[n])), n
    ref = oracle_result(("w", wid), x, w.scale)
    compare(got, ref, w.dtype)
    _identities(got, x, w.dtype)


@pytest.mark.parametrize("hd,S", [(64, 4096), (32, 6000)])
def test_f32_tensor_core_long_sequence(hd, S):
    """The 3xTF32 family at long sequences (many key tiles per query tile, a ragged tail at
    S = 6000): every head against the oracle, and the exact identities."""
    bh = 4
    scale = 1.0 / math.sqrt(hd)
    x = inputs.draw((bh, S, hd), "f32", seed=4242 + hd, stds=(1.0, 1.0, 1.0, 1.0))
    got = run_gpu(x, "f32", scale, impl=2)
    ref = oracle_result(("f32long", hd, S), x, scale)
    compare(got, ref, "f32")
    _identities(got, x, "f32")


RAGGED = [1, 5, 64, 100, 128, 129, 255, 256, 257, 300, 511, 777]


@pytest.mark.parametrize("S", RAGGED)
@pytest.mark.parametrize("dtype,hd,impl", [("bf16", 128, 2), ("bf16", 64, 2), ("bf16", 128, 3), ("bf16", 64, 3),
                                           ("bf16", 32, 1), ("f32", 32, 1), ("f32", 64, 1), ("f32", 128, 1),
                                           ("bf16", 128, 1), ("f32", 32, 2), ("f32", 64, 2)])
def test_ragged_and_small(S, dtype, hd, impl):
    bh = 3
    scale = 1.0 / math.sqrt(hd)
    x = inputs.draw((bh, S, hd), dtype, seed=1000 + S + hd, stds=(1.0, 1.0, 1.0, 1.0))
    got = run_gpu(x, dtype, scale, impl=impl)
    ref = oracle_result(("ragged", S, hd, dtype), x, scale)
    compare(got, ref, dtype)


@pytest.mark.parametrize("hd", [64, 128])
def test_tcgen05_and_simt_agree_with_oracle(hd):
    S, bh = 1024, 4
    scale = 1.0 / math.sqrt(hd)
    x = inputs.draw((bh, S, hd), "bf16", seed=77 + hd, stds=(2.0, 2.0, 1.0, 1.0))
    ref = oracle_result(("both", hd), x, scale)
    for impl in (1, 2, 3):
        compare(run_gpu(x, "bf16", scale, impl=impl), ref, "bf16")


@pytest.mark.parametrize("dtype,hd", [("f32", 32), ("f32", 128), ("bf16", 64), ("bf16", 128)])
def test_rowdot(dtype, hd):
    from bwd_xfa_fwd_gb300 import binding
    x = inputs.draw((5, 333, hd), dtype, seed=5, names=("q", "k"))
    o, do = to_device(x["q"], dtype), to_device(x["k"], dtype)
    d = to_f64(binding.rowdot(o, do))
    ref = np.sum(x["q"].exact * x["k"].exact, axis=-1)
    assert np.max(np.abs(d - ref)) <= 1e-5 * np.max(np.abs(ref))


@pytest.mark.parametrize("dtype,hd", [("bf16", 128), ("f32", 64), ("f32", 32)])
def test_outputs_do_not_write_outside_their_buffers(dtype, hd):
    """Canary guards around every output buffer stay untouched."""
    from bwd_xfa_fwd_gb300 import binding
    bh, S = 2, 300
    scale = 1.0 / math.sqrt(hd)
    x = inputs.draw((bh, S, hd), dtype, seed=9)
    q, k, v, do = (to_device(x[n], dtype) for n in ("q", "k", "v", "dout"))
    n = bh * S * hd
    guard = 4096

    def guarded(numel, dtype):
        buf = torch.full((numel + 2 * guard,), -7.0, device="cuda", dtype=dtype)
        return buf, buf[guard:guard + numel]

    for impl in (1, 2, 3):
        bo, out = guarded(n, q.dtype)
        bl, lse = guarded(bh * S, torch.float32)
        binding.fwd(q, k, v, scale, impl, out=out.view(bh, S, hd), lse=lse.view(bh, S))
        grads = [guarded(n, q.dtype) for _ in range(3)]
        binding.bwd(q, k, v, out.view(bh, S, hd), do, lse.view(bh, S), scale, impl,
                    grads=tuple(g[1].view(bh, S, hd) for g in grads))
        torch.cuda.synchronize()
        for buf in [bo, bl] + [g[0] for g in grads]:
            assert torch.all(buf[:guard] == -7.0) and torch.all(buf[-guard:] == -7.0)


def test_backward_is_repeatable_with_reused_workspace():
    from bwd_xfa_fwd_gb300 import binding
    bh, S, hd = 4, 512, 128
    x = inputs.draw((bh, S, hd), "bf16", seed=12)
    q, k, v, do = (to_device(x[n], "bf16") for n in ("q", "k", "v", "dout"))
    out, lse = binding.fwd(q, k, v)
    ws = torch.empty(binding.workspace_bytes(bh, S, hd, torch.bfloat16), device="cuda", dtype=torch.uint8)
    a = binding.bwd(q, k, v, out, do, lse, workspace=ws)
    a = [t.clone() for t in a]
    b = binding.bwd(q, k, v, out, do, lse, workspace=ws)
    for s, t in zip(a, b):
        # dQ is summed with fp32 atomics in a data-dependent order: equal up to rounding
        assert torch.allclose(s.float(), t.float(), rtol=0, atol=1e-2 * float(s.float().abs().max()))


@pytest.mark.parametrize("dtype,hd,S", [("bf16", 128, 1000), ("bf16", 64, 777), ("f32", 64, 777), ("f32", 32, 1000)])
def test_deterministic_backward_is_bit_reproducible(dtype, hd, S):
    """XFA_IMPL_TCGEN05_DET (bf16) and the fp32 tensor-core family form dQ without atomics:
    two runs give identical bits."""
    from bwd_xfa_fwd_gb300 import binding
    bh = 6
    x = inputs.draw((bh, S, hd), dtype, seed=31 + hd)
    q, k, v, do = (to_device(x[n], dtype) for n in ("q", "k", "v", "dout"))
    out, lse = binding.fwd(q, k, v, impl=binding.IMPL_TCGEN05_DET)
    a = [t.clone() for t in binding.bwd(q, k, v, out, do, lse, impl=binding.IMPL_TCGEN05_DET)]
    for _ in range(2):
        b = binding.bwd(q, k, v, out, do, lse, impl=binding.IMPL_TCGEN05_DET)
        for s_, t_ in zip(a, b):
            assert torch.equal(s_, t_)


@pytest.mark.parametrize("dtype,hd", [("bf16", 128), ("f32", 64)])
def test_bwd_stages_match_bwd_for_every_impl(dtype, hd):
    """prep/main/finish called one by one give what xfa_bwd gives, for each kernel family."""
    from bwd_xfa_fwd_gb300 import binding
    bh, S = 3, 300
    scale = 1.0 / math.sqrt(hd)
    x = inputs.draw((bh, S, hd), dtype, seed=41)
    q, k, v, do = (to_device(x[n], dtype) for n in ("q", "k", "v", "dout"))
    for impl in (1, 2, 3):
        out, lse = binding.fwd(q, k, v, scale, impl)
        whole = binding.bwd(q, k, v, out, do, lse, scale, impl)
        ws = torch.empty(binding.workspace_bytes(bh, S, hd, q.dtype), device="cuda", dtype=torch.uint8)
        grads = tuple(torch.empty_like(q) for _ in range(3))
        staged = binding.bwd_stages(q, k, v, out, do, lse, scale, ws, grads, impl=impl)
        torch.cuda.synchronize()
        for a_, b_ in zip(whole, staged):
            assert torch.allclose(a_.float(), b_.float(), rtol=0, atol=1e-2 * float(a_.float().abs().max()))


@pytest.mark.parametrize("dtype,hd", [(torch.float32, 128), (torch.bfloat16, 32)])
def test_unsupported_combinations_are_rejected(dtype, hd):
    """The tcgen05 families take bf16 with hd 64 / 128 and fp32 (3xTF32) with hd 32 / 64."""
    from bwd_xfa_fwd_gb300 import binding
    t = torch.zeros(1, 64, hd, device="cuda", dtype=dtype)
    for impl in (binding.IMPL_TCGEN05, binding.IMPL_TCGEN05_DET):
        with pytest.raises(binding.XfaError) as e:
            binding.fwd(t, t, t, impl=impl)
        assert e.value.code == binding.XFA_ERR_UNSUPPORTED


def test_timeout_path_reports_and_recovers():
    from bwd_xfa_fwd_gb300 import binding
    assert binding.status() == binding.XFA_OK
    assert binding.selftest_timeout(2000) == binding.XFA_OK
    assert binding.status() == binding.XFA_ERR_TIMEOUT
    assert binding.status() == binding.XFA_OK       # cleared
    w = inputs.WORKLOADS[1]
    x = inputs.workload_inputs(w)
    compare(run_gpu(x, w.dtype, w.scale), oracle_result(("w", 1), x, w.scale), w.dtype)   # context still usable


def test_tape_node_fanout_on_gpu():
    """out = flash_attention(x, x, x): the tape sums dQ + dK + dV into x.grad."""
    from bwd_xfa_fwd_gb300.tape import Var, flash_attention
    bh, S, hd = 2, 200, 64
    scale = 1.0 / math.sqrt(hd)
    xin = inputs.draw((bh, S, hd), "bf16", seed=21, names=("x", "w"))
    xv = Var(to_device(xin["x"], "bf16"))
    y = flash_attention(xv, xv, xv, scale)
    y.backward(seed=to_device(xin["w"], "bf16"))
    ref = oracle_result(("tape",), {"q": xin["x"], "k": xin["x"], "v": xin["x"], "dout": xin["w"]}, scale)
    got = {"out": to_f64(y.value), "dq": to_f64(xv.grad)}
    want = {"out": ref["out"], "dq": ref["dq"] + ref["dk"] + ref["dv"]}
    compare(got, want, "bf16", names=("out", "dq"))


def test_runs_on_the_callers_stream():
    """Every call is enqueued on the current torch stream (a side stream here); results
    match the oracle and nothing runs on the default stream."""
    from bwd_xfa_fwd_gb300 import binding
    bh, S, hd = 2, 640, 128
    scale = 1.0 / math.sqrt(hd)
    x = inputs.draw((bh, S, hd), "bf16", seed=55)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        q, k, v, do = (to_device(x[n], "bf16") for n in ("q", "k", "v", "dout"))
        out, lse = binding.fwd(q, k, v, scale)
        dq, dk, dv = binding.bwd(q, k, v, out, do, lse, scale)
    side.synchronize()
    got = {n: to_f64(t) for n, t in zip(("out", "lse", "dq", "dk", "dv"), (out, lse, dq, dk, dv))}
    compare(got, oracle_result(("side",), x, scale), "bf16")


def test_tape_node_with_deterministic_backward():
    from bwd_xfa_fwd_gb300 import binding
    from bwd_xfa_fwd_gb300.tape import Var, flash_attention
    bh, S, hd = 2, 300, 64
    scale = 1.0 / math.sqrt(hd)
    x = inputs.draw((bh, S, hd), "bf16", seed=61)
    qv, kv, vv = (Var(to_device(x[n], "bf16")) for n in ("q", "k", "v"))
    y = flash_attention(qv, kv, vv, scale, impl=binding.IMPL_TCGEN05_DET)
    y.backward(seed=to_device(x["dout"], "bf16"))
    got = {"out": to_f64(y.value), "dq": to_f64(qv.grad), "dk": to_f64(kv.grad), "dv": to_f64(vv.grad)}
    compare(got, oracle_result(("tape-det",), x, scale), "bf16", names=("out", "dq", "dk", "dv"))


def _fuzz_cases(n=int(os.environ.get("XFA_FUZZ_CASES", "24")), seed=2024):
    """Seeded random cases; XFA_FUZZ_CASES raises their number for a longer soak.  The
    dropout rate comes from a second generator so the other draws stay as they were."""
    rng = np.random.default_rng(seed)
    rng_drop = np.random.default_rng(seed + 1)
    rng_f32 = np.random.default_rng(seed + 2)   # fp32 kernel family
    rng_keep = np.random.default_rng(seed + 3)  # how the dropout mask travels (bf16 tensor cores)
    cases = []
    for i in range(n):
        dtype = "bf16" if i % 4 else "f32"
        hd = int(rng.choice([64, 128])) if dtype == "bf16" else int(rng.choice([32, 64, 128]))
        impl = int(rng.choice([0, 2, 3])) if dtype == "bf16" else int(rng_f32.choice([0, 1, 2] if hd < 128 else [0, 1]))
        S = int(rng.integers(1, 1400))
        bh = int(rng.integers(1, 5))
        scale = float(rng.uniform(0.02, 0.3))
        std = float(rng.choice([0.5, 1.0, 2.0, 3.0]))
        p_drop = float(rng_drop.choice([0.0, 0.0, 0.1, 0.3])) if (dtype, impl) != ("bf16", 3) else 0.0
        keep = str(rng_keep.choice(["none", "store", "fill"])) if p_drop and dtype == "bf16" else "none"
        cases.append((i, dtype, hd, impl, S, bh, scale, std, p_drop, keep))
    return cases


@pytest.mark.parametrize("case", _fuzz_cases(),
                         ids=lambda c: f"{c[0]}-{c[1]}-hd{c[2]}-impl{c[3]}-S{c[4]}-bh{c[5]}-p{c[8]}-{c[9]}")
def test_random_shapes_against_oracle(case):
    """Seeded random shapes, scales, input spreads, kernel families, dropout rates and ways
    of carrying the dropout mask (drawn twice, stored by the forward, or filled ahead)."""
    i, dtype, hd, impl, S, bh, scale, std, p_drop, keep = case
    x = inputs.draw((bh, S, hd), dtype, seed=7000 + i, stds=(std, std, 1.0, 1.0))
    drop = (p_drop, 9000 + i) if p_drop else None
    got = run_gpu(x, dtype, scale, impl=impl, dropout=drop, keep=keep)
    compare(got, oracle_result(("fuzz", i), x, scale, dropout=drop), dtype)
